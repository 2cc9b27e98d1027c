// attn_prep_fp8.cu - per-block FP8 E4M3 quantisation with optional
// incoherent processing (Hadamard transform with random signs).
//
// Sources: FlashAttention（V3）深度解析 (dtcms.com), section 4.3 (block
// quantisation, a scale per block restoring its range); the Together AI
// summary card "FlashAttention-3——利用异步与低精度加速注意力机制", section on
// incoherent processing (each head multiplied by a random orthogonal matrix,
// Hadamard x random signs, to spread outliers before quantisation).
//
// One CTA per (128-token block, head, batch); 8 warps x 16 rows; a half warp
// holds one row (d/16 values per lane, loaded 16 bytes at a time, all rows of
// the block in flight before any arithmetic).  The transform is a fast
// Walsh-Hadamard butterfly (in-lane stages, then shuffles within the half
// warp), scaled by 1/sqrt(d); the
// block amax is reduced through shared memory; codes are y * (448 / amax)
// (float32, the reciprocal rounded once per block) rounded to nearest-even and
// saturated to +-448 by the hardware conversion; descale = amax / 448.  The
// kernel is bandwidth-bound: it reads each bf16 element once and writes one
// byte per element.
//
// Two variants share the kernel:
// * rotary embedding before the transform (the summary card notes that the
//   transform can ride along with the rotary embedding, a bandwidth-bound
//   step): rotate-half form, channel c paired with c + d/2; the pair sits in
//   lanes hl and hl ^ 8 of the half warp, one shuffle per value; cos and sin
//   come from float32 tables [N, d/2] (attn_rope_table);
// * one scale per tensor (the baseline FP8 scheme): a first pass only
//   reduces the tensor's amax (atomic max of the float bits, all values >= 0),
//   a second quantises every block with that amax, and a one-CTA kernel
//   writes the descale of every block.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

// 16 bytes of bf16 input per lane; a half warp holds one row
template <int D>
__device__ __forceinline__ void load_row_part(const uint16_t* src, float (&y)[D / 16]) {
  constexpr int VEC = D / 16;
  if constexpr (VEC == 4) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
    y[0] = __uint_as_float(w.x << 16); y[1] = __uint_as_float(w.x & 0xFFFF0000u);
    y[2] = __uint_as_float(w.y << 16); y[3] = __uint_as_float(w.y & 0xFFFF0000u);
  } else {
#pragma unroll
    for (int q = 0; q < VEC / 8; ++q) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(src) + q);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        y[8 * q + 2 * i] = __uint_as_float(ws[i] << 16);
        y[8 * q + 2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
      }
    }
  }
}

// quantisation modes
enum PrepMode : int {
  kPrepBlock = 0,       // scale per 128-token block (writes codes and descales)
  kPrepTensorAmax = 1,  // per-tensor, first pass: amax only
  kPrepTensor = 2,      // per-tensor, second pass: codes from the tensor amax
};

template <int VEC>
__device__ __forceinline__ void load_f32(const float* src, float (&t)[VEC]) {
#pragma unroll
  for (int q = 0; q < VEC / 4; ++q) {
    const float4 w = __ldg(reinterpret_cast<const float4*>(src) + q);
    t[4 * q] = w.x; t[4 * q + 1] = w.y; t[4 * q + 2] = w.z; t[4 * q + 3] = w.w;
  }
}

template <int D, int MODE, bool ROPE>
__global__ void __launch_bounds__(256) prep_fp8_kernel(const uint16_t* __restrict__ x,
                                                       uint8_t* __restrict__ x8,
                                                       float* __restrict__ descale,
                                                       const int8_t* __restrict__ signs,
                                                       int sign_group, int H, int N, int nb,
                                                       int Npad, int transpose_out,
                                                       const float* __restrict__ rope_cos,
                                                       const float* __restrict__ rope_sin,
                                                       float* tensor_amax) {
  constexpr int VEC = D / 16;  // elements per lane (a half warp covers one row)
  constexpr int ITERS = 8;     // 8 warps x 2 rows x 8 iterations = 128 rows
  __shared__ float s_amax[8];
  __shared__ __align__(16) uint8_t s_t[D * 128];  // transposed block (channel-major)

  // heads vary fastest across the grid, so that CTAs running together read
  // neighbouring pieces of the same token rows ([B, N, H, d] layout)
  const int h = blockIdx.x, blk = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, hl = lane & 15;
  const int e0 = hl * VEC;  // first channel of this lane
  // row of iteration i: blk*128 + warp*16 + 2i + half
  auto row_of = [&](int i) { return blk * 128 + warp * 16 + 2 * i + half; };

  float sg[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v)
    sg[v] = signs ? (float)signs[(long long)(h / sign_group) * D + e0 + v] : 1.f;

  float y[ITERS][VEC];
  // issue every load of the block before any arithmetic on it
#pragma unroll
  for (int i = 0; i < ITERS; ++i) {
    const int n = row_of(i);
    if (n < N) {
      load_row_part<D>(x + (((long long)b * N + n) * H + h) * D + e0, y[i]);
    } else {
#pragma unroll
      for (int v = 0; v < VEC; ++v) y[i][v] = 0.f;
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < ITERS; ++i) {
    if constexpr (ROPE) {
      // (y_c, y_{c+D/2}) -> (y_c cos - y_{c+D/2} sin, y_{c+D/2} cos + y_c sin);
      // lane hl holds channels hl*VEC.., its partner lane hl ^ 8
      const int n = row_of(i);
      float cs[VEC], sn[VEC];
      if (n < N) {
        const long long off = (long long)n * (D / 2) + (hl & 7) * VEC;
        load_f32<VEC>(rope_cos + off, cs);
        load_f32<VEC>(rope_sin + off, sn);
      } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) { cs[v] = 1.f; sn[v] = 0.f; }
      }
      const bool upper = hl >= 8;
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        const float other = __shfl_xor_sync(0xffffffffu, y[i][v], 8);
        const float t = upper ? other * sn[v] : -(other * sn[v]);
        y[i][v] = fmaf(y[i][v], cs[v], t);
      }
    }
    if (signs) {
#pragma unroll
      for (int v = 0; v < VEC; ++v) y[i][v] *= sg[v];
      // butterfly stages inside the lane (channel bit < log2 VEC)
#pragma unroll
      for (int hs = 1; hs < VEC; hs <<= 1) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
          if ((v & hs) == 0) {
            const float a = y[i][v], c = y[i][v + hs];
            y[i][v] = a + c;
            y[i][v + hs] = a - c;
          }
        }
      }
      // butterfly stages across the 16 lanes of the half warp
#pragma unroll
      for (int lm = 1; lm < 16; lm <<= 1) {
        const bool upper = (hl & lm) != 0;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
          const float other = __shfl_xor_sync(0xffffffffu, y[i][v], lm);
          y[i][v] = upper ? (other - y[i][v]) : (y[i][v] + other);
        }
      }
      const float inv_sqrt_d = (D == 64) ? 0.125f : (D == 128) ? 0.08838834764831845f : 0.0625f;
#pragma unroll
      for (int v = 0; v < VEC; ++v) y[i][v] *= inv_sqrt_d;
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) amax = fmaxf(amax, fabsf(y[i][v]));
  }

  float bmax;
  if constexpr (MODE == kPrepTensor) {
    bmax = *tensor_amax;   // written by the amax pass, read-only here
  } else {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) s_amax[warp] = amax;
    __syncthreads();
    bmax = s_amax[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) bmax = fmaxf(bmax, s_amax[w]);
  }
  if constexpr (MODE == kPrepTensorAmax) {
    // non-negative floats order like their bit patterns
    if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(tensor_amax), __float_as_uint(bmax));
    return;
  }
  // codes are y * (448 / amax), the reciprocal taken once per block
  const float inv_ds = bmax > 0.f ? __fdiv_rn(448.0f, bmax) : 1.0f;
  if constexpr (MODE == kPrepBlock) {
    const float ds = bmax > 0.f ? __fdiv_rn(bmax, 448.0f) : 1.0f;
    if (threadIdx.x == 0) descale[((long long)b * H + h) * nb + blk] = ds;
  }

#pragma unroll
  for (int i = 0; i < ITERS; ++i) {
    const int n = row_of(i);
    const int nl = n - blk * 128;
    uint32_t c4[VEC / 4];
#pragma unroll
    for (int q = 0; q < VEC / 4; ++q)
      c4[q] = ptx::pack_e4m3x4(y[i][4 * q] * inv_ds, y[i][4 * q + 1] * inv_ds,
                               y[i][4 * q + 2] * inv_ds, y[i][4 * q + 3] * inv_ds);
    if (!transpose_out) {
      if (n < N) {
        uint8_t* dst = x8 + (((long long)b * N + n) * H + h) * D + e0;
        if constexpr (VEC == 4) {
          *reinterpret_cast<uint32_t*>(dst) = c4[0];
        } else if constexpr (VEC == 8) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(c4[0], c4[1]);
        } else {
          *reinterpret_cast<uint4*>(dst) = make_uint4(c4[0], c4[1], c4[2], c4[3]);
        }
      }
    } else {
      // stage codes channel-major: s_t[e][nl ^ swz(e)] (rows n >= N hold zeros);
      // the XOR swizzle puts the 16 channels a half warp writes in distinct banks
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        const int e = e0 + v;
        s_t[e * 128 + (nl ^ (((e / VEC) & 31) << 2))] = (uint8_t)((c4[v >> 2] >> (8 * (v & 3))) & 0xFF);
      }
    }
  }
  if (transpose_out) {
    __syncthreads();
    // row e of the transposed block: 128 keys = 32 lanes x 4 bytes
    const int valid = min(128, Npad - blk * 128);  // multiple of 16
    for (int e = warp; e < D; e += 8) {
      if (lane * 4 < valid) {
        uint8_t* dst = x8 + (((long long)b * H + h) * D + e) * Npad + blk * 128 + lane * 4;
        *reinterpret_cast<uint32_t*>(dst) =
            *reinterpret_cast<const uint32_t*>(&s_t[e * 128 + ((lane * 4) ^ (((e / VEC) & 31) << 2))]);
      }
    }
  }
}

// descale of every block from the tensor amax in descale[0]; one CTA, every
// thread reads descale[0] before any thread writes
__global__ void __launch_bounds__(256) prep_fill_descale_kernel(float* descale, long long n) {
  const float amax = descale[0];
  __syncthreads();
  const float ds = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  for (long long i = threadIdx.x; i < n; i += blockDim.x) descale[i] = ds;
}

// cos / sin of angle (pos0 + n) * base^(-2c/d), computed in double and
// rounded once to float32; one CTA per 64 positions
__global__ void __launch_bounds__(256) rope_table_kernel(float* __restrict__ cos_out,
                                                         float* __restrict__ sin_out, int N,
                                                         int d, double base, long long pos0) {
  __shared__ double s_freq[128];
  const int half = d / 2;
  for (int c = threadIdx.x; c < half; c += blockDim.x) s_freq[c] = pow(base, -2.0 * c / d);
  __syncthreads();
  const long long n0 = (long long)blockIdx.x * 64;
  for (int t = threadIdx.x; t < 64 * half; t += blockDim.x) {
    const long long n = n0 + t / half;
    const int c = t % half;
    if (n >= N) break;
    double sv, cv;
    sincos((double)(pos0 + n) * s_freq[c], &sv, &cv);
    cos_out[n * half + c] = (float)cv;
    sin_out[n * half + c] = (float)sv;
  }
}

template <int D, int MODE, bool ROPE>
void launch_prep_instance(dim3 grid, cudaStream_t stream, const uint16_t* xs, uint8_t* xo,
                          float* descale, const int8_t* signs, int sign_group, int H, int N,
                          int nb, int Npad, int transpose_out, const float* rc, const float* rs,
                          float* tamax) {
  prep_fp8_kernel<D, MODE, ROPE><<<grid, 256, 0, stream>>>(
      xs, xo, descale, signs, sign_group, H, N, nb, Npad, transpose_out, rc, rs, tamax);
}

template <int MODE, bool ROPE>
int launch_prep_d(int d, dim3 grid, cudaStream_t stream, const uint16_t* xs, uint8_t* xo,
                  float* descale, const int8_t* signs, int sign_group, int H, int N, int nb,
                  int Npad, int transpose_out, const float* rc, const float* rs, float* tamax) {
  switch (d) {
    case 64:
      launch_prep_instance<64, MODE, ROPE>(grid, stream, xs, xo, descale, signs, sign_group, H,
                                           N, nb, Npad, transpose_out, rc, rs, tamax);
      break;
    case 128:
      launch_prep_instance<128, MODE, ROPE>(grid, stream, xs, xo, descale, signs, sign_group, H,
                                            N, nb, Npad, transpose_out, rc, rs, tamax);
      break;
    case 256:
      launch_prep_instance<256, MODE, ROPE>(grid, stream, xs, xo, descale, signs, sign_group, H,
                                            N, nb, Npad, transpose_out, rc, rs, tamax);
      break;
    default:
      return ATTN_ERR_UNSUPPORTED;
  }
  note_launch();
  return check_launch();
}

int launch_prep_fp8(const void* x, void* x8, float* descale, int B, int H, int N, int d,
                    const int8_t* signs, int sign_group, int transpose_out, const float* rope_cos,
                    const float* rope_sin, int per_tensor, cudaStream_t stream) {
  const int nb = (N + 127) / 128;
  const int Npad = (N + 15) / 16 * 16;
  dim3 grid(H, nb, B);
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  uint8_t* xo = static_cast<uint8_t*>(x8);
  if (!per_tensor) {
    if (rope_cos)
      return launch_prep_d<kPrepBlock, true>(d, grid, stream, xs, xo, descale, signs, sign_group,
                                             H, N, nb, Npad, transpose_out, rope_cos, rope_sin,
                                             nullptr);
    return launch_prep_d<kPrepBlock, false>(d, grid, stream, xs, xo, descale, signs, sign_group,
                                            H, N, nb, Npad, transpose_out, nullptr, nullptr,
                                            nullptr);
  }
  if (rope_cos) return ATTN_ERR_UNSUPPORTED;
  // the tensor amax is accumulated in descale[0] and read from there
  cudaError_t e = cudaMemsetAsync(descale, 0, sizeof(float), stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(descale)");
  int rc = launch_prep_d<kPrepTensorAmax, false>(d, grid, stream, xs, xo, descale, signs,
                                                 sign_group, H, N, nb, Npad, transpose_out,
                                                 nullptr, nullptr, descale);
  if (rc != ATTN_OK) return rc;
  rc = launch_prep_d<kPrepTensor, false>(d, grid, stream, xs, xo, descale, signs, sign_group, H,
                                         N, nb, Npad, transpose_out, nullptr, nullptr, descale);
  if (rc != ATTN_OK) return rc;
  prep_fill_descale_kernel<<<1, 256, 0, stream>>>(descale, (long long)B * H * nb);
  note_launch();
  return check_launch();
}

int launch_rope_table(float* cos_out, float* sin_out, int N, int d, double base, long long pos0,
                      cudaStream_t stream) {
  const int blocks = (N + 63) / 64;
  rope_table_kernel<<<blocks, 256, 0, stream>>>(cos_out, sin_out, N, d, base, pos0);
  note_launch();
  return check_launch();
}

}  // namespace attn
