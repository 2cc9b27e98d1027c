// attn_prep_fp8.cu - per-block FP8 E4M3 quantisation with optional
// incoherent processing (Hadamard transform with random signs).
//
// Sources: FlashAttention（V3）深度解析 (dtcms.com), section 4.3 (block
// quantisation, a scale per block restoring its range); the Together AI
// summary card "FlashAttention-3——利用异步与低精度加速注意力机制", section on
// incoherent processing (each head multiplied by a random orthogonal matrix,
// Hadamard x random signs, to spread outliers before quantisation).
//
// One CTA per (128-token block, head, batch); 8 warps x 16 rows; a warp holds
// one row of d values (d/32 per lane).  The transform is a fast Walsh-Hadamard
// butterfly (in-lane stages, then lane shuffles), scaled by 1/sqrt(d); the
// block amax is reduced through shared memory; codes are y / descale rounded
// to nearest-even and saturated to +-448 by the hardware conversion.  The
// kernel is bandwidth-bound: it reads each bf16 element once and writes one
// byte per element.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

template <int D>
__global__ void __launch_bounds__(256) prep_fp8_kernel(const uint16_t* __restrict__ x,
                                                       uint8_t* __restrict__ x8,
                                                       float* __restrict__ descale,
                                                       const int8_t* __restrict__ signs,
                                                       int sign_group, int H, int N, int nb,
                                                       int Npad, int transpose_out) {
  constexpr int VEC = D / 32;  // elements per lane
  constexpr int ROWS = 16;     // rows per warp
  __shared__ float s_amax[8];
  __shared__ __align__(16) uint8_t s_t[D * 128];  // transposed block (channel-major)

  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = lane * VEC;  // first channel of this lane

  float sg[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v)
    sg[v] = signs ? (float)signs[(long long)(h / sign_group) * D + e0 + v] : 1.f;

  float y[ROWS][VEC];
  float amax = 0.f;
#pragma unroll
  for (int rr = 0; rr < ROWS; ++rr) {
    const int n = blk * 128 + warp * ROWS + rr;
    uint16_t raw[VEC];
    if (n < N) {
      const uint16_t* src = x + (((long long)b * N + n) * H + h) * D + e0;
      if constexpr (VEC == 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
        raw[0] = (uint16_t)(w & 0xFFFF);
        raw[1] = (uint16_t)(w >> 16);
      } else if constexpr (VEC == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(src);
        raw[0] = (uint16_t)(w.x & 0xFFFF); raw[1] = (uint16_t)(w.x >> 16);
        raw[2] = (uint16_t)(w.y & 0xFFFF); raw[3] = (uint16_t)(w.y >> 16);
      } else {
        const uint4 w = *reinterpret_cast<const uint4*>(src);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          raw[2 * q] = (uint16_t)(ws[q] & 0xFFFF);
          raw[2 * q + 1] = (uint16_t)(ws[q] >> 16);
        }
      }
    } else {
#pragma unroll
      for (int v = 0; v < VEC; ++v) raw[v] = 0;
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) y[rr][v] = __uint_as_float((uint32_t)raw[v] << 16);

    if (signs) {
#pragma unroll
      for (int v = 0; v < VEC; ++v) y[rr][v] *= sg[v];
      // butterfly stages inside the lane (channel bit < log2 VEC)
#pragma unroll
      for (int hs = 1; hs < VEC; hs <<= 1) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
          if ((v & hs) == 0) {
            const float a = y[rr][v], c = y[rr][v + hs];
            y[rr][v] = a + c;
            y[rr][v + hs] = a - c;
          }
        }
      }
      // butterfly stages across lanes (channel bit >= log2 VEC)
#pragma unroll
      for (int lm = 1; lm < 32; lm <<= 1) {
        const bool upper = (lane & lm) != 0;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
          const float other = __shfl_xor_sync(0xffffffffu, y[rr][v], lm);
          y[rr][v] = upper ? (other - y[rr][v]) : (y[rr][v] + other);
        }
      }
      const float inv_sqrt_d = (D == 64) ? 0.125f : (D == 128) ? 0.08838834764831845f : 0.0625f;
#pragma unroll
      for (int v = 0; v < VEC; ++v) y[rr][v] *= inv_sqrt_d;
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) amax = fmaxf(amax, fabsf(y[rr][v]));
  }

#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) s_amax[warp] = amax;
  __syncthreads();
  float bmax = s_amax[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) bmax = fmaxf(bmax, s_amax[w]);
  const float ds = bmax > 0.f ? __fdiv_rn(bmax, 448.0f) : 1.0f;
  if (threadIdx.x == 0) descale[((long long)b * H + h) * nb + blk] = ds;

#pragma unroll
  for (int rr = 0; rr < ROWS; ++rr) {
    const int nl = warp * ROWS + rr;
    const int n = blk * 128 + nl;
    float qv[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) qv[v] = __fdiv_rn(y[rr][v], ds);
    if (!transpose_out) {
      if (n < N) {
        uint8_t* dst = x8 + (((long long)b * N + n) * H + h) * D + e0;
        if constexpr (VEC == 2) {
          const uint32_t c4 = ptx::pack_e4m3x4(qv[0], qv[1], 0.f, 0.f);
          *reinterpret_cast<uint16_t*>(dst) = (uint16_t)(c4 & 0xFFFF);
        } else if constexpr (VEC == 4) {
          *reinterpret_cast<uint32_t*>(dst) = ptx::pack_e4m3x4(qv[0], qv[1], qv[2], qv[3]);
        } else {
          uint2 w;
          w.x = ptx::pack_e4m3x4(qv[0], qv[1], qv[2], qv[3]);
          w.y = ptx::pack_e4m3x4(qv[4], qv[5], qv[6], qv[7]);
          *reinterpret_cast<uint2*>(dst) = w;
        }
      }
    } else {
      // stage codes channel-major: s_t[e][nl]; rows n >= N hold zeros
#pragma unroll
      for (int v = 0; v < VEC; v += 2) {
        const uint32_t c4 = ptx::pack_e4m3x4(qv[v], qv[v + 1], 0.f, 0.f);
        s_t[(e0 + v) * 128 + nl] = (uint8_t)(c4 & 0xFF);
        s_t[(e0 + v + 1) * 128 + nl] = (uint8_t)((c4 >> 8) & 0xFF);
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
            *reinterpret_cast<const uint32_t*>(&s_t[e * 128 + lane * 4]);
      }
    }
  }
}

int launch_prep_fp8(const void* x, void* x8, float* descale, int B, int H, int N, int d,
                    const int8_t* signs, int sign_group, int transpose_out, cudaStream_t stream) {
  const int nb = (N + 127) / 128;
  const int Npad = (N + 15) / 16 * 16;
  dim3 grid(nb, H, B);
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  uint8_t* xo = static_cast<uint8_t*>(x8);
  switch (d) {
    case 64:
      prep_fp8_kernel<64><<<grid, 256, 0, stream>>>(xs, xo, descale, signs, sign_group, H, N, nb,
                                                    Npad, transpose_out);
      break;
    case 128:
      prep_fp8_kernel<128><<<grid, 256, 0, stream>>>(xs, xo, descale, signs, sign_group, H, N, nb,
                                                     Npad, transpose_out);
      break;
    case 256:
      prep_fp8_kernel<256><<<grid, 256, 0, stream>>>(xs, xo, descale, signs, sign_group, H, N, nb,
                                                     Npad, transpose_out);
      break;
    default:
      return ATTN_ERR_UNSUPPORTED;
  }
  note_launch();
  return check_launch();
}

}  // namespace attn
