// attn_prep_fp8.cu - per-block FP8 E4M3 quantisation with optional
// incoherent processing (Hadamard transform with random signs).
//
// Sources: FlashAttention（V3）深度解析 (dtcms.com), section 4.3 (block
// quantisation, a scale per block restoring its range); the Together AI
// summary card "FlashAttention-3——利用异步与低精度加速注意力机制", section on
// incoherent processing (each head multiplied by a random orthogonal matrix,
// Hadamard x random signs, to spread outliers before quantisation).
//
// A tile is one (128-token block, head, batch).  Persistent CTAs (two per SM
// for d <= 128) walk the tiles with heads varying fastest, taking tiles from
// a per-launch counter after their first few; each CTA keeps a ring of NS
// tiles in shared memory filled by TMA copies (one 128 x d box per tile, rows
// past N zero-filled), so the next tiles stream in while the current one is
// transformed and quantised.  8 warps x 16 rows; LPR lanes hold one row (8
// for d <= 128, 16 for d = 256), lane l owning the 16-byte chunks l, l + LPR,
// ... of 8 channels each, so that 8 lanes read 128 contiguous bytes of shared
// memory (no bank conflicts) and the rotary pair (c, c + d/2) lies in one
// lane for d >= 128; a thread holds 16 LPR / 32 consecutive rows, so that
// four of them give one 4-byte word per channel of the transposed layout.  The transform is a fast
// Walsh-Hadamard butterfly (stages over the in-lane channel bits, then
// shuffles across the LPR lanes of the row), scaled by 1/sqrt(d); the
// block amax is reduced through shared memory; descale = amax / 448 (float32);
// codes are the E4M3 rounding (nearest-even, saturated to +-448) of y /
// descale: exactly that of the quotient when y is the input itself (one
// product with a per-block reciprocal nudged to the exact quotient's side of
// every rounding midpoint, see the quantisation step), else of y * (448 /
// amax) with the reciprocal rounded once per block.  It
// reads each bf16 element once and writes one byte per element, an HBM-bound
// amount of work (two CTAs of 8 warps per SM, register and shared-memory
// limits); per-tile scalar work on the thread that issues the copies delays
// its warp at every tile barrier, so it is kept to a minimum.
//
// Two variants share the kernel:
// * rotary embedding before the transform (the summary card notes that the
//   transform can ride along with the rotary embedding, a bandwidth-bound
//   step): rotate-half form, channel c paired with c + d/2 (in the same lane
//   for d >= 128, one shuffle per value for d = 64); cos and sin come from
//   float32 tables [N, d/2] (attn_rope_table);
// * one scale per tensor (the baseline FP8 scheme): a first pass only
//   reduces the tensor's amax (atomic max of the float bits, all values >= 0),
//   a second quantises every block with that amax, and a one-CTA kernel
//   writes the descale of every block.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

// one 16-byte chunk (8 bf16 channels) from shared memory, widened to float
__device__ __forceinline__ void load_chunk(uint32_t saddr, float* y) {
  uint32_t ws[4];
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(ws[0]), "=r"(ws[1]), "=r"(ws[2]), "=r"(ws[3])
               : "r"(saddr));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    y[2 * i] = __uint_as_float(ws[i] << 16);
    y[2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
  }
}

// ring depth and CTAs per SM of the prep kernel
template <int D>
struct PrepCfg {
  static constexpr int TILE_BYTES = 128 * D * 2;   // one bf16 tile (128 rows x d)
  static constexpr int LPR = D == 256 ? 16 : 8;     // lanes per row
  static constexpr int CH = D / (8 * LPR);          // 16-byte chunks (8 channels) per lane
  static constexpr int NS = D == 64 ? 4 : 3;        // tiles in flight per CTA
  static constexpr int CTAS_PER_SM = D == 256 ? 1 : 2;
  static constexpr int TAIL = 256;                  // barriers, amax slots, stage tiles
  static int smem_bytes(int transpose_out) {
    return 128 + NS * TILE_BYTES + (transpose_out ? D * 128 : 0) + TAIL;
  }
};

constexpr long long kPrepWaitCycles = 4000000000LL;   // about 2 s


// quantisation modes
enum PrepMode : int {
  kPrepBlock = 0,       // scale per 128-token block (writes codes and descales)
  kPrepTensorAmax = 1,  // per-tensor, first pass: amax only
  kPrepTensor = 2,      // per-tensor, second pass: codes from the tensor amax
};

// Word index, within a 128-key row e of the transposed staging tile, where
// logical word kw (keys 4 kw .. 4 kw + 3) is kept: XOR-swizzled by the
// channel's 8-channel chunk so that the 32 lanes of one staging store (32
// different rows e, lanes holding 4 consecutive keys each) hit 32 banks.
template <int LPR>
__device__ __forceinline__ int tr_word(int e, int kw) {
  if constexpr (LPR == 8) {
    return kw ^ (((e >> 3) & 7) << 2);
  } else {
    const int h = (e >> 3) & 15;
    return kw ^ ((h & 1) | ((h >> 1) << 2));
  }
}

// A launch walks the tiles of up to three tensors (Q, K, V of one attention
// call) one tensor after the other, so that the ramp-up and the tail of a
// persistent launch are paid once per step instead of per tensor.
// Each CTA's first NS tiles are fixed (tile blockIdx + s * grid); every later
// tile is claimed from a counter (J.sched[0]), so that CTAs on faster SMs take
// more tiles and all of them end within about one tile of each other. The
// last CTA to finish sets the counter back to zero for the next launch.
template <int D, int MODE, bool ROPE>
__global__ void __launch_bounds__(256, PrepCfg<D>::CTAS_PER_SM)
    prep_fp8_kernel(const __grid_constant__ PrepJobs J, float* tensor_amax, unsigned int* status) {
  using PC = PrepCfg<D>;
  constexpr int LPR = PC::LPR;        // lanes per row
  constexpr int CH = PC::CH;          // chunks of 8 channels per lane
  constexpr int VEC = 8 * CH;         // channels per lane
  constexpr int RPW = 32 / LPR;       // row groups per warp
  constexpr int ITERS = 16 / RPW;     // consecutive rows per thread (8 warps x 16 rows)
  constexpr int NS = PC::NS;
  static_assert(ITERS % 4 == 0, "rows are staged for the transpose four at a time");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sraw = ptx::smem_addr(smem_raw);
  const uint32_t pad = (128u - (sraw & 127u)) & 127u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = sraw + pad;                           // NS tiles
  uint8_t* s_t = smem + NS * PC::TILE_BYTES;                   // transposed codes
  uint8_t* tail = s_t + (J.any_transpose ? D * 128 : 0);
  static_assert(NS <= 4, "tail layout");
  uint64_t* bars = reinterpret_cast<uint64_t*>(tail);          // [NS] tile landed
  float* s_amax = reinterpret_cast<float*>(tail + 32);         // [2][8], 16-byte aligned
  // [NS] tile of a stage as (tensor, head, block, batch), decoded once by the
  // thread that issues its copy; tensor -1 is the end mark
  int4* s_info = reinterpret_cast<int4*>(tail + 96);
  auto bar = [&](int i) { return ptx::smem_addr(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rsub = lane / LPR, hl = lane % LPR;
  // channel of value v = 8 j + t of this lane: 8 (hl + LPR j) + t
  auto chan = [&](int v) { return 8 * (hl + LPR * (v >> 3)) + (v & 7); };
  // row of the tile held in iteration i: rows r0 .. r0 + ITERS - 1
  const int r0 = warp * 16 + ITERS * rsub;
  const long long n_tiles = J.n_tiles;
  const long long G = gridDim.x;
  // tensor of tile t; its parameters and tensor map are read in place from
  // the kernel parameter
  auto locate = [&](long long t, int& jj, long long& tl) {
    jj = (J.n_jobs > 1 && t >= J.tile0[1] ? 1 : 0) + (J.n_jobs > 2 && t >= J.tile0[2] ? 1 : 0);
    tl = t - J.tile0[jj];
  };
  auto map_of = [&](int jj) { return &J.map[jj]; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) ptx::mbar_init(bar(i), 1);
    ptx::fence_barrier_init();
    for (int jj = 0; jj < J.n_jobs; ++jj) ptx::tma_prefetch_desc(map_of(jj));
  }
  __syncthreads();
  // (thread 0) stage st receives tile t, or the end mark when t is past the
  // last tile; the tile index is written before the arrival that completes
  // the stage's phase, so a thread that saw the phase complete reads it
  auto issue = [&](int st, long long t) {
    if (t >= n_tiles) {
      s_info[st] = make_int4(-1, 0, 0, 0);
      ptx::mbar_arrive(bar(st));
      return;
    }
    int jj;
    long long tl;
    locate(t, jj, tl);
    const PrepJob& jb = J.job[jj];
    // (a launch holds fewer than 2^31 tiles: 32-bit division)
    const unsigned ut = (unsigned)tl, uh = (unsigned)jb.H, unb = (unsigned)jb.nb;
    const unsigned r = ut / uh;
    const int th = (int)(ut - r * uh);
    const int tb = (int)(r / unb);
    const int tblk = (int)(r - (unsigned)tb * unb);
    s_info[st] = make_int4(jj, th, tblk, tb);
    ptx::mbar_arrive_expect_tx(bar(st), PC::TILE_BYTES);
    ptx::tma_load_4d(sbase + st * PC::TILE_BYTES, map_of(jj), bar(st), 0, th, tblk * 128, tb);
  };
  // (thread 0) the tile for the next refill, claimed one tile ahead of its
  // use so that the counter's round trip stays off the refill path
  long long claim = n_tiles;
  if (threadIdx.x == 0) {
    for (int k = 0; k < NS; ++k) issue(k, blockIdx.x + k * G);
    if (blockIdx.x + (NS - 1) * G < n_tiles)
      claim = NS * G + (long long)atomicAdd(J.sched, 1ull);
  }
  // (thread 0) once this CTA is done: count it, and let the last CTA of the
  // launch reset the counter (every claim of every CTA precedes its count)
  auto finish = [&]() {
    __threadfence();
    if (atomicAdd(J.sched + 1, 1ull) == (unsigned long long)(G - 1)) {
      J.sched[0] = 0;
      J.sched[1] = 0;
      __threadfence();
    }
  };

  for (long long k = 0;; ++k) {
    const int st = (int)(k % NS);
    // bounded wait for the stage; every thread takes the same decision: a
    // stage holding the end mark completed its phase before any thread got
    // here, and one holding a tile goes to the amax barrier below
    bool ok = ptx::mbar_try_wait(bar(st), (uint32_t)((k / NS) & 1));
    if (!ok) {
      const long long t0 = clock64();
      while (!(ok = ptx::mbar_try_wait_sleep(bar(st), (uint32_t)((k / NS) & 1), 100000)))
        if (clock64() - t0 > kPrepWaitCycles) break;
    }
    const int4 info = ok ? s_info[st] : make_int4(0, 0, 0, 0);
    if (info.x < 0) break;
    const PrepJob& jb = J.job[info.x];   // (read in place from the kernel parameter)
    const int H = jb.H, N = jb.N, nb = jb.nb, Npad = jb.Npad;
    const int transpose_out = jb.transpose_out, sign_group = jb.sign_group;
    uint8_t* __restrict__ x8 = jb.x8;
    float* __restrict__ descale = jb.descale;
    const int8_t* __restrict__ signs = jb.signs;
    const float* __restrict__ rope_cos = jb.rope_cos;
    const float* __restrict__ rope_sin = jb.rope_sin;
    const int h = info.y, blk = info.z, b = info.w;
    // (a thread whose wait gave up reads stale data; the block leaves at the
    // amax barrier below, before anything is stored)
    const int n0 = blk * 128 + r0;   // token of iteration 0
    const uint32_t tile = sbase + st * PC::TILE_BYTES;

    float y[ITERS][VEC];
    // the thread's rows from shared memory (rows past N were zero-filled by the copy)
#pragma unroll
    for (int i = 0; i < ITERS; ++i)
#pragma unroll
      for (int j = 0; j < CH; ++j)
        load_chunk(tile + (uint32_t)((r0 + i) * D * 2 + (hl + LPR * j) * 16), &y[i][8 * j]);

    // signs of this lane's channels: chunk j is 8 consecutive channels, one
    // 8-byte load (the host requires 8-byte aligned signs)
    float sg[VEC];
    if (signs) {
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(
            signs + (long long)(h / sign_group) * D + 8 * (hl + LPR * j)));
#pragma unroll
        for (int q = 0; q < 8; ++q)
          sg[8 * j + q] = (float)(int8_t)(((q < 4 ? w.x : w.y) >> (8 * (q & 3))) & 0xFFu);
      }
    }

    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < ITERS; ++i) {
      if (ROPE && rope_cos) {
        // (y_c, y_{c+D/2}) -> (y_c cos - y_{c+D/2} sin, y_{c+D/2} cos + y_c sin).
        // With two or more chunks per lane the partner of chunk j is chunk
        // j ^ CH/2 of the same lane; with one (d = 64) it is lane hl ^ LPR/2.
        const int n = n0 + i;
        // channels c and c + D/2 share angle c: with two or more chunks per
        // lane the upper half of the lane's values reuses the lower half's
        constexpr int HV = CH >= 2 ? VEC / 2 : VEC;
        float cs[HV], sn[HV];
        if (n < N) {
#pragma unroll
          for (int v = 0; v < HV; v += 4) {
            const int c = chan(v) % (D / 2);
            const float4 c4 = __ldg(reinterpret_cast<const float4*>(rope_cos + (long long)n * (D / 2) + c));
            const float4 s4 = __ldg(reinterpret_cast<const float4*>(rope_sin + (long long)n * (D / 2) + c));
            cs[v] = c4.x; cs[v + 1] = c4.y; cs[v + 2] = c4.z; cs[v + 3] = c4.w;
            sn[v] = s4.x; sn[v + 1] = s4.y; sn[v + 2] = s4.z; sn[v + 3] = s4.w;
          }
        } else {
#pragma unroll
          for (int v = 0; v < HV; ++v) { cs[v] = 1.f; sn[v] = 0.f; }
        }
        if constexpr (CH >= 2) {
          // value v < HV (chunk j < CH/2) pairs with v + HV (chunk j + CH/2)
#pragma unroll
          for (int v = 0; v < HV; ++v) {
            const float lo = y[i][v], hi = y[i][v + HV];
            y[i][v] = fmaf(lo, cs[v], -(hi * sn[v]));
            y[i][v + HV] = fmaf(hi, cs[v], lo * sn[v]);
          }
        } else {
          const bool upper = (hl & (LPR / 2)) != 0;
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            const float other = __shfl_xor_sync(0xffffffffu, y[i][v], LPR / 2);
            const float tt = upper ? other * sn[v] : -(other * sn[v]);
            y[i][v] = fmaf(y[i][v], cs[v], tt);
          }
        }
      }
      if (signs) {
        // the arithmetic is that of the scalar butterfly (each sum, difference
        // and product rounded once), two values per packed FP32x2 instruction
#pragma unroll
        for (int v = 0; v < VEC; v += 2)
          ptx::mul2(y[i][v], y[i][v + 1], y[i][v], y[i][v + 1], sg[v], sg[v + 1]);
        // butterfly stages over the in-lane bits of the channel (the 3 bits
        // within a chunk and the chunk-index bits above the lane bits); from
        // the second stage on, neighbouring values pair with neighbours
#pragma unroll
        for (int v = 0; v < VEC; v += 2) {
          const float a = y[i][v], c = y[i][v + 1];
          y[i][v] = a + c;
          y[i][v + 1] = a - c;
        }
#pragma unroll
        for (int hs = 2; hs < VEC; hs <<= 1) {
#pragma unroll
          for (int v = 0; v < VEC; v += 2) {
            if ((v & hs) == 0)
              ptx::addsub2(y[i][v], y[i][v + 1], y[i][v + hs], y[i][v + hs + 1], y[i][v],
                           y[i][v + 1], y[i][v + hs], y[i][v + hs + 1]);
          }
        }
        // butterfly stages across the LPR lanes of the row: the lower lane
        // keeps y + other, the upper one other - y (one FMA with +-1)
#pragma unroll
        for (int lm = 1; lm < LPR; lm <<= 1) {
          const float sgn = (hl & lm) ? -1.f : 1.f;
          float other[VEC];
#pragma unroll
          for (int v = 0; v < VEC; ++v) other[v] = __shfl_xor_sync(0xffffffffu, y[i][v], lm);
#pragma unroll
          for (int v = 0; v < VEC; v += 2)
            ptx::fma2(y[i][v], y[i][v + 1], y[i][v], y[i][v + 1], sgn, sgn, other[v], other[v + 1]);
        }
        // the 1 / sqrt(d) of the transform is applied with the quantisation scale
      }
#pragma unroll
      for (int v = 0; v < VEC; v += 2) amax = ptx::max3(amax, fabsf(y[i][v]), fabsf(y[i][v + 1]));
    }

    float bmax;
    // with the transform, y is still missing its factor 1 / sqrt(d): amax is
    // that of the scaled values, y is scaled together with the quantisation
    const float inv_sqrt_d =
        !signs ? 1.f : (D == 64) ? 0.125f : (D == 128) ? 0.08838834764831845f : 0.0625f;
    // one barrier per tile: it gathers the block amax (slots alternate by
    // tile parity, so a warp one tile ahead cannot overwrite a slot still
    // being read), makes the abort decision uniform, and frees the stage
    // (every row is in registers once all threads reached it)
    float* amax_slot = s_amax + 8 * (int)(k & 1);
    if constexpr (MODE != kPrepTensor) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (lane == 0) amax_slot[warp] = amax;
    }
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) {
        atomicOr(status, 1u);
        // wait (bounded) for the copies this CTA still has in flight
        for (long long kk = k; kk < k + NS; ++kk) {
          const int sk = (int)(kk % NS);
          if (s_info[sk].x < 0) break;
          const long long t0 = clock64();
          while (!ptx::mbar_try_wait(bar(sk), (uint32_t)((kk / NS) & 1)))
            if (clock64() - t0 > kPrepWaitCycles) break;
        }
        finish();
      }
      return;
    }
    if (threadIdx.x == 0) {
      // stage st is free: the claimed tile goes there, the next one is claimed
      issue(st, claim);
      if (claim < n_tiles) claim = NS * G + (long long)atomicAdd(J.sched, 1ull);
    }
    if constexpr (MODE == kPrepTensor) {
      bmax = *tensor_amax;   // written by the amax pass, read-only here
    } else {
      const float4 a0 = *reinterpret_cast<const float4*>(amax_slot);
      const float4 a1 = *reinterpret_cast<const float4*>(amax_slot + 4);
      bmax = fmaxf(ptx::max3(a0.x, a0.y, a0.z), ptx::max3(a0.w, a1.x, a1.y));
      bmax = ptx::max3(bmax, a1.z, a1.w);
      if (signs) bmax *= inv_sqrt_d;
    }
    if constexpr (MODE == kPrepTensorAmax) {
      // non-negative floats order like their bit patterns
      if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(tensor_amax), __float_as_uint(bmax));
      continue;
    }
    // codes are E4M3(y / descale), descale = amax / 448 rounded to float32.
    // Without the transform or rotation y is the bfloat16 input itself, and
    // the code of the exact quotient is reached with one product per value:
    // with x and amax bfloat16, x * 448 / amax is either exactly an E4M3
    // rounding midpoint or at least 2^-13 (relative) away from every one, and
    // x / descale differs from it by the descale's own rounding only. So the
    // reciprocal is nudged by 4 ulps (about 2^-21, far above the rounding of
    // the product) to the side where the descale's rounding puts the exact
    // quotient: a midpoint then rounds the way the exact quotient does, and
    // no other value changes its code. When the descale is exact, ties must
    // go to even: a reciprocal that is exact too keeps them on the midpoint,
    // else one correction step q + (x - q * descale) / descale (the residual
    // is exact in one FMA) lands exactly on a midpoint that the quotient
    // equals and within an ulp elsewhere. With the transform or
    // rotation y carries float32 rounding already and the codes are y *
    // (448 / amax), the reciprocal taken once per block (times 1 / sqrt(d)
    // with the transform).
    float inv_ds = bmax > 0.f ? __fdiv_rn(448.0f, bmax) : 1.0f;
    const float ds = bmax > 0.f ? __fdiv_rn(bmax, 448.0f) : 1.0f;
    bool divide = false;
    if (!rope_cos && !signs && bmax > 0.f) {
      const float dd = fmaf(ds, 448.0f, -bmax);   // sign of descale * 448 - amax, exact
      if (dd > 0.f) inv_ds = __uint_as_float(__float_as_uint(inv_ds) - 4u);
      else if (dd < 0.f) inv_ds = __uint_as_float(__float_as_uint(inv_ds) + 4u);
      else divide = fmaf(inv_ds, ds, -1.0f) != 0.f;
    }
    if (signs) inv_ds *= inv_sqrt_d;
    if constexpr (MODE == kPrepBlock) {
      if (threadIdx.x == 0) descale[((long long)b * H + h) * nb + blk] = ds;
    }

    // codes, four rows at a time: word q of row i holds channels 4q .. 4q + 3
    // of the lane
#pragma unroll
    for (int g = 0; g < ITERS / 4; ++g) {
      uint32_t c4[4][VEC / 4];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const int i = 4 * g + ii;
        if (!divide) {
#pragma unroll
          for (int q = 0; q < VEC / 4; ++q) {
            float p0, p1, p2, p3;
            ptx::mul2(p0, p1, y[i][4 * q], y[i][4 * q + 1], inv_ds, inv_ds);
            ptx::mul2(p2, p3, y[i][4 * q + 2], y[i][4 * q + 3], inv_ds, inv_ds);
            c4[ii][q] = ptx::pack_e4m3x4(p0, p1, p2, p3);
          }
        } else {
          auto quot = [&](float x) {
            const float q0 = x * inv_ds;
            const float res = fmaf(-q0, ds, x);
            return res == 0.f ? q0 : fmaf(res, inv_ds, q0);   // (keeps the sign of a zero)
          };
#pragma unroll
          for (int q = 0; q < VEC / 4; ++q)
            c4[ii][q] = ptx::pack_e4m3x4(quot(y[i][4 * q]), quot(y[i][4 * q + 1]),
                                         quot(y[i][4 * q + 2]), quot(y[i][4 * q + 3]));
        }
        if (!transpose_out) {
          const int n = n0 + i;
          if (n < N) {
            // chunk j of the lane: 8 codes at channel 8 (hl + LPR j)
            uint8_t* dst = x8 + (((long long)b * N + n) * H + h) * D;
#pragma unroll
            for (int j = 0; j < CH; ++j)
              *reinterpret_cast<uint2*>(dst + 8 * (hl + LPR * j)) =
                  make_uint2(c4[ii][2 * j], c4[ii][2 * j + 1]);
          }
        }
      }
      if (transpose_out) {
        // stage codes channel-major: row e of s_t holds the 128 keys of
        // channel e. The lane's rows are consecutive keys, so four rows give
        // one 4-byte word per channel: a 4 x 4 byte transpose of the words of
        // four rows (rows n >= N hold zeros)
        const int kw = (r0 + 4 * g) >> 2;
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q) {
          const uint32_t lo01 = __byte_perm(c4[0][q], c4[1][q], 0x5140);
          const uint32_t hi01 = __byte_perm(c4[0][q], c4[1][q], 0x7362);
          const uint32_t lo23 = __byte_perm(c4[2][q], c4[3][q], 0x5140);
          const uint32_t hi23 = __byte_perm(c4[2][q], c4[3][q], 0x7362);
          const uint32_t w[4] = {__byte_perm(lo01, lo23, 0x5410), __byte_perm(lo01, lo23, 0x7632),
                                 __byte_perm(hi01, hi23, 0x5410), __byte_perm(hi01, hi23, 0x7632)};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int e = chan(4 * q + c);
            reinterpret_cast<uint32_t*>(s_t)[e * 32 + tr_word<LPR>(e, kw)] = w[c];
          }
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
              reinterpret_cast<const uint32_t*>(s_t)[e * 32 + tr_word<LPR>(e, lane)];
        }
      }
    }
  }
  if (threadIdx.x == 0) finish();
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
int launch_prep_instance(const PrepJobs& J, int sm_count, float* tensor_amax,
                         unsigned int* status, cudaStream_t stream) {
  auto kern = prep_fp8_kernel<D, MODE, ROPE>;
  // the kernel decodes tile indices in 32-bit arithmetic
  if (J.n_tiles >= ((long long)1 << 31)) return ATTN_ERR_UNSUPPORTED;
  const int smem = PrepCfg<D>::smem_bytes(J.any_transpose);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prep)");
  const long long cap = (long long)PrepCfg<D>::CTAS_PER_SM * sm_count;
  const int grid = (int)(J.n_tiles < cap ? J.n_tiles : cap);
  kern<<<grid, 256, smem, stream>>>(J, tensor_amax, status);
  note_launch();
  return check_launch();
}

template <int MODE, bool ROPE>
int launch_prep_d(int d, const PrepJobs& J, int sm_count, float* tensor_amax, unsigned int* status,
                  cudaStream_t stream) {
  switch (d) {
    case 64: return launch_prep_instance<64, MODE, ROPE>(J, sm_count, tensor_amax, status, stream);
    case 128: return launch_prep_instance<128, MODE, ROPE>(J, sm_count, tensor_amax, status, stream);
    case 256: return launch_prep_instance<256, MODE, ROPE>(J, sm_count, tensor_amax, status, stream);
    default: return ATTN_ERR_UNSUPPORTED;
  }
}

PrepJob prep_job(void* x8, float* descale, int B, int H, int N, const int8_t* signs,
                 int sign_group, int transpose_out, const float* rope_cos,
                 const float* rope_sin) {
  PrepJob jb{};
  jb.x8 = static_cast<uint8_t*>(x8);
  jb.descale = descale;
  jb.signs = signs;
  jb.sign_group = sign_group;
  jb.rope_cos = rope_cos;
  jb.rope_sin = rope_sin;
  jb.H = H;
  jb.N = N;
  jb.nb = (N + 127) / 128;
  jb.Npad = (N + 15) / 16 * 16;
  jb.transpose_out = transpose_out;
  jb.n_tiles = (long long)B * jb.nb * H;
  return jb;
}

void prep_order(PrepJobs& J) {
  J.n_tiles = 0;
  for (int i = 0; i < 3; ++i) {
    J.tile0[i] = J.n_tiles;
    if (i < J.n_jobs) J.n_tiles += J.job[i].n_tiles;
  }
}

int launch_prep_jobs(const PrepJobs& J, int d, int sm_count, unsigned int* status,
                     cudaStream_t stream) {
  bool rope = false;
  for (int i = 0; i < J.n_jobs; ++i) rope = rope || J.job[i].rope_cos != nullptr;
  if (rope) return launch_prep_d<kPrepBlock, true>(d, J, sm_count, nullptr, status, stream);
  return launch_prep_d<kPrepBlock, false>(d, J, sm_count, nullptr, status, stream);
}

int launch_prep_fp8(const CUtensorMap& map_x, void* x8, float* descale, int B, int H, int N, int d,
                    const int8_t* signs, int sign_group, int transpose_out, const float* rope_cos,
                    const float* rope_sin, int per_tensor, int sm_count, unsigned int* status,
                    unsigned long long* sched, cudaStream_t stream) {
  PrepJobs J{};
  J.sched = sched;
  J.map[0] = map_x;
  J.job[0] = prep_job(x8, descale, B, H, N, signs, sign_group, transpose_out, rope_cos, rope_sin);
  J.n_jobs = 1;
  J.any_transpose = transpose_out;
  prep_order(J);
  if (!per_tensor) return launch_prep_jobs(J, d, sm_count, status, stream);
  if (rope_cos) return ATTN_ERR_UNSUPPORTED;
  // the tensor amax is accumulated in descale[0] and read from there
  cudaError_t e = cudaMemsetAsync(descale, 0, sizeof(float), stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(descale)");
  int rc = launch_prep_d<kPrepTensorAmax, false>(d, J, sm_count, descale, status, stream);
  if (rc != ATTN_OK) return rc;
  rc = launch_prep_d<kPrepTensor, false>(d, J, sm_count, descale, status, stream);
  if (rc != ATTN_OK) return rc;
  prep_fill_descale_kernel<<<1, 256, 0, stream>>>(descale, (long long)B * H * J.job[0].nb);
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
