// splitkv_merge.cu - combines the partial results of a split key range.
//
// Each split s of a query row's keys leaves O_s (already divided by its own
// row sum) and LSE_s.  The merge rule of "FlashAttention（V3）深度解析"
// section 4.2 (m = max(m_a, m_b), z = z_a e^(m_a - m) + z_b e^(m_b - m)),
// applied with m_s = LSE_s and z_s = 1, gives
//     M = max_s LSE_s,  w_s = exp(LSE_s - M),
//     O = sum_s w_s O_s / sum_s w_s,  LSE = M + ln sum_s w_s.
// Many rows: one warp per query row; the partial rows are read with coalesced
// float loads, the output row is rounded to the input type.  Few rows (decode:
// one query per head): one CTA per row, its warps taking the splits
// round-robin with a running (max, sum, O) each, combined through shared
// memory, so that all splits of a row are read at once.  Bandwidth bound:
// n_splits x (d + 1) x 4 bytes read and 2 d + 4 bytes written per row.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

template <int D, bool BF16>
__global__ void __launch_bounds__(256) splitkv_merge_kernel(const float* __restrict__ o_part,
                                                            const float* __restrict__ lse_part,
                                                            uint16_t* __restrict__ o,
                                                            float* __restrict__ lse, int n_splits,
                                                            int Hq, int Nq, long long rows) {
  constexpr int VEC = D / 32;  // elements of the row per lane
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    float m = -CUDART_INF_F;
    for (int sp = lane; sp < n_splits; sp += 32) m = fmaxf(m, __ldg(lse_part + sp * rows + r));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
    float wsum = 0.f;
    for (int sp = 0; sp < n_splits; ++sp) {
      const float w = expf(__ldg(lse_part + sp * rows + r) - m);
      wsum += w;
      const float* src = o_part + (sp * rows + r) * D + lane * VEC;
#pragma unroll
      for (int v = 0; v < VEC; ++v) acc[v] = fmaf(w, __ldg(src + v), acc[v]);
    }
    const float inv = 1.f / wsum;
    const long long bh = r / Nq;
    const int i = (int)(r - bh * Nq);
    const long long b = bh / Hq;
    const int hq = (int)(bh - b * Hq);
    uint16_t* dst = o + ((b * Nq + i) * Hq + hq) * D + lane * VEC;
#pragma unroll
    for (int v = 0; v < VEC; v += 2) {
      const uint32_t pk = BF16 ? ptx::pack_bf16x2(acc[v] * inv, acc[v + 1] * inv)
                               : ptx::pack_f16x2(acc[v] * inv, acc[v + 1] * inv);
      *reinterpret_cast<uint32_t*>(dst + v) = pk;
    }
    if (lane == 0) lse[r] = m + logf(wsum);
  }
}

// one CTA (WARPS warps) per query row
template <int D, bool BF16, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) splitkv_merge_row_kernel(
    const float* __restrict__ o_part, const float* __restrict__ lse_part, uint16_t* __restrict__ o,
    float* __restrict__ lse, int n_splits, int Hq, int Nq, long long rows) {
  constexpr int VEC = D / 32;
  __shared__ float s_m[WARPS], s_z[WARPS];
  __shared__ float s_acc[WARPS][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long r = blockIdx.x;
  float m = -CUDART_INF_F, z = 0.f, acc[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
  for (int sp = warp; sp < n_splits; sp += WARPS) {
    const float ls = __ldg(lse_part + sp * rows + r);
    const float* src = o_part + (sp * rows + r) * D + lane * VEC;
    float x[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) x[v] = __ldg(src + v);
    // merge rule: new max, rescale what is held, add this split with weight 1
    const float mn = fmaxf(m, ls);
    const float a = expf(m - mn), w = expf(ls - mn);
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = acc[v] * a + w * x[v];
    z = z * a + w;
    m = mn;
  }
  if (lane == 0) { s_m[warp] = m; s_z[warp] = z; }
#pragma unroll
  for (int v = 0; v < VEC; ++v) s_acc[warp][lane * VEC + v] = acc[v];
  __syncthreads();
  if (warp == 0) {
    float mt = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) mt = fmaxf(mt, s_m[w]);
    float zt = 0.f, out[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) out[v] = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      const float f = s_z[w] > 0.f ? expf(s_m[w] - mt) : 0.f;   // warps without a split hold z = 0
      zt += f * s_z[w];
#pragma unroll
      for (int v = 0; v < VEC; ++v) out[v] += f * s_acc[w][lane * VEC + v];
    }
    const float inv = 1.f / zt;
    const long long bh = r / Nq;
    const int i = (int)(r - bh * Nq);
    const long long b = bh / Hq;
    const int hq = (int)(bh - b * Hq);
    uint16_t* dst = o + ((b * Nq + i) * Hq + hq) * D + lane * VEC;
#pragma unroll
    for (int v = 0; v < VEC; v += 2) {
      const uint32_t pk = BF16 ? ptx::pack_bf16x2(out[v] * inv, out[v + 1] * inv)
                               : ptx::pack_f16x2(out[v] * inv, out[v + 1] * inv);
      *reinterpret_cast<uint32_t*>(dst + v) = pk;
    }
    if (lane == 0) lse[r] = mt + logf(zt);
  }
}

int launch_splitkv_merge(const float* o_part, const float* lse_part, void* o, float* lse,
                         int n_splits, int B, int Hq, int Nq, int d, int dtype, int sm_count,
                         cudaStream_t stream) {
  const long long rows = (long long)B * Hq * Nq;
  uint16_t* out = static_cast<uint16_t*>(o);
  const bool bf16 = dtype == ATTN_BF16;
  if (rows <= (long long)sm_count * 4 && n_splits >= 8) {
    // few rows: a CTA per row reads all of a row's splits at once
#define ATTN_MERGE_ROW(DD)                                                                     \
  (bf16 ? (splitkv_merge_row_kernel<DD, true, 8><<<(int)rows, 256, 0, stream>>>(              \
               o_part, lse_part, out, lse, n_splits, Hq, Nq, rows), 0)                        \
        : (splitkv_merge_row_kernel<DD, false, 8><<<(int)rows, 256, 0, stream>>>(             \
               o_part, lse_part, out, lse, n_splits, Hq, Nq, rows), 0))
    switch (d) {
      case 64: ATTN_MERGE_ROW(64); break;
      case 128: ATTN_MERGE_ROW(128); break;
      case 256: ATTN_MERGE_ROW(256); break;
      default: return ATTN_ERR_UNSUPPORTED;
    }
#undef ATTN_MERGE_ROW
    note_launch();
    return check_launch();
  }
  long long blocks = (rows + 7) / 8;
  const long long cap = (long long)sm_count * 8;
  if (blocks > cap) blocks = cap;
#define ATTN_MERGE(DD)                                                                         \
  (bf16 ? (splitkv_merge_kernel<DD, true><<<(int)blocks, 256, 0, stream>>>(                    \
               o_part, lse_part, out, lse, n_splits, Hq, Nq, rows), 0)                        \
        : (splitkv_merge_kernel<DD, false><<<(int)blocks, 256, 0, stream>>>(                   \
               o_part, lse_part, out, lse, n_splits, Hq, Nq, rows), 0))
  switch (d) {
    case 64: ATTN_MERGE(64); break;
    case 128: ATTN_MERGE(128); break;
    case 256: ATTN_MERGE(256); break;
    default: return ATTN_ERR_UNSUPPORTED;
  }
#undef ATTN_MERGE
  note_launch();
  return check_launch();
}

}  // namespace attn
