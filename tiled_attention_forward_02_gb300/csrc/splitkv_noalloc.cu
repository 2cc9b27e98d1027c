// splitkv_noalloc.cu - attn_fwd_splitkv_noalloc: the split-key-range forward
// for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: code running while a CUDA graph is
// being captured (an allocation would break or end the capture), programs
// whose device memory belongs to a pool or arena they manage themselves, and
// runtimes that forbid allocation on the request path so that latency and
// memory use stay fixed.  attn_fwd_splitkv needs a workspace for its
// per-split partial results, and the library's other entry points allocate a
// status word on their first call on a device.  This entry point does
// neither: its partial results and its status word live in the fixed array
// below, which is part of the library's device image, so every GPU that loads
// the library holds it until the process exits.
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "attn_fwd_kernel.cuh"
#include "internal.h"

namespace attn {
namespace {

// Fixed scratch: the first 256 bytes hold the status word, the rest the FP32
// partial rows (O / l, then LSE) of the splits.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;   // 16 MiB
constexpr size_t kNoAllocStatusBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
struct NoAllocDevice {
  bool ready = false;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
};
std::mutex g_na_mutex;
NoAllocDevice g_na_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_na_encode = nullptr;

// One-time set-up for the current device: attributes, the tensor-map encoder
// and the device address of the scratch array.  Allocates nothing.
int noalloc_setup(NoAllocDevice** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  NoAllocDevice& st = g_na_dev[dev];
  if (!st.ready) {
    if ((e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev)) ||
        (e = cudaDeviceGetAttribute(&st.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) ||
        (e = cudaDeviceGetAttribute(&st.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)))
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (!g_na_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return cuda_fail(e != cudaSuccess ? e : cudaErrorNotSupported,
                         "cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)");
      g_na_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    // the array's name is only a host-side stand-in: ask for its device address
    void* ptr = nullptr;
    if ((e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    // the status word must start at zero (the partial rows are always
    // written before they are read)
    if ((e = cudaMemset(ptr, 0, kNoAllocStatusBytes)) != cudaSuccess)
      return cuda_fail(e, "cudaMemset(no-alloc status word)");
    st.scratch = static_cast<unsigned char*>(ptr);
    st.ready = true;
  }
  if (st.cc_major != 10 || st.cc_minor != 3) return ATTN_ERR_UNSUPPORTED;
  *out = &st;
  return ATTN_OK;
}

int na_map_bshd(CUtensorMap* map, CUtensorMapDataType dt, const void* base, int B, int64_t N,
                int H, int d, int heads = 1) {
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2,
                                 (cuuint64_t)N * H * d * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)heads, (cuuint32_t)(128 / heads), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_na_encode(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

bool na_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                                        float* lse, int B, int Hq, int Hkv, int64_t Nq,
                                        int64_t Nk, int d, int num_splits, float scale, int dtype,
                                        void* stream) {
  if (B < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale) || num_splits < 1) return ATTN_ERR_INVALID_ARG;
  if (Nq > ((int64_t)1 << 30) || Nk > ((int64_t)1 << 30)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || Nq == 0) return ATTN_OK;
  if (Nk == 0) return ATTN_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!na_aligned(q, 128) || !na_aligned(k, 128) || !na_aligned(v, 128) || !na_aligned(o, 128) ||
      !na_aligned(lse, 16))
    return ATTN_ERR_MISALIGNED;

  // split layout: as many splits as asked, at most one per 128-key tile
  const int tiles = (int)((Nk + 127) / 128);
  const int n_req = num_splits > tiles ? tiles : num_splits;
  const int split_tiles = (tiles + n_req - 1) / n_req;
  const int eff = (tiles + split_tiles - 1) / split_tiles;
  const int64_t rows = (int64_t)eff * B * Hq * Nq;
  const int64_t o_bytes = (rows * d * 4 + 255) / 256 * 256;
  if (eff > 1 && (size_t)(o_bytes + rows * 4) > kNoAllocScratchBytes - kNoAllocStatusBytes)
    return ATTN_ERR_SCRATCH;

  NoAllocDevice* st = nullptr;
  int rc = noalloc_setup(&st);
  if (rc != ATTN_OK) return rc;
  const int qst = fwd_q_tiles(d);
  const int group = Hq / Hkv;
  const int pack_g = splitkv_pack(group, eff, Nq, d);
  const int64_t n_mb = (Nq * pack_g + qst * 128 - 1) / (qst * 128);
  const int64_t units = (int64_t)B * (Hq / pack_g) * n_mb * eff;
  if (units > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;

  const CUtensorMapDataType tdt =
      dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mq, mk, mv;
  if ((rc = na_map_bshd(&mq, tdt, q, B, Nq, Hq, d, pack_g)) ||
      (rc = na_map_bshd(&mk, tdt, k, B, Nk, Hkv, d)) ||
      (rc = na_map_bshd(&mv, tdt, v, B, Nk, Hkv, d)))
    return rc;

  FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = Hq / Hkv;
  p.Nq = (int)Nq;
  p.Nk = (int)Nk;
  p.n_kv_tiles = tiles;
  p.n_mblocks = (int)n_mb;
  p.n_units = (int)units;
  p.nqb = (int)((Nq + 127) / 128);
  p.nkb = tiles;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = reinterpret_cast<unsigned int*>(st->scratch);
  p.active_stages = (Nq * pack_g <= 128) ? 1 : qst;
  p.pack_g = pack_g;
  p.n_splits = eff;
  p.split_tiles = split_tiles;
  float* o_part = reinterpret_cast<float*>(st->scratch + kNoAllocStatusBytes);
  float* lse_part = reinterpret_cast<float*>(st->scratch + kNoAllocStatusBytes + o_bytes);
  p.o_part = eff > 1 ? o_part : nullptr;
  p.lse_part = eff > 1 ? lse_part : nullptr;
  const int grid = (int)(units < st->sm_count ? units : st->sm_count);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int mode = (eff > 1 || pack_g > 1) ? 2 : 0;
  rc = dtype == ATTN_BF16 ? launch_fwd_bf16(d, mode, mq, mk, mv, p, grid, s)
                          : launch_fwd_f16(d, mode, mq, mk, mv, p, grid, s);
  if (rc != ATTN_OK || eff == 1) return rc;
  return launch_splitkv_merge(o_part, lse_part, o, lse, eff, B, Hq, (int)Nq, d, dtype,
                              st->sm_count, s);
}
