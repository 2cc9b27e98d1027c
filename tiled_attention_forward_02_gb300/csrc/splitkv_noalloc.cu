// splitkv_noalloc.cu - attn_fwd_splitkv_noalloc: the split-key-range forward
// for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: programs whose device memory belongs
// to a pool or arena they manage themselves (a library allocation would
// compete with that pool, or fail once it holds the whole device), and
// runtimes that forbid allocation on the request path because an allocation
// can block, synchronise the device or fail under memory pressure, which
// breaks their latency and memory bounds.  attn_fwd_splitkv needs a
// workspace for its per-split partial results, and the library's other entry
// points allocate a status word on their first call on a device.  This entry
// point does neither: its partial results and its status word live in the
// fixed array below, which is part of the library's device image, so every
// GPU that loads the library holds it until the process exits.
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

// One-time set-up for the current device: attributes, the tensor-map encoder
// and the device address of the scratch array.  Allocates nothing.
int noalloc_setup(NoAllocDevice** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  int rc = resolve_encoder();
  if (rc != ATTN_OK) return rc;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  NoAllocDevice& st = g_na_dev[dev];
  if (!st.ready) {
    if ((rc = device_attrs(dev, &st.sm_count, &st.cc_major, &st.cc_minor)) != ATTN_OK) return rc;
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

}  // namespace

int noalloc_take_status(int dev, unsigned int* word) {
  *word = 0;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_OK;
  unsigned char* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_na_mutex);
    if (g_na_dev[dev].ready) scratch = g_na_dev[dev].scratch;
  }
  if (!scratch) return ATTN_OK;
  cudaError_t e = cudaMemcpy(word, scratch, sizeof(unsigned int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(no-alloc status word)");
  if (*word != 0 && (e = cudaMemset(scratch, 0, sizeof(unsigned int))) != cudaSuccess)
    return cuda_fail(e, "cudaMemset(no-alloc status word)");
  return ATTN_OK;
}

}  // namespace attn

using namespace attn;

extern "C" int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                                        float* lse, int B, int Hq, int Hkv, int64_t Nq,
                                        int64_t Nk, int d, int num_splits, float scale, int dtype,
                                        void* stream) {
  int rc = check_common(B, Hq, Hkv, Nq, Nk, 0, scale);
  if (rc < 0) return rc;
  if (num_splits < 1) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (rc == 1) return ATTN_OK;  // empty problem
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 128) || !aligned(k, 128) || !aligned(v, 128) || !aligned(o, 128) ||
      !aligned(lse, 16))
    return ATTN_ERR_MISALIGNED;

  // split layout: as many splits as asked, at most one per 128-key tile
  int split_tiles = 0, eff = 1;
  split_layout(Nk, num_splits, &split_tiles, &eff);
  if (eff > 1 &&
      (size_t)splitkv_bytes(B, Hq, Nq, d, eff) > kNoAllocScratchBytes - kNoAllocStatusBytes)
    return ATTN_ERR_SCRATCH;

  NoAllocDevice* st = nullptr;
  if ((rc = noalloc_setup(&st)) != ATTN_OK) return rc;
  const int pack_g = splitkv_pack(Hq / Hkv, eff, Nq, d);
  const CUtensorMapDataType tdt =
      dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mq, mk, mv;
  if ((rc = map_bshd(&mq, tdt, 2, q, B, Nq, Hq, d, 64, pack_g)) ||
      (rc = map_bshd(&mk, tdt, 2, k, B, Nk, Hkv, d, 64, 1)) ||
      (rc = map_bshd(&mv, tdt, 2, v, B, Nk, Hkv, d, 64, 1)))
    return rc;

  FwdParams p{};
  p.o = o;
  p.lse = lse;
  int grid = 0;
  unsigned int* status = reinterpret_cast<unsigned int*>(st->scratch);
  if ((rc = fill_params(p, d, B, Hq, Hkv, Nq, Nk, scale, st->sm_count, status, &grid, eff,
                        split_tiles, pack_g)) != ATTN_OK)
    return rc;
  float* o_part = reinterpret_cast<float*>(st->scratch + kNoAllocStatusBytes);
  float* lse_part = reinterpret_cast<float*>(st->scratch + kNoAllocStatusBytes +
                                             splitkv_lse_offset(B, Hq, Nq, d, eff));
  p.o_part = eff > 1 ? o_part : nullptr;
  p.lse_part = eff > 1 ? lse_part : nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int mode = (eff > 1 || pack_g > 1) ? 2 : 0;
  rc = dtype == ATTN_BF16 ? launch_fwd_bf16(d, mode, mq, mk, mv, p, grid, s)
                          : launch_fwd_f16(d, mode, mq, mk, mv, p, grid, s);
  if (rc != ATTN_OK || eff == 1) return rc;
  return launch_splitkv_merge(o_part, lse_part, o, lse, eff, B, Hq, (int)Nq, d, dtype,
                              st->sm_count, s);
}
