// api.cu - the C ABI (include/attn.h): argument validation, one-time device
// set-up, TMA tensor-map encoding, kernel dispatch and error reporting.
// No torch types cross this boundary; every pointer is a plain device
// pointer owned by the caller.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "attn_fwd_kernel.cuh"
#include "internal.h"

namespace attn {

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxRows = (int64_t)1 << 30;  // TMA coordinates are int32; keep head-room

struct DeviceState {
  bool ready = false;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  int smem_optin = 0;
  unsigned int* status = nullptr;  // device status word (timeouts, internal checks)
  // tile counters of the prep launches: kPrepSlots pairs (next tile,
  // finished CTAs), each left at zero by the launch that used it
  unsigned long long* prep_sched = nullptr;
};
constexpr int kPrepSlots = 64;
constexpr size_t kStatusBlockBytes = 256 + kPrepSlots * 2 * sizeof(unsigned long long);

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<int64_t> g_launches{0};
std::atomic<unsigned> g_prep_seq{0};

// the tile counter of one prep call: slots are taken in turn, so that up to
// kPrepSlots prep launches may run at the same time (on different streams)
// without sharing a counter
unsigned long long* prep_slot(const DeviceState* st) {
  return st->prep_sched + 2 * (g_prep_seq.fetch_add(1) % kPrepSlots);
}
thread_local char g_cuda_msg[256] = "no CUDA error recorded";

// one-time per-device set-up; returns 0 or an error code
int device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  int rc = resolve_encoder();
  if (rc != ATTN_OK) return rc;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    if ((rc = device_attrs(dev, &st.sm_count, &st.cc_major, &st.cc_minor)) != ATTN_OK) return rc;
    if ((e = cudaDeviceGetAttribute(&st.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)))
      return cuda_fail(e, "cudaDeviceGetAttribute");
    // one allocation: the status word, then the prep launches' tile counters
    void* blk = nullptr;
    if ((e = cudaMalloc(&blk, kStatusBlockBytes)) != cudaSuccess)
      return cuda_fail(e, "cudaMalloc(status word)");
    if ((e = cudaMemset(blk, 0, kStatusBlockBytes)) != cudaSuccess)
      return cuda_fail(e, "cudaMemset(status word)");
    st.status = static_cast<unsigned int*>(blk);
    st.prep_sched = reinterpret_cast<unsigned long long*>(static_cast<char*>(blk) + 256);
    st.ready = true;
  }
  // the kernels are built for sm_103a only
  if (st.cc_major != 10 || st.cc_minor != 3) return ATTN_ERR_UNSUPPORTED;
  *out = &st;
  return ATTN_OK;
}

}  // namespace

int resolve_encoder() {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode) return ATTN_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
    return cuda_fail(e != cudaSuccess ? e : cudaErrorNotSupported,
                     "cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)");
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return ATTN_OK;
}

int device_attrs(int dev, int* sm_count, int* cc_major, int* cc_minor) {
  cudaError_t e;
  if ((e = cudaDeviceGetAttribute(sm_count, cudaDevAttrMultiProcessorCount, dev)) ||
      (e = cudaDeviceGetAttribute(cc_major, cudaDevAttrComputeCapabilityMajor, dev)) ||
      (e = cudaDeviceGetAttribute(cc_minor, cudaDevAttrComputeCapabilityMinor, dev)))
    return cuda_fail(e, "cudaDeviceGetAttribute");
  return ATTN_OK;
}

int encode(CUtensorMap* map, CUtensorMapDataType dt, const void* base, const cuuint64_t dims[4],
           const cuuint64_t strides[3], const cuuint32_t box[4], CUtensorMapSwizzle swizzle) {
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_cuda_msg, sizeof(g_cuda_msg), "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

// BSHD tensor [B, N, H, d] as TMA dims (d, H, N, B); box = `heads` heads x
// 128 / heads rows (128 rows in all), `inner` elements of d: 128 bytes for
// the 128-byte swizzle, or 64 bytes (a whole FP8 row of d = 64) for the
// 64-byte swizzle
int map_bshd(CUtensorMap* map, CUtensorMapDataType dt, int esz, const void* base, int B, int64_t N,
             int H, int d, int inner, int heads) {
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)d * esz, (cuuint64_t)H * d * esz,
                                 (cuuint64_t)N * H * d * esz};
  const cuuint32_t box[4] = {(cuuint32_t)inner, (cuuint32_t)heads, (cuuint32_t)(128 / heads), 1};
  return encode(map, dt, base, dims, strides, box,
                inner * esz == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
}

namespace {

// prep input [B, N, H, d] bf16 as dims (d, H, N, B); box = one head's 128 rows
// of d elements, unswizzled (row r of the tile at r * d * 2 bytes)
int map_prep(CUtensorMap* map, const void* base, int B, int64_t N, int H, int d) {
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2,
                                 (cuuint64_t)N * H * d * 2};
  const cuuint32_t box[4] = {(cuuint32_t)d, 1, 128, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_NONE);
}

// transposed value tensor [B, H, d, Npad] (bytes) as dims (Npad, d, H, B);
// box = 128 keys x d channels
int map_vt(CUtensorMap* map, const void* base, int B, int H, int d, int64_t Npad) {
  const cuuint64_t dims[4] = {(cuuint64_t)Npad, (cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)Npad, (cuuint64_t)d * Npad,
                                 (cuuint64_t)H * d * Npad};
  const cuuint32_t box[4] = {128, (cuuint32_t)d, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

// checks shared by the forward entry points; returns 1 for an empty problem
int check_common(int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int causal, float scale) {
  if (B < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (Nq > kMaxRows || Nk > kMaxRows) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || Nq == 0) return 1;
  if (Nk == 0) return ATTN_ERR_INVALID_ARG;
  return 0;
}

int fill_params(FwdParams& p, int d, int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, float scale,
                int sm_count, unsigned int* status, int* grid, int n_splits, int split_tiles,
                int pack_g) {
  const int qst = fwd_q_tiles(d);
  // pack_g query heads share each tile: Nq * pack_g packed rows per head group
  const int64_t n_mb = (Nq * pack_g + qst * 128 - 1) / (qst * 128);
  const int64_t units = (int64_t)B * (Hq / pack_g) * n_mb * n_splits;
  if (units > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = Hq / Hkv;
  p.Nq = (int)Nq;
  p.Nk = (int)Nk;
  p.n_kv_tiles = (int)((Nk + 127) / 128);
  p.n_mblocks = (int)n_mb;
  p.n_units = (int)units;
  p.nqb = (int)((Nq + 127) / 128);
  p.nkb = (int)((Nk + 127) / 128);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  p.active_stages = (Nq * pack_g <= 128) ? 1 : qst;   // a second tile would hold only padding
  p.pack_g = pack_g;
  p.n_splits = n_splits;
  p.split_tiles = split_tiles > 0 ? split_tiles : p.n_kv_tiles;
  *grid = (int)(units < sm_count ? units : sm_count);
  return ATTN_OK;
}

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_cuda_msg, sizeof(g_cuda_msg), "%s: %s (%s)", where, cudaGetErrorName(e),
           cudaGetErrorString(e));
  return ATTN_ERR_CUDA;
}

int check_launch() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "kernel launch");
}

}  // namespace attn

using namespace attn;

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int Hq, int Hkv, int64_t Nq, int64_t Nk, int d, int causal, float scale,
                        int dtype, void* stream) {
  int rc = check_common(B, Hq, Hkv, Nq, Nk, causal, scale);
  if (rc < 0) return rc;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (rc == 1) return ATTN_OK;  // empty problem
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 128) || !aligned(k, 128) || !aligned(v, 128) || !aligned(o, 128) ||
      !aligned(lse, 16))
    return ATTN_ERR_MISALIGNED;

  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != ATTN_OK) return rc;
  // few query rows under grouped-query attention (decode-like, non-causal):
  // the query heads of a group share the rows of a tile (the split instance
  // with one split), so each key/value head is streamed once per group
  const int pack_g = causal ? 1 : splitkv_pack(Hq / Hkv, 1, Nq, d);
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
  if ((rc = fill_params(p, d, B, Hq, Hkv, Nq, Nk, scale, st->sm_count, st->status, &grid, 1, 0,
                        pack_g)) != ATTN_OK)
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int mode = pack_g > 1 ? 2 : causal;
  return dtype == ATTN_BF16 ? launch_fwd_bf16(d, mode, mq, mk, mv, p, grid, s)
                            : launch_fwd_f16(d, mode, mq, mk, mv, p, grid, s);
}

extern "C" int attn_fwd_fp8(const void* q8, const void* k8, const void* v8t,
                            const float* q_descale, const float* k_descale,
                            const float* v_descale, void* o, float* lse, int B, int Hq, int Hkv,
                            int64_t Nq, int64_t Nk, int d, int causal, float scale, int hadamard,
                            void* stream) {
  int rc = check_common(B, Hq, Hkv, Nq, Nk, causal, scale);
  if (rc < 0) return rc;
  if (hadamard != 0 && hadamard != 1) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (rc == 1) return ATTN_OK;
  if (!q8 || !k8 || !v8t || !q_descale || !k_descale || !v_descale || !o || !lse)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(q8, 128) || !aligned(k8, 128) || !aligned(v8t, 128) || !aligned(o, 128) ||
      !aligned(lse, 16) || !aligned(q_descale, 16) || !aligned(k_descale, 16) ||
      !aligned(v_descale, 16))
    return ATTN_ERR_MISALIGNED;

  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != ATTN_OK) return rc;
  const int64_t Npad = (Nk + 15) / 16 * 16;
  const int inner = d == 64 ? 64 : 128;   // bytes of a row chunk (64-byte rows at d = 64)
  CUtensorMap mq, mk, mv;
  if ((rc = map_bshd(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q8, B, Nq, Hq, d, inner, 1)) ||
      (rc = map_bshd(&mk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, k8, B, Nk, Hkv, d, inner, 1)) ||
      (rc = map_vt(&mv, v8t, B, Hkv, d, Npad)))
    return rc;
  FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.q_descale = q_descale;
  p.k_descale = k_descale;
  p.v_descale = v_descale;
  int grid = 0;
  if ((rc = fill_params(p, d, B, Hq, Hkv, Nq, Nk, scale, st->sm_count, st->status, &grid, 1, 0,
                        1)) != ATTN_OK)
    return rc;
  return launch_fwd_e4m3(d, causal, mq, mk, mv, p, grid, static_cast<cudaStream_t>(stream));
}

namespace {
// argument checks shared by the prep variants
int check_prep(const void* x, const void* x8, const float* descale, int B, int H, int64_t N,
               int d, const int8_t* signs, int sign_heads, int transpose_out) {
  if (B < 0 || H < 1 || N < 0) return ATTN_ERR_INVALID_ARG;
  if (transpose_out != 0 && transpose_out != 1) return ATTN_ERR_INVALID_ARG;
  if (signs && (sign_heads < 1 || H % sign_heads != 0)) return ATTN_ERR_INVALID_ARG;
  if (N > kMaxRows) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (B > 65535 || (N + 127) / 128 > 65535) return ATTN_ERR_UNSUPPORTED;  // grid y/z limits
  if (B == 0 || N == 0) return ATTN_OK;
  if (!x || !x8 || !descale) return ATTN_ERR_INVALID_ARG;
  if (!aligned(x, 128) || !aligned(x8, 128) || !aligned(descale, 16)) return ATTN_ERR_MISALIGNED;
  if (signs && !aligned(signs, 8)) return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}
}  // namespace

extern "C" int attn_prep_fp8(const void* x, void* x8, float* descale, int B, int H, int64_t N,
                             int d, const int8_t* signs, int sign_heads, int transpose_out,
                             void* stream) {
  int rc = check_prep(x, x8, descale, B, H, N, d, signs, sign_heads, transpose_out);
  if (rc != ATTN_OK || B == 0 || N == 0) return rc;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != ATTN_OK) return rc;
  CUtensorMap mx;
  if ((rc = map_prep(&mx, x, B, N, H, d)) != ATTN_OK) return rc;
  const int group = signs ? H / sign_heads : 1;
  return launch_prep_fp8(mx, x8, descale, B, H, (int)N, d, signs, group, transpose_out, nullptr,
                         nullptr, 0, st->sm_count, st->status, prep_slot(st),
                         static_cast<cudaStream_t>(stream));
}

extern "C" int attn_prep_fp8_per_tensor(const void* x, void* x8, float* descale, int B, int H,
                                        int64_t N, int d, const int8_t* signs, int sign_heads,
                                        int transpose_out, void* stream) {
  int rc = check_prep(x, x8, descale, B, H, N, d, signs, sign_heads, transpose_out);
  if (rc != ATTN_OK || B == 0 || N == 0) return rc;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != ATTN_OK) return rc;
  CUtensorMap mx;
  if ((rc = map_prep(&mx, x, B, N, H, d)) != ATTN_OK) return rc;
  const int group = signs ? H / sign_heads : 1;
  return launch_prep_fp8(mx, x8, descale, B, H, (int)N, d, signs, group, transpose_out, nullptr,
                         nullptr, 1, st->sm_count, st->status, prep_slot(st),
                         static_cast<cudaStream_t>(stream));
}

extern "C" int attn_prep_fp8_qkv(const void* q, const void* k, const void* v, void* q8, void* k8,
                                 void* v8t, float* q_descale, float* k_descale, float* v_descale,
                                 int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
                                 const int8_t* signs, const float* rope_cos, const float* rope_sin,
                                 void* stream) {
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if ((rope_cos == nullptr) != (rope_sin == nullptr)) return ATTN_ERR_INVALID_ARG;
  int rc;
  if ((rc = check_prep(q, q8, q_descale, B, Hq, Nq, d, signs, Hkv, 0)) ||
      (rc = check_prep(k, k8, k_descale, B, Hkv, Nk, d, signs, Hkv, 0)) ||
      (rc = check_prep(v, v8t, v_descale, B, Hkv, Nk, d, nullptr, 1, 1)))
    return rc;
  if (rope_cos && (!aligned(rope_cos, 16) || !aligned(rope_sin, 16))) return ATTN_ERR_MISALIGNED;
  if (B == 0 || (Nq == 0 && Nk == 0)) return ATTN_OK;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != ATTN_OK) return rc;
  // Q, K, V as three tensors of one launch (Q and K: per-block codes with the
  // optional rotation and transform; V: transposed codes)
  PrepJobs J{};
  int n = 0;
  auto add = [&](const void* x, void* x8, float* ds, int H, int64_t N, const int8_t* sg,
                 int group, int tr, bool rot) -> int {
    if (N == 0) return ATTN_OK;
    const int r = map_prep(&J.map[n], x, B, N, H, d);
    if (r != ATTN_OK) return r;
    J.job[n] = prep_job(x8, ds, B, H, (int)N, sg, group, tr, rot ? rope_cos : nullptr,
                        rot ? rope_sin : nullptr);
    ++n;
    return ATTN_OK;
  };
  if ((rc = add(q, q8, q_descale, Hq, Nq, signs, Hq / Hkv, 0, true)) ||
      (rc = add(k, k8, k_descale, Hkv, Nk, signs, 1, 0, true)) ||
      (rc = add(v, v8t, v_descale, Hkv, Nk, nullptr, 1, 1, false)))
    return rc;
  J.n_jobs = n;
  J.any_transpose = Nk > 0 ? 1 : 0;
  prep_order(J);
  J.sched = prep_slot(st);
  return launch_prep_jobs(J, d, st->sm_count, st->status, static_cast<cudaStream_t>(stream));
}

extern "C" int attn_rope_table(float* rope_cos, float* rope_sin, int64_t N, int d, double base,
                               int64_t pos0, void* stream) {
  if (N < 0 || N > kMaxRows || d < 2 || d > 256 || (d & 1)) return ATTN_ERR_INVALID_ARG;
  if (!(base > 1.0) || !isfinite(base) || pos0 < 0 || pos0 > ((int64_t)1 << 40))
    return ATTN_ERR_INVALID_ARG;
  if (N == 0) return ATTN_OK;
  if (!rope_cos || !rope_sin) return ATTN_ERR_INVALID_ARG;
  if (!aligned(rope_cos, 4) || !aligned(rope_sin, 4)) return ATTN_ERR_MISALIGNED;
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != ATTN_OK) return rc;
  return launch_rope_table(rope_cos, rope_sin, (int)N, d, base, (long long)pos0,
                           static_cast<cudaStream_t>(stream));
}

extern "C" int attn_prep_fp8_rope(const void* x, void* x8, float* descale, int B, int H,
                                  int64_t N, int d, const float* rope_cos, const float* rope_sin,
                                  const int8_t* signs, int sign_heads, void* stream) {
  int rc = check_prep(x, x8, descale, B, H, N, d, signs, sign_heads, 0);
  if (rc != ATTN_OK || B == 0 || N == 0) return rc;
  if (!rope_cos || !rope_sin) return ATTN_ERR_INVALID_ARG;
  if (!aligned(rope_cos, 16) || !aligned(rope_sin, 16)) return ATTN_ERR_MISALIGNED;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != ATTN_OK) return rc;
  CUtensorMap mx;
  if ((rc = map_prep(&mx, x, B, N, H, d)) != ATTN_OK) return rc;
  const int group = signs ? H / sign_heads : 1;
  return launch_prep_fp8(mx, x8, descale, B, H, (int)N, d, signs, group, 0, rope_cos, rope_sin, 0,
                         st->sm_count, st->status, prep_slot(st), static_cast<cudaStream_t>(stream));
}

namespace attn {
// query heads packed per tile row group by the split instance: a GQA group
// whose size divides 128, with several splits, or with one split when the
// packed rows fit the unit's query tiles (decode-like shapes)
int splitkv_pack(int group, int eff_splits, int64_t Nq, int d) {
  if (group > 128 || 128 % group != 0) return 1;
  if (eff_splits > 1) return group;
  return (int64_t)Nq * group <= (int64_t)fwd_q_tiles(d) * 128 ? group : 1;
}
}  // namespace attn

namespace attn {
// key tiles per split and the number of non-empty splits for a request
void split_layout(int64_t Nk, int num_splits, int* split_tiles, int* eff_splits) {
  const int tiles = (int)((Nk + 127) / 128);
  int n = num_splits < 1 ? 1 : (num_splits > tiles ? tiles : num_splits);
  const int per = (tiles + n - 1) / n;
  *split_tiles = per;
  *eff_splits = (tiles + per - 1) / per;
}

int64_t splitkv_bytes(int64_t B, int64_t Hq, int64_t Nq, int64_t d, int64_t splits) {
  return splitkv_lse_offset(B, Hq, Nq, d, splits) + splits * B * Hq * Nq * 4;
}

int64_t splitkv_lse_offset(int64_t B, int64_t Hq, int64_t Nq, int64_t d, int64_t splits) {
  const int64_t rows = splits * B * Hq * Nq;
  return (rows * d * 4 + 255) / 256 * 256;   // the LSE part starts 256-byte aligned
}
}  // namespace attn

extern "C" size_t attn_splitkv_workspace_bytes(int B, int Hq, int64_t Nq, int d, int num_splits) {
  if (B < 0 || Hq < 1 || Nq < 0 || d < 1 || num_splits < 1) return 0;
  return (size_t)splitkv_bytes(B, Hq, Nq, d, num_splits);
}

extern "C" int attn_splitkv_default_splits(int B, int Hq, int Hkv, int64_t Nq, int64_t Nk,
                                           int d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Nq < 1 || Nk < 1) return 1;
  DeviceState* st = nullptr;
  if (device_state(&st) != ATTN_OK) return 1;
  const int qst = fwd_q_tiles(d);
  const int group = Hq / Hkv;
  const int pack_g = (group <= 128 && 128 % group == 0) ? group : 1;   // as attn_fwd_splitkv
  const int64_t units =
      (int64_t)B * (Hq / pack_g) * ((Nq * pack_g + qst * 128 - 1) / (qst * 128));
  const int64_t tiles = (Nk + 127) / 128;
  int64_t n = (st->sm_count + units - 1) / units;   // enough units for one wave
  if (n > tiles) n = tiles;
  if (n > 256) n = 256;
  return (int)(n < 1 ? 1 : n);
}

extern "C" int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
                                int num_splits, float scale, int dtype, void* workspace,
                                size_t workspace_bytes, void* stream) {
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
  int split_tiles = 0, eff = 1;
  split_layout(Nk, num_splits, &split_tiles, &eff);
  if (eff > 1) {
    if (!workspace) return ATTN_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return ATTN_ERR_MISALIGNED;
    if ((int64_t)workspace_bytes < splitkv_bytes(B, Hq, Nq, d, eff)) return ATTN_ERR_INVALID_ARG;
  }
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != ATTN_OK) return rc;
  // the split instance packs a GQA group into the rows of one query tile so
  // that each key/value head is streamed once per split; with one split it
  // is used for that alone when the packed rows fit the unit's query tiles
  // (decode-like shapes), and writes O and LSE directly
  const int group = Hq / Hkv;
  const int pack_g = splitkv_pack(group, eff, Nq, d);
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
  if ((rc = fill_params(p, d, B, Hq, Hkv, Nq, Nk, scale, st->sm_count, st->status, &grid, eff,
                        split_tiles, pack_g)) != ATTN_OK)
    return rc;
  float* o_part = nullptr;
  float* lse_part = nullptr;
  if (eff > 1) {
    o_part = static_cast<float*>(workspace);
    lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        splitkv_lse_offset(B, Hq, Nq, d, eff));
  }
  p.o_part = o_part;
  p.lse_part = lse_part;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // 2: split instance (partial results when eff > 1, else O and LSE directly)
  const int mode = (eff > 1 || pack_g > 1) ? 2 : 0;
  rc = dtype == ATTN_BF16 ? launch_fwd_bf16(d, mode, mq, mk, mv, p, grid, s)
                          : launch_fwd_f16(d, mode, mq, mk, mv, p, grid, s);
  if (rc != ATTN_OK || eff == 1) return rc;
  return launch_splitkv_merge(o_part, lse_part, o, lse, eff, B, Hq, (int)Nq, d, dtype,
                              st->sm_count, s);
}

extern "C" int attn_get_status(void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  if ((e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return cuda_fail(e, "cudaStreamSynchronize");
  // the allocated status word, if an allocating entry point set it up
  unsigned int* status = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_dev[dev].ready) status = g_dev[dev].status;
  }
  unsigned int word = 0;
  if (status) {
    if ((e = cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost)) != cudaSuccess)
      return cuda_fail(e, "cudaMemcpy(status word)");
    if (word != 0 && (e = cudaMemset(status, 0, sizeof(word))) != cudaSuccess)
      return cuda_fail(e, "cudaMemset(status word)");
  }
  // the no-alloc entry point's status word (inside its fixed array)
  unsigned int na_word = 0;
  int rc = noalloc_take_status(dev, &na_word);
  if (rc != ATTN_OK) return rc;
  word |= na_word;
  if (word == 0) return ATTN_OK;
  return (word & kStatusTimeout) ? ATTN_ERR_TIMEOUT : ATTN_ERR_DEVICE;
}

extern "C" const char* attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "success";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported head dimension, element type or device";
    case ATTN_ERR_MISALIGNED: return "pointer not aligned (128 bytes for tensors, 16 for vectors)";
    case ATTN_ERR_CUDA: return g_cuda_msg;
    case ATTN_ERR_TIMEOUT: return "a kernel wait expired (bounded wait timeout)";
    case ATTN_ERR_DEVICE: return "a kernel reported an internal consistency error";
    case ATTN_ERR_SCRATCH: return "problem needs more scratch than the fixed no-alloc array holds";
    default: return "unknown error code";
  }
}

extern "C" int64_t attn_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

namespace attn {
namespace {
// one warp waits, with the kernels' own bounded wait, on an mbarrier whose
// phase never completes: the wait gives up after its budget, sets the abort
// flag and the timeout bit of the status word, and the kernel returns
__global__ void bounded_wait_selftest_kernel(unsigned int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_addr(&bar), 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  const Ctl ctl{&abort_flag, status};
  warp_wait_bar(ptx::smem_addr(&bar), 0, ctl);
}
}  // namespace
}  // namespace attn

extern "C" int attn_selftest_bounded_wait(void* stream) {
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != ATTN_OK) return rc;
  attn::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(st->status);
  note_launch();
  return check_launch();
}
