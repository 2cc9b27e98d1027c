// internal.h - host-side declarations shared by the C-ABI layer (api.cu)
// and the kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn.h"  // include/ is on the include path

namespace attn {

struct FwdParams;

// counts one kernel launch (attn_launch_count)
void note_launch();
// turns the launch status into a return code, keeping the CUDA message
int check_launch();
// records a CUDA error text for attn_strerror and returns ATTN_ERR_CUDA
int cuda_fail(cudaError_t e, const char* where);

// fused forward launchers, one per element type; `grid` is the number of
// persistent CTAs; d and causal select the template instance (causal 2:
// non-causal with a split key range, writing FP32 partial results)
int launch_fwd_f16(int d, int causal, const CUtensorMap& q, const CUtensorMap& k,
                   const CUtensorMap& v, const FwdParams& p, int grid, cudaStream_t stream);
int launch_fwd_bf16(int d, int causal, const CUtensorMap& q, const CUtensorMap& k,
                    const CUtensorMap& v, const FwdParams& p, int grid, cudaStream_t stream);
int launch_fwd_e4m3(int d, int causal, const CUtensorMap& q, const CUtensorMap& k,
                    const CUtensorMap& v, const FwdParams& p, int grid, cudaStream_t stream);

// query tiles per work unit of the fused forward (tensor-memory budget)
inline int fwd_q_tiles(int d) { return d == 256 ? 1 : 2; }

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// --- host helpers that allocate nothing (api.cu); the no-alloc entry point
// uses them too
// resolves cuTensorMapEncodeTiled once per process
int resolve_encoder();
// number of SMs and compute capability of device `dev`
int device_attrs(int dev, int* sm_count, int* cc_major, int* cc_minor);
// argument checks of the forward entry points; 1 for an empty problem
int check_common(int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int causal, float scale);
// BSHD tensor [B, N, H, d] as a 4-D tensor map (d, H, N, B) with a box of
// `heads` heads x 128 / heads rows x `inner` elements, 128-byte swizzle
// (64-byte swizzle for 64-byte rows: inner x element size = 64)
int map_bshd(CUtensorMap* map, CUtensorMapDataType dt, int esz, const void* base, int B, int64_t N,
             int H, int d, int inner, int heads);
// forward parameters and persistent grid size for a problem
int fill_params(FwdParams& p, int d, int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, float scale,
                int sm_count, unsigned int* status, int* grid, int n_splits, int split_tiles,
                int pack_g);
// key tiles per split and the number of non-empty splits for a request
void split_layout(int64_t Nk, int num_splits, int* split_tiles, int* eff_splits);
// bytes of split partial results (O / l rows, then LSE rows from a 256-byte
// aligned offset)
int64_t splitkv_bytes(int64_t B, int64_t Hq, int64_t Nq, int64_t d, int64_t splits);
int64_t splitkv_lse_offset(int64_t B, int64_t Hq, int64_t Nq, int64_t d, int64_t splits);
// reads and clears the no-alloc entry point's status word of device `dev`
// (0 if that entry point was never set up there); allocates nothing
int noalloc_take_status(int dev, unsigned int* word);

// query heads the split instance packs into a tile's rows (api.cu)
int splitkv_pack(int group, int eff_splits, int64_t Nq, int d);

// combines split partial results (O / l per split, LSE per split) into o, lse
int launch_splitkv_merge(const float* o_part, const float* lse_part, void* o, float* lse,
                         int n_splits, int B, int Hq, int Nq, int d, int dtype, int sm_count,
                         cudaStream_t stream);

// One tensor of an FP8 prep launch (per-block mode): codes x8 (BSHD, or
// [B, H, d, Npad] when transpose_out), descales [B, H, nb], optional signs
// [H / sign_group, d] and rotary tables [N, d/2]; n_tiles = B x nb x H tiles
// (heads fastest, then 128-token blocks, then batch).
struct PrepJob {
  uint8_t* x8;
  float* descale;
  const int8_t* signs;
  const float* rope_cos;
  const float* rope_sin;
  long long n_tiles;
  int sign_group, H, N, nb, Npad, transpose_out;
};
// up to three tensors in one launch; map[i]: tensor i's bf16 input as
// (d, H, N, B), box d x 1 x 128 x 1, no swizzle; sched: the launch's tile
// counter and finished-CTA count, both zero before the launch (the kernel
// leaves them zero)
// Launch tile t is tile t - tile0[j] of tensor j, tile0[j] <= t < tile0[j + 1]
// (the tensors one after the other).
struct PrepJobs {
  CUtensorMap map[3];
  PrepJob job[3];
  int n_jobs;
  int any_transpose;
  long long n_tiles;
  long long tile0[3];
  unsigned long long* sched;
};
PrepJob prep_job(void* x8, float* descale, int B, int H, int N, const int8_t* signs,
                 int sign_group, int transpose_out, const float* rope_cos, const float* rope_sin);
// n_tiles and tile0 of J from its jobs
void prep_order(PrepJobs& J);
int launch_prep_jobs(const PrepJobs& J, int d, int sm_count, unsigned int* status,
                     cudaStream_t stream);

// per_tensor: one scale for the tensor (descale[0] is used as the amax
// accumulator, then every block's descale is written); rope_cos / rope_sin:
// NULL or float32 [N, d/2] tables, rotation before the transform
// map_x: x [B, N, H, d] bf16 as TMA dims (d, H, N, B), box d x 1 x 128 x 1,
// no swizzle (encode_prep_map)
int launch_prep_fp8(const CUtensorMap& map_x, void* x8, float* descale, int B, int H, int N, int d,
                    const int8_t* signs, int sign_group, int transpose_out, const float* rope_cos,
                    const float* rope_sin, int per_tensor, int sm_count, unsigned int* status,
                    unsigned long long* sched, cudaStream_t stream);
int launch_rope_table(float* cos_out, float* sin_out, int N, int d, double base, long long pos0,
                      cudaStream_t stream);

}  // namespace attn
