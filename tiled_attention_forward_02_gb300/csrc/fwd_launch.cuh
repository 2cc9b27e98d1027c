// fwd_launch.cuh - template launch helpers for the fused forward kernel;
// included by the per-element-type translation units only.
#pragma once

#include "attn_fwd_kernel.cuh"
#include "internal.h"

namespace attn {

template <int D, int DT, bool CAUSAL, bool SPLIT>
int launch_fwd_instance(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                        const FwdParams& p, int grid, cudaStream_t stream) {
  using C = FwdCfg<D, DT>;
  auto kern = attn_fwd_kernel<D, DT, CAUSAL, SPLIT>;
  if constexpr (C::QST == 2) {
    // the register split inside the kernel must fit in the block's pool,
    // otherwise setmaxnreg.inc would wait forever: refuse to launch instead
    cudaFuncAttributes fa;
    cudaError_t ea = cudaFuncGetAttributes(&fa, kern);
    if (ea != cudaSuccess) return cuda_fail(ea, "cudaFuncGetAttributes");
    if (fa.numRegs < C::LAUNCH_REGS) return ATTN_ERR_DEVICE;
  }
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
  kern<<<grid, C::NTHREADS, C::SMEM_BYTES, stream>>>(q, k, v, p);
  note_launch();
  return check_launch();
}

// causal: 0 or 1; 2 = non-causal with the key range split (FP32 partial results)
template <int DT, int D>
int launch_fwd_d(int causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                 const FwdParams& p, int grid, cudaStream_t stream) {
  switch (causal) {
    case 0: return launch_fwd_instance<D, DT, false, false>(q, k, v, p, grid, stream);
    case 1: return launch_fwd_instance<D, DT, true, false>(q, k, v, p, grid, stream);
    default:
      if constexpr (DT == DT_E4M3) return ATTN_ERR_UNSUPPORTED;
      else return launch_fwd_instance<D, DT, false, true>(q, k, v, p, grid, stream);
  }
}

template <int DT>
int launch_fwd_dt(int d, int causal, const CUtensorMap& q, const CUtensorMap& k,
                  const CUtensorMap& v, const FwdParams& p, int grid, cudaStream_t stream) {
  switch (d) {
    case 64: return launch_fwd_d<DT, 64>(causal, q, k, v, p, grid, stream);
    case 128: return launch_fwd_d<DT, 128>(causal, q, k, v, p, grid, stream);
    case 256: return launch_fwd_d<DT, 256>(causal, q, k, v, p, grid, stream);
    default: return ATTN_ERR_UNSUPPORTED;
  }
}

}  // namespace attn
