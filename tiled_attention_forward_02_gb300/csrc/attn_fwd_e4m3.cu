// attn_fwd_e4m3.cu - fused forward kernel instances for e4m3 operands.
#include "fwd_launch.cuh"

namespace attn {

int launch_fwd_e4m3(int d, int causal, const CUtensorMap& q, const CUtensorMap& k,
                   const CUtensorMap& v, const FwdParams& p, int grid, cudaStream_t stream) {
  return launch_fwd_dt<DT_E4M3>(d, causal, q, k, v, p, grid, stream);
}

}  // namespace attn
