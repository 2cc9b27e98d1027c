// attn_fwd_f16.cu - fused forward kernel instances for f16 operands.
#include "fwd_launch.cuh"

namespace attn {

int launch_fwd_f16(int d, int causal, const CUtensorMap& q, const CUtensorMap& k,
                   const CUtensorMap& v, const FwdParams& p, int grid, cudaStream_t stream) {
  return launch_fwd_dt<DT_F16>(d, causal, q, k, v, p, grid, stream);
}

}  // namespace attn
