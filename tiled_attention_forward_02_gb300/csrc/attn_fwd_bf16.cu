// attn_fwd_bf16.cu - fused forward kernel instances for bf16 operands.
#include "fwd_launch.cuh"

namespace attn {

int launch_fwd_bf16(int d, int causal, const CUtensorMap& q, const CUtensorMap& k,
                   const CUtensorMap& v, const FwdParams& p, int grid, cudaStream_t stream) {
  return launch_fwd_dt<DT_BF16>(d, causal, q, k, v, p, grid, stream);
}

}  // namespace attn
