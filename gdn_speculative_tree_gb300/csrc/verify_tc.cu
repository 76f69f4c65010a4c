// verify_tc.cu -- launchers of the tensor-core verification kernel
// (verify_tc.cuh) for an fp32 state pool; a bf16 pool is dispatched to
// verify_tc_bf16state.cu, so the two sets of instances compile in parallel.
#include "verify_tc.cuh"

namespace treewy {

cudaError_t launch_verify_tc(const treewy_batch& b, const VerifyMaps& maps, int npm,
                             cudaStream_t stream) {
  if (b.flags & TREEWY_FLAG_STATE_BF16) return launch_verify_tc_bf16state(b, maps, nullptr, npm, stream);
  return launch_tc<false>(b, maps, nullptr, npm, stream);
}

cudaError_t launch_commit_verify_tc(const treewy_batch& next, const PrevRound& prev,
                                    const VerifyMaps& maps, int npm, cudaStream_t stream) {
  if (next.flags & TREEWY_FLAG_STATE_BF16)
    return launch_verify_tc_bf16state(next, maps, &prev, npm, stream);
  return launch_tc<false>(next, maps, &prev, npm, stream);
}

}  // namespace treewy
