// verify_tc_bf16state.cu -- instances of the tensor-core verification kernel
// (verify_tc.cuh) for a bf16 state pool: S0 arrives by TMA directly in the
// operand layout of the first product, and a fused commit rounds S_a to bf16.
#include "verify_tc.cuh"

namespace treewy {

cudaError_t launch_verify_tc_bf16state(const treewy_batch& b, const VerifyMaps& maps,
                                       const PrevRound* prev, int npm, cudaStream_t stream) {
  return launch_tc<true>(b, maps, prev, npm, stream);
}

}  // namespace treewy
