// gdn_tree_tc.cu -- tensor-core (tcgen05) contraction of the tree verifier.
#include "gdn_internal.cuh"

namespace gdn {

bool tc_contract_eligible(const VerifyArgs&) { return false; }

cudaError_t launch_tree_contract_tc(const VerifyArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gdn
