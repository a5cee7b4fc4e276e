// bf16 tree attention launchers.
#include "tc.h"

namespace stp {

cudaError_t tc_fwd(const AttnArgs& a, cudaStream_t s) { return simt_fwd(a, true, s); }
cudaError_t tc_bwd(const AttnArgs& a, cudaStream_t s) { return simt_bwd(a, true, s); }

}  // namespace stp
