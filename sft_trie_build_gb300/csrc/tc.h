// Tensor-core (tcgen05) tree-attention launchers, bf16, head_dim 128.
#pragma once

#include <cuda_runtime.h>

#include "simt.h"

namespace stp {

cudaError_t tc_fwd(const AttnArgs& a, cudaStream_t s);
cudaError_t tc_bwd(const AttnArgs& a, cudaStream_t s);

}  // namespace stp
