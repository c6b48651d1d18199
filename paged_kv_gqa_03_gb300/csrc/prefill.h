// prefill.h — host entry points of the two tcgen05 prefill kernels.
#pragma once

#include "internal.h"

namespace pkv {

// One CTA per work item (prefill_tiles.cu); same contract as launch_prefill,
// which runs the persistent kernel (prefill.cu).
cudaError_t launch_prefill_tiles(const PrefillParams &p, int cache_dtype, const CUtensorMap &tmK,
                                 const CUtensorMap &tmV, cudaStream_t stream);

}  // namespace pkv
