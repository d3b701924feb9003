// Chunked causal prefill on tcgen05 tensor cores (filled in below).
#include "pa_internal.h"

namespace pa {

bool prefill_supported(const AttnArgs &) { return false; }

cudaError_t launch_prefill(const AttnArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace pa
