// MLA decode on tcgen05 tensor cores (filled in below).
#include "pa_internal.h"

namespace pa {

bool mla_supported(const AttnArgs &) { return false; }

cudaError_t launch_mla(const AttnArgs &, bool, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace pa
