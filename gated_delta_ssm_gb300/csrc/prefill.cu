// prefill.cu -- chunked prefill (placeholder until the chunk kernel lands).
#include "gdn_kernels.h"

namespace gdn {

cudaError_t launch_prefill(const PrefillArgs &, bool, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gdn
