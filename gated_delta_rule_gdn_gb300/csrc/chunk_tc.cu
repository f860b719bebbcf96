// Fused tcgen05/TMA chunk kernel (scalar gate): placeholder until the kernel lands.
#include "internal.h"

namespace gdn {

const char* tc_chunk_unsupported_reason(const ChunkArgs&) { return "the tcgen05 kernel is not built yet"; }

cudaError_t launch_chunk_tc(const ChunkArgs&, cudaStream_t) { return cudaErrorNotSupported; }

cudaError_t tc_read_and_clear_status(unsigned* value, bool) {
    *value = 0;
    return cudaSuccess;
}

}  // namespace gdn
