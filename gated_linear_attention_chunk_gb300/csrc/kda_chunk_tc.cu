// Chunked (64-token) KDA forward on tcgen05 tensor cores.  (Placeholder until
// the kernel lands: reports the shape as unsupported so every prefill runs
// through the token-sequential kernel.)
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {

bool chunk_tc_supported(int, int, int) { return false; }

cudaError_t launch_chunk_tc(const ChunkParams &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace kda
