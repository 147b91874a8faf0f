// Tensor-core (tcgen05) chunk prefill: not built yet; the launcher reports
// the shape as unsupported so that AUTO selects the CUDA-core kernel.
#include "kda_internal.h"

namespace kda {

bool chunk_tc_supported(int, int, bool) { return false; }
size_t chunk_tc_scratch_bytes(int, int, int, int) { return 0; }
cudaError_t launch_chunk_tc(const ChunkArgs &, cudaStream_t) { return cudaErrorInvalidValue; }

}  // namespace kda
