// chunk.cu -- chunked causal suffix attention (placeholder until written).
#include "kvc_internal.h"

namespace kvc {
cudaError_t launch_chunk(kvc_handle*, const void*, void*, int, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace kvc
