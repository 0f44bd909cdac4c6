// decode_fast.cu -- bf16 split-K decode kernel (placeholder until written).
#include "kvc_internal.h"

namespace kvc {
bool fast_decode_supported(const DecodeArgs&) { return false; }
cudaError_t launch_decode_fast(const DecodeArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace kvc
