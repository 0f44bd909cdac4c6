// int8.cu -- fused INT8 decode with the witness bound (placeholder until written).
#include "kvc_internal.h"

namespace kvc {
cudaError_t launch_int8_decode(kvc_handle*, const void*, void*, float*, float*, float*, cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace kvc
