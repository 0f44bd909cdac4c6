// decode_noalloc.cu -- kvc_decode_attn_noalloc: decode attention whose split-K
// scratch lives in a fixed array inside this library instead of the caller's
// state buffer.
//
// Some callers cannot call cudaMalloc at all while they decode. Examples:
//  - a serving engine that reserved all device memory for its KV pool at start-up;
//  - an embedding runtime whose allocator owns every device buffer;
//  - host code that must not block on the allocator's device synchronisation.
// They hand over the cache, q and out buffers they already own, and this entry
// point needs nothing else.  The scratch is a file-scope __device__ array, so
// every GPU that loads the library keeps KVC_NOALLOC_SCRATCH_BYTES reserved
// until the process exits.
//
// In host code, the array's name is only a host-side stand-in, not a device
// address.  The device address is fetched once per device with
// cudaGetSymbolAddress, with that device current, and passed to the kernels.
#include <cmath>
#include <mutex>

#include "kvc_internal.h"

namespace kvc {
bool fast_decode_supported(const DecodeArgs& a);
}

namespace {

// Partials of one call: (m, l) pairs [B][Hq][splits], then accumulators
// [B][Hq][splits][d], 256-byte aligned.  Every call shares this array.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KVC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on device `dev` (which must be current).
cudaError_t scratch_address(int dev, void** out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int kvc_decode_attn_noalloc(kvc_t h, const void* d_q, void* d_out, kvc_stream_t stream) {
    using namespace kvc;
    if (!h || !d_q || !d_out) return KVC_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(d_q) & 15u) || (reinterpret_cast<uintptr_t>(d_out) & 15u)) return KVC_ERR_ARG;
    const Shape& s = h->sh;
    if (s.int8) return KVC_ERR_UNSUPPORTED;
    for (int b = 0; b < s.B; ++b)
        if (h->np[b] < 1) return KVC_ERR_ARG;
    if (s.ring && h->ring_needs_append) return KVC_ERR_ARG;

    // scratch this call needs; refuse anything beyond the fixed array
    const size_t rows = (size_t)s.B * s.Hq * s.max_splits;
    const size_t ml_bytes = (rows * sizeof(float2) + 255) & ~(size_t)255;
    const size_t need = ml_bytes + rows * s.d * sizeof(float);
    if (need > (size_t)KVC_NOALLOC_SCRATCH_BYTES) return KVC_ERR_CAPACITY;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVC_ERR_CUDA;
    if (dev != h->device) return KVC_ERR_ARG;
    void* base = nullptr;
    if (scratch_address(dev, &base) != cudaSuccess) return KVC_ERR_CUDA;

    DecodeArgs a{};
    a.q = d_q;
    a.k = h->state + h->L.k;
    a.v = h->state + h->L.v;
    a.next_pos = reinterpret_cast<const int32_t*>(h->state + h->L.next_pos);
    a.rope = s.rope ? reinterpret_cast<const float2*>(h->state + h->L.rope) : nullptr;
    a.part_ml = static_cast<float2*>(base);
    a.part_acc = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + ml_bytes);
    a.hdr = reinterpret_cast<uint32_t*>(h->state + h->L.hdr);
    a.table = s.pages ? reinterpret_cast<const int32_t*>(h->state + h->L.table) : nullptr;
    a.B = s.B; a.Hq = s.Hq; a.Hkv = s.Hkv; a.g = s.g; a.d = s.d; a.S = s.S; a.W = s.W;
    a.max_splits = s.max_splits; a.split = s.split; a.gqa = s.gqa; a.ring = s.ring; a.bf16 = s.bf16;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.d));
    CombineArgs c{};
    c.part_ml = a.part_ml; c.part_acc = a.part_acc; c.next_pos = a.next_pos; c.out = d_out;
    c.B = s.B; c.Hq = s.Hq; c.d = s.d; c.S = s.S; c.W = s.W; c.max_splits = s.max_splits;
    c.split = s.split; c.ring = s.ring; c.bf16 = s.out_bf16;
    c.align_lo = s.pages > 0 && s.gqa;
    const bool fast = s.split == kFastSplit && fast_decode_supported(a);
    if (launch_decode(a, c, fast, h->has_kv_maps ? &h->kv_maps : nullptr, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return KVC_ERR_CUDA;
    return KVC_OK;
}
