// kvc_api.cu -- the C ABI (include/kvc.h): argument checks, state layout, host
// mirror of next_position, RoPE table, and kernel launches.
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "async_copy.h"
#include "kvc_internal.h"

namespace kvc {

cudaError_t allow_smem(const void* kernel, size_t bytes) {
    // each thread remembers the grants it made (a few kernels): no lock on the launch path;
    // setting the attribute again from another thread is harmless
    struct Grant { const void* kernel; int device; size_t bytes; };
    thread_local std::vector<Grant> granted;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    for (const Grant& g : granted)
        if (g.kernel == kernel && g.device == dev && g.bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) granted.push_back(Grant{kernel, dev, bytes});
    return e;
}

cudaError_t launch_append_rows_counts(const AppendArgs& a, const int32_t* counts, cudaStream_t st);
bool fast_decode_supported(const DecodeArgs& a);
cudaError_t launch_int8_decode(kvc_handle* h, const void* q, void* out, float* cmax, float* tanh_out,
                               float* ct, cudaStream_t st);

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// One CTA waits on an mbarrier that nothing arrives at: the bounded wait gives up and
// flags the error word, as a kernel whose copy never lands would.
__global__ void wait_path_kernel(uint32_t* hdr) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0)) atomicOr(hdr, kErrWait);
}

}  // namespace

bool make_shape(const kvc_config& c, Shape* s) {
    if (c.dtype != KVC_F32 && c.dtype != KVC_BF16) return false;
    if (c.layout != KVC_CONTIGUOUS && c.layout != KVC_RING) return false;
    if (c.kv_quant != KVC_QUANT_NONE && c.kv_quant != KVC_QUANT_INT8 && c.kv_quant != KVC_QUANT_INT8_DITHER)
        return false;
    if (c.batch < 1 || c.n_q_heads < 1 || c.n_kv_heads < 1) return false;
    if (c.n_q_heads % c.n_kv_heads) return false;
    if (c.head_dim < 2 || c.head_dim > 256 || (c.head_dim & 1)) return false;
    if (c.capacity < 1 || c.window < 0 || c.max_position < 0 || c.max_chunk < 0) return false;
    if (c.out_dtype != 0 && c.out_dtype != KVC_F32 + 1 && c.out_dtype != KVC_BF16 + 1) return false;
    if (!(c.rope_base >= 0.f) || std::isinf(c.rope_base)) return false;
    const bool ring = c.layout == KVC_RING;
    if (ring && c.window != 0 && c.window != c.capacity) return false;
    const bool int8 = c.kv_quant != KVC_QUANT_NONE;
    const bool dither = c.kv_quant == KVC_QUANT_INT8_DITHER;
    // the dither counter packs the KV head and the layer into 16 bits each
    if (dither && (c.layer_index < 0 || c.layer_index > 65535 || c.n_kv_heads > 65536)) return false;
    if (int8 && (c.dtype != KVC_BF16 || c.head_dim % kBands || c.capacity % kQBlock)) return false;
    // the gated fallback's pool serves contiguous caches attending to their whole history
    if (c.int8_exact_blocks < 0 ||
        ((!int8 || dither || ring || c.window != 0) && c.int8_exact_blocks != 0))
        return false;
    if (c.page_pool < 0 || (c.page_pool > 0 && c.capacity % kPage)) return false;
    if (c.page_pool > 0 && c.int8_exact_blocks != 0) return false;   // the gate's pool: unpaged caches
    if (c.int8_split != 0 && (!int8 || c.int8_split % 64 != 0 || c.int8_split < kInt8Split ||
                              c.int8_split > kInt8SplitLong))
        return false;
    if (c.store_slots < 0 || (c.store_slots > 0 && int8)) return false;
    if (int8) {
        const int g = c.n_q_heads / c.n_kv_heads;
        if ((c.head_dim != 64 && c.head_dim != 128) || (g != 1 && g != 2 && g != 4 && g != 8)) return false;
    }
    const bool rope = c.rope_base > 0.f;
    int P = 0;
    if (rope) {
        P = c.max_position ? c.max_position : (ring ? 0 : c.capacity);
        if (P < 1) return false;
    }
    s->B = c.batch; s->Hq = c.n_q_heads; s->Hkv = c.n_kv_heads; s->g = c.n_q_heads / c.n_kv_heads;
    s->d = c.head_dim; s->S = c.capacity; s->W = ring ? c.capacity : c.window;
    s->P = P; s->ring = ring; s->int8 = int8; s->rope = rope; s->bf16 = c.dtype == KVC_BF16;
    s->dither = dither;
    s->elem = s->bf16 ? 2 : 4;
    s->max_chunk = c.max_chunk;
    s->xpool = c.int8_exact_blocks;
    s->pages = c.page_pool;
    s->store_slots = c.store_slots;
    s->out_bf16 = c.out_dtype == 0 ? s->bf16 : c.out_dtype == KVC_BF16 + 1;
    s->split = kGenericSplit;
    if (s->bf16 && !int8 && (s->d == 64 || s->d == 128) && s->g <= 8) s->split = kFastSplit;
    // (its tensor copies address cache rows with signed 32-bit coordinates)
    const long long rows = s->pages ? (long long)s->pages * s->Hkv * kPage : (long long)s->B * s->Hkv * s->S;
    const long long keys = (s->W > 0 && s->W < s->S) ? s->W : s->S;
    s->gqa = s->bf16 && !int8 && gqa_decode_supported(s->d, s->g) && rows < (1ll << 31);
    if (s->gqa) s->split = keys >= kGqaLongKeys ? kGqaSplitLong : kGqaSplit;
    // the generic decode holds a CTA's g queries and g x split scores in shared memory
    if (!int8 && s->split == kGenericSplit && (size_t)s->g * (s->d + kGenericSplit) * 4 > kMaxSmemPerBlock)
        return false;
    // a paged cache may start its splits up to one page before the window
    s->max_splits = (int)((keys + s->split - 1) / s->split) + (s->pages > 0 ? 1 : 0);
    if (int8) {
        // quantized splits (longer ones for long caches: less start-up per byte; a longer
        // split measured faster than one that fills the SMs' last wave of CTAs better), one
        // split for the exact tail rows and, with a pool, the splits of the exact-block decode
        const long long qkeys = int8_qkeys(*s);
        s->split = c.int8_split ? c.int8_split : qkeys >= kInt8LongKeys ? kInt8SplitLong : kInt8Split;
        s->max_splits = (int)((qkeys + s->split - 1) / s->split) + 1 + (s->xpool > 0 ? kExactSplits : 0);
    }
    return true;
}

Layout make_layout(const Shape& s) {
    Layout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
    const size_t B = s.B, Hkv = s.Hkv, S = s.S, d = s.d, Hq = s.Hq;
    L.hdr = take(256);
    L.next_pos = take(B * 4);
    L.pos = take(B * S * 4);
    if (!s.int8) {
        const size_t rows = s.pages ? (size_t)s.pages * Hkv * kPage : B * Hkv * S;
        L.k = take(rows * d * s.elem);
        L.v = take(rows * d * s.elem);
        if (s.pages) L.table = take(B * (S / kPage) * 4);
    } else {
        // quantized blocks: [B][Hkv][S/16], or [pages][Hkv] on a paged cache
        const size_t blocks = s.pages ? (size_t)s.pages * Hkv : B * Hkv * (S / kQBlock);
        L.kq = take(blocks * kQBlock * d);
        L.vq = take(blocks * kQBlock * d);
        L.sk = take(blocks * 4);
        L.sv = take(blocks * 4);
        if (!s.dither) L.wit = take(blocks * kQBlock * kBands * 2);
        if (s.pages) L.table = take(B * (S / kPage) * 4);
        L.ktail = take(B * Hkv * kQBlock * d * 2);
        L.vtail = take(B * Hkv * kQBlock * d * 2);
        L.xmap = take(B * Hkv * (S / kQBlock) * 4);
        L.xn = take(B * Hkv * 4);
        L.xlist = take(B * Hkv * kMaxRestored * 4);
        L.xent = take(B * Hkv * kMaxRestored * 4);
        L.xpool = take((size_t)s.xpool * 2 * kQBlock * d * 2);
    }
    L.req_id = take(B * 4);
    L.arrive = take(B * 4);
    L.rope = take((size_t)s.P * (d / 2) * 8);
    L.part_ml = take(B * Hq * s.max_splits * 8);
    L.part_acc = take(B * Hq * s.max_splits * d * 4);
    if (s.int8) L.part_c = take(B * Hq * s.max_splits * 4);
    if (s.ring && s.bf16 && !s.int8 && s.max_chunk > 0)
        L.cws = take(2 * B * Hkv * (size_t)chunk_ws_rows(s) * d * 2);
    if (s.store_slots > 0) {
        L.store_stride = align256(2 * Hkv * S * d * s.elem + S * 4);
        L.store = take((size_t)s.store_slots * L.store_stride);
    }
    L.total = o;
    return L;
}

}  // namespace kvc

using namespace kvc;

namespace {

inline cudaStream_t S_(kvc_stream_t s) { return static_cast<cudaStream_t>(s); }

template <typename T>
T* at(kvc_handle* h, size_t off) { return reinterpret_cast<T*>(h->state + off); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// {cos, sin} of angle p * base^(-(2i)/d) (double), each rounded once to fp32.
void rope_table(double base, int d, int P, float2* out) {
    const int half = d / 2;
    std::vector<double> theta(half);
    for (int i = 0; i < half; ++i) theta[i] = std::pow(base, (double)(-2 * i) / (double)d);
    for (int p = 0; p < P; ++p)
        for (int i = 0; i < half; ++i) {
            const double ang = (double)p * theta[i];
            out[(size_t)p * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        }
}

AppendArgs append_args(kvc_handle* h, const void* k, const void* v, int n) {
    const Shape& s = h->sh;
    AppendArgs a{};
    a.k = k; a.v = v; a.n = n;
    a.sb = (size_t)s.Hkv * n * s.d; a.sh = (size_t)n * s.d; a.sr = s.d;   // [B][Hkv][n][d]
    a.next_pos = at<int32_t>(h, h->L.next_pos);
    a.pos = at<int32_t>(h, h->L.pos);
    if (!s.int8) { a.kc = h->state + h->L.k; a.vc = h->state + h->L.v; }
    else {
        a.kq = at<int8_t>(h, h->L.kq); a.vq = at<int8_t>(h, h->L.vq);
        a.sk = at<float>(h, h->L.sk); a.sv = at<float>(h, h->L.sv);
        a.wit = s.dither ? nullptr : at<__half>(h, h->L.wit);
        a.ktail = at<__nv_bfloat16>(h, h->L.ktail); a.vtail = at<__nv_bfloat16>(h, h->L.vtail);
    }
    a.rope = s.rope ? at<float2>(h, h->L.rope) : nullptr;
    a.hdr = at<uint32_t>(h, h->L.hdr);
    a.table = s.pages ? at<int32_t>(h, h->L.table) : nullptr;
    a.req_id = at<uint32_t>(h, h->L.req_id);
    a.key0 = h->cfg.dither_key_lo; a.key1 = h->cfg.dither_key_hi;
    a.layer_ctr = 65536u * (uint32_t)h->cfg.layer_index;
    a.B = s.B; a.Hkv = s.Hkv; a.d = s.d; a.S = s.S; a.P = s.P;
    a.ring = s.ring; a.bf16 = s.bf16; a.int8 = s.int8; a.dither = s.dither;
    a.arrive = at<int32_t>(h, h->L.arrive);
    // a one-token append into an INT8 cache quantizes a block per KV head every 16th row: up to
    // 8 CTAs per request share that work; a bf16/fp32 append is one CTA per request (its arrival
    // fence and counter cost more than the rows: sliding-window GQA step 0.1626 against 0.1594 ms)
    a.hpc = s.int8 ? (s.Hkv + 7) / 8 : s.Hkv;
    return a;
}

// Highest position the append of counts[b] rows would reach must fit.
int check_capacity(kvc_handle* h, const int32_t* counts, int n) {
    const Shape& s = h->sh;
    for (int b = 0; b < s.B; ++b) {
        const long long c = counts ? counts[b] : n;
        if (c <= 0) continue;
        const long long last = (long long)h->np[b] + c - 1;
        if (last > 0x7ffffffeLL) return KVC_ERR_CAPACITY;
        if (!s.ring && last >= s.S) return KVC_ERR_CAPACITY;
        if (s.rope && last >= s.P) return KVC_ERR_CAPACITY;
    }
    return KVC_OK;
}

}  // namespace

extern "C" {

const char* kvc_strerror(int code) {
    switch (code) {
        case KVC_OK: return "ok";
        case KVC_ERR_ARG: return "invalid argument";
        case KVC_ERR_CAPACITY: return "cache capacity or RoPE table exceeded";
        case KVC_ERR_EVICTED: return "rows needed after the trim are no longer held exactly";
        case KVC_ERR_CUDA: return "CUDA runtime error";
        case KVC_ERR_UNSUPPORTED: return "not supported for this configuration";
        case KVC_ERR_DEVICE: return "a kernel reported an error";
        default: return "unknown status";
    }
}

int kvc_state_bytes(const kvc_config* cfg, size_t* bytes) {
    if (!cfg || !bytes) return KVC_ERR_ARG;
    Shape s;
    if (!make_shape(*cfg, &s)) return KVC_ERR_ARG;
    *bytes = make_layout(s).total;
    return KVC_OK;
}

int kvc_create(const kvc_config* cfg, void* d_state, size_t bytes, kvc_stream_t stream, kvc_t* out) {
    if (!cfg || !d_state || !out) return KVC_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(d_state) & 255u) return KVC_ERR_ARG;
    Shape s;
    if (!make_shape(*cfg, &s)) return KVC_ERR_ARG;
    Layout L = make_layout(s);
    if (bytes < L.total) return KVC_ERR_ARG;
    kvc_handle* h = new (std::nothrow) kvc_handle();
    if (!h) return KVC_ERR_ARG;
    h->cfg = *cfg; h->sh = s; h->L = L; h->state = static_cast<char*>(d_state); h->bytes = bytes;
    h->np.assign(s.B, 0);
    h->store_n.assign(s.store_slots, -1);
    h->ring_needs_append = false;
    h->has_kv_maps = false;
    if (s.gqa) {
        // the GQA decode reads 16-row tiles of the K and V caches by tensor copy
        const cuuint64_t dims[2] = {(cuuint64_t)s.d,
                                    s.pages ? (cuuint64_t)s.pages * s.Hkv * kPage : (cuuint64_t)s.B * s.Hkv * s.S};
        const cuuint64_t strides[1] = {(cuuint64_t)s.d * 2};
        const cuuint32_t box[2] = {64, 16};
        if (!make_tensor_map_bf16(&h->kv_maps.k, h->state + L.k, 2, dims, strides, box) ||
            !make_tensor_map_bf16(&h->kv_maps.v, h->state + L.v, 2, dims, strides, box)) {
            delete h;
            return KVC_ERR_CUDA;
        }
        h->has_kv_maps = true;
    }
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
        delete h;
        return KVC_ERR_CUDA;
    }
    cudaStream_t st = S_(stream);
    cudaError_t e = cudaMemsetAsync(h->state, 0, L.total, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->state + L.pos, 0xff, (size_t)s.B * s.S * 4, st);
    if (e == cudaSuccess && s.pages) {
        // every logical page unmapped; the free pages in a fixed shuffled order, so
        // that requests' pages interleave in the pool
        e = cudaMemsetAsync(h->state + L.table, 0xff, (size_t)s.B * (s.S / kPage) * 4, st);
        h->table_h.assign((size_t)s.B * (s.S / kPage), -1);
        h->page_free.resize(s.pages);
        for (int i = 0; i < s.pages; ++i) h->page_free[i] = i;
        uint64_t x = 0x9E3779B97F4A7C15ull;
        for (int i = s.pages - 1; i > 0; --i) {
            x ^= x << 13; x ^= x >> 7; x ^= x << 17;
            std::swap(h->page_free[i], h->page_free[x % (uint64_t)(i + 1)]);
        }
    }
    if (e == cudaSuccess) {
        // request IDs of the dither counters: b until set
        h->req_id_h.resize(s.B);
        for (int b = 0; b < s.B; ++b) h->req_id_h[b] = (uint32_t)b;
        e = cudaMemcpyAsync(h->state + L.req_id, h->req_id_h.data(), (size_t)s.B * 4, cudaMemcpyHostToDevice, st);
    }
    if (e == cudaSuccess && s.int8) {
        const size_t nb = (size_t)s.B * s.Hkv * (s.S / kQBlock);
        e = cudaMemsetAsync(h->state + L.xmap, 0xff, nb * 4, st);
        h->xmap_h.assign(nb, -1);
        h->xn_h.assign((size_t)s.B * s.Hkv, 0);
        h->xlist_h.assign((size_t)s.B * s.Hkv * kMaxRestored, 0);
        h->xent_h.assign((size_t)s.B * s.Hkv * kMaxRestored, 0);
        for (int i = s.xpool - 1; i >= 0; --i) h->xfree.push_back(i);
    }
    if (e == cudaSuccess && s.rope) {
        std::vector<float2> tab((size_t)s.P * (s.d / 2));
        rope_table((double)cfg->rope_base, s.d, s.P, tab.data());
        e = cudaMemcpyAsync(h->state + L.rope, tab.data(), tab.size() * sizeof(float2),
                            cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) { delete h; return KVC_ERR_CUDA; }
    *out = h;
    return KVC_OK;
}

int kvc_destroy(kvc_t h) {
    if (!h) return KVC_ERR_ARG;
    delete h;
    return KVC_OK;
}

int kvc_append(kvc_t h, const void* d_k, const void* d_v, kvc_stream_t stream) {
    if (!h || !on_device(h) || !d_k || !d_v || !aligned16(d_k) || !aligned16(d_v)) return KVC_ERR_ARG;
    int rc = check_capacity(h, nullptr, 1);
    if (rc) return rc;
    if (h->sh.pages) {
        std::vector<int> to(h->np.begin(), h->np.end());
        for (auto& t : to) ++t;
        if (map_pages(h, std::vector<int>(h->np.begin(), h->np.end()), to, S_(stream), &rc) != cudaSuccess)
            return KVC_ERR_CUDA;
        if (rc) return rc;
    }
    AppendArgs a = append_args(h, d_k, d_v, 1);
    if (launch_append_token(a, S_(stream)) != cudaSuccess) return KVC_ERR_CUDA;
    for (auto& p : h->np) ++p;
    h->ring_needs_append = false;
    return KVC_OK;
}

int kvc_append_rows(kvc_t h, const void* d_k, const void* d_v, int32_t n, const int32_t* h_counts,
                    kvc_stream_t stream) {
    if (!h || !on_device(h) || n < 0 || !aligned16(d_k) || !aligned16(d_v)) return KVC_ERR_ARG;
    if (n == 0) return KVC_OK;
    if (!d_k || !d_v) return KVC_ERR_ARG;
    const Shape& s = h->sh;
    h->counts.assign(s.B, n);
    if (h_counts)
        for (int b = 0; b < s.B; ++b) {
            if (h_counts[b] < 0 || h_counts[b] > n) return KVC_ERR_ARG;
            h->counts[b] = h_counts[b];
        }
    int rc = check_capacity(h, h->counts.data(), n);
    if (rc) return rc;
    if (s.pages) {
        std::vector<int> from(h->np.begin(), h->np.end()), to(from);
        for (int b = 0; b < s.B; ++b) to[b] += h->counts[b];
        if (map_pages(h, from, to, S_(stream), &rc) != cudaSuccess) return KVC_ERR_CUDA;
        if (rc) return rc;
    }
    AppendArgs a = append_args(h, d_k, d_v, n);
    if (launch_append_rows_counts(a, h->counts.data(), S_(stream)) != cudaSuccess) return KVC_ERR_CUDA;
    bool any = false;
    for (int b = 0; b < s.B; ++b) { h->np[b] += h->counts[b]; any |= h->counts[b] > 0; }
    if (any) h->ring_needs_append = false;
    return KVC_OK;
}

int kvc_decode_attn(kvc_t h, const void* d_q, void* d_out, float* d_cmax, float* d_tanh, float* d_ct,
                    kvc_stream_t stream) {
    if (!h || !on_device(h) || !d_q || !d_out || !aligned16(d_q) || !aligned16(d_out)) return KVC_ERR_ARG;
    const Shape& s = h->sh;
    for (int b = 0; b < s.B; ++b)
        if (h->np[b] < 1) return KVC_ERR_ARG;                 // nothing cached to attend to
    if (s.ring && h->ring_needs_append) return KVC_ERR_ARG;
    cudaStream_t st = S_(stream);
    if (s.dither && (d_cmax || d_tanh || d_ct)) return KVC_ERR_ARG;      // Tier B returns no bound
    if (s.int8) {
        if (launch_int8_decode(h, d_q, d_out, d_cmax, d_tanh, d_ct, st) != cudaSuccess) return KVC_ERR_CUDA;
        return KVC_OK;
    }
    if (d_ct) return KVC_ERR_ARG;
    DecodeArgs a{};
    a.q = d_q; a.k = h->state + h->L.k; a.v = h->state + h->L.v;
    a.next_pos = at<int32_t>(h, h->L.next_pos);
    a.rope = s.rope ? at<float2>(h, h->L.rope) : nullptr;
    a.part_ml = at<float2>(h, h->L.part_ml);
    a.part_acc = at<float>(h, h->L.part_acc);
    a.hdr = at<uint32_t>(h, h->L.hdr);
    a.table = s.pages ? at<int32_t>(h, h->L.table) : nullptr;
    a.B = s.B; a.Hq = s.Hq; a.Hkv = s.Hkv; a.g = s.g; a.d = s.d; a.S = s.S; a.W = s.W;
    a.max_splits = s.max_splits; a.split = s.split; a.gqa = s.gqa; a.ring = s.ring; a.bf16 = s.bf16;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.d));
    CombineArgs c{};
    c.part_ml = a.part_ml; c.part_acc = a.part_acc; c.next_pos = a.next_pos; c.out = d_out;
    c.B = s.B; c.Hq = s.Hq; c.d = s.d; c.S = s.S; c.W = s.W; c.max_splits = s.max_splits;
    c.split = s.split; c.ring = s.ring; c.bf16 = s.out_bf16;
    c.align_lo = s.pages > 0 && s.gqa;
    const bool fast = s.split == kFastSplit && fast_decode_supported(a);
    if (launch_decode(a, c, fast, h->has_kv_maps ? &h->kv_maps : nullptr, st) != cudaSuccess) return KVC_ERR_CUDA;
    if (d_cmax && cudaMemsetAsync(d_cmax, 0, (size_t)s.B * s.Hq * 4, st) != cudaSuccess) return KVC_ERR_CUDA;
    if (d_tanh && cudaMemsetAsync(d_tanh, 0, (size_t)s.B * s.Hq * 4, st) != cudaSuccess) return KVC_ERR_CUDA;
    return KVC_OK;
}

int kvc_trim(kvc_t h, const int32_t* h_cut, kvc_stream_t stream) {
    if (!h || !on_device(h) || !h_cut) return KVC_ERR_ARG;
    const Shape& s = h->sh;
    for (int b = 0; b < s.B; ++b) {
        const int cut = h_cut[b], np = h->np[b];
        if (cut < 0 || cut > np) return KVC_ERR_ARG;
        if (s.ring) {
            const int lo = cut - s.S + 1 > 0 ? cut - s.S + 1 : 0;
            const int resident = np - s.S > 0 ? np - s.S : 0;
            if (!(lo == cut || lo >= resident)) return KVC_ERR_EVICTED;
        }
        if (s.int8 && (cut % kQBlock) && cut < (np / kQBlock) * kQBlock) return KVC_ERR_EVICTED;
    }
    if (launch_trim_cuts(at<int32_t>(h, h->L.next_pos), at<int32_t>(h, h->L.pos), h_cut, s.B, s.S, s.ring,
                         S_(stream)) != cudaSuccess)
        return KVC_ERR_CUDA;
    if (s.int8 && int8_drop_restored(h, h_cut, S_(stream)) != cudaSuccess) return KVC_ERR_CUDA;
    if (s.pages && !s.ring) {
        // a contiguous cache returns the pages that lie wholly past the cut
        bool freed = false;
        const int npg = s.S / kPage;
        for (int b = 0; b < s.B; ++b)
            for (int lp = (h_cut[b] + kPage - 1) / kPage; lp < npg; ++lp) {
                int32_t& e = h->table_h[(size_t)b * npg + lp];
                if (e < 0) continue;
                h->page_free.push_back(e);
                e = -1;
                freed = true;
            }
        if (freed && cudaMemcpyAsync(h->state + h->L.table, h->table_h.data(), h->table_h.size() * 4,
                                     cudaMemcpyHostToDevice, S_(stream)) != cudaSuccess)
            return KVC_ERR_CUDA;
    }
    for (int b = 0; b < s.B; ++b) h->np[b] = h_cut[b];
    if (s.ring) h->ring_needs_append = true;
    return KVC_OK;
}

int kvc_chunk_attn(kvc_t h, const void* d_q, const void* d_k, const void* d_v, int32_t n, void* d_out,
                   kvc_stream_t stream) {
    if (!h || !on_device(h) || !d_q || !d_k || !d_v || !d_out || n < 1) return KVC_ERR_ARG;
    if (!aligned16(d_q) || !aligned16(d_k) || !aligned16(d_v) || !aligned16(d_out)) return KVC_ERR_ARG;
    const Shape& s = h->sh;
    if (!chunk_supported(s)) return KVC_ERR_UNSUPPORTED;
    if (n > s.max_chunk) return KVC_ERR_ARG;
    int rc = check_capacity(h, nullptr, n);
    if (rc) return rc;
    cudaStream_t st = S_(stream);
    if (s.pages) {
        std::vector<int> from(h->np.begin(), h->np.end()), to(from);
        for (auto& t : to) t += n;
        if (map_pages(h, from, to, st, &rc) != cudaSuccess) return KVC_ERR_CUDA;
        if (rc) return rc;
    }
    h->counts.assign(s.B, n);
    AppendArgs a = append_args(h, d_k, d_v, n);
    a.sb = (size_t)n * s.Hkv * s.d; a.sh = s.d; a.sr = (size_t)s.Hkv * s.d;   // [B][n][Hkv][d]
    if (s.ring) {
        // a ring would evict rows that the early suffix queries still need: the suffix is
        // staged beside the resident rows, attended, and only then appended
        if (launch_chunk(h, d_q, d_k, d_v, d_out, n, st) != cudaSuccess) return KVC_ERR_CUDA;
        if (launch_append_rows_counts(a, h->counts.data(), st) != cudaSuccess) return KVC_ERR_CUDA;
        for (auto& p : h->np) p += n;
        h->ring_needs_append = false;
        return KVC_OK;
    }
    // the suffix rows join the cache first (rotated keys, positions cut .. cut+n-1) ...
    if (launch_append_rows_counts(a, h->counts.data(), st) != cudaSuccess) return KVC_ERR_CUDA;
    for (auto& p : h->np) p += n;
    // ... then every suffix query attends over its window
    if (launch_chunk(h, d_q, d_k, d_v, d_out, n, st) != cudaSuccess) return KVC_ERR_CUDA;
    return KVC_OK;
}

int kvc_export_bytes(kvc_t h, int32_t which, size_t* bytes) {
    if (!h || !bytes) return KVC_ERR_ARG;
    const Shape& s = h->sh;
    const size_t B = s.B, Hkv = s.Hkv, S = s.S, d = s.d;
    switch (which) {
        case KVC_EXPORT_K: case KVC_EXPORT_V:
            if (s.int8) return KVC_ERR_ARG;
            *bytes = B * Hkv * S * d * s.elem; return KVC_OK;
        case KVC_EXPORT_POSITIONS: *bytes = B * S * 4; return KVC_OK;
        case KVC_EXPORT_PAGE_TABLE:
            if (!s.pages) return KVC_ERR_ARG;
            *bytes = B * (S / kPage) * 4; return KVC_OK;
        case KVC_EXPORT_NEXT_POSITION: *bytes = B * 4; return KVC_OK;
        default: break;
    }
    if (!s.int8) return KVC_ERR_ARG;
    switch (which) {
        case KVC_EXPORT_KQ: case KVC_EXPORT_VQ: *bytes = B * Hkv * S * d; return KVC_OK;
        case KVC_EXPORT_SK: case KVC_EXPORT_SV: *bytes = B * Hkv * (S / kQBlock) * 4; return KVC_OK;
        case KVC_EXPORT_WITNESS:
            if (s.dither) return KVC_ERR_ARG;
            *bytes = B * Hkv * S * kBands * 2; return KVC_OK;
        case KVC_EXPORT_KTAIL: case KVC_EXPORT_VTAIL: *bytes = B * Hkv * kQBlock * d * 2; return KVC_OK;
        case KVC_EXPORT_XMAP: *bytes = B * Hkv * (S / kQBlock) * 4; return KVC_OK;
        default: return KVC_ERR_ARG;
    }
}

int kvc_export(kvc_t h, int32_t which, void* h_dst, size_t bytes, kvc_stream_t stream) {
    size_t need = 0;
    int rc = kvc_export_bytes(h, which, &need);
    if (rc) return rc;
    if (!h_dst || bytes != need || !on_device(h)) return KVC_ERR_ARG;
    size_t off = 0;
    switch (which) {
        case KVC_EXPORT_K: off = h->L.k; break;
        case KVC_EXPORT_V: off = h->L.v; break;
        case KVC_EXPORT_POSITIONS: off = h->L.pos; break;
        case KVC_EXPORT_NEXT_POSITION: off = h->L.next_pos; break;
        case KVC_EXPORT_KQ: off = h->L.kq; break;
        case KVC_EXPORT_VQ: off = h->L.vq; break;
        case KVC_EXPORT_SK: off = h->L.sk; break;
        case KVC_EXPORT_SV: off = h->L.sv; break;
        case KVC_EXPORT_WITNESS: off = h->L.wit; break;
        case KVC_EXPORT_KTAIL: off = h->L.ktail; break;
        case KVC_EXPORT_VTAIL: off = h->L.vtail; break;
        case KVC_EXPORT_XMAP: off = h->L.xmap; break;
        case KVC_EXPORT_PAGE_TABLE: off = h->L.table; break;
        default: return KVC_ERR_ARG;
    }
    cudaStream_t st = S_(stream);
    if (h->sh.pages && (which == KVC_EXPORT_K || which == KVC_EXPORT_V)) {
        // gather the logical [B][Hkv][S][d] rows through the block table (zeros where unmapped)
        const Shape& s = h->sh;
        const size_t rowb = (size_t)s.d * s.elem, npg = s.S / kPage;
        std::vector<uint8_t> pool((size_t)s.pages * s.Hkv * kPage * rowb);
        if (cudaMemcpyAsync(pool.data(), h->state + off, pool.size(), cudaMemcpyDeviceToHost, st) != cudaSuccess)
            return KVC_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return KVC_ERR_CUDA;
        uint8_t* out = static_cast<uint8_t*>(h_dst);
        std::memset(out, 0, need);
        for (int b = 0; b < s.B; ++b)
            for (size_t lp = 0; lp < npg; ++lp) {
                const int page = h->table_h[b * npg + lp];
                if (page < 0) continue;
                for (int hh = 0; hh < s.Hkv; ++hh)
                    std::memcpy(out + (((size_t)b * s.Hkv + hh) * s.S + lp * kPage) * rowb,
                                pool.data() + (((size_t)page * s.Hkv + hh) * kPage) * rowb, kPage * rowb);
            }
        return KVC_OK;
    }
    const bool codes = which == KVC_EXPORT_KQ || which == KVC_EXPORT_VQ;
    const bool paged_blocks = h->sh.pages && h->sh.int8 &&
                              (codes || which == KVC_EXPORT_SK || which == KVC_EXPORT_SV || which == KVC_EXPORT_WITNESS);
    std::vector<uint8_t> raw(codes ? need : 0);
    void* dst = codes ? static_cast<void*>(raw.data()) : h_dst;
    if (paged_blocks) {
        // quantized blocks live in pages ([pages][Hkv] blocks): gather them into the logical
        // [B][Hkv][capacity/16] block order through the host mirror of the block table
        const Shape& s = h->sh;
        const size_t npg = s.S / kPage, per = need / ((size_t)s.B * s.Hkv * npg);
        std::vector<uint8_t> pool((size_t)s.pages * s.Hkv * per);
        if (cudaMemcpyAsync(pool.data(), h->state + off, pool.size(), cudaMemcpyDeviceToHost, st) != cudaSuccess)
            return KVC_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return KVC_ERR_CUDA;
        uint8_t* o = static_cast<uint8_t*>(dst);
        std::memset(o, 0, need);
        for (int b = 0; b < s.B; ++b)
            for (size_t lp = 0; lp < npg; ++lp) {
                const int page = h->table_h[b * npg + lp];
                if (page < 0) continue;
                for (int hh = 0; hh < s.Hkv; ++hh)
                    std::memcpy(o + (((size_t)b * s.Hkv + hh) * npg + lp) * per,
                                pool.data() + ((size_t)page * s.Hkv + hh) * per, per);
            }
    } else {
        if (cudaMemcpyAsync(dst, h->state + off, need, cudaMemcpyDeviceToHost, st) != cudaSuccess) return KVC_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return KVC_ERR_CUDA;
    }
    if (codes) {
        // stored biased in the decode's block order; exported signed, token-major [S][d]
        const int d = h->sh.d;
        const size_t blocks = need / ((size_t)kQBlock * d);
        int8_t* out = static_cast<int8_t*>(h_dst);
        for (size_t blk = 0; blk < blocks; ++blk) {
            const uint8_t* src = raw.data() + blk * kQBlock * d;
            int8_t* o = out + blk * kQBlock * d;
            for (int t = 0; t < kQBlock; ++t)
                for (int x = 0; x < d; ++x) {
                    const int at = which == KVC_EXPORT_KQ ? kq_offset(d, t, x) : vq_offset(d, t, x);
                    o[t * d + x] = (int8_t)((int)src[at] - 128);
                }
        }
    }
    return KVC_OK;
}

int kvc_set_request_id(kvc_t h, int32_t b, uint32_t request_id, kvc_stream_t stream) {
    if (!h || !on_device(h) || b < 0 || b >= h->sh.B || !h->sh.dither || h->np[b] != 0) return KVC_ERR_ARG;
    h->req_id_h[b] = request_id;
    if (cudaMemcpyAsync(h->state + h->L.req_id + (size_t)b * 4, &h->req_id_h[b], 4, cudaMemcpyHostToDevice,
                        S_(stream)) != cudaSuccess)
        return KVC_ERR_CUDA;
    return KVC_OK;
}

int kvc_next_positions(kvc_t h, int32_t* h_out) {
    if (!h || !h_out) return KVC_ERR_ARG;
    std::memcpy(h_out, h->np.data(), h->np.size() * 4);
    return KVC_OK;
}

int kvc_device_status(kvc_t h, kvc_stream_t stream, int32_t* h_status) {
    if (!h || !on_device(h) || !h_status) return KVC_ERR_ARG;
    cudaStream_t st = S_(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, h->state + h->L.hdr, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return KVC_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KVC_ERR_CUDA;
    if (word && cudaMemsetAsync(h->state + h->L.hdr, 0, 4, st) != cudaSuccess) return KVC_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KVC_ERR_CUDA;
    *h_status = (int32_t)word;
    return KVC_OK;
}

int kvc_check_wait_path(kvc_t h, kvc_stream_t stream) {
    if (!h || !on_device(h)) return KVC_ERR_ARG;
    wait_path_kernel<<<1, 32, 0, S_(stream)>>>(at<uint32_t>(h, h->L.hdr));
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

int kvc_prefix_cut(const int64_t* h_old_ids, int32_t n_old, const int64_t* h_new_ids, int32_t n_new,
                   int32_t ring, int32_t* h_cut) {
    if (!h_cut || n_new < 1 || n_old < 0 || !h_new_ids || (n_old > 0 && !h_old_ids)) return KVC_ERR_ARG;
    int32_t lcp = 0;
    const int32_t m = n_old < n_new ? n_old : n_new;
    while (lcp < m && h_old_ids[lcp] == h_new_ids[lcp]) ++lcp;
    int32_t cut = lcp;
    if (ring) cut = (lcp == n_old && n_new > n_old) ? n_old : 0;
    if (cut > n_new - 1) cut = n_new - 1;
    *h_cut = cut;
    return KVC_OK;
}

}  // extern "C"
