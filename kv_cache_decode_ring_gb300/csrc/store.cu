// store.cu -- prefix store ([PREFIX] "LLM 機制實驗（五）：改了歷史，能否只重算變化的後綴？",
// "查詢流程與快取所有權"): the host policy object that picks the stored prefill a
// query reuses and how many of its rows, and the device copies of one request's
// rows between the cache and a store slot of the state buffer.
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "kvc_internal.h"

struct kvc_pstore {
    struct Entry {
        bool used = false;
        uint64_t seq = 0;              // insertion order; larger = more recent
        std::vector<int64_t> ids;
        std::string scope;
        std::vector<uint8_t> sig;
    };
    int32_t ring = 0;
    uint64_t seq = 0;
    std::vector<Entry> e;
};

namespace kvc {
namespace {

// A CTA copies 128 rows of K and V (64 KB at d = 128, bf16); each thread has eight
// 16-byte units of K and eight of V in flight before it stores (two CTAs an SM by
// registers: 128 KB in flight an SM).  64 rows and four units a thread reached 0.87 of
// the copy bandwidth, this shape 0.96.
constexpr int kStoreRows = 128;        // cache rows per CTA of the copy kernel
constexpr int kStoreThreads = 256;
constexpr int kStoreUnroll = 8;        // row units a thread loads before it stores
constexpr int kStoreBatch = 64;        // requests per launch of a batched load

struct StoreItem {
    int slot;                          // store slot (-1: load of nothing)
    int b;                             // request
    int cut;                           // load: rows at positions below cut are kept
    int rows;                          // slots [0, rows) may hold a row to copy
};

struct StoreArgs {
    char* kc; char* vc;                // cache rows (unpaged runs or pages)
    const int32_t* table;              // paged caches: block table, else nullptr
    int32_t* pos;                      // cache positions [B][S]
    int32_t* next_pos;
    char* store;                       // store slot 0; slot i at store + i * stride
    size_t stride;                     // bytes per store slot: K [Hkv][S][d], V, positions [S]
    int Hkv, S, row_bytes;
    int ring;                          // ring layout: a slot's position is read, else it is the slot
    int load;                          // 1: store slot -> request; 0: request -> store slot
    int n;                             // items
    StoreItem item[kStoreBatch];
};

// grid (ceil(max rows / kStoreRows), Hkv + 1, items): plane y < Hkv copies KV head y's
// rows of item z, plane Hkv its positions (and, on a load, next_position).
// Save: every slot holding a row (position >= 0) goes to the store slot, with the
// positions array.  Load: the store slot's rows at positions [0, cut) come back;
// every other slot of the request is marked empty.
template <typename U>
__global__ void __launch_bounds__(kStoreThreads) store_copy_kernel(const StoreArgs a) {
    const StoreItem it = a.item[blockIdx.z];
    const int h = blockIdx.y;
    const size_t half = (size_t)a.Hkv * a.S * a.row_bytes;
    char* sbase = it.slot >= 0 ? a.store + (size_t)it.slot * a.stride : nullptr;
    const int32_t* spos = sbase ? reinterpret_cast<const int32_t*>(sbase + 2 * half) : nullptr;
    int32_t* pb = a.pos + (size_t)it.b * a.S;
    if (h == a.Hkv) {
        for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < a.S; s += gridDim.x * blockDim.x) {
            if (a.load) {
                const int p = spos ? spos[s] : -1;
                pb[s] = (p >= 0 && p < it.cut) ? p : -1;
            } else {
                reinterpret_cast<int32_t*>(sbase + 2 * half)[s] = pb[s];
            }
        }
        if (a.load && blockIdx.x == 0 && threadIdx.x == 0) a.next_pos[it.b] = it.cut;
        return;
    }
    if (!sbase) return;
    const int upr = a.row_bytes / (int)sizeof(U);        // units per row
    const int s0 = blockIdx.x * kStoreRows;
    if (s0 >= it.rows) return;
    const int nrows = it.rows - s0 < kStoreRows ? it.rows - s0 : kStoreRows;
    const int total = nrows * upr;
    const int32_t* held = a.load ? spos : pb;            // the side whose rows are read
    // K and V of a row sit at the same offset from their bases on either side
    const char* fk = a.load ? sbase : a.kc;              // copied from
    const char* fv = a.load ? sbase + half : a.vc;
    char* tk = a.load ? a.kc : sbase;                    // copied to
    char* tv = a.load ? a.vc : sbase + half;
    constexpr size_t kNone = ~(size_t)0;
    for (int base = threadIdx.x; base < total; base += kStoreUnroll * kStoreThreads) {
        U kx[kStoreUnroll], vx[kStoreUnroll];
        size_t to[kStoreUnroll];                          // byte offset of the unit's destination
#pragma unroll
        for (int j = 0; j < kStoreUnroll; ++j) {
            to[j] = kNone;
            const int i = base + j * kStoreThreads;
            if (i >= total) continue;
            const int s = s0 + i / upr, u = i % upr;
            // a contiguous cache holds position s in slot s for s below its length (rows):
            // its copies start without waiting for a position
            const int p = a.ring ? held[s] : s;
            if (p < 0 || (a.load && p >= it.cut)) continue;
            const size_t crow = kv_row(a.table, it.b, h, s, a.Hkv, a.S);
            const size_t srow = (size_t)h * a.S + s;
            const size_t co = crow * a.row_bytes + (size_t)u * sizeof(U), so = srow * a.row_bytes + (size_t)u * sizeof(U);
            const size_t from = a.load ? so : co;
            to[j] = a.load ? co : so;
            kx[j] = *reinterpret_cast<const U*>(fk + from);
            vx[j] = *reinterpret_cast<const U*>(fv + from);
        }
#pragma unroll
        for (int j = 0; j < kStoreUnroll; ++j)
            if (to[j] != kNone) {
                *reinterpret_cast<U*>(tk + to[j]) = kx[j];
                *reinterpret_cast<U*>(tv + to[j]) = vx[j];
            }
    }
}

cudaError_t launch_store_copy(const StoreArgs& a, cudaStream_t st) {
    int rows = 0;
    for (int i = 0; i < a.n; ++i) rows = a.item[i].rows > rows ? a.item[i].rows : rows;
    const int blocks = rows > 0 ? (rows + kStoreRows - 1) / kStoreRows : 1;
    dim3 grid(blocks, a.Hkv + 1, a.n);
    if (a.row_bytes % 16 == 0) store_copy_kernel<uint4><<<grid, kStoreThreads, 0, st>>>(a);
    else store_copy_kernel<uint32_t><<<grid, kStoreThreads, 0, st>>>(a);
    return cudaGetLastError();
}

StoreArgs store_args(kvc_handle* h, int load) {
    const Shape& s = h->sh;
    StoreArgs a{};
    a.kc = h->state + h->L.k; a.vc = h->state + h->L.v;
    a.table = s.pages ? reinterpret_cast<const int32_t*>(h->state + h->L.table) : nullptr;
    a.pos = reinterpret_cast<int32_t*>(h->state + h->L.pos);
    a.next_pos = reinterpret_cast<int32_t*>(h->state + h->L.next_pos);
    a.store = h->state + h->L.store;
    a.stride = h->L.store_stride;
    a.Hkv = s.Hkv; a.S = s.S; a.row_bytes = s.d * s.elem; a.ring = s.ring;
    a.load = load;
    return a;
}

bool valid_ids(const int64_t* ids, int32_t n) { return ids && n >= 1; }

bool valid_key(const char* scope, const void* sig, int32_t sig_bytes) {
    return scope && sig_bytes >= 0 && (sig_bytes == 0 || sig);
}

bool same_key(const kvc_pstore::Entry& e, const char* scope, const void* sig, int32_t sig_bytes) {
    return e.scope == scope && e.sig.size() == (size_t)sig_bytes &&
           (sig_bytes == 0 || std::memcmp(e.sig.data(), sig, sig_bytes) == 0);
}

}  // namespace
}  // namespace kvc

using namespace kvc;

extern "C" {

int kvc_pstore_create(const kvc_config* cfg, int32_t capacity, kvc_pstore_t* out) {
    if (!cfg || !out || capacity < 1) return KVC_ERR_ARG;
    Shape s;
    if (!make_shape(*cfg, &s)) return KVC_ERR_ARG;
    kvc_pstore* ps = new (std::nothrow) kvc_pstore();
    if (!ps) return KVC_ERR_ARG;
    ps->ring = s.ring;
    ps->e.resize(capacity);
    *out = ps;
    return KVC_OK;
}

int kvc_pstore_destroy(kvc_pstore_t ps) {
    if (!ps) return KVC_ERR_ARG;
    delete ps;
    return KVC_OK;
}

int kvc_pstore_insert(kvc_pstore_t ps, const int64_t* h_ids, int32_t n_ids, const char* scope,
                      const void* h_sig, int32_t sig_bytes, int32_t* h_slot) {
    if (!ps || !h_slot || !valid_ids(h_ids, n_ids) || !valid_key(scope, h_sig, sig_bytes)) return KVC_ERR_ARG;
    int slot = -1;
    for (size_t i = 0; i < ps->e.size() && slot < 0; ++i)
        if (!ps->e[i].used) slot = (int)i;
    if (slot < 0) {                                   // full: the oldest entry makes room
        slot = 0;
        for (size_t i = 1; i < ps->e.size(); ++i)
            if (ps->e[i].seq < ps->e[slot].seq) slot = (int)i;
    }
    kvc_pstore::Entry& e = ps->e[slot];
    e.used = true;
    e.seq = ++ps->seq;
    e.ids.assign(h_ids, h_ids + n_ids);
    e.scope = scope;
    e.sig.assign(static_cast<const uint8_t*>(h_sig), static_cast<const uint8_t*>(h_sig) + sig_bytes);
    *h_slot = slot;
    return KVC_OK;
}

int kvc_pstore_lookup(kvc_pstore_t ps, const int64_t* h_ids, int32_t n_ids, const char* scope,
                      const void* h_sig, int32_t sig_bytes, int32_t* h_slot, int32_t* h_cut) {
    if (!ps || !h_slot || !h_cut || !valid_ids(h_ids, n_ids) || !valid_key(scope, h_sig, sig_bytes))
        return KVC_ERR_ARG;
    int best = -1, best_cut = 0;
    uint64_t best_seq = 0;
    for (size_t i = 0; i < ps->e.size(); ++i) {
        const kvc_pstore::Entry& e = ps->e[i];
        if (!e.used || !same_key(e, scope, h_sig, sig_bytes)) continue;
        int32_t cut = 0;
        kvc_prefix_cut(e.ids.data(), (int32_t)e.ids.size(), h_ids, n_ids, ps->ring, &cut);
        if (cut > best_cut || (cut == best_cut && cut > 0 && e.seq > best_seq)) {
            best = (int)i; best_cut = cut; best_seq = e.seq;
        }
    }
    *h_slot = best;
    *h_cut = best_cut;
    return KVC_OK;
}

int kvc_store_save(kvc_t h, int32_t slot, int32_t b, int32_t n, kvc_stream_t stream) {
    if (!h || !on_device(h)) return KVC_ERR_ARG;
    const Shape& s = h->sh;
    if (s.store_slots == 0) return KVC_ERR_UNSUPPORTED;
    if (slot < 0 || slot >= s.store_slots || b < 0 || b >= s.B || n < 1 || n != h->np[b]) return KVC_ERR_ARG;
    StoreArgs a = store_args(h, 0);
    a.n = 1;
    a.item[0] = StoreItem{slot, b, 0, s.ring ? s.S : n};
    if (launch_store_copy(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ERR_CUDA;
    h->store_n[slot] = n;
    return KVC_OK;
}

int kvc_store_load_batch(kvc_t h, int32_t n, const int32_t* h_slots, const int32_t* h_b, const int32_t* h_cuts,
                         kvc_stream_t stream) {
    if (!h || !on_device(h) || n < 0) return KVC_ERR_ARG;
    const Shape& s = h->sh;
    if (s.store_slots == 0) return KVC_ERR_UNSUPPORTED;
    if (n == 0) return KVC_OK;
    if (!h_slots || !h_b || !h_cuts) return KVC_ERR_ARG;
    // every item is checked before anything changes
    std::vector<char> seen(s.B, 0);
    for (int i = 0; i < n; ++i) {
        const int slot = h_slots[i], b = h_b[i], cut = h_cuts[i];
        if (b < 0 || b >= s.B || seen[b] || slot < -1 || slot >= s.store_slots) return KVC_ERR_ARG;
        seen[b] = 1;
        const int len = slot < 0 ? 0 : h->store_n[slot];
        if (len < 0 || cut < 0 || cut > len) return KVC_ERR_ARG;
        if (s.ring && cut > 0) {
            // the token at `cut` attends to [cut - S + 1, cut); the slot holds [len - S, len)
            const int lo = cut - s.S + 1 > 0 ? cut - s.S + 1 : 0;
            const int resident = len - s.S > 0 ? len - s.S : 0;
            if (lo < resident) return KVC_ERR_EVICTED;
        }
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (s.pages) {
        // the requests give back all their pages and map those that the kept rows need
        const int npg = s.S / kPage;
        std::vector<int> from(h->np.begin(), h->np.end()), to(from);
        long long need = 0, held = 0;
        for (int i = 0; i < n; ++i) {
            const int b = h_b[i], len = h_slots[i] < 0 ? 0 : h->store_n[h_slots[i]];
            const long long lo = s.ring && len > s.S ? len - s.S : 0;
            from[b] = (int)lo; to[b] = h_cuts[i];
            for (int lp = 0; lp < npg; ++lp) {
                need += page_touched(s, lp, lo, h_cuts[i]) ? 1 : 0;
                held += h->table_h[(size_t)b * npg + lp] >= 0 ? 1 : 0;
            }
        }
        if (need > held + (long long)h->page_free.size()) return KVC_ERR_CAPACITY;
        for (int i = 0; i < n; ++i)
            for (int lp = 0; lp < npg; ++lp) {
                int32_t& e = h->table_h[(size_t)h_b[i] * npg + lp];
                if (e >= 0) { h->page_free.push_back(e); e = -1; }
            }
        int rc = KVC_OK;
        if (map_pages(h, from, to, st, &rc) != cudaSuccess) return KVC_ERR_CUDA;
        if (rc) return rc;               // not reached: the count above guarantees the pages
        if (cudaMemcpyAsync(h->state + h->L.table, h->table_h.data(), h->table_h.size() * 4,
                            cudaMemcpyHostToDevice, st) != cudaSuccess)
            return KVC_ERR_CUDA;
    }
    for (int i0 = 0; i0 < n; i0 += kStoreBatch) {
        StoreArgs a = store_args(h, 1);
        a.n = n - i0 < kStoreBatch ? n - i0 : kStoreBatch;
        for (int j = 0; j < a.n; ++j) {
            const int slot = h_slots[i0 + j], cut = h_cuts[i0 + j];
            a.item[j] = StoreItem{slot, h_b[i0 + j], cut, slot < 0 ? 0 : (s.ring ? s.S : cut)};
        }
        if (launch_store_copy(a, st) != cudaSuccess) return KVC_ERR_CUDA;
    }
    for (int i = 0; i < n; ++i) h->np[h_b[i]] = h_cuts[i];
    if (s.ring) h->ring_needs_append = true;
    return KVC_OK;
}

int kvc_store_load(kvc_t h, int32_t slot, int32_t b, int32_t cut, kvc_stream_t stream) {
    return kvc_store_load_batch(h, 1, &slot, &b, &cut, stream);
}

}  // extern "C"
