// kvc_internal.h -- state layout, handle, kernel argument blocks and device
// helpers shared by the libkvc translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <vector>

#include "../../include/kvc.h"

namespace kvc {

constexpr int kQBlock = 16;           // tokens per INT8 quantization block
constexpr int kPage = 16;             // slots per page of a paged cache
constexpr int kBands = 16;            // witness bands per key row
constexpr int kGenericSplit = 64;     // keys per split, generic decode kernel
constexpr size_t kMaxSmemPerBlock = 232448;   // dynamic shared memory a block may be granted (227 KB)
constexpr int kFastSplit = 128;       // keys per split, bf16 fast decode kernel
constexpr int kInt8Split = 1024;      // keys per quantized split, INT8 decode kernel ...
constexpr int kInt8SplitLong = 2048;  // ... and for caches of kInt8LongKeys slots or more
constexpr int kInt8LongKeys = 16384;
// keys per split of the bf16 decode kernel for 4 or 8 heads per KV head: longer splits
// when a request may attend to many keys (less per-CTA start-up per byte), shorter ones
// otherwise (enough CTAs to fill the GPU)
constexpr int kGqaSplit = 1024;
constexpr int kGqaSplitLong = 2048;
constexpr int kGqaLongKeys = 16384;
constexpr int kMaxRestored = 1024;    // INT8 blocks restored to full precision per (request, KV head)
constexpr int kExactBlocksPerCta = 64; // restored blocks one CTA of the exact-block decode serves
constexpr int kExactSplits = kMaxRestored / kExactBlocksPerCta;   // their split slots per query head
constexpr uint32_t kErrPosition = 1u; // device error bits (sticky, cleared by kvc_device_status)
constexpr uint32_t kErrWait = 2u;
constexpr uint32_t kErrRange = 4u;    // a chunk-attention operand beyond the fp16 range

// Byte offsets of the arrays inside the caller's state buffer (256-B aligned).
struct Layout {
    size_t hdr;       // uint32[64]: [0] error word, [1] work counter, [2] done counter
    size_t next_pos;  // int32 [B]
    size_t pos;       // int32 [B][S]
    size_t k, v;      // [B][Hkv][S][d] cache dtype (non-INT8); paged: [pages][Hkv][16][d]
    size_t table;     // int32 [B][S/16] physical page of each logical page, -1 = none (paged)
    size_t kq, vq;    // int8 [B][Hkv][S][d]                   (INT8)
    size_t sk, sv;    // f32  [B][Hkv][S/16]                   (INT8)
    size_t wit;       // f16  [B][Hkv][S][16]                  (INT8)
    size_t ktail, vtail;  // bf16 [B][Hkv][16][d]              (INT8)
    size_t xmap;      // int32 [B][Hkv][S/16] pool entry of a restored block, -1 = quantized (INT8)
    size_t xn;        // int32 [B][Hkv] restored blocks per (request, KV head)        (INT8)
    size_t xlist;     // int32 [B][Hkv][kMaxRestored] their block indices, then      (INT8)
    size_t xent;      // int32 [B][Hkv][kMaxRestored] their pool entries              (INT8)
    size_t xpool;     // bf16 [pool][2][16 d] K and V rows, xk_offset / xv_offset     (INT8)
    size_t rope;      // float2 [P][d/2] {cos, sin}
    size_t part_ml;   // float2 [B][Hq][max_splits] {m (log2 domain), l}
    size_t part_acc;  // float  [B][Hq][max_splits][d]
    size_t part_c;    // float  [B][Hq][max_splits] max_t c_t of the split   (INT8)
    size_t req_id;    // uint32 [B] request IDs of the dither counters (Tier B)
    size_t arrive;    // int32 [B] CTAs of a one-token append done (0 between calls)
    size_t cws;       // ring caches with kvc_chunk_attn: K then V staging [B][Hkv][chunk_ws_rows][d] bf16
    size_t store;     // store slots: each K, V [Hkv][S][d] cache dtype, then positions int32 [S]
    size_t store_stride;  // bytes per store slot
    size_t total;
};

struct Shape {
    int B, Hq, Hkv, g, d, S, W;  // W = attention window in positions (0 = full)
    int P;                       // RoPE table rows (0 = no RoPE)
    int elem;                    // bytes per cache element (non-INT8)
    bool ring, int8, rope, bf16;
    bool dither;                 // INT8 Tier B: subtractive dither, no witnesses
    bool out_bf16;               // attention outputs in bf16 (else fp32)
    int split;                   // keys per split of the decode kernel in use
    int max_splits;
    int max_chunk;               // largest suffix of kvc_chunk_attn (0 = none)
    int xpool;                   // entries of the INT8 exact-block pool
    int pages;                   // pages of a paged cache (0 = not paged)
    bool gqa;                    // the bf16 GQA decode kernel serves the shape
    int store_slots;             // saved-prefill slots (0 = none)
};

// INT8 decode: the slots its quantized splits cover.  A window of W positions on a
// contiguous cache touches at most W/16 + 2 blocks; a ring or an unwindowed cache, all S.
inline long long int8_qkeys(const Shape& s) {
    return (!s.ring && s.W > 0 && (long long)s.W + 2 * kQBlock < s.S) ? (long long)s.W + 2 * kQBlock : s.S;
}
// ... and the columns of its grid: the quantized splits of `split` tokens, then the exact-tail split
inline int int8_grid(const Shape& s) {
    const long long bps = s.split / kQBlock;
    return (int)(((int8_qkeys(s) + kQBlock - 1) / kQBlock + bps - 1) / bps) + 1;
}

bool make_shape(const kvc_config& c, Shape* s);
// Rows per (request, KV head) of a ring's chunk staging: positions from the cut rounded
// down to 16 up to the last suffix row rounded up to 16.
inline int chunk_ws_rows(const Shape& s) { return ((s.max_chunk + 15) & ~15) + 32; }
Layout make_layout(const Shape& s);

// Arguments of the decode kernels (everything by value; no host pointers).
struct DecodeArgs {
    const void* q;        // [B][Hq][d] cache dtype
    const void* k;        // cache rows (non-INT8)
    const void* v;
    const int32_t* next_pos;
    const float2* rope;   // nullptr = no RoPE
    float2* part_ml;
    float* part_acc;
    uint32_t* hdr;
    const int32_t* table; // paged caches: the block table (else nullptr)
    int B, Hq, Hkv, g, d, S, W, max_splits, split;
    int gqa;              // the GQA decode kernel serves the shape (split kGqaSplit or kGqaSplitLong)
    int ring;
    int bf16;             // cache dtype (1 = bf16, 0 = fp32)
    float scale_log2;     // log2(e) / sqrt(d)
};

struct CombineArgs {
    const float2* part_ml;
    const float* part_acc;
    const int32_t* next_pos;
    void* out;            // [B][Hq][d] cache dtype
    int B, Hq, d, S, W, max_splits, split, ring, bf16;
    int align_lo;         // splits start at the window start rounded down to a page
};

struct AppendArgs {
    const void* k;        // row r of KV head h of request b at b*sb + h*sh + r*sr
    const void* v;
    int n;                // rows in the input per request
    size_t sb, sh, sr;    // element strides of the input (row elements are contiguous)
    int32_t* next_pos;
    int32_t* pos;
    void* kc;             // cache rows (non-INT8)
    void* vc;
    int8_t* kq; int8_t* vq; float* sk; float* sv; __half* wit;
    __nv_bfloat16* ktail; __nv_bfloat16* vtail;
    const float2* rope;
    uint32_t* hdr;
    const int32_t* table; // paged caches: the block table (else nullptr)
    const uint32_t* req_id;   // Tier B: request IDs
    uint32_t key0, key1;      // Tier B: Philox key
    uint32_t layer_ctr;       // Tier B: 65536 * layer
    int B, Hkv, d, S, P, ring, bf16, int8, dither;
    int32_t* arrive;          // [B] one-token append: CTAs of the request done (0 between calls)
    int hpc;                  // one-token append: KV heads per CTA
};

// Tensor maps over the whole K and V caches, rows [B*Hkv*S][d] bf16, boxes of 64
// elements x 16 rows, 128-byte swizzle (the GQA decode's tiles).
struct KvMaps {
    CUtensorMap k, v;
};

// bf16 tensor map with 128-byte swizzle (cuTensorMapEncodeTiled); false on failure
bool make_tensor_map_bf16(CUtensorMap* tm, void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                          const cuuint32_t* box);

// ---- launchers (one per translation unit) ----------------------------------
cudaError_t launch_append_token(const AppendArgs& a, cudaStream_t st);
// INT8 gated fallback (int8_gate.cu): drop restored blocks that a trim removed
cudaError_t int8_drop_restored(kvc_handle* h, const int32_t* h_cut, cudaStream_t st);
// paged caches (append.cu): map the pages that slots [from, to) of each request need
cudaError_t map_pages(kvc_handle* h, const std::vector<int>& from, const std::vector<int>& to, cudaStream_t st,
                      int* status);
cudaError_t launch_trim_cuts(int32_t* next_pos, int32_t* pos, const int32_t* cuts, int B, int S, int ring,
                             cudaStream_t st);

// Whether logical page lp holds a slot of positions [lo, hi) (slot = position on a
// contiguous cache, position mod S on a ring of S slots).
inline bool page_touched(const Shape& s, int lp, long long lo, long long hi) {
    if (hi <= lo) return false;
    const long long p0 = (long long)lp * kPage, p1 = p0 + kPage - 1;
    if (!s.ring) return p0 < hi && p1 >= lo;
    if (hi - lo >= s.S) return true;
    const long long a0 = lo % s.S, a1 = (hi - 1) % s.S;     // possibly wrapping
    return a0 <= a1 ? (p0 <= a1 && p1 >= a0) : (p1 >= a0 || p0 <= a1);
}
// INT8 exact-block decode (int8_exact.cu): the restored blocks' splits
cudaError_t launch_int8_exact(kvc_handle* h, const void* q, float* ct, cudaStream_t st);
// maps: required when the GQA kernel serves the shape (Shape::gqa)
cudaError_t launch_decode(const DecodeArgs& d, const CombineArgs& c, bool fast, const KvMaps* maps, cudaStream_t st);
bool chunk_supported(const Shape& s);
bool gqa_decode_supported(int d, int g);
cudaError_t launch_decode_gqa(const DecodeArgs& a, const KvMaps& maps, cudaStream_t st);
// Chunked suffix attention (chunk.cu).  A contiguous cache has already appended the n
// suffix rows; a ring first stages them (rotated) next to its resident rows and
// appends them after the attention (the caller does).
cudaError_t launch_chunk(kvc_handle* h, const void* q, const void* k, const void* v, void* out, int n,
                         cudaStream_t st);

// ---- INT8 code storage --------------------------------------------------------
// Inside one 16-token block of one (request, KV head) the 16*d code bytes are
// stored biased, u = c + 128 (bit pattern c ^ 0x80), so that the decode turns a
// byte into the fp16 value 1024 + u with one byte permute.  Byte offsets of code
// (token t of the block, dim x), for d in {64, 128}:
//  K: token-major rows of d bytes; at d = 128 the 16-byte chunks of odd rows are
//     swapped pairwise (chunk c at c ^ 1), so that the decode's 16-byte row loads
//     hit every bank group once.
//  V: ordered for the decode's P.V operand fragments: lane L = 4 (x mod 8) + t/4
//     owns a d/2-byte run holding word f = x/8 (tokens 4 (t/4) .. +3 of dim x),
//     its 16-byte chunks XOR-swizzled by lane so that 8 lanes' loads hit 8 groups.
__host__ __device__ __forceinline__ int kq_offset(int d, int t, int x) {
    const int sw = d == 128 ? (t & 1) : 0;
    return t * d + (((x >> 4) ^ sw) << 4) + (x & 15);
}
__host__ __device__ __forceinline__ int vq_offset(int d, int t, int x) {
    const int lane = 4 * (x & 7) + (t >> 2), f = x >> 3;
    const int cpr = d / 32;                          // 16-byte chunks per lane run
    const int swz = (lane / (8 / cpr)) % cpr;
    return lane * (d / 2) + (((f >> 2) ^ swz) << 4) + ((f & 3) << 2) + (t & 3);
}

// Restored (exact) blocks live in the pool as bf16 in the order of the exact-block
// decode's MMA operand fragments; byte offsets inside the K half and the V half of a
// pool entry for (token t of the block, dim x), d in {64, 128}:
//  K: rows of 2d bytes; the 16-byte chunk c (8 dims) of row t sits at c ^ s, with
//     s = 2 (c / 8) + (t mod 2) at d = 128 and s = t mod 2 at d = 64;
//  V: lane L = 4 (x mod 8) + t/4 owns d/16 chunks of 16 bytes, one per group of 16
//     dims (x/16), XOR-swizzled by lane; inside a chunk the words are (dim 16i + L/4:
//     tokens 4 (L mod 4) + 0,1), (... + 2,3), (dim 16i + 8 + L/4: + 0,1), (... + 2,3).
__host__ __device__ __forceinline__ int xk_offset(int d, int t, int x) {
    const int c = x >> 3;
    const int s = d == 128 ? (((c >> 3) << 1) | (t & 1)) : (t & 1);
    return t * 2 * d + ((c ^ s) << 4) + (x & 7) * 2;
}
__host__ __device__ __forceinline__ int xv_offset(int d, int t, int x) {
    const int lane = 4 * (x & 7) + (t >> 2), i = x >> 4, j = (x >> 3) & 1, q = t & 3;
    const int swz = d == 128 ? (lane & 7) : ((lane >> 1) & 3);
    return lane * (d / 16) * 16 + ((i ^ swz) << 4) + (j * 2 + (q >> 1)) * 4 + (q & 1) * 2;
}

// ---- device helpers -----------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
// 1, 2, 3", SC 2011): ten rounds of two 32x32 -> 64-bit products of counter words 0
// and 2, recombined with words 1 and 3 and the key by xor; the key is bumped by the
// Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Programmatic dependent launch.  A kernel started by launch_dep may be scheduled while
// the previous kernel in the stream is still running; it calls dep_wait() before it reads
// or writes any global memory, and that returns once the previous kernel has completed
// with its writes visible, so stream order holds.  dep_release() lets the next such
// kernel be scheduled early (it still waits for this one to complete).  Both are no-ops
// in a kernel launched the ordinary way.
__device__ __forceinline__ void dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void dep_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Grants `kernel` `bytes` of dynamic shared memory on the current device, once per
// (kernel, device, size) and calling thread (kvc_api.cu).  Kernels above 48 KB need it;
// each kernel always asks for the same size, so no grant ever narrows another.
cudaError_t allow_smem(const void* kernel, size_t bytes);

template <typename... Params, typename... Args>
inline cudaError_t launch_dep(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__device__ __forceinline__ float ld_elem(const void* p, size_t i, int bf16) {
    return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i])
                : static_cast<const float*>(p)[i];
}

// RoPE on one interleaved pair, fp32, each product and the sum rounded once:
//   y0 = x0*c - x1*s,  y1 = x1*c + x0*s.
__device__ __forceinline__ void rope_pair(float x0, float x1, float2 cs, float& y0, float& y1) {
    y0 = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y));
    y1 = __fadd_rn(__fmul_rn(x1, cs.x), __fmul_rn(x0, cs.y));
}

// Row (in rows of d elements) holding slot `slot` of (request b, KV head h): a
// request's own run of S rows, or row slot % 16 of the head's part of its page.
__device__ __forceinline__ size_t kv_row(const int32_t* table, int b, int h, int slot, int Hkv, int S) {
    if (!table) return ((size_t)b * Hkv + h) * S + slot;
    int page = table[(size_t)b * (S / kPage) + slot / kPage];
    page = page < 0 ? 0 : page;       // never taken: every slot read or written is mapped first
    return ((size_t)page * Hkv + h) * kPage + (slot % kPage);
}

// INT8 tier: the complete 16-position blocks that the newest token of a request (at
// len - 1) attends to.  A contiguous cache stores block n in block slot n; a ring of S
// slots (S a multiple of 16) stores block n in block slot n mod (S/16), so a slot
// holds the newest complete block congruent to it.  Physical block slots [blo, bhi)
// hold the blocks read; positions below `lo` (the window start) are masked, which can
// only cut into the first of them.  The rows [nfull, len) of the incomplete block live
// in the exact tail.
struct Int8Window {
    int blo, bhi;      // physical block slots read
    int lo;            // first visible position
    int nfb;           // complete blocks written so far (absolute count)
    int nbk;           // block slots of the cache
};
__host__ __device__ __forceinline__ Int8Window int8_window(int len, int S, int W, int ring) {
    Int8Window w;
    w.nfb = len / kQBlock;
    w.nbk = S / kQBlock;
    w.lo = (W > 0 && len > W) ? len - W : 0;
    if (ring) { w.blo = 0; w.bhi = w.nfb < w.nbk ? w.nfb : w.nbk; }
    else { w.blo = w.lo / kQBlock; w.bhi = w.nfb; }
    if (w.bhi < w.blo) w.bhi = w.blo;
    return w;
}
// Linear index of the quantization block in block slot k of (request b, KV head h):
// blocks [B][Hkv][S/16], or, on a paged cache (a 16-slot page is one block), the
// page the block table maps times Hkv plus h.  Codes sit at 16 d bytes per block,
// witnesses at 16 x 16 halves, scales at one float.
__host__ __device__ __forceinline__ size_t int8_block(const int32_t* table, int b, int h, int k, int Hkv, int S) {
    if (!table) return ((size_t)b * Hkv + h) * (S / kQBlock) + k;
    int page = table[(size_t)b * (S / kQBlock) + k];
    page = page < 0 ? 0 : page;       // never taken: every block read or written is mapped first
    return (size_t)page * Hkv + h;
}

// Absolute block number held by physical block slot k.
__host__ __device__ __forceinline__ int int8_abs_block(const Int8Window& w, int k, int ring) {
    if (!ring || w.nfb <= w.nbk) return k;
    return (w.nfb - 1) - ((w.nfb - 1 - k) % w.nbk);
}

// Cached key slots of request b attended by its newest token (next_position - 1):
// a ring holds the window in slots [0, min(len, W)); a contiguous cache in
// slots [len - min(len, W), len).
__device__ __forceinline__ void key_range(int len, int S, int W, int ring, int& lo, int& hi) {
    if (ring) { lo = 0; hi = len < S ? len : S; }
    else { hi = len; lo = (W > 0 && len > W) ? len - W : 0; }
}

}  // namespace kvc

// Opaque handle behind kvc_t.
struct kvc_handle {
    kvc_config cfg;
    kvc::Shape sh;
    kvc::Layout L;
    char* state;
    size_t bytes;
    int device;
    int num_sms;
    std::vector<int32_t> np;      // host mirror of next_position
    bool ring_needs_append;        // a ring was trimmed and has not appended since
    std::vector<int32_t> counts;   // host staging for append_rows counts
    kvc::KvMaps kv_maps;           // built at create when the GQA decode serves the shape
    bool has_kv_maps;
    // INT8 gated fallback: host mirrors of the block map and the per-head counts, and
    // the free pool entries
    std::vector<int32_t> xmap_h, xn_h, xfree;
    std::vector<int32_t> xlist_h, xent_h;   // mirrors of the per-head lists
    // paged caches: host mirror of the block table and the free pages
    std::vector<int32_t> table_h, page_free;
    // prefix store: rows saved in each store slot (-1 = empty)
    std::vector<int32_t> store_n;
    // Tier B: host mirror of the request IDs
    std::vector<uint32_t> req_id_h;
};

// Calls that enqueue device work run with the handle's device current (its buffers live
// there); anything else is refused with KVC_ERR_ARG rather than launched elsewhere.
inline bool on_device(const kvc_handle* h) {
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess && dev == h->device;
}
