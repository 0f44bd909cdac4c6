// chunk.cu -- chunked causal (or sliding-window) suffix attention on tcgen05.
//
// [PREFIX] "哪些東西必須一起裁剪": after the cache is trimmed to `cut`, the
// suffix tokens[cut:] are computed in one chunk from next_position = cut:
// suffix query i sits at position p = cut + i and attends to cached positions
// [max(0, p - W + 1), p] (W = 0: all), exactly what a one-token decode at p
// would see ([LEAN] §2.1 masks).  On a contiguous cache the suffix K/V rows are
// appended first, so every key a query needs is in the cache.  A ring of W slots
// would evict, while appending, rows that the early suffix queries still need
// ([LEAN] §3.4): there the suffix rows are staged, rotated, in a workspace that
// also holds the resident rows from the cut rounded down to 16, the queries read
// positions below that from the ring and the rest from the workspace, and the
// suffix is appended to the ring afterwards.
//
// This is a dense contraction, so it runs on the 5th-generation tensor cores.
//  * CTA = 128 query rows of two query heads that share one KV head (two "slots";
//    the second is idle when the group has an odd number of heads).  Both slots
//    read the same K and V tiles of 128 keys, walked backwards from the diagonal.
//  * 16 warps: warps 0-3 and 4-7 run the softmax of slot 0 and slot 1 (thread =
//    query row = tensor-memory lane); warps 8-11, 14 and 15 convert K and V tiles from
//    bf16 to fp16 in shared memory; warp 12 issues the tensor copies; one thread of
//    warp 13 issues every tcgen05.mma.  Register shares: 184 for the softmax warps, 72 for
//    the others (setmaxnreg).
//  * Tensor memory (512 columns): S of slot 0 and slot 1 in [0, 128) and
//    [128, 256), fp32; the softmax writes P as fp16 pairs over the first 64 columns
//    of its S buffer (the A operand of P.V); O of slot 0 and 1 in [256, 384) and
//    [384, 512).  Q of both slots sits in shared memory (A operand of S = Q K^T).
//  * Operands are fp16 on both products: the rotated query times log2(e)/sqrt(d)
//    (relative error 2^-11), the softmax weights (<= 2^8), and the K and V rows,
//    which are exact in fp16 for magnitudes in [2^-14, 65504] (smaller ones lose
//    relative precision, at most 2^-25 absolute).  A query, key or value of
//    magnitude 65520 or more would overflow: the kernel flags the device error word
//    (kErrRange) and the call's output is not valid.
//  * Rows of a tile outside the keys the CTA attends to (before the earliest
//    window start, past the last suffix row, or before position 0) are zeroed by
//    the converters, so a masked weight of 0 never meets a non-finite value.
//  * Pipeline per slot: S(j) -> softmax(j) -> P.V(j) -> S(j+1) (S(j+1) overwrites
//    the columns P.V(j) reads, so it waits for P.V(j) to complete); the two slots
//    interleave on the tensor pipe, so one slot's MMAs run while the other's
//    softmax works.
//  * A row's reference maximum moves only when a tile exceeds it by more than 2^8
//    (log2 domain), so weights stay <= 2^8 and O is rarely rescaled (by the
//    softmax thread itself: at that point no P.V of its slot is in flight).
//  * Key tiles start on 16-key boundaries.  A contiguous cache is read with two
//    128-row tensor copies per tile; paged caches and rings with one 16-row copy per
//    16 positions and half (from the page the block table gives, the ring slot, or
//    the staging rows), skipping positions before 0.
//  * CTAs are taken longest first (a host-sorted table of (request, query tile)
//    items in the kernel parameters), the head pairs of one KV head adjacent so
//    that they read its tiles from L2.
// Every mbarrier wait is bounded; on expiry the kernel flags the device error
// word, skips the remaining work, waits (bounded) for its copies and MMAs in
// flight and still frees its tensor memory.  tcgen05.ld/st are warp-collective:
// every lane of a warp issues them.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <utility>
#include <vector>

#include "async_copy.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kBM = 128;            // query rows per slot
constexpr int kBN = 128;            // keys per tile
constexpr int kD = 128;             // head dim of this kernel
constexpr int kSlots = 2;           // query heads per CTA (sharing a KV head)
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;
constexpr int kThreads = 16 * 32;
constexpr int kConvWarps = 6;       // warps 8-11, 14 and 15
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr float kLazyMax = 8.f;     // log2-domain headroom of a row's reference maximum
constexpr int kTileB = kBN * kD * 2;     // 32 KB: two 64-dim halves of [128 rows][128 B]
constexpr int kHalfB = kTileB / 2;
constexpr int kGroupB = 16 * 128;        // 16 rows of one half
constexpr int kRegSoftmax = 184, kRegOther = 72;
static_assert(4 * 32 * (2 * kRegSoftmax + 2 * kRegOther) == 65536, "register split sums to the launch's registers");

constexpr int OFF_Q = 0;                               // Q of the two slots (fp16, 128-byte swizzle)
constexpr int OFF_K = OFF_Q + kSlots * kTileB;         // K stages
constexpr int OFF_V = OFF_K + kKStages * kTileB;       // V stages
constexpr int OFF_BAR = OFF_V + kVStages * kTileB;
enum {
    B_KFULL = 0,                        // [stage] K copied
    B_KCONV = B_KFULL + kKStages,       // [stage] K converted (every converter warp)
    B_KFREE = B_KCONV + kKStages,       // [stage] both S MMAs of the tile complete
    B_VFULL = B_KFREE + kKStages,
    B_VCONV = B_VFULL + kVStages,
    B_VFREE = B_VCONV + kVStages,       // [stage] both P.V MMAs of the tile complete
    B_SFULL = B_VFREE + kVStages,       // [slot] S complete
    B_PFULL = B_SFULL + kSlots,         // [slot] P written (4 softmax warps)
    B_ODONE = B_PFULL + kSlots,         // [slot] P.V complete
    B_QREADY = B_ODONE + kSlots,        // Q of both slots in shared memory (8 softmax warps)
    B_DONE = B_QREADY + 1,              // every MMA issued so far complete (abort path)
    kBars = B_DONE + 1
};
constexpr int OFF_MISC = OFF_BAR + 8 * kBars;          // tensor memory base, abort flag
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;       // + alignment slack of the dynamic base
static_assert(SMEM_BYTES <= 232448, "shared memory per block");
constexpr int kMaxItems = 2048;                        // (request, query tile) items in the order table
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kF16Limit = 65520.f;                   // rounds to infinity in fp16

struct ChunkArgs {
    const int32_t* next_pos;   // after the append: cut + n
    const __nv_bfloat16* q;    // [B][n][Hq][d], not rotated
    const float2* rope;        // nullptr = no RoPE
    void* out;                 // [B][n][Hq][d]
    uint32_t* hdr;
    const int32_t* table;      // paged caches: block table [B][S/16] (else nullptr)
    int B, Hq, Hkv, g, S, W, n, out_bf16;
    int ring;                  // keys below the cut (rounded down to 16) from the ring, the rest staged
    int n_appended;            // suffix rows next_position already counts (contiguous: n; ring: 0)
    int ws_rows;               // staging rows per (request, KV head) (ring)
    int tiles;                 // query tiles per request
    int pairs;                 // head pairs per KV head, ceil(g / 2)
    float scale_log2;
    int n_items;               // 0: natural order; else items[] = (request << 16 | tile), longest first
    uint32_t items[kMaxItems];
};

// ---- tcgen05 wrappers -------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle, sm_100 format:
// start address >> 4 (bits 0-13), leading-dimension byte offset >> 4 (16-29),
// stride-dimension byte offset >> 4 (32-45), version 1 (46-47), layout 2 =
// SWIZZLE_128B (61-63).  K-major operands: 8-row groups 1024 B apart (SBO).
// MN-major operands additionally step `lbo` bytes to the next 64 MN elements.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(1024u >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16 with A and B fp16 (format 0 in bits 7-9 and
// 10-12) and D fp32 (bit 4); B MN-major when b_mn (bit 16), N >> 3 (bits 17-22),
// M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t instr_desc_f16(int M, int N, bool b_mn) {
    return (1u << 4) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (tensor memory) (+)= A (shared memory descriptor) . B (shared memory descriptor)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, int acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// D (tensor memory) (+)= A (tensor memory, 16-bit pairs along columns, row m in
// lane m) . B (shared memory descriptor)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, int acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive 32-bit columns of this thread's tensor-memory lane (no wait)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// the same, into fp32 registers
__device__ __forceinline__ void tmem_ld32f(uint32_t taddr, float* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]),
          "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15]),
          "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]),
          "=f"(v[24]), "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
          "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
          "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
          "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x with the hardware approximation (relative error about 2^-22; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// two fp32 values rounded to fp16 (nearest even), a in the low half
__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
    __half2 t = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
}

// Non-blocking check that phase `parity` of an mbarrier has completed.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait (about one second) that polls without suspending: for the single
// thread that issues the MMAs, whose reaction time is on every tile's critical path.
__device__ __forceinline__ bool mbar_spin(uint64_t* bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (mbar_test(bar, parity)) return true;
        if ((it & 1023u) == 1023u && global_ns() - t0 > 1000000000ull) break;
    }
    return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}


// Convert one stage (a K or V tile) from bf16 to fp16 in place.  The kConvThreads
// converter threads take 16-byte chunks t, t + kConvThreads, ..., four at a time (all
// loads first); a chunk's row is its key (chunk q: half q / 1024, row (q mod 1024) / 8).
// Rows whose key lies outside [klo, khi] are zeroed.  `hmax` keeps the largest fp16
// magnitude written (infinity once a value overflowed).
__device__ __forceinline__ void convert_tile(unsigned char* tile, int t, int kb, int klo, int khi, __half2& hmax) {
    constexpr int kChunks = kTileB / 16;
    const bool all_valid = kb >= klo && kb + kBN - 1 <= khi;
#pragma unroll 1
    for (int q0 = t; q0 < kChunks; q0 += 4 * kConvThreads) {
        uint4 u[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int q = q0 + e * kConvThreads;
            if (q < kChunks) u[e] = *reinterpret_cast<const uint4*>(tile + 16 * q);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int q = q0 + e * kConvThreads;
            if (q >= kChunks) continue;
            const int key = kb + ((q & 1023) >> 3);
            uint4 o = make_uint4(0u, 0u, 0u, 0u);
            if (all_valid || (key >= klo && key <= khi)) {
                uint32_t w[4] = {u[e].x, u[e].y, u[e].z, u[e].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    w[k] = pack_f16(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
                    hmax = __hmax2(hmax, __habs2(*reinterpret_cast<const __half2*>(&w[k])));
                }
                o = make_uint4(w[0], w[1], w[2], w[3]);
            }
            *reinterpret_cast<uint4*>(tile + 16 * q) = o;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    chunk_attn_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmWK, const __grid_constant__ CUtensorMap tmWV,
                      const __grid_constant__ ChunkArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* sQ = smem + OFF_Q;
    unsigned char* sK = smem + OFF_K;
    unsigned char* sV = smem + OFF_V;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA's (request, query tile) item and head pair
    const int per_item = a.Hkv * a.pairs;
    const int item = blockIdx.x / per_item, hp = blockIdx.x % per_item;
    const int kvh = hp / a.pairs, pi = hp % a.pairs;
    const int nslots = (2 * pi + 1 < a.g) ? 2 : 1;
    int b, tile;
    if (a.n_items > 0) { b = (int)(a.items[item] >> 16); tile = (int)(a.items[item] & 0xFFFFu); }
    else { b = item / a.tiles; tile = item % a.tiles; }
    const int i0 = tile * kBM;
    const int np = a.next_pos[b];
    const int cut = np - a.n_appended;
    const int rows = min(kBM, a.n - i0);
    const int p_first = cut + i0, p_last = cut + i0 + rows - 1;
    // keys the CTA attends to: [kmin, p_last]; tiles end at kt (16-aligned) and walk back
    const int kmin = a.W > 0 ? max(0, p_first - a.W + 1) : 0;
    const int key_lo_max = a.W > 0 ? max(0, p_last - a.W + 1) : 0;
    const int kt = (p_last + 16) & ~15;
    const int ntiles = (kt - (kmin & ~15) + kBN - 1) / kBN;

    if (tid == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bar[B_KFULL + s], 1); mbar_init(&bar[B_KCONV + s], kConvWarps);
            mbar_init(&bar[B_KFREE + s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bar[B_VFULL + s], 1); mbar_init(&bar[B_VCONV + s], kConvWarps);
            mbar_init(&bar[B_VFREE + s], 1);
        }
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&bar[B_SFULL + s], 1); mbar_init(&bar[B_PFULL + s], 4); mbar_init(&bar[B_ODONE + s], 1);
        }
        mbar_init(&bar[B_QREADY], 8);
        mbar_init(&bar[B_DONE], 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    // every warpgroup changes its register share together
    if (warp < 8) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegSoftmax));
    else asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegOther));

    auto kbase = [&](int j) { return kt - kBN * (j + 1); };   // first key of tile j

    if (warp < 8) {
        // ================= softmax: warp w serves slot w / 4, rows 32 (w % 4) .. + 31
        const int slot = warp >> 2, lg = warp & 3;
        const int row = 32 * lg + lane;
        const uint32_t lane_off = (uint32_t)(32 * lg) << 16;
        const uint32_t tS = tmem + 128 * slot + lane_off;
        const uint32_t tO = tmem + kColO + 128 * slot + lane_off;
        const bool slot_valid = slot < nslots;
        const int hq = kvh * a.g + 2 * pi + slot;
        const int p = cut + i0 + row;
        const bool row_valid = slot_valid && row < rows;
        const int key_lo = a.W > 0 ? max(0, p - a.W + 1) : 0;
        bool fail = false;
        {
            // the row's query, rotated at p in fp32, times log2(e)/sqrt(d), rounded to fp16
            // and stored in the slot's Q tile (128-byte swizzle: 16-byte chunk c of row r at
            // c ^ (r mod 8)), two 64-dim halves with all loads of a half in one round trip
            float qmax = 0.f;
            unsigned char* qt = sQ + slot * kTileB;
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                uint4 qv[8];
                float4 rv[16];
#pragma unroll
                for (int c = 0; c < 8; ++c) qv[c] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int c = 0; c < 16; ++c) rv[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (row_valid) {
                    const uint4* qrow = reinterpret_cast<const uint4*>(
                        a.q + (((size_t)b * a.n + i0 + row) * a.Hq + hq) * kD + 64 * hf);
#pragma unroll
                    for (int c = 0; c < 8; ++c) qv[c] = __ldg(qrow + c);
                    if (a.rope) {
                        const float4* rp = reinterpret_cast<const float4*>(a.rope + (size_t)p * (kD / 2) + 32 * hf);
#pragma unroll
                        for (int c = 0; c < 16; ++c) rv[c] = __ldg(rp + c);
                    }
                }
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t wq[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
                    uint32_t h4[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float x0 = __uint_as_float(wq[k] << 16), x1 = __uint_as_float(wq[k] & 0xffff0000u);
                        float y0 = x0, y1 = x1;
                        if (a.rope) {
                            const float4 r4 = rv[(4 * c + k) >> 1];
                            rope_pair(x0, x1, ((4 * c + k) & 1) ? make_float2(r4.z, r4.w) : make_float2(r4.x, r4.y),
                                      y0, y1);
                        }
                        y0 = __fmul_rn(y0, a.scale_log2);
                        y1 = __fmul_rn(y1, a.scale_log2);
                        qmax = fmaxf(qmax, fmaxf(fabsf(y0), fabsf(y1)));
                        h4[k] = row_valid ? pack_f16(y0, y1) : 0u;
                    }
                    *reinterpret_cast<uint4*>(qt + hf * kHalfB + row * 128 + ((c ^ (row & 7)) << 4)) =
                        make_uint4(h4[0], h4[1], h4[2], h4[3]);
                }
            }
            if (row_valid && qmax >= kF16Limit) atomicOr(a.hdr, kErrRange);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_QREADY]);
        }
        float m_ref = -INFINITY, l = 0.f;
        if (slot_valid) {
            for (int j = 0; j < ntiles; ++j) {
                bool w = mbar_wait(&bar[B_SFULL + slot], (uint32_t)(j & 1)) && !*abort_flag;
                if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
                fence_after();
                float s[kBN];
                tmem_ld32f(tS, s);
                tmem_ld32f(tS + 32, s + 32);
                tmem_ld32f(tS + 64, s + 64);
                tmem_ld32f(tS + 96, s + 96);
                tmem_wait_ld();
                const int kb = kbase(j);
                if (!(kb >= key_lo_max && kb + kBN - 1 <= p_first && row_valid)) {
                    // some key of the tile is masked for some row of the CTA
#pragma unroll
                    for (int c = 0; c < kBN; ++c) {
                        const bool vis = row_valid && kb + c >= key_lo && kb + c <= p;
                        s[c] = vis ? s[c] : -INFINITY;
                    }
                }
                // row maximum: eight independent chains of three-input maxima, then a tree
                float m8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) m8[e] = fmaxf(s[e], s[8 + e]);
#pragma unroll
                for (int c = 16; c < kBN; c += 16)
#pragma unroll
                    for (int e = 0; e < 8; ++e) m8[e] = fmax3(m8[e], s[c + e], s[c + 8 + e]);
                const float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                // the reference maximum moves only when the tile exceeds it by more than kLazyMax;
                // then O (complete up to P.V of tile j - 1: S of this tile waited for it) is rescaled
                bool grow = false;
                float alpha = 1.f;
                if (mx > m_ref + kLazyMax) {
                    grow = m_ref != -INFINITY;
                    alpha = grow ? ex2(m_ref - mx) : 1.f;
                    m_ref = mx;
                }
                if (__any_sync(0xffffffffu, grow)) {
                    const float f = grow ? alpha : 1.f;
#pragma unroll 1
                    for (int c = 0; c < kD; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(tO + c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tmem_st32(tO + c, o);
                    }
                    tmem_wait_st();
                }
                const float base = m_ref == -INFINITY ? 0.f : m_ref;
                uint32_t pk[kBN / 2];
                float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
                const float2 nb2 = make_float2(-base, -base);
#pragma unroll
                for (int e = 0; e < kBN / 2; ++e) {
                    const float2 x = __fadd2_rn(make_float2(s[2 * e], s[2 * e + 1]), nb2);    // s - base, packed
                    const float p0 = ex2(x.x), p1 = ex2(x.y);                                  // masked keys: 0
                    rs[e & 3] = __fadd2_rn(rs[e & 3], make_float2(p0, p1));
                    pk[e] = pack_f16(p0, p1);
                }
                const float2 r01 = __fadd2_rn(rs[0], rs[1]), r23 = __fadd2_rn(rs[2], rs[3]);
                const float2 r4 = __fadd2_rn(r01, r23);
                l = l * alpha + (r4.x + r4.y);
                tmem_st32(tS, pk);
                tmem_st32(tS + 32, pk + 32);
                tmem_wait_st();
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[B_PFULL + slot]);
            }
            // the last P.V complete before O is read
            if (!fail && ntiles > 0) {
                const bool w = mbar_wait(&bar[B_ODONE + slot], (uint32_t)((ntiles - 1) & 1));
                fail = !__all_sync(0xffffffffu, w);
            }
            if (fail) {
                if (lane == 0) atomicOr(a.hdr, kErrWait);
                *abort_flag = 1;
            } else if (!*abort_flag) {
                // epilogue: O / l
                fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const size_t orow = (((size_t)b * a.n + i0 + row) * a.Hq + hq) * kD;
#pragma unroll 1
                for (int c = 0; c < kD; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(tO + c, o);
                    tmem_wait_ld();
                    if (!row_valid) continue;
                    if (a.out_bf16) {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow + c);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint32_t u[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                __nv_bfloat162 t2 = __floats2bfloat162_rn(__uint_as_float(o[8 * e + 2 * k]) * inv,
                                                                          __uint_as_float(o[8 * e + 2 * k + 1]) * inv);
                                u[k] = *reinterpret_cast<uint32_t*>(&t2);
                            }
                            dst[e] = make_uint4(u[0], u[1], u[2], u[3]);
                        }
                    } else {
                        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow + c);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                                 __uint_as_float(o[4 * e + 2]) * inv,
                                                 __uint_as_float(o[4 * e + 3]) * inv);
                    }
                }
            }
        }
    } else if (warp < kWarpTma || warp > kWarpMma) {
        // ================= converters (warps 8-11, 14, 15): K and V tiles bf16 -> fp16 in place
        const int t = warp < kWarpTma ? tid - 8 * 32 : tid - 10 * 32;
        __half2 hmax = __float2half2_rn(0.f);
        bool ok = true;
        for (int j = 0; j < ntiles && ok; ++j) {
            const int kb = kbase(j);
            const int ks = j % kKStages, vs = j % kVStages;
            ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_KFULL + ks], (uint32_t)((j / kKStages) & 1)) &&
                                             !*abort_flag);
            if (!ok) break;
            convert_tile(sK + ks * kTileB, t, kb, kmin, p_last, hmax);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_KCONV + ks]);
            ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_VFULL + vs], (uint32_t)((j / kVStages) & 1)) &&
                                             !*abort_flag);
            if (!ok) break;
            convert_tile(sV + vs * kTileB, t, kb, kmin, p_last, hmax);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_VCONV + vs]);
        }
        if (!ok) {
            if (lane == 0) atomicOr(a.hdr, kErrWait);
            *abort_flag = 1;
        }
        const float2 hm = __half22float2(hmax);
        if (__any_sync(0xffffffffu, fmaxf(hm.x, hm.y) >= kF16Limit) && lane == 0) atomicOr(a.hdr, kErrRange);
    } else if (warp == kWarpTma) {
        // ================= tensor copies of K and V tiles
        if (lane == 0) {
            const int head_row0 = (b * a.Hkv + kvh) * a.S;
            const int npages = a.S / kPage;
            // one tile of one tensor into `dst`: two 128-row copies (contiguous cache) or one
            // 16-row copy per 16 positions and half: the page of a paged cache, the slot of a
            // ring, or the staging rows at and after the ring's cut rounded down to 16
            // (positions before 0 are skipped)
            const int cal = cut & ~15;
            const int ws_row0 = (b * a.Hkv + kvh) * a.ws_rows;
            auto load_tile = [&](const CUtensorMap* tm, const CUtensorMap* tmw, unsigned char* dst, uint64_t* full,
                                 int kb) {
                if (!a.table && !a.ring) {
                    mbar_arrive_expect_tx(full, kTileB);
                    tma_load_2d(dst, tm, 0, head_row0 + kb, full);
                    tma_load_2d(dst + kHalfB, tm, 64, head_row0 + kb, full);
                    return;
                }
                const int g0 = kb < 0 ? (-kb) / 16 : 0;
                mbar_arrive_expect_tx(full, (uint32_t)(kBN / 16 - g0) * 2 * kGroupB);
                for (int gi = g0; gi < kBN / 16; ++gi) {
                    const int pos = kb + 16 * gi;
                    const CUtensorMap* m = tm;
                    int r;
                    if (a.ring && pos >= cal) {
                        m = tmw;
                        r = ws_row0 + (pos - cal);
                    } else {
                        const int slot = a.ring ? pos % a.S : pos;
                        if (a.table) {
                            int page = a.table[(size_t)b * npages + slot / kPage];
                            page = page < 0 ? 0 : page;      // never taken: every page the CTA reads is mapped
                            r = (page * a.Hkv + kvh) * kPage;
                        } else {
                            r = head_row0 + slot;
                        }
                    }
                    tma_load_2d(dst + gi * kGroupB, m, 0, r, full);
                    tma_load_2d(dst + kHalfB + gi * kGroupB, m, 64, r, full);
                }
            };
            bool ok = true;
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < ntiles && ok; ++j) {
                const int ks = j % kKStages, vs = j % kVStages;
                if (j >= kKStages) ok = mbar_wait(&bar[B_KFREE + ks], (uint32_t)((j / kKStages - 1) & 1));
                if (!ok || *abort_flag) { ok = false; break; }
                load_tile(&tmK, &tmWK, sK + ks * kTileB, &bar[B_KFULL + ks], kbase(j));
                k_issued = j + 1;
                if (j >= kVStages) ok = mbar_wait(&bar[B_VFREE + vs], (uint32_t)((j / kVStages - 1) & 1));
                if (!ok || *abort_flag) { ok = false; break; }
                load_tile(&tmV, &tmWV, sV + vs * kTileB, &bar[B_VFULL + vs], kbase(j));
                v_issued = j + 1;
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(a.hdr, kErrWait);
                // the last copy issued into each stage lands before the CTA can exit
                for (int t = max(0, k_issued - kKStages); t < k_issued; ++t)
                    mbar_wait(&bar[B_KFULL + t % kKStages], (uint32_t)((t / kKStages) & 1));
                for (int t = max(0, v_issued - kVStages); t < v_issued; ++t)
                    mbar_wait(&bar[B_VFULL + t % kVStages], (uint32_t)((t / kVStages) & 1));
            }
        }
    } else if (warp == kWarpMma) {
        // ================= one thread issues every MMA, whichever is ready first
        if (lane == 0) {
            constexpr uint32_t idesc_qk = instr_desc_f16(kBM, kBN, false);
            constexpr uint32_t idesc_pv = instr_desc_f16(kBM, kD, true);
            // descriptors of slot 0 / stage 0; other slots, stages and k-steps move only the
            // start address field (bytes / 16, no carry: shared addresses stay below 256 KB)
            const uint64_t qdesc0 = smem_desc(smem_u32(sQ), 16), kdesc0 = smem_desc(smem_u32(sK), 16);
            const uint64_t vdesc0 = smem_desc(smem_u32(sV), kHalfB);
            auto koff = [](int s) { return (uint64_t)(((s >> 2) * kHalfB + (s & 3) * 32) >> 4); };
            // S_i(j) = Q_i K_j^T into S buffer i (dims 16 s .. + 15 per instruction)
            auto issue_s = [&](int i, int j) {
                const uint64_t qd = qdesc0 + (uint64_t)(i * (kTileB >> 4));
                const uint64_t kd = kdesc0 + (uint64_t)((j % kKStages) * (kTileB >> 4));
#pragma unroll
                for (int s = 0; s < kD / 16; ++s) mma_ss(tmem + 128 * i, qd + koff(s), kd + koff(s), idesc_qk, s > 0);
                mma_commit(&bar[B_SFULL + i]);
            };
            // O_i += P_i(j) V_j: keys 16 s .. + 15 of P sit in columns 8 s .. + 7 of S buffer i
            auto issue_pv = [&](int i, int j) {
                const uint64_t vd = vdesc0 + (uint64_t)((j % kVStages) * (kTileB >> 4));
#pragma unroll
                for (int s = 0; s < kBN / 16; ++s)
                    mma_ts(tmem + kColO + 128 * i, tmem + 128 * i + 8 * s, vd + (uint64_t)((s * 2048) >> 4), idesc_pv,
                           (j > 0 || s > 0));
                mma_commit(&bar[B_ODONE + i]);
            };
            // per slot: S(j) -> [softmax writes P(j)] -> P.V(j) -> S(j + 1) once P.V(j) is
            // complete (S(j + 1) overwrites the P columns P.V(j) reads); the slots alternate
            auto wait_ok = [&](uint64_t* bar_, uint32_t parity) { return mbar_spin(bar_, parity) && !*abort_flag; };
            bool ok = wait_ok(&bar[B_QREADY], 0) && wait_ok(&bar[B_KCONV], 0);
            if (ok) {
                fence_after();
                for (int i = 0; i < nslots; ++i) issue_s(i, 0);
                mma_commit(&bar[B_KFREE]);
            }
            for (int j = 0; j < ntiles && ok; ++j) {
                const int vs = j % kVStages, ks1 = (j + 1) % kKStages;
                ok = wait_ok(&bar[B_VCONV + vs], (uint32_t)((j / kVStages) & 1));
                for (int i = 0; i < nslots && ok; ++i) {
                    ok = wait_ok(&bar[B_PFULL + i], (uint32_t)(j & 1));
                    if (!ok) break;
                    fence_after();
                    issue_pv(i, j);
                    if (j + 1 < ntiles) {
                        if (i == 0) ok = wait_ok(&bar[B_KCONV + ks1], (uint32_t)(((j + 1) / kKStages) & 1));
                        if (ok) ok = wait_ok(&bar[B_ODONE + i], (uint32_t)(j & 1));
                        if (!ok) break;
                        fence_after();
                        issue_s(i, j + 1);
                    }
                }
                if (!ok) break;
                mma_commit(&bar[B_VFREE + vs]);                       // both P.V of tile j issued
                if (j + 1 < ntiles) mma_commit(&bar[B_KFREE + ks1]);  // both S of tile j + 1 issued
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(a.hdr, kErrWait);
            }
            // no tensor-core operation may still target our columns when they are freed:
            // a commit tracks every MMA this thread issued
            mma_commit(&bar[B_DONE]);
            mbar_wait(&bar[B_DONE], 0);
        }
    }
    fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        __syncwarp();
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ---- ring staging --------------------------------------------------------------
struct StageArgs {
    const __nv_bfloat16* kc;   // cache rows
    const __nv_bfloat16* vc;
    const int32_t* table;      // paged: block table (else nullptr)
    const __nv_bfloat16* k;    // suffix [B][n][Hkv][d], keys not rotated
    const __nv_bfloat16* v;
    const float2* rope;        // nullptr = no RoPE
    __nv_bfloat16* wk;         // staging [B][Hkv][ws_rows][d]
    __nv_bfloat16* wv;
    const int32_t* next_pos;   // the cut (before the append)
    int Hkv, S, n, ws_rows;
};

// Staging row r of (request b, KV head h) holds position cal + r, cal = cut rounded
// down to 16: rows below the cut copied from the ring, suffix rows rotated at their
// position (fp32, each product and sum rounded once, then bf16 round to nearest:
// the append's arithmetic).  16 bytes per thread, 8 rows per CTA of 128 threads.
__global__ void __launch_bounds__(128) chunk_stage_kernel(const StageArgs a) {
    const int b = blockIdx.z, h = blockIdx.y;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 4), c = threadIdx.x & 15;
    const int cut = a.next_pos[b], cal = cut & ~15;
    if (r >= cut - cal + a.n) return;
    const int pos = cal + r;
    uint4 ko, vo;
    if (pos < cut) {
        const size_t src = kv_row(a.table, b, h, pos % a.S, a.Hkv, a.S) * kD + 8 * (size_t)c;
        ko = *reinterpret_cast<const uint4*>(a.kc + src);
        vo = *reinterpret_cast<const uint4*>(a.vc + src);
    } else {
        const size_t src = (((size_t)b * a.n + (pos - cut)) * a.Hkv + h) * kD + 8 * (size_t)c;
        ko = __ldg(reinterpret_cast<const uint4*>(a.k + src));
        vo = __ldg(reinterpret_cast<const uint4*>(a.v + src));
        if (a.rope) {
            const float4* rp = reinterpret_cast<const float4*>(a.rope + (size_t)pos * (kD / 2) + 4 * c);
            const float4 c0 = __ldg(rp), c1 = __ldg(rp + 1);
            uint32_t w[4] = {ko.x, ko.y, ko.z, ko.w};
            const float2 cs[4] = {make_float2(c0.x, c0.y), make_float2(c0.z, c0.w), make_float2(c1.x, c1.y),
                                  make_float2(c1.z, c1.w)};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 x2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
                float y0, y1;
                rope_pair(__low2float(x2), __high2float(x2), cs[e], y0, y1);
                const __nv_bfloat162 o2 = __floats2bfloat162_rn(y0, y1);
                w[e] = *reinterpret_cast<const uint32_t*>(&o2);
            }
            ko = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    const size_t dst = (((size_t)b * a.Hkv + h) * a.ws_rows + r) * kD + 8 * (size_t)c;
    *reinterpret_cast<uint4*>(a.wk + dst) = ko;
    *reinterpret_cast<uint4*>(a.wv + dst) = vo;
}

// ---- tensor maps -----------------------------------------------------------
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

}  // namespace

bool make_tensor_map_bf16(CUtensorMap* tm, void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                          const cuuint32_t* box) {
    EncodeTiled enc = encoder();
    if (!enc) return false;
    cuuint32_t es[3] = {1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool chunk_supported(const Shape& s) { return s.bf16 && !s.int8 && s.d == kD && (!s.ring || s.S % 16 == 0); }

cudaError_t launch_chunk(kvc_handle* h, const void* q, const void* k, const void* v, void* out, int n,
                         cudaStream_t st) {
    const Shape& s = h->sh;
    const int ws = chunk_ws_rows(s);
    CUtensorMap tk, tv, twk, twv;
    const cuuint64_t rows = s.pages ? (cuuint64_t)s.pages * s.Hkv * kPage : (cuuint64_t)s.B * s.Hkv * s.S;
    const cuuint64_t kdims[2] = {(cuuint64_t)s.d, rows};
    const cuuint64_t kstr[1] = {(cuuint64_t)s.d * 2};
    const cuuint32_t kbox[2] = {64, (s.pages || s.ring) ? (cuuint32_t)kPage : (cuuint32_t)kBN};
    if (!make_tensor_map_bf16(&tk, h->state + h->L.k, 2, kdims, kstr, kbox) ||
        !make_tensor_map_bf16(&tv, h->state + h->L.v, 2, kdims, kstr, kbox))
        return cudaErrorInvalidValue;
    twk = tk; twv = tv;
    if (s.ring) {
        // staging rows, then the suffix attention reads them beside the ring
        const size_t half = (size_t)s.B * s.Hkv * ws * s.d;
        __nv_bfloat16* wk = reinterpret_cast<__nv_bfloat16*>(h->state + h->L.cws);
        const cuuint64_t wdims[2] = {(cuuint64_t)s.d, (cuuint64_t)s.B * s.Hkv * ws};
        const cuuint32_t wbox[2] = {64, (cuuint32_t)kPage};
        if (!make_tensor_map_bf16(&twk, wk, 2, wdims, kstr, wbox) ||
            !make_tensor_map_bf16(&twv, wk + half, 2, wdims, kstr, wbox))
            return cudaErrorInvalidValue;
        StageArgs sa{};
        sa.kc = reinterpret_cast<const __nv_bfloat16*>(h->state + h->L.k);
        sa.vc = reinterpret_cast<const __nv_bfloat16*>(h->state + h->L.v);
        sa.table = s.pages ? reinterpret_cast<const int32_t*>(h->state + h->L.table) : nullptr;
        sa.k = static_cast<const __nv_bfloat16*>(k);
        sa.v = static_cast<const __nv_bfloat16*>(v);
        sa.rope = s.rope ? reinterpret_cast<const float2*>(h->state + h->L.rope) : nullptr;
        sa.wk = wk;
        sa.wv = wk + half;
        sa.next_pos = reinterpret_cast<const int32_t*>(h->state + h->L.next_pos);
        sa.Hkv = s.Hkv; sa.S = s.S; sa.n = n; sa.ws_rows = ws;
        chunk_stage_kernel<<<dim3((n + 15 + 7) / 8, s.Hkv, s.B), 128, 0, st>>>(sa);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (cudaError_t e = allow_smem(reinterpret_cast<const void*>(chunk_attn_kernel), SMEM_BYTES)) return e;
    // ChunkArgs carries the order table: it lives in static storage, not on the stack
    static thread_local ChunkArgs a;
    a = ChunkArgs{};
    a.next_pos = reinterpret_cast<const int32_t*>(h->state + h->L.next_pos);
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.rope = s.rope ? reinterpret_cast<const float2*>(h->state + h->L.rope) : nullptr;
    a.out = out; a.hdr = reinterpret_cast<uint32_t*>(h->state + h->L.hdr);
    a.table = s.pages ? reinterpret_cast<const int32_t*>(h->state + h->L.table) : nullptr;
    a.B = s.B; a.Hq = s.Hq; a.Hkv = s.Hkv; a.g = s.g; a.S = s.S; a.W = s.W; a.n = n; a.out_bf16 = s.out_bf16;
    a.ring = s.ring; a.n_appended = s.ring ? 0 : n; a.ws_rows = ws;
    a.tiles = (n + kBM - 1) / kBM;
    a.pairs = (s.g + 1) / 2;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.d));
    // longest first: a (request, tile) item's work is its number of key tiles, from the
    // host mirror of next_position (already advanced past the appended suffix)
    const int items = s.B * a.tiles;
    if (items <= kMaxItems && s.B <= 65536 && a.tiles <= 65536) {
        std::vector<std::pair<int, uint32_t>> w(items);
        for (int b = 0; b < s.B; ++b)
            for (int t = 0; t < a.tiles; ++t) {
                const int cut = h->np[b] - a.n_appended, i0 = t * kBM, rows = std::min(kBM, n - i0);
                const int p_first = cut + i0, p_last = p_first + rows - 1;
                const int kmin = s.W > 0 ? std::max(0, p_first - s.W + 1) : 0;
                const int kt = (p_last + 16) & ~15;
                w[b * a.tiles + t] = {-((kt - (kmin & ~15) + kBN - 1) / kBN), ((uint32_t)b << 16) | (uint32_t)t};
            }
        std::stable_sort(w.begin(), w.end(),
                         [](const std::pair<int, uint32_t>& x, const std::pair<int, uint32_t>& y) {
                             return x.first < y.first;
                         });
        for (int i = 0; i < items; ++i) a.items[i] = w[i].second;
        a.n_items = items;
    }
    chunk_attn_kernel<<<dim3(items * s.Hkv * a.pairs), kThreads, SMEM_BYTES, st>>>(tk, tv, twk, twv, a);
    return cudaGetLastError();
}

}  // namespace kvc
