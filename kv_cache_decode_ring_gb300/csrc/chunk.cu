// chunk.cu -- chunked causal (or sliding-window) suffix attention on tcgen05.
//
// [PREFIX] "哪些東西必須一起裁剪": after the cache is trimmed to `cut`, the
// suffix tokens[cut:] are computed in one chunk from next_position = cut:
// suffix query i sits at position p = cut + i and attends to cached positions
// [max(0, p - W + 1), p] (W = 0: all), exactly what a one-token decode at p
// would see ([LEAN] §2.1 masks).  The suffix K/V rows are appended to the
// contiguous cache first, so every key a query needs lies in one contiguous
// run of cache rows.
//
// This is a dense contraction, so it runs on the 5th-generation tensor cores:
//  * CTA = 128 query rows of one query head (4 warps, thread = row); tiles of
//    64 keys;
//  * K and V tiles arrive by TMA (128-byte swizzle), each stage refilled as soon
//    as the MMA that read it completes; each softmax warp rotates its rows' query
//    half from global memory (fp32 rule of the cache keys, times log2(e)/sqrt(d))
//    and stores it into tensor memory as bf16 hi and lo;
//  * CTAs are taken longest first (a host-sorted table of (request, query tile)
//    items in the kernel parameters), the query heads of one item adjacent so that
//    heads sharing a KV head read its tiles from L2;
//  * S = Q K^T and O += P V are tcgen05.mma (bf16 in, fp32 accumulate) issued
//    by one thread into tensor memory (two 64-column S buffers, 128-column O);
//  * software pipeline: S of tile j + 1 is issued before the softmax of tile j
//    and P V of tile j after it, so the tensor cores work while the threads run
//    the softmax; two P buffers let P of tile j + 1 be written while P V of
//    tile j still reads its own;
//  * each thread reads its S row from tensor memory, applies the causal and
//    window masks by absolute position, runs the online softmax in fp32 (log2
//    domain) and writes its P row to shared memory for the next MMA.  A row's
//    reference maximum moves only when a tile exceeds it by more than 2^8, so
//    the O rescale in tensor memory (which must wait for the pending P V) is
//    rare;
//  * the rotated query and P are not exact in bf16, so each enters its MMA as
//    two bf16 terms (hi, lo) accumulated in fp32 (about 16 significant bits);
//  * K/V tiles are walked backwards from the diagonal;
//  * tcgen05.ld/st are warp-collective: every lane of a warp issues them.
// Every mbarrier wait is bounded; on expiry the kernel flags the device error
// word, skips the remaining work and still frees its tensor memory.
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

constexpr int kBM = 128;          // query rows per CTA
constexpr int kBN = 128;          // keys per tile
constexpr int kD = 128;           // head dim of this kernel
constexpr int kSoftmaxWarps = 8;   // two per tensor-memory lane group
constexpr int kThreads = (kSoftmaxWarps + 1) * 32;   // + one producer warp
constexpr int kKStages = 3;       // K tile stages (free once S of the tile is complete)
constexpr int kVStages = 2;       // V tile stages (free once P V of the tile is complete)
constexpr float kLazyMax = 8.f;   // log2-domain headroom of a row's reference maximum
constexpr int kTileB = 128 * kD * 2;     // 32 KB: two 64-dim halves of [128 rows][128 B]
constexpr int kHalfB = kTileB / 2;
// Operands that are not exact bf16 (the rotated query and the softmax weights)
// enter the MMAs as two bf16 terms, hi = bf16(x) and lo = bf16(x - hi), both
// accumulated in fp32: about 16 significant bits instead of 8.
constexpr int OFF_X = 0;                              // row-maximum exchange [2][2][kBM] floats
constexpr int OFF_L = OFF_X + 4 * kBM * 4;            // row sums of the two halves [2][kBM]
constexpr int OFF_K = 4096;                           // kKStages K tiles (1024-aligned)
constexpr int OFF_V = OFF_K + kKStages * kTileB;      // kVStages V tiles
constexpr int OFF_BAR = OFF_V + kVStages * kTileB;    // k[3], v[2], s[2], o[2], p[2], done, q in tmem
constexpr int kBars = kKStages + kVStages + 2 + 2 + 2 + 1 + 1;
constexpr int kMaxItems = 2048;                       // (request, query tile) items in the order table
constexpr int OFF_MISC = OFF_BAR + 8 * kBars;         // tensor memory base, abort flag
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory per block");
// Tensor memory (512 columns, 128 lanes = query rows):
//   S/P buffers [0, 128), [128, 256): S of a tile in fp32; the softmax warp serving
//     keys 64 h .. + 63 overwrites its 64 columns with P as bf16 pairs (hi in the first
//     32, lo in the next 32), the A operand of P V;
//   O [256, 384) fp32; Q hi [384, 448) and Q lo [448, 512) as bf16 pairs, the A
//   operand of S.  Only K and V tiles are shared-memory operands.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256, kColQ = 384, kColQlo = 448;

struct ChunkArgs {
    const int32_t* next_pos;   // after the append: cut + n
    const __nv_bfloat16* q;    // [B][n][Hq][d], not rotated
    const float2* rope;        // nullptr = no RoPE
    void* out;                 // [B][n][Hq][d]
    uint32_t* hdr;
    int B, Hq, Hkv, g, S, W, n, out_bf16;
    int tiles;                 // query tiles per request
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

// Instruction descriptor, kind::f16: D fp32 (bit 4), A and B bf16 (bits 7, 10),
// B MN-major when b_mn (bit 16), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// D (tensor memory) (+)= A (tensor memory, bf16 pairs along columns, row m in lane m)
// . B (shared memory descriptor)
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            int acc) {
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

// 32 consecutive fp32 columns of this thread's tensor-memory lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
          "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
          "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
          "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
          "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
          "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
          "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
          "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
          "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
          "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
          "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x with the hardware approximation (relative error about 2^-22; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 16 consecutive 32-bit columns of this thread's tensor-memory lane
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
          "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t* v) {
    tmem_st16(taddr, v);
    tmem_st16(taddr + 16, v + 16);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Barrier `id` over the 64 threads of a warp pair; returns the OR of `pred` over them.
__device__ __forceinline__ bool pair_sync_or(int id, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.red.or.pred q, %2, 64, p;\n"
        " selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r) : "r"((uint32_t)pred), "r"(id) : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    chunk_attn_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ ChunkArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* sK = smem + OFF_K;
    unsigned char* sV = smem + OFF_V;
    float* xmax = reinterpret_cast<float*>(smem + OFF_X);   // [parity][half][row]
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* bk = bar;                      // [stage] K tile landed
    uint64_t* bv = bk + kKStages;            // [stage] V tile landed
    uint64_t* bs = bv + kVStages;            // [buffer] S = Q K^T complete
    uint64_t* bo = bs + 2;                   // [buffer] O += P V complete
    uint64_t* bp = bo + 2;                   // [buffer] P written by the 8 softmax warps
    uint64_t* bdone = bp + 2;                // every MMA issued so far complete (abort path)
    uint64_t* bqt = bdone + 1;               // Q copied into tensor memory by the 8 softmax warps
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA's (request, query tile, query head)
    int b, tile;
    const int hq = blockIdx.x % a.Hq, item = blockIdx.x / a.Hq;
    if (a.n_items > 0) { b = (int)(a.items[item] >> 16); tile = (int)(a.items[item] & 0xFFFFu); }
    else { b = item / a.tiles; tile = item % a.tiles; }
    const int i0 = tile * kBM;
    const int kvh = hq / a.g;
    const int np = a.next_pos[b];
    const int cut = np - a.n;
    const int rows = min(kBM, a.n - i0);
    const int p_first = cut + i0, p_last = cut + i0 + rows - 1;
    const int lo = a.W > 0 ? max(0, p_first - a.W + 1) : 0;
    const int ntiles = (p_last + 1 - lo + kBN - 1) / kBN;
    const int head_row0 = (b * a.Hkv + kvh) * a.S;

    if (tid == 0) {
        for (int i = 0; i < kBars; ++i) mbar_init(&bar[i], 1);
        for (int i = 0; i < 2; ++i) mbar_init(&bp[i], kSoftmaxWarps);
        mbar_init(bqt, kSoftmaxWarps);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kSoftmaxWarps) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tO = tmem + kColO;

    if (warp == kSoftmaxWarps) {
        // ================= producer: one thread issues every copy and every MMA
        if (lane == 0) {
            constexpr uint32_t idesc_qk = instr_desc(kBM, kBN, false);
            constexpr uint32_t idesc_pv = instr_desc(kBM, kD, true);
            auto kbase_of = [&](int j) { return p_last + 1 - kBN * (j + 1); };
            auto load_k = [&](int j) {
                const int st = j % kKStages;
                mbar_arrive_expect_tx(&bk[st], kTileB);
                tma_load_2d(sK + st * kTileB, &tmK, 0, head_row0 + kbase_of(j), &bk[st]);
                tma_load_2d(sK + st * kTileB + kHalfB, &tmK, 64, head_row0 + kbase_of(j), &bk[st]);
            };
            auto load_v = [&](int j) {
                const int st = j % kVStages;
                mbar_arrive_expect_tx(&bv[st], kTileB);
                tma_load_2d(sV + st * kTileB, &tmV, 0, head_row0 + kbase_of(j), &bv[st]);
                tma_load_2d(sV + st * kTileB + kHalfB, &tmV, 64, head_row0 + kbase_of(j), &bv[st]);
            };
            // descriptors of stage 0; stage and k-step offsets move only the start address
            // field (bytes / 16, no carry: shared addresses stay below 256 KB)
            const uint64_t kdesc0 = smem_desc(smem_u32(sK), 16), vdesc0 = smem_desc(smem_u32(sV), kHalfB);
            // S_j = Q_hi K_j^T + Q_lo K_j^T into S/P buffer j % 2 (Q: dims 16 s .. + 15 in
            // columns 8 s .. + 7 of its region)
            auto issue_s = [&](int j) {
                const uint64_t kd = kdesc0 + (uint64_t)((j % kKStages) * (kTileB >> 4));
                const uint32_t d = tmem + 128 * (j & 1);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s)
                    mma_bf16_ts(d, tmem + kColQ + 8 * s, kd + (uint64_t)(((s >> 2) * kHalfB + (s & 3) * 32) >> 4),
                                idesc_qk, s > 0);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s)
                    mma_bf16_ts(d, tmem + kColQlo + 8 * s, kd + (uint64_t)(((s >> 2) * kHalfB + (s & 3) * 32) >> 4),
                                idesc_qk, 1);
                mma_commit(&bs[j & 1]);
            };
            // O += P_hi V_j + P_lo V_j: keys 16 s2 .. + 15 of P sit in columns
            // 64 (s2 / 4) + 8 (s2 % 4) .. + 7 of S/P buffer j % 2 (lo 32 columns further)
            auto issue_pv = [&](int j) {
                const uint32_t pb = tmem + 128 * (j & 1);
                const uint64_t vd = vdesc0 + (uint64_t)((j % kVStages) * (kTileB >> 4));
#pragma unroll
                for (int s2 = 0; s2 < kBN / 16; ++s2)
                    mma_bf16_ts(tO, pb + 64 * (s2 >> 2) + 8 * (s2 & 3), vd + (uint64_t)((s2 * 2048) >> 4), idesc_pv,
                                (j > 0 || s2 > 0));
#pragma unroll
                for (int s2 = 0; s2 < kBN / 16; ++s2)
                    mma_bf16_ts(tO, pb + 64 * (s2 >> 2) + 32 + 8 * (s2 & 3), vd + (uint64_t)((s2 * 2048) >> 4),
                                idesc_pv, 1);
                mma_commit(&bo[j & 1]);
            };

            bool ok = true;
            // copies issued and awaited so far (an abort drains the rest before exit)
            int k_issued = 0, v_issued = 0, k_waited = 0, v_waited = 0;
            for (int j = 0; j < kKStages && j < ntiles; ++j) { load_k(j); k_issued = j + 1; }
            for (int j = 0; j < kVStages && j < ntiles; ++j) { load_v(j); v_issued = j + 1; }
            ok = mbar_wait(bqt, 0);                  // the softmax warps stored Q into tensor memory
            for (int j = 0; j < 2 && j < ntiles && ok; ++j) {
                ok = mbar_wait(&bk[j], 0);
                if (ok) { k_waited = j + 1; fence_after(); issue_s(j); }
            }
            for (int j = 0; j < ntiles && ok; ++j) {
                if (*abort_flag) { ok = false; break; }
                // P_j written: the softmax warps read S_j, so S_j is complete and the K stage
                // of tile j is free: fetch K of tile j + kKStages
                ok = mbar_wait(&bp[j & 1], (uint32_t)((j >> 1) & 1));
                if (!ok) break;
                if (j + kKStages < ntiles) { load_k(j + kKStages); k_issued = j + kKStages + 1; }
                // O += P_j V_j
                ok = mbar_wait(&bv[j % kVStages], (uint32_t)((j / kVStages) & 1));
                if (!ok) break;
                v_waited = j + 1;
                fence_after();
                issue_pv(j);
                if (j + 2 < ntiles) {
                    // S_{j+2} overwrites P_j's buffer: wait for P V_j (which also frees the
                    // V stage of tile j), then fetch V of tile j + 2 and issue S_{j+2}
                    ok = mbar_wait(&bo[j & 1], (uint32_t)((j >> 1) & 1));
                    if (!ok) break;
                    load_v(j + 2);
                    v_issued = j + 3;
                    ok = mbar_wait(&bk[(j + 2) % kKStages], (uint32_t)(((j + 2) / kKStages) & 1));
                    if (!ok) break;
                    k_waited = j + 3;
                    fence_after();
                    issue_s(j + 2);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(a.hdr, kErrWait);
                // let every copy still in flight land before the CTA can exit
                for (int t = k_waited; t < k_issued; ++t) mbar_wait(&bk[t % kKStages], (uint32_t)((t / kKStages) & 1));
                for (int t = v_waited; t < v_issued; ++t) mbar_wait(&bv[t % kVStages], (uint32_t)((t / kVStages) & 1));
            }
        }
    } else {
        // ================= softmax warps: warp w serves rows 32 (w % 4) .. + 31 (its
        // tensor-memory lanes) and keys 64 (w / 4) .. + 63 of every tile; the two warps of
        // a row pair exchange their halves' maxima through shared memory
        const int lg = warp & 3, hf = warp >> 2;
        const int row = 32 * lg + lane;            // query row = tensor-memory lane
        const uint32_t lane_off = (uint32_t)(32 * lg) << 16;
        const int p = cut + i0 + row;               // its absolute position
        const bool row_valid = row < rows;
        const int key_lo = a.W > 0 ? max(0, p - a.W + 1) : 0;
        const int key_lo_max = a.W > 0 ? max(0, p_last - a.W + 1) : 0;   // the CTA's largest key_lo
        const int pair_bar = 1 + lg;               // named barrier of the pair (0 = __syncthreads)
        float m_ref = -INFINITY, l = 0.f;
        bool fail = false;
        {
            // this warp's half of its row's query (dims 64 hf .. + 63): rotated at the row's
            // position in fp32, times log2(e)/sqrt(d), split into bf16 hi = bf16(y) and
            // lo = bf16(y - hi), stored into tensor memory as bf16 pairs along columns
            uint32_t qh[32], ql[32];
            if (row_valid) {
                // every load first (one round trip): 8 x 16 B of the query half, 16 x 16 B
                // of its {cos, sin} pairs
                const uint4* qrow = reinterpret_cast<const uint4*>(
                    a.q + (((size_t)b * a.n + i0 + row) * a.Hq + hq) * kD + 64 * hf);
                uint4 qv[8];
                float4 rv[16];
#pragma unroll
                for (int c = 0; c < 8; ++c) qv[c] = __ldg(qrow + c);
                if (a.rope) {
                    const float4* rp = reinterpret_cast<const float4*>(a.rope + (size_t)p * (kD / 2) + 32 * hf);
#pragma unroll
                    for (int c = 0; c < 16; ++c) rv[c] = __ldg(rp + c);
                }
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t wq[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const __nv_bfloat162 x2 = *reinterpret_cast<const __nv_bfloat162*>(&wq[k]);
                        const float x0 = __low2float(x2), x1 = __high2float(x2);
                        float y0 = x0, y1 = x1;
                        if (a.rope) {
                            const float4 r4 = rv[(4 * c + k) >> 1];
                            rope_pair(x0, x1, ((4 * c + k) & 1) ? make_float2(r4.z, r4.w) : make_float2(r4.x, r4.y),
                                      y0, y1);
                        }
                        y0 = __fmul_rn(y0, a.scale_log2);
                        y1 = __fmul_rn(y1, a.scale_log2);
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(y0, y1);
                        qh[4 * c + k] = *reinterpret_cast<const uint32_t*>(&h2);
                        ql[4 * c + k] = pack_bf16(__fsub_rn(y0, __low2float(h2)), __fsub_rn(y1, __high2float(h2)));
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) { qh[e] = 0u; ql[e] = 0u; }
            }
            tmem_st32u(tmem + kColQ + 32 * hf + lane_off, qh);
            tmem_st32u(tmem + kColQlo + 32 * hf + lane_off, ql);
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bqt);
        }
        for (int j = 0; j < ntiles; ++j) {
            // (1) S_j complete; this warp's 64 scores of the row
            bool w = !fail && mbar_wait(&bs[j & 1], (uint32_t)((j >> 1) & 1)) && !*abort_flag;
            w = __all_sync(0xffffffffu, w);
            float sm[kBN / 2];
            float mx = -INFINITY;
            const int kb = p_last + 1 - kBN * (j + 1) + 64 * hf;         // first key of this half
            const uint32_t tSj = tmem + 128 * (j & 1) + 64 * hf + lane_off;
            if (w) {
                fence_after();
                tmem_ld32(tSj, sm);
                tmem_ld32(tSj + 32, sm + 32);
                if (kb - 64 * hf >= key_lo_max && kb - 64 * hf + kBN - 1 <= p_first) {
                    // every key of the tile is visible to every row of the CTA
#pragma unroll
                    for (int c = 0; c < kBN / 2; ++c) mx = fmaxf(mx, sm[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < kBN / 2; ++c) {
                        const bool vis = row_valid && kb + c >= key_lo && kb + c <= p;
                        sm[c] = vis ? sm[c] : -INFINITY;
                        mx = fmaxf(mx, sm[c]);
                    }
                }
            }
            // (2) exchange the halves' maxima (and any failure) with the partner warp
            xmax[((j & 1) * 2 + hf) * kBM + row] = mx;
            if (pair_sync_or(pair_bar, !w)) { fail = true; break; }
            mx = fmaxf(mx, xmax[((j & 1) * 2 + (1 - hf)) * kBM + row]);
            // (3) the reference maximum moves only when the tile exceeds it by more than kLazyMax
            bool grow = false;
            float alpha = 1.f;
            if (mx > m_ref + kLazyMax) {           // also the first visible tile (m_ref = -inf)
                grow = m_ref != -INFINITY;        // O and l hold earlier tiles only then
                alpha = grow ? exp2f(m_ref - mx) : 1.f;
                m_ref = mx;
            }
            const float base = m_ref == -INFINITY ? 0.f : m_ref;
            float2 rs2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kBN / 2; c += 2) {
                sm[c] = ex2(sm[c] - base);         // masked keys: 0
                sm[c + 1] = ex2(sm[c + 1] - base);
                rs2 = __fadd2_rn(rs2, make_float2(sm[c], sm[c + 1]));
            }
            l = l * alpha + (rs2.x + rs2.y);
            // (4) O may be rescaled only once P V of tile j - 1 is complete
            // (tcgen05.ld/st: whole warps)
            const bool any_grow = __any_sync(0xffffffffu, grow);
            if (any_grow) {
                if (!__all_sync(0xffffffffu, mbar_wait(&bo[(j - 1) & 1], (uint32_t)(((j - 1) >> 1) & 1)))) {
                    fail = true;                   // the partner learns at the next exchange
                } else {
                    fence_after();
                    const float f = grow ? alpha : 1.f;
#pragma unroll
                    for (int c = 0; c < kD / 2; c += 32) {
                        float o[32];
                        tmem_ld32(tO + lane_off + 64 * hf + c, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= f;
                        tmem_st32(tO + lane_off + 64 * hf + c, o);
                    }
                }
            }
            if (fail) continue;                    // skip the write; the next exchange ends the loop
            // (5) this warp's 64 keys of the P row over its own S columns: hi and lo bf16
            // pairs (keys 64 hf + 2 e, + 1 in column e; lo 32 columns further)
            uint32_t hi[32], lo2[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float2 x = make_float2(sm[2 * e], sm[2 * e + 1]);
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(x.x, x.y);
                const float2 r = __ffma2_rn(__bfloat1622float2(h2), make_float2(-1.f, -1.f), x);   // x - hi, exact
                hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
                lo2[e] = pack_bf16(r.x, r.y);
            }
            tmem_st32u(tSj, hi);
            tmem_st32u(tSj + 32, lo2);
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bp[j & 1]);
        }
        // the last P V complete before O is read
        if (!fail && ntiles > 0) {
            const bool w = mbar_wait(&bo[(ntiles - 1) & 1], (uint32_t)(((ntiles - 1) >> 1) & 1));
            fail = !__all_sync(0xffffffffu, w);
        }
        if (fail) {
            if (lane == 0) atomicOr(a.hdr, kErrWait);
            *abort_flag = 1;
        }
        // partial row sums of the two halves
        reinterpret_cast<float*>(smem + OFF_L)[hf * kBM + row] = l;
    }
    __syncthreads();
    const bool aborted = *abort_flag != 0;
    if (warp < kSoftmaxWarps && !aborted) {
        // ---- epilogue: O / l; warp w stores columns 64 (w / 4) .. + 63 of its rows
        const int lg = warp & 3, hf = warp >> 2;
        const int row = 32 * lg + lane;
        const uint32_t lane_off = (uint32_t)(32 * lg) << 16;
        fence_after();
        const float* lsum = reinterpret_cast<const float*>(smem + OFF_L);
        const float L = lsum[row] + lsum[kBM + row];
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const size_t orow = (((size_t)b * a.n + i0 + row) * a.Hq + hq) * kD + 64 * hf;
#pragma unroll
        for (int c = 0; c < kD / 2; c += 32) {
            float o[32];
            tmem_ld32(tO + lane_off + 64 * hf + c, o);
            if (row >= rows) continue;
            if (a.out_bf16) {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow + c);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint4 u;
                    u.x = pack_bf16(o[8 * e + 0] * inv, o[8 * e + 1] * inv);
                    u.y = pack_bf16(o[8 * e + 2] * inv, o[8 * e + 3] * inv);
                    u.z = pack_bf16(o[8 * e + 4] * inv, o[8 * e + 5] * inv);
                    u.w = pack_bf16(o[8 * e + 6] * inv, o[8 * e + 7] * inv);
                    dst[e] = u;
                }
            } else {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow + c);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    dst[e] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv, o[4 * e + 3] * inv);
            }
        }
    }
    if (warp == kSoftmaxWarps && aborted && lane == 0) {
        // make sure no tensor-core operation still targets our columns before freeing
        // them: a commit tracks every MMA this thread issued
        mma_commit(bdone);
        mbar_wait(bdone, 0);
    }
    fence_before();
    __syncthreads();
    if (warp == kSoftmaxWarps) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
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

bool chunk_supported(const Shape& s) { return s.bf16 && !s.int8 && !s.ring && s.d == kD; }

cudaError_t launch_chunk(kvc_handle* h, const void* q, void* out, int n, cudaStream_t st) {
    const Shape& s = h->sh;
    CUtensorMap tk, tv;
    const cuuint64_t kdims[2] = {(cuuint64_t)s.d, (cuuint64_t)s.B * s.Hkv * s.S};
    const cuuint64_t kstr[1] = {(cuuint64_t)s.d * 2};
    const cuuint32_t kbox[2] = {64, kBN};
    if (!make_tensor_map_bf16(&tk, h->state + h->L.k, 2, kdims, kstr, kbox) ||
        !make_tensor_map_bf16(&tv, h->state + h->L.v, 2, kdims, kstr, kbox))
        return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(chunk_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    // ChunkArgs carries the order table: it lives in static storage, not on the stack
    static thread_local ChunkArgs a;
    a = ChunkArgs{};
    a.next_pos = reinterpret_cast<const int32_t*>(h->state + h->L.next_pos);
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.rope = s.rope ? reinterpret_cast<const float2*>(h->state + h->L.rope) : nullptr;
    a.out = out; a.hdr = reinterpret_cast<uint32_t*>(h->state + h->L.hdr);
    a.B = s.B; a.Hq = s.Hq; a.Hkv = s.Hkv; a.g = s.g; a.S = s.S; a.W = s.W; a.n = n; a.out_bf16 = s.out_bf16;
    a.tiles = (n + kBM - 1) / kBM;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.d));
    // longest first: a (request, tile) item's work is its number of key tiles, from the
    // host mirror of next_position (already advanced past the appended suffix)
    const int items = s.B * a.tiles;
    if (items <= kMaxItems && s.B <= 65536 && a.tiles <= 65536) {
        std::vector<std::pair<int, uint32_t>> w(items);
        for (int b = 0; b < s.B; ++b)
            for (int t = 0; t < a.tiles; ++t) {
                const int cut = h->np[b] - n, i0 = t * kBM, rows = std::min(kBM, n - i0);
                const int p_first = cut + i0, p_last = p_first + rows - 1;
                const int lo = s.W > 0 ? std::max(0, p_first - s.W + 1) : 0;
                w[b * a.tiles + t] = {-((p_last + 1 - lo + kBN - 1) / kBN), ((uint32_t)b << 16) | (uint32_t)t};
            }
        std::stable_sort(w.begin(), w.end(),
                         [](const std::pair<int, uint32_t>& x, const std::pair<int, uint32_t>& y) {
                             return x.first < y.first;
                         });
        for (int i = 0; i < items; ++i) a.items[i] = w[i].second;
        a.n_items = items;
    }
    chunk_attn_kernel<<<dim3(items * s.Hq), kThreads, SMEM_BYTES, st>>>(tk, tv, a);
    return cudaGetLastError();
}

}  // namespace kvc
