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
//  * Q, K, V tiles arrive by TMA (128-byte swizzle); three K and three V stages;
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

#include <cmath>
#include <mutex>

#include "async_copy.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kBM = 128;          // query rows per CTA
constexpr int kBN = 64;           // keys per tile
constexpr int kD = 128;           // head dim of this kernel
constexpr int kSoftmaxWarps = 8;   // two per tensor-memory lane group
constexpr int kThreads = (kSoftmaxWarps + 1) * 32;   // + one producer warp
constexpr int kStages = 3;        // K and V tile stages
constexpr float kLazyMax = 8.f;   // log2-domain headroom of a row's reference maximum
constexpr int kQTile = kBM * kD * 2;     // 32 KB: two 64-dim halves of [128 rows][128 B]
constexpr int kQHalf = kQTile / 2;
constexpr int kKVTile = kBN * kD * 2;    // 16 KB: two 64-dim halves of [64 rows][128 B]
constexpr int kKVHalf = kKVTile / 2;
constexpr int kPTile = kBM * kBN * 2;    // 16 KB: [128 rows][64 keys] bf16, one 128-B swizzle column
// Operands that are not exact bf16 (the rotated query and the softmax weights)
// enter the MMAs as two bf16 terms, hi = bf16(x) and lo = bf16(x - hi), both
// accumulated in fp32: about 16 significant bits instead of 8.
constexpr int OFF_Q = 0;                          // Q hi
constexpr int OFF_QLO = OFF_Q + kQTile;           // Q lo
constexpr int OFF_K = OFF_QLO + kQTile;           // kStages K tiles
constexpr int OFF_V = OFF_K + kStages * kKVTile;  // kStages V tiles
constexpr int OFF_P = OFF_V + kStages * kKVTile;  // 2 buffers of (P hi, P lo)
constexpr int OFF_BAR = OFF_P + 4 * kPTile;       // q, k[3], v[3], s[2], o[2], p[2], done
constexpr int kBars = 14;
constexpr int OFF_MISC = OFF_BAR + 8 * kBars;     // tensor memory base, abort flag
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory per block");
constexpr uint32_t kTmemCols = 256;               // S buffers: [0, 64), [64, 128); O: [128, 256)

struct ChunkArgs {
    const int32_t* next_pos;   // after the append: cut + n
    void* out;                 // [B][n][Hq][d]
    uint32_t* hdr;
    int B, Hq, Hkv, g, S, W, n, out_bf16;
    float scale_log2;
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

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, int acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
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

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    chunk_attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQlo,
                      const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const ChunkArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* sQ = smem + OFF_Q;
    unsigned char* sQlo = smem + OFF_QLO;
    unsigned char* sK = smem + OFF_K;
    unsigned char* sV = smem + OFF_V;
    unsigned char* sP = smem + OFF_P;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* bq = bar;          // Q landed
    uint64_t* bk = bar + 1;      // [stage] K tile landed
    uint64_t* bv = bar + 4;      // [stage] V tile landed
    uint64_t* bs = bar + 7;      // [buffer] S = Q K^T complete
    uint64_t* bo = bar + 9;      // [buffer] O += P V complete (P buffer and V stage free again)
    uint64_t* bp = bar + 11;     // [buffer] P written and S read by the 8 softmax warps
    uint64_t* bdone = bar + 13;  // every MMA issued so far complete (abort path)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, hq = blockIdx.y, i0 = blockIdx.x * kBM;
    const int kvh = hq / a.g;
    const int np = a.next_pos[b];
    const int cut = np - a.n;
    const int rows = min(kBM, a.n - i0);
    const int p_first = cut + i0, p_last = cut + i0 + rows - 1;
    const int lo = a.W > 0 ? max(0, p_first - a.W + 1) : 0;
    const int ntiles = (p_last + 1 - lo + kBN - 1) / kBN;
    const int head_row0 = (b * a.Hkv + kvh) * a.S;

    if (tid == 0) {
        for (int i = 0; i < kBars; ++i) mbar_init(&bar[i], i == 11 || i == 12 ? kSoftmaxWarps : 1);
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
    const uint32_t tO = tmem + 128;

    if (warp == kSoftmaxWarps) {
        // ================= producer: one thread issues every copy and every MMA
        if (lane == 0) {
            constexpr uint32_t idesc_qk = instr_desc(kBM, kBN, false);
            constexpr uint32_t idesc_pv = instr_desc(kBM, kD, true);
            auto kbase_of = [&](int j) { return p_last + 1 - kBN * (j + 1); };
            auto load_k = [&](int j) {
                const int st = j % kStages;
                mbar_arrive_expect_tx(&bk[st], kKVTile);
                tma_load_2d(sK + st * kKVTile, &tmK, 0, head_row0 + kbase_of(j), &bk[st]);
                tma_load_2d(sK + st * kKVTile + kKVHalf, &tmK, 64, head_row0 + kbase_of(j), &bk[st]);
            };
            auto load_v = [&](int j) {
                const int st = j % kStages;
                mbar_arrive_expect_tx(&bv[st], kKVTile);
                tma_load_2d(sV + st * kKVTile, &tmV, 0, head_row0 + kbase_of(j), &bv[st]);
                tma_load_2d(sV + st * kKVTile + kKVHalf, &tmV, 64, head_row0 + kbase_of(j), &bv[st]);
            };
            // S_j = Q_hi K_j^T + Q_lo K_j^T into S buffer j % 2
            auto issue_s = [&](int j) {
                const uint32_t q0 = smem_u32(sQ), q1 = smem_u32(sQlo), k0 = smem_u32(sK + (j % kStages) * kKVTile);
                const uint32_t d = tmem + 64 * (j & 1);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s) {
                    const uint32_t oq = (s >> 2) * kQHalf + (s & 3) * 32, ok = (s >> 2) * kKVHalf + (s & 3) * 32;
                    mma_bf16(d, smem_desc(q0 + oq, 16), smem_desc(k0 + ok, 16), idesc_qk, s > 0);
                }
#pragma unroll
                for (int s = 0; s < kD / 16; ++s) {
                    const uint32_t oq = (s >> 2) * kQHalf + (s & 3) * 32, ok = (s >> 2) * kKVHalf + (s & 3) * 32;
                    mma_bf16(d, smem_desc(q1 + oq, 16), smem_desc(k0 + ok, 16), idesc_qk, 1);
                }
                mma_commit(&bs[j & 1]);
            };
            // O += P_hi V_j + P_lo V_j (P buffer j % 2)
            auto issue_pv = [&](int j) {
                const uint32_t ph = smem_u32(sP + (j & 1) * 2 * kPTile), pl = ph + kPTile;
                const uint32_t v0 = smem_u32(sV + (j % kStages) * kKVTile);
#pragma unroll
                for (int s2 = 0; s2 < kBN / 16; ++s2)
                    mma_bf16(tO, smem_desc(ph + s2 * 32, 16), smem_desc(v0 + s2 * 2048, kKVHalf), idesc_pv,
                             (j > 0 || s2 > 0));
#pragma unroll
                for (int s2 = 0; s2 < kBN / 16; ++s2)
                    mma_bf16(tO, smem_desc(pl + s2 * 32, 16), smem_desc(v0 + s2 * 2048, kKVHalf), idesc_pv, 1);
                mma_commit(&bo[j & 1]);
            };

            bool ok = true;
            // copies issued and awaited so far (an abort drains the rest before exit)
            int k_issued = 0, v_issued = 0, k_waited = 0, v_waited = 0;
            bool q_waited = false;
            mbar_arrive_expect_tx(bq, 2 * kQTile);
            tma_load_3d(sQ, &tmQ, 0, hq, b * a.n + i0, bq);
            tma_load_3d(sQ + kQHalf, &tmQ, 64, hq, b * a.n + i0, bq);
            tma_load_3d(sQlo, &tmQlo, 0, hq, b * a.n + i0, bq);
            tma_load_3d(sQlo + kQHalf, &tmQlo, 64, hq, b * a.n + i0, bq);
            for (int j = 0; j < kStages && j < ntiles; ++j) { load_k(j); load_v(j); k_issued = v_issued = j + 1; }
            ok = q_waited = mbar_wait(bq, 0);
            for (int j = 0; j < 2 && j < ntiles && ok; ++j) {
                ok = mbar_wait(&bk[j], 0);
                if (ok) { k_waited = j + 1; fence_after(); issue_s(j); }
            }
            for (int j = 0; j < ntiles && ok; ++j) {
                if (*abort_flag) { ok = false; break; }
                // K stage of tile j is free once S_j is complete: fetch tile j + kStages
                ok = mbar_wait(&bs[j & 1], (uint32_t)((j >> 1) & 1));
                if (!ok) break;
                if (j + kStages < ntiles) { load_k(j + kStages); k_issued = j + kStages + 1; }
                // V stage of tile j - 2 is free once its P V is complete: fetch tile j + 1
                if (j >= 2 && j + 1 < ntiles) {
                    ok = mbar_wait(&bo[j & 1], (uint32_t)(((j - 2) >> 1) & 1));
                    if (!ok) break;
                    load_v(j + 1);
                    v_issued = j + 2;
                }
                // O += P_j V_j once the softmax warps wrote P_j and V_j landed
                ok = mbar_wait(&bp[j & 1], (uint32_t)((j >> 1) & 1)) &&
                     mbar_wait(&bv[j % kStages], (uint32_t)((j / kStages) & 1));
                if (!ok) break;
                v_waited = j + 1;
                fence_after();
                issue_pv(j);
                // S_{j+2} into S buffer j % 2 (read by the softmax warps: bp above)
                if (j + 2 < ntiles) {
                    ok = mbar_wait(&bk[(j + 2) % kStages], (uint32_t)(((j + 2) / kStages) & 1));
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
                if (!q_waited) mbar_wait(bq, 0);
                for (int t = k_waited; t < k_issued; ++t) mbar_wait(&bk[t % kStages], (uint32_t)((t / kStages) & 1));
                for (int t = v_waited; t < v_issued; ++t) mbar_wait(&bv[t % kStages], (uint32_t)((t / kStages) & 1));
            }
        }
    } else {
        // ================= softmax warps: warp w serves rows 32 (w % 4) .. + 31 (its
        // tensor-memory lanes) and keys 32 (w / 4) .. + 31 of every tile
        const int lg = warp & 3, hf = warp >> 2;
        const int row = 32 * lg + lane;            // query row = tensor-memory lane
        const uint32_t lane_off = (uint32_t)(32 * lg) << 16;
        const int p = cut + i0 + row;               // its absolute position
        const bool row_valid = row < rows;
        const int key_lo = a.W > 0 ? max(0, p - a.W + 1) : 0;
        const int key_lo_max = a.W > 0 ? max(0, p_last - a.W + 1) : 0;   // the CTA's largest key_lo
        float m_ref = -INFINITY, l = 0.f;
        bool fail = false;
        for (int j = 0; j < ntiles; ++j) {
            bool w = mbar_wait(&bs[j & 1], (uint32_t)((j >> 1) & 1)) && !*abort_flag;
            if (!__all_sync(0xffffffffu, w)) { fail = true; break; }
            fence_after();
            // both warps of a row pair read the whole tile, so they agree on its maximum
            float sm[kBN / 2], so[kBN / 2];
            const uint32_t tSj = tmem + 64 * (j & 1) + lane_off;
            tmem_ld32(tSj + 32 * hf, sm);
            tmem_ld32(tSj + 32 * (1 - hf), so);
            const int kb = p_last + 1 - kBN * (j + 1);
            const int km = kb + 32 * hf, ko = kb + 32 * (1 - hf);    // first key of each half
            float mx = -INFINITY;
            if (kb >= key_lo_max && kb + kBN - 1 <= p_first) {
                // every key of the tile is visible to every row of the CTA
#pragma unroll
                for (int c = 0; c < kBN / 2; ++c) mx = fmaxf(mx, fmaxf(sm[c], so[c]));
            } else {
#pragma unroll
                for (int c = 0; c < kBN / 2; ++c) {
                    const bool vm = row_valid && km + c >= key_lo && km + c <= p;
                    const bool vo = row_valid && ko + c >= key_lo && ko + c <= p;
                    sm[c] = vm ? sm[c] : -INFINITY;
                    mx = fmaxf(mx, fmaxf(sm[c], vo ? so[c] : -INFINITY));
                }
            }
            // the reference maximum moves only when the tile exceeds it by more than kLazyMax
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
            // P buffer j % 2 was last read by P V of tile j - 2; O may be rescaled only
            // once P V of tile j - 1 is complete (tcgen05.ld/st: whole warps)
            const bool any_grow = __any_sync(0xffffffffu, grow);
            bool w2 = j < 2 || mbar_wait(&bo[j & 1], (uint32_t)(((j - 2) >> 1) & 1));
            if (any_grow) w2 = w2 && mbar_wait(&bo[(j - 1) & 1], (uint32_t)(((j - 1) >> 1) & 1));
            if (!__all_sync(0xffffffffu, w2)) { fail = true; break; }
            if (any_grow) {
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
            // this warp's 32 keys of the P row -> shared memory as hi and lo bf16 terms,
            // K-major 128-byte swizzle
            unsigned char* sPhi = sP + (j & 1) * 2 * kPTile;
#pragma unroll
            for (int c = 0; c < kBN / 16; ++c) {
                uint32_t hi[4], lo2[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x = make_float2(sm[8 * c + 2 * e], sm[8 * c + 2 * e + 1]);
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(x.x, x.y);
                    const float2 r = __ffma2_rn(__bfloat1622float2(h2), make_float2(-1.f, -1.f), x);   // x - hi, exact
                    hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
                    lo2[e] = pack_bf16(r.x, r.y);
                }
                const int off = row * 128 + (((4 * hf + c) ^ (row & 7)) * 16);
                *reinterpret_cast<uint4*>(sPhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(sPhi + kPTile + off) = make_uint4(lo2[0], lo2[1], lo2[2], lo2[3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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
        // partial row sums meet in the (now idle) K stages
        reinterpret_cast<float*>(sK)[hf * kBM + row] = l;
    }
    __syncthreads();
    const bool aborted = *abort_flag != 0;
    if (warp < kSoftmaxWarps && !aborted) {
        // ---- epilogue: O / l; warp w stores columns 64 (w / 4) .. + 63 of its rows
        const int lg = warp & 3, hf = warp >> 2;
        const int row = 32 * lg + lane;
        const uint32_t lane_off = (uint32_t)(32 * lg) << 16;
        fence_after();
        const float L = reinterpret_cast<const float*>(sK)[row] + reinterpret_cast<const float*>(sK)[kBM + row];
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

// Query rows rotated at their positions (fp32 rule of the cache keys), times
// log2(e)/sqrt(d) (so that Q K^T is the logit in the log2 domain), split into
// bf16 hi = bf16(y) and lo = bf16(y - hi).
__global__ void rope_q_kernel(const __nv_bfloat16* q, __nv_bfloat16* qr, __nv_bfloat16* qlo,
                              const int32_t* next_pos, const float2* rope, int n, int Hq, int d, float scale) {
    const int b = blockIdx.y;
    const int cut = next_pos[b] - n;
    const size_t per_b = (size_t)n * Hq * (d / 2);
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < per_b; idx += (size_t)gridDim.x * blockDim.x) {
        const int i = (int)(idx / ((size_t)Hq * (d / 2)));
        const int pr = (int)(idx % (d / 2));
        const size_t off = (size_t)b * n * Hq * d + idx * 2;
        const float x0 = __bfloat162float(q[off]), x1 = __bfloat162float(q[off + 1]);
        float y0 = x0, y1 = x1;
        if (rope) rope_pair(x0, x1, rope[(size_t)(cut + i) * (d / 2) + pr], y0, y1);
        y0 *= scale;
        y1 *= scale;
        const __nv_bfloat16 h0 = __float2bfloat16_rn(y0), h1 = __float2bfloat16_rn(y1);
        qr[off] = h0;
        qr[off + 1] = h1;
        qlo[off] = __float2bfloat16_rn(y0 - __bfloat162float(h0));
        qlo[off + 1] = __float2bfloat16_rn(y1 - __bfloat162float(h1));
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
    __nv_bfloat16* qr = reinterpret_cast<__nv_bfloat16*>(h->state + h->L.qrot);
    __nv_bfloat16* qlo = qr + (size_t)s.B * s.max_chunk * s.Hq * s.d;
    const int32_t* np = reinterpret_cast<const int32_t*>(h->state + h->L.next_pos);
    const float2* rope = s.rope ? reinterpret_cast<const float2*>(h->state + h->L.rope) : nullptr;
    const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.d));
    rope_q_kernel<<<dim3(128, s.B), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(q), qr, qlo, np, rope, n, s.Hq,
                                                  s.d, scale_log2);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    CUtensorMap tq, tql, tk, tv;
    const cuuint64_t qdims[3] = {(cuuint64_t)s.d, (cuuint64_t)s.Hq, (cuuint64_t)s.B * n};
    const cuuint64_t qstr[2] = {(cuuint64_t)s.d * 2, (cuuint64_t)s.Hq * s.d * 2};
    const cuuint32_t qbox[3] = {64, 1, kBM};
    const cuuint64_t kdims[2] = {(cuuint64_t)s.d, (cuuint64_t)s.B * s.Hkv * s.S};
    const cuuint64_t kstr[1] = {(cuuint64_t)s.d * 2};
    const cuuint32_t kbox[2] = {64, kBN};
    if (!make_tensor_map_bf16(&tq, qr, 3, qdims, qstr, qbox) || !make_tensor_map_bf16(&tql, qlo, 3, qdims, qstr, qbox) ||
        !make_tensor_map_bf16(&tk, h->state + h->L.k, 2, kdims, kstr, kbox) ||
        !make_tensor_map_bf16(&tv, h->state + h->L.v, 2, kdims, kstr, kbox))
        return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        e = cudaFuncSetAttribute(chunk_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    ChunkArgs a{};
    a.next_pos = np; a.out = out; a.hdr = reinterpret_cast<uint32_t*>(h->state + h->L.hdr);
    a.B = s.B; a.Hq = s.Hq; a.Hkv = s.Hkv; a.g = s.g; a.S = s.S; a.W = s.W; a.n = n; a.out_bf16 = s.out_bf16;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.d));
    chunk_attn_kernel<<<dim3((n + kBM - 1) / kBM, s.Hq, s.B), kThreads, SMEM_BYTES, st>>>(tq, tql, tk, tv, a);
    return cudaGetLastError();
}

}  // namespace kvc
