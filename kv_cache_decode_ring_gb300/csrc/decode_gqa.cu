// decode_gqa.cu -- split-K decode attention for bf16 caches with 4 or 8 query
// heads per KV head (head_dim 64 or 128), on sm_103a.
//
// Same mathematics as decode.cu ([LOOP] §三 step; [LEAN] §2.1 window mask), with
// the per-split partials (m, l, acc) merged by the combine kernel.
//
// CTA = 4 warps = a split of 1024 keys (2048 for caches whose requests may attend
// to 16384 keys or more).  A warp streams its 16 (32) tiles of 16 keys through
// two shared-memory stages (three CTAs per SM): a tile is d/64 tensor copies of 64 dims x
// 16 rows from K and as many from V, written with the 128-byte swizzle (16-byte
// chunk c of row r at c ^ (r mod 8)), so the 8 row addresses of an ldmatrix fall
// into 8 different bank groups.  Rows past the window's last key are copied too
// (the cache is zero-initialised, so they are finite) and their scores masked.
// Both contractions run on the tensor cores (mma m16n8k16, bf16 operands, fp32
// accumulation), operands loaded straight from the stage with ldmatrix:
//  * scores, transposed: S^T[16 keys][cols] = K[16][d] . Q^T[d][cols], where the
//    columns are (head, hi) and (head, lo): the rotated query times
//    log2(e)/sqrt(d), split into two bf16 parts (about 16 significant bits).
//    Lane L receives the whole scores of head L%4 (and 4 + L%4) for keys L/4 and
//    L/4 + 8;
//  * P.V, transposed: O^T[d][cols] += V^T[d][16] . P^T[16][cols] (V^T by
//    ldmatrix.trans), P as bf16 hi + lo.  Lane L accumulates the same heads it
//    scored, so the online-softmax rescale is local to the lane.
// The reference maximum moves only when a tile exceeds it by more than 2^8 (log2
// domain), so weights stay <= 2^8 and the accumulators are rarely rescaled.
// Every mbarrier wait is bounded (about 1 s); on expiry the device error word is
// set and the split's arithmetic is skipped.
#include "async_copy.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kWarps = 4;
constexpr int kTileKeys = 16;                            // keys per stage
constexpr int kStages = 2;                               // per warp (three CTAs per SM: more warps in flight)
constexpr float kLazyMax = 8.f;                          // log2-domain headroom of the reference maximum
static_assert(kGqaSplit % (kWarps * kTileKeys) == 0 && kGqaSplitLong % (kWarps * kTileKeys) == 0, "split shape");
static_assert(kGqaSplitLong / (kWarps * kTileKeys) <= 32, "a warp's tiles (their pages) fit in its lanes");

// 2^x with the hardware approximation (relative error about 2^-22; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// D (16x8, fp32) += A (16x16, bf16, row) . B (16x8, bf16, col)
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi)
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

template <int D, int G>
struct GqaCfg {
    static constexpr int KS = D / 16;                    // k-steps of the scores = m-tiles of P.V
    static constexpr int NT = (2 * G + 7) / 8;           // 8-column tiles of (head, hi|lo) columns
    static constexpr int NBOX = D / 64;                  // tensor-copy boxes per 16-row tile
    static constexpr int BOXB = kTileKeys * 128;         // bytes of one box (16 rows of 64 bf16)
    static constexpr int HALF = NBOX * BOXB;             // K (or V) rows of one stage
    static constexpr int STAGEB = 2 * HALF;
    static constexpr int WARPB = kStages * STAGEB;
    static constexpr int PARTB = G * (D + 2) * 4;
    static_assert(PARTB <= WARPB, "partial must fit in the warp's stages");
    // P^T staging per warp and column tile: 8 rows (columns) of 16 keys, bf16, 48-byte
    // stride (the lanes' 2-byte stores and 4-byte fragment loads are conflict-free)
    static constexpr int PRSTR = 48;
    static constexpr int PTILE = 8 * PRSTR;
    static constexpr int OFF_P = kWarps * WARPB;                          // [warp][NT] P^T staging
    static constexpr int PBYTES = kWarps * NT * PTILE > G * D * 4 ? kWarps * NT * PTILE : G * D * 4;
    static constexpr int OFF_Q = OFF_P + ((PBYTES + 15) / 16) * 16;      // bf16 query [2G][D]
    static constexpr int OFF_BAR = OFF_Q + 2 * G * D * 2;                 // [warp][stage]
    static constexpr size_t SMEM = OFF_BAR + kWarps * kStages * 8 + 1024;   // + base alignment
    static_assert(HALF % 1024 == 0 && OFF_P % 1024 == 0, "swizzled boxes need 1024-byte alignment");
};

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32, 3)
    decode_gqa_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const DecodeArgs a) {
    using C = GqaCfg<D, G>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* sPm = smem + C::OFF_P;
    __nv_bfloat16* sQb = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_Q);   // row 2h hi, 2h + 1 lo
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
    dep_wait();                                          // launched dependent: see launch_dep
    dep_release();
    const int len = a.next_pos[b];
    int lo, hi;
    key_range(len, a.S, a.W, a.ring, lo, hi);
    // a paged cache aligns its tiles to pages (keys before the window are masked)
    const int lo_t = a.table ? (lo & ~(kPage - 1)) : lo;
    const int kSplit = a.split;                          // keys per CTA
    const int tpw = kSplit / (kWarps * kTileKeys);       // tiles per warp
    const int nsplit = (hi - lo_t + kSplit - 1) / kSplit;
    if (split >= nsplit) return;

    const int head_row0 = (b * a.Hkv + kvh) * a.S;       // tensor-map row of key slot 0 (unpaged)
    unsigned char* myS = smem + warp * C::WARPB;
    uint64_t* myBar = bar + warp * kStages;
    // keys of this warp's tile i: 16 consecutive rows, tiles of the 4 warps interleaved
    auto tile_k0 = [&](int i) { return lo_t + split * kSplit + (i * kWarps + warp) * kTileKeys; };
    auto tile_nk = [&](int i) { return max(0, min(kTileKeys, hi - tile_k0(i))); };
    // paged: lane i holds the page of the warp's tile i (a tile is one page), all loaded in
    // one round trip at the start instead of one table read before each tile's copies
    int tpage = 0;
    if (a.table && lane < tpw && tile_nk(lane) > 0)
        tpage = a.table[(size_t)b * (a.S / kPage) + tile_k0(lane) / kPage];
    // lane 0: the tile's K and V boxes (always 16 full rows) on the stage's barrier;
    // called by the whole warp
    auto issue = [&](int i) {
        const int pg = __shfl_sync(0xffffffffu, tpage, i & 31);
        if (lane == 0 && tile_nk(i) > 0) {
            const int sg = i % kStages;
            unsigned char* st = myS + sg * C::STAGEB;
            // page < 0 is never taken: every slot read is mapped
            const int row = a.table ? ((pg < 0 ? 0 : pg) * a.Hkv + kvh) * kPage : head_row0 + tile_k0(i);
            mbar_arrive_expect_tx(&myBar[sg], (uint32_t)C::STAGEB);
#pragma unroll
            for (int j = 0; j < C::NBOX; ++j) {
                tma_load_2d(st + j * C::BOXB, &tmK, 64 * j, row, &myBar[sg]);
                tma_load_2d(st + C::HALF + j * C::BOXB, &tmV, 64 * j, row, &myBar[sg]);
            }
        }
    };
    if (lane == 0) {
#pragma unroll
        for (int sg = 0; sg < kStages; ++sg) mbar_init(&myBar[sg], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < kStages; ++i) issue(i);

    // the query of the G heads, rotated at t = len - 1, times log2(e)/sqrt(d), as
    // bf16 hi + lo rows (fp32 staging in the P area meanwhile)
    {
        float* qf = reinterpret_cast<float*>(sPm);
        const int t = len - 1;
        for (int idx = threadIdx.x; idx < G * D / 2; idx += blockDim.x) {
            const int h = idx / (D / 2), i = idx % (D / 2);
            const size_t off = ((size_t)b * a.Hq + (size_t)kvh * G + h) * D + 2 * i;
            const float x0 = ld_elem(a.q, off, 1), x1 = ld_elem(a.q, off + 1, 1);
            float y0 = x0, y1 = x1;
            if (a.rope) rope_pair(x0, x1, a.rope[(size_t)t * (D / 2) + i], y0, y1);
            qf[h * D + 2 * i] = y0 * a.scale_log2;
            qf[h * D + 2 * i + 1] = y1 * a.scale_log2;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
            const int h = idx / D, i = idx % D;
            __nv_bfloat16 qh, ql;
            split_bf16(qf[idx], qh, ql);
            sQb[(2 * h) * D + i] = qh;
            sQb[(2 * h + 1) * D + i] = ql;
        }
        __syncthreads();
    }

    // ---- per-lane fragments: g = L/4 (MMA group), qd = L%4
    const int g = lane >> 2, qd = lane & 3;
    uint32_t qb[C::NT][C::KS][2];                 // Q^T operand: column 8 nt + g, k-step s
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
        for (int s = 0; s < C::KS; ++s) {
            const __nv_bfloat16* row = sQb + (8 * nt + g) * D + 16 * s + 2 * qd;
            qb[nt][s][0] = *reinterpret_cast<const uint32_t*>(row);
            qb[nt][s][1] = *reinterpret_cast<const uint32_t*>(row + 8);
        }
    // ldmatrix row addresses: matrix mi = lane / 8 supplies row rr = lane % 8 (+ 8);
    // 16-byte chunk c of a row sits at c ^ rr
    const int mi = lane >> 3, rr = lane & 7;
    const uint32_t krow = (uint32_t)((rr + 8 * (mi & 1)) * 128), kch = (uint32_t)(mi >> 1);
    const uint32_t vrow = (uint32_t)((rr + 8 * (mi >> 1)) * 128), vch = (uint32_t)(mi & 1);
    unsigned char* myPm = sPm + warp * C::NT * C::PTILE;

    float m_w[C::NT], l_w[C::NT];
    float acc[C::KS][C::NT][4];
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) { m_w[nt] = -INFINITY; l_w[nt] = 0.f; }
#pragma unroll
    for (int mt = 0; mt < C::KS; ++mt)
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;

    for (int i = 0; i < tpw; ++i) {
        const int nk = tile_nk(i);
        if (nk == 0) break;                       // later tiles of this warp are empty too
        const int kmin = lo - tile_k0(i);         // keys of the tile before the window
        const int sg = i % kStages;
        const uint32_t par = (uint32_t)((i / kStages) & 1);
        unsigned char* tK = myS + sg * C::STAGEB;
        unsigned char* tV = tK + C::HALF;
        if (!mbar_wait(&myBar[sg], par)) {
            // give up: flag it, and let this stage's copy and the later stages'
            // (if issued) land before the stages are reused for the partial
            if (lane == 0) atomicOr(a.hdr, kErrWait);
            mbar_wait(&myBar[sg], par);
            for (int j = i + 1; j < i + kStages && j < tpw; ++j)
                if (tile_nk(j) > 0) mbar_wait(&myBar[j % kStages], (uint32_t)((j / kStages) & 1));
            break;
        }
        // ---- scores S^T = K Q^T
        const uint32_t kbase = smem_u32(tK) + krow;
        float sacc[C::NT][4];
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
        for (int s = 0; s < C::KS; ++s) {
            uint32_t af[4];
            ldsm_x4(af, kbase + (s >> 2) * C::BOXB + (((uint32_t)(((s & 3) << 1)) + kch) ^ (uint32_t)rr) * 16);
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt) mma_bf16(sacc[nt], af, qb[nt][s][0], qb[nt][s][1]);
        }
        // ---- online softmax of the lane's heads over keys g, g + 8; weights into the
        // P^T staging as bf16 hi + lo
        float alpha[C::NT];
        bool rescale = false;
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
            const float s0 = g < nk && g >= kmin ? sacc[nt][0] + sacc[nt][1] : -INFINITY;
            const float s1 = g + 8 < nk && g + 8 >= kmin ? sacc[nt][2] + sacc[nt][3] : -INFINITY;
            float bm = fmaxf(s0, s1);
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
            const float mn = bm > m_w[nt] + kLazyMax ? bm : m_w[nt];
            alpha[nt] = ex2(m_w[nt] - mn);            // 0 while the maximum was -inf
            rescale |= alpha[nt] != 1.f;
            m_w[nt] = mn;
            const float e0 = ex2(s0 - mn), e1 = ex2(s1 - mn);     // masked keys: 0
            l_w[nt] = fmaf(l_w[nt], alpha[nt], e0 + e1);
            __nv_bfloat16 h0, l0, h1, l1;
            split_bf16(e0, h0, l0);
            split_bf16(e1, h1, l1);
            unsigned char* pt = myPm + nt * C::PTILE;
            *reinterpret_cast<__nv_bfloat16*>(pt + (2 * qd) * C::PRSTR + 2 * g) = h0;
            *reinterpret_cast<__nv_bfloat16*>(pt + (2 * qd + 1) * C::PRSTR + 2 * g) = l0;
            *reinterpret_cast<__nv_bfloat16*>(pt + (2 * qd) * C::PRSTR + 2 * (g + 8)) = h1;
            *reinterpret_cast<__nv_bfloat16*>(pt + (2 * qd + 1) * C::PRSTR + 2 * (g + 8)) = l1;
        }
        if (__any_sync(0xffffffffu, rescale) && i > 0) {     // at i = 0 the accumulators are 0
#pragma unroll
            for (int mt = 0; mt < C::KS; ++mt)
#pragma unroll
                for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[mt][nt][e] *= alpha[nt];
        }
        __syncwarp();
        // ---- P.V: O^T += V^T P^T; B operand = P^T column g, keys 2 qd, +1 and 2 qd + 8, +9
        uint32_t pb[C::NT][2];
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
            const unsigned char* pr = myPm + nt * C::PTILE + g * C::PRSTR + 4 * qd;
            pb[nt][0] = *reinterpret_cast<const uint32_t*>(pr);
            pb[nt][1] = *reinterpret_cast<const uint32_t*>(pr + 16);
        }
        const uint32_t vbase = smem_u32(tV) + vrow;
#pragma unroll
        for (int mt = 0; mt < C::KS; ++mt) {
            uint32_t af[4];
            ldsm_x4_trans(af, vbase + (mt >> 2) * C::BOXB + (((uint32_t)(((mt & 3) << 1)) + vch) ^ (uint32_t)rr) * 16);
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt) mma_bf16(acc[mt][nt], af, pb[nt][0], pb[nt][1]);
        }
        // this stage and the staging are free once every lane is past its reads
        __syncwarp();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (i + kStages < tpw) issue(i + kStages);
    }

    // ---- this warp's partial into its own stage buffers (every issued tile was
    // waited for): l summed over the 8 lanes of a head; output = hi + lo columns
    __syncwarp();
    float* part_w = reinterpret_cast<float*>(myS);        // [G][2 + D]
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
        float l = l_w[nt];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        const int h = 4 * nt + qd;
#pragma unroll
        for (int mt = 0; mt < C::KS; ++mt) {
            part_w[h * (D + 2) + 2 + 16 * mt + g] = acc[mt][nt][0] + acc[mt][nt][1];
            part_w[h * (D + 2) + 2 + 16 * mt + 8 + g] = acc[mt][nt][2] + acc[mt][nt][3];
        }
        if (g == 0) { part_w[h * (D + 2)] = m_w[nt]; part_w[h * (D + 2) + 1] = l; }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int h = idx / D, i = idx % D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            mx = fmaxf(mx, reinterpret_cast<const float*>(smem + w * C::WARPB)[h * (D + 2)]);
        float l = 0.f, sacc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float* pw = reinterpret_cast<const float*>(smem + w * C::WARPB) + h * (D + 2);
            const float f = pw[0] == -INFINITY ? 0.f : exp2f(pw[0] - mx);
            l += pw[1] * f;
            sacc += pw[2 + i] * f;
        }
        const size_t row = ((size_t)b * a.Hq + (size_t)kvh * G + h) * a.max_splits + split;
        a.part_acc[row * D + i] = sacc;
        if (i == 0) a.part_ml[row] = make_float2(mx, l);
    }
}

template <int D, int G>
cudaError_t launch_t(const DecodeArgs& a, const KvMaps& m, cudaStream_t st) {
    using C = GqaCfg<D, G>;
    if (cudaError_t e = allow_smem(reinterpret_cast<const void*>(decode_gqa_kernel<D, G>), C::SMEM)) return e;
    return launch_dep(decode_gqa_kernel<D, G>, dim3(a.max_splits, a.Hkv, a.B), dim3(kWarps * 32), C::SMEM, st,
                      m.k, m.v, a);
}

}  // namespace

bool gqa_decode_supported(int d, int g) { return (d == 64 || d == 128) && (g == 4 || g == 8); }

cudaError_t launch_decode_gqa(const DecodeArgs& a, const KvMaps& m, cudaStream_t st) {
#define KVC_CASE(D, G) \
    if (a.d == D && a.g == G) return launch_t<D, G>(a, m, st);
    KVC_CASE(128, 4) KVC_CASE(128, 8) KVC_CASE(64, 4) KVC_CASE(64, 8)
#undef KVC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kvc
