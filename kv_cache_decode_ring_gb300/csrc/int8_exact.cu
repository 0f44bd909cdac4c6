// int8_exact.cu -- decode attention over the INT8 blocks restored to full precision.
//
// [WITCERT] "SGLang 生产级落地与闭环门控修复": a block swapped back in from the
// full-precision backing store is lossless, so its tokens carry c_t = 0.  The gated
// fallback (int8_gate.cu) keeps such blocks, bf16 and unchanged, in a pool and lists
// them per (request, KV head); the quantized INT8 decode skips them and this kernel
// serves them.  Its per-split partials (m, l, acc; c = 0) join the INT8 combine.
//
// Kernel shape: CTA = 4 warps = up to 64 listed blocks of one (request, KV head);
// each warp streams 16 of them, one pool entry (16 K rows + 16 V rows, 8 KB at
// d = 128) per bulk copy, through three shared-memory stages.  Both contractions are
// bf16 mma.sync (m16n8k16, fp32 accumulation), operands read in the fragment order
// the pool stores (xk_offset / xv_offset):
//  * scores S^T[16 tokens][cols] = K . Q^T, columns (head, hi | lo) of the rotated
//    query times log2(e)/sqrt(d) split into two bf16 terms;
//  * O^T[d][cols] += V^T . P^T with the weights as bf16 hi + lo.
// Lane L holds the scores and the output of head L % 4 (and 4 + L % 4); the
// reference maximum moves only when a block exceeds it by more than 2^8.
#include <cmath>

#include "async_copy.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kWarps = 4;
constexpr int kTiles = 16;                 // blocks per warp
constexpr int kStages = 3;                 // per warp
constexpr float kLazyMax = 8.f;
static_assert(kWarps * kTiles == kExactBlocksPerCta, "CTA shape");

struct ExactArgs {
    const void* q;
    const __nv_bfloat16* xpool;
    const int32_t* xn;
    const int32_t* xlist;
    const int32_t* xent;
    const int32_t* next_pos;
    const float2* rope;
    float2* part_ml;
    float* part_acc;
    float* part_c;
    float* ct;          // nullable
    uint32_t* hdr;
    int B, Hq, Hkv, d, S, max_splits;
    int split;          // tokens per quantized split of the INT8 decode
    float scale_log2;
};

// D (16x8, fp32) += A (16x16, bf16, row) . B (16x8, bf16, col)
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^x with the hardware approximation (relative error about 2^-22; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi)
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

__device__ __forceinline__ int prow(int n) { return 32 * n + (n >= 4 ? 16 : 0); }

template <int D, int G>
struct XC {
    static constexpr int KS = D / 16;               // k-steps of the scores = m-tiles of P.V
    static constexpr int NT = (2 * G + 7) / 8;      // 8-column tiles of (head, hi|lo) columns
    static constexpr int CPQ = D / 32;              // 16-byte K chunks per (row, lane quad)
    static constexpr int EB = 2 * kQBlock * D * 2;  // bytes of one pool entry
    static constexpr int WARPB = kStages * EB;
    static constexpr int PARTF = G * (D + 3);
    static_assert(PARTF * 4 <= WARPB, "partial must fit in the warp's stages");
    static constexpr int PROWB = 288;               // P^T staging per column tile (see prow)
    static constexpr int OFF_P = kWarps * WARPB;
    static constexpr int PBYTES = kWarps * NT * PROWB > G * D * 4 ? kWarps * NT * PROWB : G * D * 4;
    static constexpr int OFF_QB = OFF_P + ((PBYTES + 15) / 16) * 16;   // bf16 query [2G][D]
    static constexpr int OFF_BAR = OFF_QB + 2 * G * D * 2;
    static constexpr size_t SMEM = OFF_BAR + kWarps * kStages * 8 + 128;
};

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32) int8_exact_kernel(const ExactArgs a) {
    using C = XC<D, G>;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* sPm = smem + C::OFF_P;
    __nv_bfloat16* sQb = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_QB);   // row 2h hi, 2h + 1 lo
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, kvh = blockIdx.y;
    const size_t bh = (size_t)b * a.Hkv + kvh;
    const int nx = a.xn[bh];
    const int base = blockIdx.x * kExactBlocksPerCta;
    if (base >= nx) return;
    const int len = a.next_pos[b];
    const int nfull = len & ~(kQBlock - 1);
    const int split = (nfull + a.split - 1) / a.split + 1 + blockIdx.x;
    const int t_q = len - 1;
    const size_t rowq0 = (size_t)b * a.Hq + (size_t)kvh * G;

    unsigned char* myS = smem + warp * C::WARPB;
    uint64_t* myBar = bar + warp * kStages;
    auto li = [&](int i) { return base + i * kWarps + warp; };             // list index of tile i
    auto tile_ok = [&](int i) { return li(i) < nx; };
    auto issue = [&](int i) {
        if (lane == 0 && tile_ok(i)) {
            const int e = a.xent[bh * kMaxRestored + li(i)];
            const int sg = i % kStages;
            mbar_arrive_expect_tx(&myBar[sg], (uint32_t)C::EB);
            bulk_copy_g2s(myS + sg * C::EB, a.xpool + (size_t)e * (C::EB / 2), C::EB, &myBar[sg]);
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

    // the rotated query times log2(e)/sqrt(d), as bf16 hi + lo rows
    {
        float* qf = reinterpret_cast<float*>(sPm);
        for (int idx = threadIdx.x; idx < G * D / 2; idx += blockDim.x) {
            const int h = idx / (D / 2), i = idx % (D / 2);
            const size_t off = (rowq0 + h) * D + 2 * i;
            const float x0 = ld_elem(a.q, off, 1), x1 = ld_elem(a.q, off + 1, 1);
            float y0 = x0, y1 = x1;
            if (a.rope) rope_pair(x0, x1, a.rope[(size_t)t_q * (D / 2) + i], y0, y1);
            qf[h * D + 2 * i] = y0 * a.scale_log2;
            qf[h * D + 2 * i + 1] = y1 * a.scale_log2;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
            const int h = idx / D, i = idx % D;
            __nv_bfloat16 hi, lo;
            split_bf16(qf[idx], hi, lo);
            sQb[(2 * h) * D + i] = hi;
            sQb[(2 * h + 1) * D + i] = lo;
        }
        __syncthreads();
    }

    const int g = lane >> 2, qd = lane & 3;
    uint32_t qb[C::NT][C::KS][2];                  // Q^T operand: column 8 nt + g, dims qd (D/4) + 4 s ..
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
        const int n = 8 * nt + g;
#pragma unroll
        for (int s = 0; s < C::KS; ++s) {
            uint2 v = make_uint2(0u, 0u);
            if (n < 2 * G) v = *reinterpret_cast<const uint2*>(sQb + n * D + qd * (D / 4) + 4 * s);
            qb[nt][s][0] = v.x;
            qb[nt][s][1] = v.y;
        }
    }
    constexpr int CPR = D / 16;                    // 16-byte V chunks of a lane
    const int vswz = D == 128 ? (lane & 7) : ((lane >> 1) & 3);
    unsigned char* myPm = sPm + warp * C::NT * C::PROWB;
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

    for (int i = 0; i < kTiles; ++i) {
        if (!tile_ok(i)) break;
        const int sg = i % kStages;
        const uint32_t par = (uint32_t)((i / kStages) & 1);
        const unsigned char* tK = myS + sg * C::EB;
        const unsigned char* tV = tK + C::EB / 2;
        if (!mbar_wait(&myBar[sg], par)) {
            if (lane == 0) atomicOr(a.hdr, kErrWait);
            mbar_wait(&myBar[sg], par);
            for (int j = i + 1; j < i + kStages && j < kTiles; ++j)
                if (tile_ok(j)) mbar_wait(&myBar[j % kStages], (uint32_t)((j / kStages) & 1));
            break;
        }
        const int blk = a.xlist[bh * kMaxRestored + li(i)];
        // ---- scores: K rows g and g + 8, chunks CPQ qd .. + CPQ - 1 (swizzled)
        uint32_t kw0[2 * C::CPQ][2], kw1[2 * C::CPQ][2];
#pragma unroll
        for (int j = 0; j < C::CPQ; ++j) {
            const int c = C::CPQ * qd + j;
            const int s0 = D == 128 ? (((c >> 3) << 1) | (g & 1)) : (g & 1);
            const uint4 u0 = *reinterpret_cast<const uint4*>(tK + g * 2 * D + ((c ^ s0) << 4));
            const uint4 u1 = *reinterpret_cast<const uint4*>(tK + (g + 8) * 2 * D + ((c ^ s0) << 4));
            kw0[2 * j][0] = u0.x; kw0[2 * j][1] = u0.y; kw0[2 * j + 1][0] = u0.z; kw0[2 * j + 1][1] = u0.w;
            kw1[2 * j][0] = u1.x; kw1[2 * j][1] = u1.y; kw1[2 * j + 1][0] = u1.z; kw1[2 * j + 1][1] = u1.w;
        }
        float sacc[C::NT][4];
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
        for (int s = 0; s < C::KS; ++s)
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt)
                mma_bf16(sacc[nt], kw0[s][0], kw1[s][0], kw0[s][1], kw1[s][1], qb[nt][s][0], qb[nt][s][1]);
        // ---- online softmax of the lane's heads over tokens g, g + 8
        float alpha[C::NT];
        bool rescale = false;
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
            const float s0 = sacc[nt][0] + sacc[nt][1];
            const float s1 = sacc[nt][2] + sacc[nt][3];
            float bm = fmaxf(s0, s1);
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
            const float mn = bm > m_w[nt] + kLazyMax ? bm : m_w[nt];
            alpha[nt] = ex2(m_w[nt] - mn);            // 0 while the maximum was -inf
            rescale |= alpha[nt] != 1.f;
            m_w[nt] = mn;
            const float e0 = ex2(s0 - mn), e1 = ex2(s1 - mn);
            l_w[nt] = fmaf(l_w[nt], alpha[nt], e0 + e1);
            __nv_bfloat16 h0, l0, h1, l1;
            split_bf16(e0, h0, l0);
            split_bf16(e1, h1, l1);
            unsigned char* pt = myPm + nt * C::PROWB;
            *reinterpret_cast<__nv_bfloat16*>(pt + prow(2 * qd) + 2 * g) = h0;
            *reinterpret_cast<__nv_bfloat16*>(pt + prow(2 * qd + 1) + 2 * g) = l0;
            *reinterpret_cast<__nv_bfloat16*>(pt + prow(2 * qd) + 2 * (g + 8)) = h1;
            *reinterpret_cast<__nv_bfloat16*>(pt + prow(2 * qd + 1) + 2 * (g + 8)) = l1;
        }
        if (a.ct)                                   // restored tokens: c_t = 0
            for (int idx = lane; idx < G * kQBlock; idx += 32)
                a.ct[(rowq0 + idx / kQBlock) * a.S + (size_t)blk * kQBlock + idx % kQBlock] = 0.f;
        if (__any_sync(0xffffffffu, rescale) && i > 0) {
#pragma unroll
            for (int mt = 0; mt < C::KS; ++mt)
#pragma unroll
                for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[mt][nt][e] *= alpha[nt];
        }
        __syncwarp();
        // ---- P.V: O^T += V^T P^T
        uint2 pb[C::NT];
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt)
            pb[nt] = *reinterpret_cast<const uint2*>(myPm + nt * C::PROWB + prow(g) + 8 * qd);
#pragma unroll
        for (int mt = 0; mt < C::KS; ++mt) {
            const uint4 u = *reinterpret_cast<const uint4*>(tV + lane * CPR * 16 + ((mt ^ vswz) << 4));
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt) mma_bf16(acc[mt][nt], u.x, u.z, u.y, u.w, pb[nt].x, pb[nt].y);
        }
        __syncwarp();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (i + kStages < kTiles) issue(i + kStages);
    }

    // ---- this warp's partial, then the CTA's split
    __syncwarp();
    float* part_w = reinterpret_cast<float*>(myS);             // [G][3 + D]
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
        float l = l_w[nt];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        const int hq = 4 * nt + qd;
        if (hq < G) {
#pragma unroll
            for (int mt = 0; mt < C::KS; ++mt) {
                part_w[hq * (D + 3) + 3 + 16 * mt + g] = acc[mt][nt][0] + acc[mt][nt][1];
                part_w[hq * (D + 3) + 3 + 16 * mt + 8 + g] = acc[mt][nt][2] + acc[mt][nt][3];
            }
            if (g == 0) { part_w[hq * (D + 3)] = m_w[nt]; part_w[hq * (D + 3) + 1] = l; }
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int h = idx / D, i = idx % D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            mx = fmaxf(mx, reinterpret_cast<const float*>(smem + w * C::WARPB)[h * (D + 3)]);
        float l = 0.f, sacc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float* pwp = reinterpret_cast<const float*>(smem + w * C::WARPB) + h * (D + 3);
            const float f = pwp[0] == -INFINITY ? 0.f : exp2f(pwp[0] - mx);
            l += pwp[1] * f;
            sacc += pwp[3 + i] * f;
        }
        const size_t row = (rowq0 + h) * a.max_splits + split;
        a.part_acc[row * D + i] = sacc;
        if (i == 0) { a.part_ml[row] = make_float2(mx, l); a.part_c[row] = 0.f; }
    }
}

template <int D, int G>
cudaError_t launch_t(const ExactArgs& a, int nx_ctas, cudaStream_t st) {
    using C = XC<D, G>;
    if (cudaError_t e = allow_smem(reinterpret_cast<const void*>(int8_exact_kernel<D, G>), C::SMEM)) return e;
    int8_exact_kernel<D, G><<<dim3(nx_ctas, a.Hkv, a.B), kWarps * 32, C::SMEM, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_int8_exact(kvc_handle* h, const void* q, float* ct, cudaStream_t st) {
    const Shape& s = h->sh;
    int max_xn = 0;
    for (int v : h->xn_h) max_xn = v > max_xn ? v : max_xn;
    if (max_xn == 0) return cudaSuccess;
    ExactArgs a{};
    a.q = q;
    a.xpool = reinterpret_cast<const __nv_bfloat16*>(h->state + h->L.xpool);
    a.xn = reinterpret_cast<const int32_t*>(h->state + h->L.xn);
    a.xlist = reinterpret_cast<const int32_t*>(h->state + h->L.xlist);
    a.xent = reinterpret_cast<const int32_t*>(h->state + h->L.xent);
    a.next_pos = reinterpret_cast<const int32_t*>(h->state + h->L.next_pos);
    a.rope = s.rope ? reinterpret_cast<const float2*>(h->state + h->L.rope) : nullptr;
    a.part_ml = reinterpret_cast<float2*>(h->state + h->L.part_ml);
    a.part_acc = reinterpret_cast<float*>(h->state + h->L.part_acc);
    a.part_c = reinterpret_cast<float*>(h->state + h->L.part_c);
    a.ct = ct;
    a.hdr = reinterpret_cast<uint32_t*>(h->state + h->L.hdr);
    a.B = s.B; a.Hq = s.Hq; a.Hkv = s.Hkv; a.d = s.d; a.S = s.S; a.max_splits = s.max_splits;
    a.split = s.split;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.d));
    const int nx_ctas = (max_xn + kExactBlocksPerCta - 1) / kExactBlocksPerCta;
#define KVC_CASE(D, G) \
    if (s.d == D && s.g == G) return launch_t<D, G>(a, nx_ctas, st);
    KVC_CASE(128, 1) KVC_CASE(128, 2) KVC_CASE(128, 4) KVC_CASE(128, 8)
    KVC_CASE(64, 1) KVC_CASE(64, 2) KVC_CASE(64, 4) KVC_CASE(64, 8)
#undef KVC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kvc
