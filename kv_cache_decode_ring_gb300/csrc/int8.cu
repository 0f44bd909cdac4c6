// int8.cu -- fused INT8 decode attention with the witness bound.
//
// [WITCERT] "频带酉性与双层证书": for every cached token t the decode step also
// returns c_t = (1/sqrt d) sum_b ||q_b|| w_{t,b} >= |q . r_t| / sqrt(d), the
// largest logit perturbation the quantization residual r_t can cause, and per
// query head tanh(max_t c_t) >= the attention total variation
// ("为什么在线监控 KV 误差如此困难？": TV <= tanh(max |eps|)).
// "SGLang 生产级落地与闭环门控修复": per-block scales are token-independent, so
// they fold into scalars: the score of key t in block m is s_K[m] (q . code_t),
// and block m contributes s_V[m] sum_t p_t code_t to the output.
//
// Layout read per (request, KV head): K codes int8 [S][d], V codes int8 per
// 16-token block dim-major [S/16][d][16], scales fp32 [S/16], witnesses fp16
// [S][16], exact bf16 tail [16][d] for the rows of the incomplete block.
//
// Kernel shape: CTA = 4 warps = a split of 256 tokens (16 blocks); each warp
// streams its 4 blocks through two shared-memory stages (codes and witnesses by
// bulk copy on the stage's mbarrier), so copies overlap arithmetic; online
// softmax over the warp's blocks, warps merged at the end.  One extra split
// handles the exact tail rows (c_t = 0 there).
//
// Arithmetic, chosen to spend few instructions per cached byte:
//  * scores: the rotated fp32 query of each head is carried as a 16-bit
//    integer q ~ s_q (256 hi + lo) (s_q = max|q| / 32767, round to nearest);
//    dp4a on the raw K codes gives the exact int32 dot product per head, then
//    one multiply by s_q * s_K * log2(e)/sqrt(d);
//  * P.V: per block and head the weights are carried as 16-bit integers
//    relative to the block's largest weight, and dp4a over 4 tokens of one dim
//    at a time (the dim-major V layout) gives the exact int32 block sum, scaled
//    back by max_p * s_V / 32767 into fp32 accumulators;
//  * the bound with every operation rounded toward +inf from the fp32 query
//    (band norms, products with the witnesses, their sum, an upward 1/sqrt(d));
//    tanh gets two ulps of headroom over CUDA tanhf's documented error.
// The integer query and weights change the output by about 2^-16 relative,
// far inside the bf16 tolerance; the bound is evaluated with the fp32 query.
#include <cmath>

#include "async_copy.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kWarps = 4;
constexpr int kTilesPerWarp = 4;           // one 16-token block per tile
static_assert(kWarps * kTilesPerWarp * kQBlock == kInt8Split, "split shape");

struct Int8Args {
    const void* q;
    const int8_t* kq;
    const int8_t* vq;
    const float* sk;
    const float* sv;
    const __half* wit;
    const __nv_bfloat16* ktail;
    const __nv_bfloat16* vtail;
    const int32_t* next_pos;
    const float2* rope;
    float2* part_ml;
    float* part_acc;
    float* part_c;
    float* ct;          // nullable: c_t per token [B][Hq][S]
    uint32_t* hdr;
    int B, Hq, Hkv, d, S, max_splits;
    float scale_log2;   // log2(e)/sqrt(d)
    float inv_sqrt_d_up;
};

struct Int8CombineArgs {
    const float2* part_ml;
    const float* part_acc;
    const float* part_c;
    const int32_t* next_pos;
    void* out;
    float* cmax;        // nullable
    float* tanh_out;    // nullable
    int B, Hq, d, max_splits, out_bf16;
};

// dp4a with unsigned bytes in a and signed bytes in b
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

template <int D, int G>
struct I8 {
    static constexpr int LPR = D / 16;            // score lanes per row, 16 codes each
    static constexpr int RPP = 32 / LPR;          // key groups per warp for the scores
    static constexpr int KPG = kQBlock / RPP;     // keys per group per block
    static constexpr int KB0 = 2 * LPR / G;
    static constexpr int KB = KB0 < KPG ? (KB0 < 1 ? 1 : KB0) : KPG;
    static constexpr int M = KB * G;              // int32 partial scores per lane per batch
    // finished scores per lane per batch; with fewer partials than lanes (M < LPR) the
    // last reduction steps are all-reduces and LPR/M lanes share each score
    static constexpr int OUT = M >= LPR ? M / LPR : 1;
    static constexpr int SHARE = M >= LPR ? 1 : LPR / M;
    static constexpr int DPL = D / 32;            // output dims per lane for P.V
    static constexpr int CB = kQBlock * D;        // bytes of one block's codes (K or V)
    static constexpr int WB = kQBlock * kBands * 2;
    static constexpr int STAGEB = 2 * CB + WB;
    static constexpr int WARPB = 2 * STAGEB;
    static constexpr int PARTF = G * (D + 3);     // floats of one warp's partial (m, l, c, acc)
    static_assert(KPG >= 1 && (M % LPR == 0 || LPR % M == 0), "batch shape");
    static_assert(PARTF * 4 <= WARPB, "partial must fit in the warp's stages");
    // after the warps' stages: scores [warp][16][G] (the fp32 query during preparation),
    // weight bytes [warp][G][2][16], query bytes [2][G][D/4] words, band norms [G][16],
    // score factors [G], barriers [warp][2]
    static constexpr int OFF_P = kWarps * WARPB;
    static constexpr int PBYTES = (kWarps * kQBlock * G > G * D ? kWarps * kQBlock * G : G * D) * 4;
    static constexpr int OFF_PW = OFF_P + PBYTES;
    static constexpr int OFF_QW = OFF_PW + kWarps * G * 2 * kQBlock;
    static constexpr int OFF_NQ = OFF_QW + 2 * G * (D / 4) * 4;
    static constexpr int OFF_F = OFF_NQ + G * kBands * 4;
    static constexpr int OFF_BAR = OFF_F + ((G * 4 + 15) / 16) * 16;
    static constexpr size_t SMEM = OFF_BAR + kWarps * 2 * 8 + 128;
};

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32, G >= 8 ? (D >= 128 ? 2 : 3) : 4) int8_decode_kernel(const Int8Args a) {
    using C = I8<D, G>;
    extern __shared__ __align__(128) unsigned char smem[];
    float* sP = reinterpret_cast<float*>(smem + C::OFF_P);              // [warp][16][G]
    unsigned char* sPW = smem + C::OFF_PW;                               // [warp][G][2][16] weight bytes
    uint32_t* sQW = reinterpret_cast<uint32_t*>(smem + C::OFF_QW);      // [2][G][D/4] query bytes
    float* sNQ = reinterpret_cast<float*>(smem + C::OFF_NQ);            // [G][16] band norms
    float* sF = reinterpret_cast<float*>(smem + C::OFF_F);              // [G] score factors
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);     // [warp][2]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
    const int len = a.next_pos[b];
    const int nfull = len & ~(kQBlock - 1);
    const int nsq = (nfull + kInt8Split - 1) / kInt8Split;
    const bool tail_split = split == nsq;
    if (split > nsq || (tail_split && len == nfull)) return;
    const int t_q = len - 1;
    const size_t rowq0 = (size_t)b * a.Hq + (size_t)kvh * G;    // first query row of the group

    if (tail_split) {
        // ---- exact bf16 tail rows [nfull, len): warp 0, lane = row; c_t = 0
        if (warp != 0) return;
        const int nt = len - nfull;
        float* qs = reinterpret_cast<float*>(smem);          // [G][D] scaled query
        float* pt = qs + G * D;                              // [16][G]
        for (int idx = lane; idx < G * D / 2; idx += 32) {
            const int h = idx / (D / 2), i = idx % (D / 2);
            const size_t off = (rowq0 + h) * D + 2 * i;
            const float x0 = ld_elem(a.q, off, 1), x1 = ld_elem(a.q, off + 1, 1);
            float y0 = x0, y1 = x1;
            if (a.rope) rope_pair(x0, x1, a.rope[(size_t)t_q * (D / 2) + i], y0, y1);
            qs[h * D + 2 * i] = y0 * a.scale_log2;
            qs[h * D + 2 * i + 1] = y1 * a.scale_log2;
        }
        __syncwarp();
        const size_t tail0 = ((size_t)b * a.Hkv + kvh) * kQBlock * D;
        float s[G];
#pragma unroll
        for (int h = 0; h < G; ++h) s[h] = -INFINITY;
        if (lane < nt) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float acc = 0.f;
                for (int i = 0; i < D; ++i) acc = fmaf(qs[h * D + i], __bfloat162float(a.ktail[tail0 + lane * D + i]), acc);
                s[h] = acc;
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float mx = s[h];
            for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float p = lane < nt ? exp2f(s[h] - mx) : 0.f;
            float l = p;
            for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
            if (lane < kQBlock) pt[lane * G + h] = p;
            const size_t row = (rowq0 + h) * a.max_splits + split;
            if (lane == 0) { a.part_ml[row] = make_float2(mx, l); a.part_c[row] = 0.f; }
            if (a.ct && lane < nt) a.ct[(rowq0 + h) * a.S + nfull + lane] = 0.f;
        }
        __syncwarp();
        for (int idx = lane; idx < G * D; idx += 32) {
            const int h = idx / D, i = idx % D;
            float acc = 0.f;
            for (int t = 0; t < nt; ++t) acc = fmaf(pt[t * G + h], __bfloat162float(a.vtail[tail0 + t * D + i]), acc);
            a.part_acc[((rowq0 + h) * a.max_splits + split) * D + i] = acc;
        }
        return;
    }

    // ---- quantized split ----------------------------------------------------
    const size_t bh = (size_t)b * a.Hkv + kvh;
    const size_t row0 = bh * a.S;
    unsigned char* myS = smem + warp * C::WARPB;
    uint64_t* myBar = bar + warp * 2;
    // block of this warp's tile i (tiles of the 4 warps interleaved)
    auto tile_blk = [&](int i) { return (split * kInt8Split) / kQBlock + i * kWarps + warp; };
    auto tile_ok = [&](int i) { return (tile_blk(i) + 1) * kQBlock <= nfull; };
    auto issue = [&](int i) {
        if (lane == 0 && tile_ok(i)) {
            const size_t p0 = (size_t)tile_blk(i) * kQBlock;
            unsigned char* st = myS + (i & 1) * C::STAGEB;
            mbar_arrive_expect_tx(&myBar[i & 1], (uint32_t)C::STAGEB);
            bulk_copy_g2s(st, a.kq + (row0 + p0) * D, C::CB, &myBar[i & 1]);
            bulk_copy_g2s(st + C::CB, a.vq + (row0 + p0) * D, C::CB, &myBar[i & 1]);
            bulk_copy_g2s(st + 2 * C::CB, a.wit + (row0 + p0) * kBands, C::WB, &myBar[i & 1]);
        }
    };
    if (lane == 0) {
        mbar_init(&myBar[0], 1);
        mbar_init(&myBar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    issue(0);
    issue(1);

    // ---- query preparation, once per CTA while the copies fly: rotated fp32
    // query; per head its 16-bit integer copy for the scores and the band norms
    // of the fp32 query, rounded up, for the bound
    float* qf = sP;                                           // [G][D] until the scores use it
    for (int idx = threadIdx.x; idx < G * D / 2; idx += blockDim.x) {
        const int h = idx / (D / 2), i = idx % (D / 2);
        const size_t off = (rowq0 + h) * D + 2 * i;
        const float x0 = ld_elem(a.q, off, 1), x1 = ld_elem(a.q, off + 1, 1);
        float y0 = x0, y1 = x1;
        if (a.rope) rope_pair(x0, x1, a.rope[(size_t)t_q * (D / 2) + i], y0, y1);
        qf[h * D + 2 * i] = y0;
        qf[h * D + 2 * i + 1] = y1;
    }
    __syncthreads();
    for (int h = warp; h < G; h += kWarps) {
        float amax = 0.f;
        for (int i = lane; i < D; i += 32) amax = fmaxf(amax, fabsf(qf[h * D + i]));
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float inv = amax > 0.f ? 32767.f / amax : 0.f;
        for (int wd = lane; wd < D / 4; wd += 32) {
            uint32_t hi = 0, lo = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int qi = max(-32767, min(32767, __float2int_rn(qf[h * D + 4 * wd + e] * inv)));
                hi |= (uint32_t)((qi >> 8) & 0xff) << (8 * e);
                lo |= (uint32_t)(qi & 0xff) << (8 * e);
            }
            sQW[h * (D / 4) + wd] = hi;
            sQW[G * (D / 4) + h * (D / 4) + wd] = lo;
        }
        if (lane < kBands) {
            float ss = 0.f;
            for (int e = lane * (D / kBands); e < (lane + 1) * (D / kBands); ++e)
                ss = __fadd_ru(ss, __fmul_ru(qf[h * D + e], qf[h * D + e]));
            sNQ[h * kBands + lane] = __fsqrt_ru(ss);
        }
        if (lane == 0) sF[h] = (amax > 0.f ? amax / 32767.f : 0.f) * a.scale_log2;
    }
    __syncthreads();
    const int r = lane % C::LPR, grp = lane / C::LPR;
    uint32_t qhi[G][4], qlo[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            qhi[h][e] = sQW[h * (D / 4) + r * 4 + e];
            qlo[h][e] = sQW[G * (D / 4) + h * (D / 4) + r * 4 + e];
        }

    float* myP = sP + warp * kQBlock * G;
    unsigned char* myPW = sPW + warp * G * 2 * kQBlock;
    float m_w[G], l_w[G], c_w[G], acc[G][C::DPL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m_w[h] = -INFINITY; l_w[h] = 0.f; c_w[h] = 0.f;
#pragma unroll
        for (int e = 0; e < C::DPL; ++e) acc[h][e] = 0.f;
    }
    for (int i = 0; i < kTilesPerWarp; ++i) {
        if (!tile_ok(i)) break;                   // later tiles of this warp are empty too
        const unsigned char* tK = myS + (i & 1) * C::STAGEB;
        const unsigned char* tV = tK + C::CB;
        const __half* tW = reinterpret_cast<const __half*>(tK + 2 * C::CB);
        const int blk = tile_blk(i);
        const int p0 = blk * kQBlock;
        if (!mbar_wait(&myBar[i & 1], (uint32_t)((i >> 1) & 1))) {
            // give up: flag it, and let this stage's copy and the other stage's
            // (if issued) land before the stages are reused for the partial
            if (lane == 0) atomicOr(a.hdr, kErrWait);
            mbar_wait(&myBar[i & 1], (uint32_t)((i >> 1) & 1));
            if (i + 1 < kTilesPerWarp && tile_ok(i + 1)) mbar_wait(&myBar[(i + 1) & 1], (uint32_t)(((i + 1) >> 1) & 1));
            break;
        }
        const float s_k = a.sk[bh * (a.S / kQBlock) + blk];
        const float s_v = a.sv[bh * (a.S / kQBlock) + blk];
        // ---- scores: exact int32 dot products of the query bytes with the codes
#pragma unroll
        for (int kb = 0; kb < C::KPG; kb += C::KB) {
            int part[C::M];
#pragma unroll
            for (int k = 0; k < C::KB; ++k) {
                const int t = grp * C::KPG + kb + k;
                const uint4 u = *reinterpret_cast<const uint4*>(tK + t * D + r * 16);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    int hs = __dp4a((int)qhi[h][0], (int)u.x, 0);
                    int ls = dp4a_us(qlo[h][0], u.x, 0);
                    hs = __dp4a((int)qhi[h][1], (int)u.y, hs);
                    ls = dp4a_us(qlo[h][1], u.y, ls);
                    hs = __dp4a((int)qhi[h][2], (int)u.z, hs);
                    ls = dp4a_us(qlo[h][2], u.z, ls);
                    hs = __dp4a((int)qhi[h][3], (int)u.w, hs);
                    ls = dp4a_us(qlo[h][3], u.w, ls);
                    part[k * G + h] = hs * 256 + ls;
                }
            }
#pragma unroll
            for (int mask = C::LPR / 2, cnt = C::M; mask >= 1; mask >>= 1, cnt >>= 1) {
                if (cnt >= 2) {
                    const bool upper = (r & mask) != 0;
#pragma unroll
                    for (int j = 0; j < cnt / 2; ++j) {
                        const int keep = upper ? part[j + cnt / 2] : part[j];
                        const int send = upper ? part[j] : part[j + cnt / 2];
                        part[j] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
                    }
                } else {
                    part[0] += __shfl_xor_sync(0xffffffffu, part[0], mask);
                }
            }
            if (r % C::SHARE == 0) {
#pragma unroll
                for (int j = 0; j < C::OUT; ++j) {
                    const int o = r / C::SHARE * C::OUT + j;
                    const int t = grp * C::KPG + kb + o / G;
                    const int h = o % G;
                    myP[t * G + h] = (float)part[j] * (sF[h] * s_k);
                }
            }
        }
        __syncwarp();
        // ---- two heads per pass, lane = (token lane & 15, head h + lane / 16):
        // online softmax, weights as 16-bit integers relative to the block maximum,
        // and the bound of the token
        // (one head: both halves evaluate head 0 and only the lower half writes)
        constexpr int HP = G >= 2 ? 2 : 1;
        const int t = lane & 15, half = lane >> 4;
        const bool writer = G >= 2 || half == 0;
        float alpha[G], wscale[G];
#pragma unroll
        for (int h = 0; h < G; h += HP) {
            const int hh = G >= 2 ? h + half : 0;
            const float s = myP[t * G + hh];
            float mx = s;
#pragma unroll
            for (int o = 8; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_lo = __shfl_sync(0xffffffffu, mx, 0), m_hi = __shfl_sync(0xffffffffu, mx, 16);
            const float mn0 = fmaxf(m_w[h], m_lo);
            const float mn1 = G >= 2 ? fmaxf(m_w[(h + 1) % G], m_hi) : mn0;
            const float mn = half ? mn1 : mn0;
            const float p = exp2f(s - mn);
            float ls = p, pm = p;
#pragma unroll
            for (int o = 8; o; o >>= 1) {
                ls += __shfl_xor_sync(0xffffffffu, ls, o);
                pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, o));
            }
            // 16-bit weight bytes: w = rint(p / pm * 32767) = 256 hi + lo
            const int wi = pm > 0.f ? min(32767, __float2int_rn(p * (32767.f / pm))) : 0;
            if (writer) {
                myPW[(hh * 2 + 0) * kQBlock + t] = (unsigned char)(wi >> 8);
                myPW[(hh * 2 + 1) * kQBlock + t] = (unsigned char)(wi & 0xff);
            }
            const float l_lo = __shfl_sync(0xffffffffu, ls, 0), l_hi = __shfl_sync(0xffffffffu, ls, 16);
            const float pm_lo = __shfl_sync(0xffffffffu, pm, 0), pm_hi = __shfl_sync(0xffffffffu, pm, 16);
            alpha[h] = exp2f(m_w[h] - mn0);           // 0 while the maximum was -inf
            l_w[h] = l_w[h] * alpha[h] + l_lo;
            m_w[h] = mn0;
            wscale[h] = pm_lo * s_v * (1.f / 32767.f);
            if constexpr (G >= 2) {
                alpha[h + 1] = exp2f(m_w[h + 1] - mn1);
                l_w[h + 1] = l_w[h + 1] * alpha[h + 1] + l_hi;
                m_w[h + 1] = mn1;
                wscale[h + 1] = pm_hi * s_v * (1.f / 32767.f);
            }
            // the bound of token t for head hh, every operation rounded up
            const uint4* wr = reinterpret_cast<const uint4*>(tW + t * kBands);
            const float4* nq = reinterpret_cast<const float4*>(sNQ + hh * kBands);
            float c = 0.f;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                const uint4 u = wr[c2];
                const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
                const float4 n0 = nq[2 * c2], n1 = nq[2 * c2 + 1];
                const float nn[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ww[e]));
                    c = __fmaf_ru(nn[2 * e], f.x, c);
                    c = __fmaf_ru(nn[2 * e + 1], f.y, c);
                }
            }
            c = __fmul_ru(c, a.inv_sqrt_d_up);
            if (a.ct && writer) a.ct[(rowq0 + hh) * a.S + p0 + t] = c;
            float cm = c;
#pragma unroll
            for (int o = 8; o; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
            c_w[h] = fmaxf(c_w[h], __shfl_sync(0xffffffffu, cm, 0));
            if constexpr (G >= 2) c_w[h + 1] = fmaxf(c_w[h + 1], __shfl_sync(0xffffffffu, cm, 16));
        }
        __syncwarp();
        // ---- P.V: lane owns dims lane + 32 j; dp4a over 4 tokens of one dim at a time
        const uint32_t* pw = reinterpret_cast<const uint32_t*>(myPW);
#pragma unroll
        for (int j = 0; j < C::DPL; ++j) {
            const uint4 v = *reinterpret_cast<const uint4*>(tV + (lane + 32 * j) * kQBlock);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const uint4 wh = *reinterpret_cast<const uint4*>(pw + (h * 2 + 0) * 4);
                const uint4 wl = *reinterpret_cast<const uint4*>(pw + (h * 2 + 1) * 4);
                int hs = dp4a_us(wh.x, v.x, 0);
                int ls = dp4a_us(wl.x, v.x, 0);
                hs = dp4a_us(wh.y, v.y, hs);
                ls = dp4a_us(wl.y, v.y, ls);
                hs = dp4a_us(wh.z, v.z, hs);
                ls = dp4a_us(wl.z, v.z, ls);
                hs = dp4a_us(wh.w, v.w, hs);
                ls = dp4a_us(wl.w, v.w, ls);
                acc[h][j] = fmaf(acc[h][j], alpha[h], (float)(hs * 256 + ls) * wscale[h]);
            }
        }
        // this stage is free once every lane is past its reads: refill it
        __syncwarp();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (i + 2 < kTilesPerWarp) issue(i + 2);
    }
    // ---- this warp's partial into its stage buffers (all issued copies were awaited)
    __syncwarp();
    float* part_w = reinterpret_cast<float*>(myS);             // [G][3 + D]
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int j = 0; j < C::DPL; ++j) part_w[h * (D + 3) + 3 + lane + 32 * j] = acc[h][j];
        if (lane == 0) {
            part_w[h * (D + 3)] = m_w[h];
            part_w[h * (D + 3) + 1] = l_w[h];
            part_w[h * (D + 3) + 2] = c_w[h];
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int h = idx / D, i = idx % D;
        float mx = -INFINITY, cm = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float* pwp = reinterpret_cast<const float*>(smem + w * C::WARPB) + h * (D + 3);
            mx = fmaxf(mx, pwp[0]);
            cm = fmaxf(cm, pwp[2]);
        }
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
        if (i == 0) { a.part_ml[row] = make_float2(mx, l); a.part_c[row] = cm; }
    }
}

// tanh(x) rounded up: CUDA's tanhf is within 2 ulps, so two steps toward +inf
// give an upper bound; tanh never exceeds 1.
__device__ __forceinline__ float tanh_up(float x) {
    float t = tanhf(x);
    t = nextafterf(nextafterf(t, 2.f), 2.f);
    return fminf(t, 1.f);
}

__global__ void __launch_bounds__(128) int8_combine_kernel(const Int8CombineArgs c) {
    const int hq = blockIdx.x, b = blockIdx.y;
    const int len = c.next_pos[b];
    const int nfull = len & ~(kQBlock - 1);
    const int ns = (nfull + kInt8Split - 1) / kInt8Split + (len > nfull ? 1 : 0);
    const int nsq = (nfull + kInt8Split - 1) / kInt8Split;
    const size_t row = (size_t)b * c.Hq + hq;
    // the tail split sits at index nsq; the quantized ones at 0..nsq-1
    float mx = -INFINITY, cm = 0.f;
    for (int s = 0; s < ns; ++s) {
        const int idx = s < nsq ? s : nsq;
        mx = fmaxf(mx, c.part_ml[row * c.max_splits + idx].x);
        cm = fmaxf(cm, c.part_c[row * c.max_splits + idx]);
    }
    float L = 0.f;
    for (int s = 0; s < ns; ++s) {
        const float2 ml = c.part_ml[row * c.max_splits + s];
        L += ml.y * exp2f(ml.x - mx);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int i = threadIdx.x; i < c.d; i += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < ns; ++s)
            acc = fmaf(c.part_acc[(row * c.max_splits + s) * c.d + i], exp2f(c.part_ml[row * c.max_splits + s].x - mx), acc);
        const float o = acc * inv;
        if (c.out_bf16) static_cast<__nv_bfloat16*>(c.out)[row * c.d + i] = __float2bfloat16_rn(o);
        else static_cast<float*>(c.out)[row * c.d + i] = o;
    }
    if (threadIdx.x == 0) {
        if (c.cmax) c.cmax[row] = cm;
        if (c.tanh_out) c.tanh_out[row] = tanh_up(cm);
    }
}

template <int D, int G>
cudaError_t launch_t(const Int8Args& a, cudaStream_t st) {
    using C = I8<D, G>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(int8_decode_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    int8_decode_kernel<D, G><<<dim3(a.max_splits, a.Hkv, a.B), kWarps * 32, C::SMEM, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_int8_decode(kvc_handle* h, const void* q, void* out, float* cmax, float* tanh_out, float* ct,
                               cudaStream_t st) {
    const Shape& s = h->sh;
    Int8Args a{};
    a.q = q;
    a.kq = reinterpret_cast<const int8_t*>(h->state + h->L.kq);
    a.vq = reinterpret_cast<const int8_t*>(h->state + h->L.vq);
    a.sk = reinterpret_cast<const float*>(h->state + h->L.sk);
    a.sv = reinterpret_cast<const float*>(h->state + h->L.sv);
    a.wit = reinterpret_cast<const __half*>(h->state + h->L.wit);
    a.ktail = reinterpret_cast<const __nv_bfloat16*>(h->state + h->L.ktail);
    a.vtail = reinterpret_cast<const __nv_bfloat16*>(h->state + h->L.vtail);
    a.next_pos = reinterpret_cast<const int32_t*>(h->state + h->L.next_pos);
    a.rope = s.rope ? reinterpret_cast<const float2*>(h->state + h->L.rope) : nullptr;
    a.part_ml = reinterpret_cast<float2*>(h->state + h->L.part_ml);
    a.part_acc = reinterpret_cast<float*>(h->state + h->L.part_acc);
    a.part_c = reinterpret_cast<float*>(h->state + h->L.part_c);
    a.ct = ct;
    a.hdr = reinterpret_cast<uint32_t*>(h->state + h->L.hdr);
    a.B = s.B; a.Hq = s.Hq; a.Hkv = s.Hkv; a.d = s.d; a.S = s.S; a.max_splits = s.max_splits;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.d));
    a.inv_sqrt_d_up = std::nextafter((float)(1.0 / std::sqrt((double)s.d)), 1.0f);
    cudaError_t e = cudaErrorInvalidValue;
#define KVC_CASE(D, G) \
    if (s.d == D && s.g == G) e = launch_t<D, G>(a, st);
    KVC_CASE(128, 1) KVC_CASE(128, 2) KVC_CASE(128, 4) KVC_CASE(128, 8)
    KVC_CASE(64, 1) KVC_CASE(64, 2) KVC_CASE(64, 4) KVC_CASE(64, 8)
#undef KVC_CASE
    if (e != cudaSuccess) return e;
    Int8CombineArgs c{};
    c.part_ml = a.part_ml; c.part_acc = a.part_acc; c.part_c = a.part_c; c.next_pos = a.next_pos;
    c.out = out; c.cmax = cmax; c.tanh_out = tanh_out;
    c.B = s.B; c.Hq = s.Hq; c.d = s.d; c.max_splits = s.max_splits; c.out_bf16 = s.out_bf16;
    int8_combine_kernel<<<dim3(s.Hq, s.B), 128, 0, st>>>(c);
    return cudaGetLastError();
}

}  // namespace kvc
