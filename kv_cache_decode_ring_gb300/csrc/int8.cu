// int8.cu -- fused INT8 decode attention with the witness bound.
//
// [WITCERT] "频带酉性与双层证书": for every cached token t the decode step also
// returns c_t = (1/sqrt d) sum_b ||q_b|| w_{t,b} >= |q . r_t| / sqrt(d), the
// largest logit perturbation the quantization residual r_t can cause, and per
// query head tanh(max_t c_t) >= the attention total variation
// ("为什么在线监控 KV 误差如此困难？": TV <= tanh(max |eps|)).
// "SGLang 生产级落地与闭环门控修复": per-block scales are token-independent, so
// they fold into scalars: the score of key t in block m is s_K[m] (q . code_t),
// and its value contributes p_t s_V[m] code_t.
//
// Layout read per (request, KV head): codes int8 [S][d] (K and V), scales fp32
// [S/16], witnesses fp16 [S][16], exact bf16 tail [16][d] for the rows of the
// incomplete block.  Quantized splits cover [0, 16*floor(len/16)) in 128-key
// CTAs (4 warps x 32 keys = 2 blocks per warp); one extra split handles the
// tail rows exactly (c_t = 0 there).
//
// Arithmetic:
//  * codes -> fp32 exactly: bias the bytes by 128, place each in the low
//    mantissa of 2^23 with a byte permute, subtract 2^23 + 128;
//  * scores and P.V in fp32 as in the bf16 kernel (reduce-scatter across the
//    lanes of a row);
//  * the bound with every operation rounded toward +inf: band norms of the
//    rotated fp32 query (sum of squares, square root), products with the fp16
//    witnesses, their sum, times an upward-rounded 1/sqrt(d); tanh gets two
//    ulps of headroom over CUDA tanhf's documented error, capped at 1.
#include <cmath>

#include "async_copy.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kWarps = 8;
constexpr int kTile = 32;       // keys per warp = two blocks
static_assert(kWarps * kTile == kInt8Split, "split shape");

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

// 4 int8 codes in one word -> 4 exact fp32 values.
__device__ __forceinline__ void s8x4_to_f32(uint32_t w, float* f) {
    const uint32_t u = w ^ 0x80808080u;
    f[0] = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7650)) - 8388736.0f;
    f[1] = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7651)) - 8388736.0f;
    f[2] = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7652)) - 8388736.0f;
    f[3] = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7653)) - 8388736.0f;
}

// dp4a with unsigned bytes in a and signed bytes in b
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

template <int D, int G>
struct I8 {
    static constexpr int LPR = D / 16;            // score lanes per row, 16 codes (one 16-B load) each
    static constexpr int RPP = 32 / LPR;          // key groups per warp for the scores
    static constexpr int KPG = kTile / RPP;       // keys per group
    static constexpr int KB0 = 2 * LPR / G;
    static constexpr int KB = KB0 < KPG ? (KB0 < 1 ? 1 : KB0) : KPG;
    static constexpr int M = KB * G;              // int32 partial scores per lane per batch
    static constexpr int OUT = M / LPR;           // finished scores per lane per batch
    static constexpr int LPR2 = D / 8;            // P.V lanes per row, 8 codes each
    static constexpr int RPP2 = 32 / LPR2;
    static constexpr int TILEB = kTile * D;       // one warp's codes (K or V)
    static constexpr int WITB = kTile * kBands * 2;
    static constexpr int WARPB = 2 * TILEB + WITB;
    static constexpr int PARTF = G * (D + 3);     // floats of one warp's partial (m, l, c, acc)
    static_assert(M % LPR == 0 && OUT >= 1, "batch shape");
    static_assert(PARTF * 4 <= WARPB, "partial must fit in the warp's tiles");
    // shared memory after the warps' tiles: scores [warp][kTile][G] (also the fp32 query
    // during preparation), query bytes hi/lo [G][D/4] words, band norms [G][16],
    // score factors [G], barriers [warp]
    static constexpr int OFF_P = kWarps * WARPB;
    static constexpr int PBYTES = (kWarps * kTile * G > G * D ? kWarps * kTile * G : G * D) * 4;
    static constexpr int OFF_QW = OFF_P + PBYTES;
    static constexpr int OFF_NQ = OFF_QW + 2 * G * (D / 4) * 4;
    static constexpr int OFF_F = OFF_NQ + G * kBands * 4;
    static constexpr int OFF_BAR = OFF_F + ((G * 4 + 15) / 16) * 16;
    static constexpr size_t SMEM = OFF_BAR + kWarps * 8 + 128;
};

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32, 2) int8_decode_kernel(const Int8Args a) {
    using C = I8<D, G>;
    extern __shared__ __align__(128) unsigned char smem[];
    float* sP = reinterpret_cast<float*>(smem + C::OFF_P);              // [warp][kTile][G]
    uint32_t* sQW = reinterpret_cast<uint32_t*>(smem + C::OFF_QW);      // [2][G][D/4] query bytes
    float* sNQ = reinterpret_cast<float*>(smem + C::OFF_NQ);            // [G][16] band norms
    float* sF = reinterpret_cast<float*>(smem + C::OFF_F);              // [G] score factors
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);     // [warp]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
    const int len = a.next_pos[b];
    const int nfull = len & ~(kQBlock - 1);
    const int nsq = (nfull + kInt8Split - 1) / kInt8Split;
    const bool tail_split = split == nsq;
    if (split > nsq || (tail_split && len == nfull)) return;
    const int t_q = len - 1;
    const size_t rowq0 = (size_t)b * a.Hq + (size_t)kvh * G;    // first query row of the group

    if (threadIdx.x < kWarps) mbar_init(&bar[threadIdx.x], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();

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
    const int r = lane % C::LPR, grp = lane / C::LPR;          // score mapping
    const int r2 = lane % C::LPR2, grp2 = lane / C::LPR2;      // P.V mapping
    unsigned char* myK = smem + warp * C::WARPB;
    unsigned char* myV = myK + C::TILEB;
    const __half* myW = reinterpret_cast<const __half*>(myV + C::TILEB);
    float* myP = sP + warp * kTile * G;
    const int k0 = split * kInt8Split + warp * kTile;
    const int nk = max(0, min(kTile, nfull - k0));
    const size_t row0 = ((size_t)b * a.Hkv + kvh) * a.S;
    if (lane == 0 && nk > 0) {
        mbar_arrive_expect_tx(&bar[warp], (uint32_t)(2 * nk * D + nk * kBands * 2));
        bulk_copy_g2s(myK, a.kq + (row0 + k0) * D, (uint32_t)(nk * D), &bar[warp]);
        bulk_copy_g2s(myV, a.vq + (row0 + k0) * D, (uint32_t)(nk * D), &bar[warp]);
        bulk_copy_g2s((void*)myW, a.wit + (row0 + k0) * kBands, (uint32_t)(nk * kBands * 2), &bar[warp]);
    }

    // ---- query preparation, once per CTA while the copies fly:
    //  rotated fp32 query; per head a 16-bit integer copy q ~ s_q * (256 hi + lo) for the
    //  scores (exact int32 dot products with the codes); band norms of the fp32 query,
    //  rounded up, for the bound
    float* qf = sP;                                           // [G][D] before the scores use it
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
        const float sq = amax > 0.f ? amax / 32767.f : 0.f;
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
        if (lane == 0) sF[h] = sq * a.scale_log2;
    }
    __syncthreads();
    uint32_t qhi[G][4], qlo[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            qhi[h][e] = sQW[h * (D / 4) + r * 4 + e];
            qlo[h][e] = sQW[G * (D / 4) + h * (D / 4) + r * 4 + e];
        }

    float m_w[G], l_w[G], c_w[G], acc[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m_w[h] = -INFINITY; l_w[h] = 0.f; c_w[h] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
    }
    bool ok = true;
    if (nk > 0) {
        ok = mbar_wait(&bar[warp], 0);
        if (!ok) {
            if (lane == 0) atomicOr(a.hdr, kErrWait);
            mbar_wait(&bar[warp], 0);
        }
    }
    if (nk > 0 && ok) {
        const float* skb = a.sk + ((size_t)b * a.Hkv + kvh) * (a.S / kQBlock) + k0 / kQBlock;
        const float* svb = a.sv + ((size_t)b * a.Hkv + kvh) * (a.S / kQBlock) + k0 / kQBlock;
        // ---- scores: exact int32 dot products of the query bytes with the codes
#pragma unroll
        for (int kb = 0; kb < C::KPG; kb += C::KB) {
            int part[C::M];
#pragma unroll
            for (int k = 0; k < C::KB; ++k) {
                const int t = grp * C::KPG + kb + k;
                const uint4 u = *reinterpret_cast<const uint4*>(myK + t * D + r * 16);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    int hi = __dp4a((int)qhi[h][0], (int)u.x, 0);
                    int lo = dp4a_us(qlo[h][0], u.x, 0);
                    hi = __dp4a((int)qhi[h][1], (int)u.y, hi);
                    lo = dp4a_us(qlo[h][1], u.y, lo);
                    hi = __dp4a((int)qhi[h][2], (int)u.z, hi);
                    lo = dp4a_us(qlo[h][2], u.z, lo);
                    hi = __dp4a((int)qhi[h][3], (int)u.w, hi);
                    lo = dp4a_us(qlo[h][3], u.w, lo);
                    part[k * G + h] = hi * 256 + lo;
                }
            }
#pragma unroll
            for (int mask = C::LPR / 2, cnt = C::M; mask >= 1; mask >>= 1, cnt >>= 1) {
                const bool upper = (r & mask) != 0;
#pragma unroll
                for (int j = 0; j < cnt / 2; ++j) {
                    const int keep = upper ? part[j + cnt / 2] : part[j];
                    const int send = upper ? part[j] : part[j + cnt / 2];
                    part[j] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
                }
            }
#pragma unroll
            for (int j = 0; j < C::OUT; ++j) {
                const int o = r * C::OUT + j;
                const int t = grp * C::KPG + kb + o / G;
                const int h = o % G;
                myP[t * G + h] = (t < nk) ? (float)part[j] * (sF[h] * skb[t / kQBlock]) : -INFINITY;
            }
        }
        __syncwarp();
        // ---- lane = key: softmax weights, the value scale folded into p, and the bound
        float pk[G];
        float smax[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float sv = myP[lane * G + h];
            float mx = sv;
#pragma unroll
            for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            smax[h] = mx;
            pk[h] = exp2f(sv - mx);                   // masked keys: 2^-inf = 0
        }
        if (lane < nk) {
            const float vs = svb[lane / kQBlock];
            const uint4* wr = reinterpret_cast<const uint4*>(myW + lane * kBands);
            float wf[kBands];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                const uint4 u = wr[c2];
                const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ww[e]));
                    wf[c2 * 8 + 2 * e] = f.x;
                    wf[c2 * 8 + 2 * e + 1] = f.y;
                }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                myP[lane * G + h] = pk[h] * vs;
                float c = 0.f;
#pragma unroll
                for (int bb = 0; bb < kBands; ++bb) c = __fmaf_ru(sNQ[h * kBands + bb], wf[bb], c);
                c = __fmul_ru(c, a.inv_sqrt_d_up);
                c_w[h] = fmaxf(c_w[h], c);
                if (a.ct) a.ct[(rowq0 + h) * a.S + k0 + lane] = c;
            }
        } else {
#pragma unroll
            for (int h = 0; h < G; ++h) myP[lane * G + h] = 0.f;
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float l = pk[h];
            float cm = c_w[h];
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                l += __shfl_xor_sync(0xffffffffu, l, o);
                cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
            }
            m_w[h] = smax[h];
            l_w[h] = l;
            c_w[h] = cm;
        }
        __syncwarp();
        // ---- P.V: lane owns dims [8 r2, 8 r2 + 8) of every head, keys of its group
        for (int t = grp2; t < nk; t += C::RPP2) {
            const uint2 u = *reinterpret_cast<const uint2*>(myV + t * D + r2 * 8);
            float x[8];
            s8x4_to_f32(u.x, x);
            s8x4_to_f32(u.y, x + 4);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float p = myP[t * G + h];
                const float2 pp = make_float2(p, p);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float2 r_ = __ffma2_rn(pp, make_float2(x[e], x[e + 1]), make_float2(acc[h][e], acc[h][e + 1]));
                    acc[h][e] = r_.x;
                    acc[h][e + 1] = r_.y;
                }
            }
        }
#pragma unroll
        for (int mask = C::LPR2; mask < 32; mask <<= 1)
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], mask);
    }
    __syncwarp();
    float* part_w = reinterpret_cast<float*>(myK);             // [G][3 + D]
    if (grp2 == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int e = 0; e < 8; ++e) part_w[h * (D + 3) + 3 + r2 * 8 + e] = acc[h][e];
            if (r2 == 0) {
                part_w[h * (D + 3)] = m_w[h];
                part_w[h * (D + 3) + 1] = l_w[h];
                part_w[h * (D + 3) + 2] = c_w[h];
            }
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int h = idx / D, i = idx % D;
        float mx = -INFINITY, cm = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float* pw = reinterpret_cast<const float*>(smem + w * C::WARPB) + h * (D + 3);
            mx = fmaxf(mx, pw[0]);
            cm = fmaxf(cm, pw[2]);
        }
        float l = 0.f, sacc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float* pw = reinterpret_cast<const float*>(smem + w * C::WARPB) + h * (D + 3);
            const float f = pw[0] == -INFINITY ? 0.f : exp2f(pw[0] - mx);
            l += pw[1] * f;
            sacc += pw[3 + i] * f;
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
