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

constexpr int kWarps = 4;
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

template <int D, int G>
struct I8 {
    static constexpr int LPR = D / 8;             // lanes per row, 8 codes (8 bytes) each
    static constexpr int RPP = 32 / LPR;          // key groups per warp
    static constexpr int KPG = kTile / RPP;       // keys per group
    static constexpr int KB0 = 2 * LPR / G;
    static constexpr int KB = KB0 < KPG ? (KB0 < 1 ? 1 : KB0) : KPG;
    static constexpr int M = KB * G;
    static constexpr int OUT = M / LPR;
    static constexpr int BW = D / kBands;         // dims per band
    static constexpr int TILEB = kTile * D;       // one warp's codes (K or V)
    static constexpr int WITB = kTile * kBands * 2;
    static constexpr int WARPB = 2 * TILEB + WITB;
    static constexpr int PARTF = G * (D + 3);     // floats of one warp's partial (m, l, c, acc)
    static_assert(M % LPR == 0 && OUT >= 1, "batch shape");
    static_assert(PARTF * 4 <= WARPB, "partial must fit in the warp's tiles");
    static constexpr size_t SMEM = (size_t)kWarps * WARPB + (size_t)kWarps * kTile * G * 4 +
                                   (size_t)kWarps * G * kBands * 4 + kWarps * 8 + 128;
};

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32, G >= 8 ? 3 : 4) int8_decode_kernel(const Int8Args a) {
    using C = I8<D, G>;
    extern __shared__ __align__(128) unsigned char smem[];
    float* sP = reinterpret_cast<float*>(smem + kWarps * C::WARPB);      // [warp][kTile][G]
    float* sNQ = sP + kWarps * kTile * G;                                 // [warp][G][16] band norms
    uint64_t* bar = reinterpret_cast<uint64_t*>(sNQ + kWarps * G * kBands);

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
    const int r = lane % C::LPR, grp = lane / C::LPR;
    unsigned char* myK = smem + warp * C::WARPB;
    unsigned char* myV = myK + C::TILEB;
    const __half* myW = reinterpret_cast<const __half*>(myV + C::TILEB);
    float* myP = sP + warp * kTile * G;
    float* myNQ = sNQ + warp * G * kBands;
    const int k0 = split * kInt8Split + warp * kTile;
    const int nk = max(0, min(kTile, nfull - k0));
    const size_t row0 = ((size_t)b * a.Hkv + kvh) * a.S;
    if (lane == 0 && nk > 0) {
        mbar_arrive_expect_tx(&bar[warp], (uint32_t)(2 * nk * D + nk * kBands * 2));
        bulk_copy_g2s(myK, a.kq + (row0 + k0) * D, (uint32_t)(nk * D), &bar[warp]);
        bulk_copy_g2s(myV, a.vq + (row0 + k0) * D, (uint32_t)(nk * D), &bar[warp]);
        bulk_copy_g2s((void*)myW, a.wit + (row0 + k0) * kBands, (uint32_t)(nk * kBands * 2), &bar[warp]);
    }

    // query: rotated fp32; scaled copy for the scores, band norms (rounded up) for the bound
    float q[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const size_t off = (rowq0 + h) * D + r * 8;
        const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + off);
        float x[8];
        bf16x8_to_f32(u, x);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float y0 = x[2 * j], y1 = x[2 * j + 1];
            if (a.rope) rope_pair(x[2 * j], x[2 * j + 1], a.rope[(size_t)t_q * (D / 2) + r * 4 + j], y0, y1);
            q[h][2 * j] = y0;
            q[h][2 * j + 1] = y1;
        }
        if (grp == 0) {
#pragma unroll
            for (int bb = 0; bb < 8 / C::BW; ++bb) {
                float ss = 0.f;
#pragma unroll
                for (int e = bb * C::BW; e < (bb + 1) * C::BW; ++e) ss = __fadd_ru(ss, __fmul_ru(q[h][e], q[h][e]));
                myNQ[h * kBands + r * (8 / C::BW) + bb] = __fsqrt_ru(ss);
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) q[h][e] *= a.scale_log2;
    }
    __syncwarp();
    // band norms of the heads whose scores this lane ends up owning
    float nq[C::OUT][kBands];
#pragma unroll
    for (int j = 0; j < C::OUT; ++j) {
        const int h = (r * C::OUT + j) % G;
#pragma unroll
        for (int bb = 0; bb < kBands; ++bb) nq[j][bb] = myNQ[h * kBands + bb];
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
#pragma unroll
        for (int kb = 0; kb < C::KPG; kb += C::KB) {
            float part[C::M];
#pragma unroll
            for (int k = 0; k < C::KB; ++k) {
                const int t = grp * C::KPG + kb + k;
                const uint2 u = *reinterpret_cast<const uint2*>(myK + t * D + r * 8);
                float x[8];
                s8x4_to_f32(u.x, x);
                s8x4_to_f32(u.y, x + 4);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float s0 = q[h][0] * x[0], s1 = q[h][1] * x[1];
#pragma unroll
                    for (int e = 2; e < 8; e += 2) {
                        s0 = fmaf(q[h][e], x[e], s0);
                        s1 = fmaf(q[h][e + 1], x[e + 1], s1);
                    }
                    part[k * G + h] = s0 + s1;
                }
            }
#pragma unroll
            for (int mask = C::LPR / 2, cnt = C::M; mask >= 1; mask >>= 1, cnt >>= 1) {
                const bool upper = (r & mask) != 0;
#pragma unroll
                for (int j = 0; j < cnt / 2; ++j) {
                    const float keep = upper ? part[j + cnt / 2] : part[j];
                    const float send = upper ? part[j] : part[j + cnt / 2];
                    part[j] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
                }
            }
#pragma unroll
            for (int j = 0; j < C::OUT; ++j) {
                const int o = r * C::OUT + j;
                const int t = grp * C::KPG + kb + o / G;
                const int h = o % G;
                if (t < nk) {
                    myP[t * G + h] = part[j] * skb[t / kQBlock];
                    // the bound for (t, h): every operation rounded up
                    const __half2* w2 = reinterpret_cast<const __half2*>(myW + t * kBands);
                    float c = 0.f;
#pragma unroll
                    for (int bb = 0; bb < kBands / 2; ++bb) {
                        const float2 w = __half22float2(w2[bb]);
                        c = __fmaf_ru(nq[j][2 * bb], w.x, c);
                        c = __fmaf_ru(nq[j][2 * bb + 1], w.y, c);
                    }
                    c = __fmul_ru(c, a.inv_sqrt_d_up);
                    c_w[h] = fmaxf(c_w[h], c);
                    if (a.ct) a.ct[(rowq0 + h) * a.S + k0 + t] = c;
                } else {
                    myP[t * G + h] = -INFINITY;
                }
            }
        }
        __syncwarp();
        // softmax over the warp's keys (lane = key); p' = p * s_V folds the value scale
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float s = myP[lane * G + h];
            float mx = s;
#pragma unroll
            for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float p = exp2f(s - mx);
            myP[lane * G + h] = lane < nk ? p * svb[lane / kQBlock] : 0.f;
            float l = p;
#pragma unroll
            for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
            m_w[h] = mx;
            l_w[h] = l;
            float cm = c_w[h];
#pragma unroll
            for (int o = 16; o; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
            c_w[h] = cm;
        }
        __syncwarp();
        for (int t = grp; t < nk; t += C::RPP) {
            const uint2 u = *reinterpret_cast<const uint2*>(myV + t * D + r * 8);
            float x[8];
            s8x4_to_f32(u.x, x);
            s8x4_to_f32(u.y, x + 4);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float p = myP[t * G + h];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(p, x[e], acc[h][e]);
            }
        }
#pragma unroll
        for (int mask = C::LPR; mask < 32; mask <<= 1)
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], mask);
    }
    __syncwarp();
    float* part_w = reinterpret_cast<float*>(myK);             // [G][3 + D]
    if (grp == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int e = 0; e < 8; ++e) part_w[h * (D + 3) + 3 + r * 8 + e] = acc[h][e];
            if (r == 0) {
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
        float l = 0.f, s = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float* pw = reinterpret_cast<const float*>(smem + w * C::WARPB) + h * (D + 3);
            const float f = pw[0] == -INFINITY ? 0.f : exp2f(pw[0] - mx);
            l += pw[1] * f;
            s += pw[3 + i] * f;
        }
        const size_t row = (rowq0 + h) * a.max_splits + split;
        a.part_acc[row * D + i] = s;
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
