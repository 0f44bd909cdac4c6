// decode_gqa.cu -- split-K decode attention for bf16 caches with 4 or 8 query
// heads per KV head (head_dim 64 or 128), on sm_103a.
//
// Same mathematics as decode.cu ([LOOP] §三 step; [LEAN] §2.1 window mask), with
// the per-split partials (m, l, acc) merged by the combine kernel.
//
// With g query heads on every K/V byte the arithmetic per byte is 4g/2 FMAs, so
// the kernel must keep HBM busy while it computes.  A warp therefore streams its
// keys through two shared-memory stages of 16 keys (K and V rows contiguous in
// the cache, one cp.async.bulk each, completing on the stage's mbarrier): while
// it computes one tile the next is in flight.  The warp keeps an online softmax
// (running maximum, sum and rescaled accumulators) over its tiles; the CTA's 4
// warps merge at the end of the 256-key split.
//  * scores: lane = (run of 16-byte chunks of the row, key group); partial dot
//    products for all g heads in packed fp32 FMAs, reduce-scatter across the
//    lanes of a row;
//  * P.V: lane = 8 output dims of every head, packed fp32 FMAs;
//  * the rotated, scaled query is prepared once per CTA in shared memory, after
//    the first copies are already in flight.
// Every mbarrier wait is bounded (about 1 s); on expiry the device error word is
// set and the split's arithmetic is skipped.
#include "async_copy.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kWarps = 4;
constexpr int kTileKeys = 16;                            // keys per stage
constexpr int kTilesPerWarp = 4;
constexpr int kSplit = kWarps * kTilesPerWarp * kTileKeys;   // 256 keys per CTA
static_assert(kSplit == kGqaSplit, "split shape");

template <int D, int G>
struct GqaCfg {
    static constexpr int QD = G <= 4 ? 16 : 8;           // score dims per lane
    static constexpr int LPR = D / QD;                   // score lanes per row
    static constexpr int RPP = 32 / LPR;                 // key groups per warp
    static constexpr int KPG = kTileKeys / RPP;          // keys per group per tile
    static constexpr int KB0 = 2 * LPR / G;
    static constexpr int KB = KB0 < KPG ? (KB0 < 1 ? 1 : KB0) : KPG;
    static constexpr int M = KB * G;
    static constexpr int OUT = M / LPR;
    static constexpr int LPR2 = D / 8;                   // P.V lanes per row
    static constexpr int RPP2 = 32 / LPR2;
    static constexpr int ROWB = D * 2;
    static constexpr int HALF = kTileKeys * ROWB;        // K (or V) rows of one stage
    static constexpr int STAGEB = 2 * HALF;
    static constexpr int WARPB = 2 * STAGEB;             // two stages
    static constexpr int PARTB = G * (D + 2) * 4;
    static_assert(KPG >= 1 && M % LPR == 0 && OUT >= 1, "batch shape");
    static_assert(PARTB <= WARPB, "partial must fit in the warp's stages");
    static constexpr int OFF_P = kWarps * WARPB;                          // scores [warp][16][G]
    static constexpr int OFF_Q = OFF_P + kWarps * kTileKeys * G * 4;      // query [G][D]
    static constexpr int OFF_BAR = OFF_Q + G * D * 4;                     // [warp][stage]
    static constexpr size_t SMEM = OFF_BAR + kWarps * 2 * 8 + 128;
};

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32, 3) decode_gqa_kernel(const DecodeArgs a) {
    using C = GqaCfg<D, G>;
    extern __shared__ __align__(128) unsigned char smem[];
    float* sP = reinterpret_cast<float*>(smem + C::OFF_P);
    float* sQ = reinterpret_cast<float*>(smem + C::OFF_Q);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
    const int len = a.next_pos[b];
    int lo, hi;
    key_range(len, a.S, a.W, a.ring, lo, hi);
    const int nsplit = (hi - lo + kSplit - 1) / kSplit;
    if (split >= nsplit) return;

    const size_t head_row0 = ((size_t)b * a.Hkv + kvh) * a.S;
    const __nv_bfloat16* Kg = static_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* Vg = static_cast<const __nv_bfloat16*>(a.v);
    unsigned char* myS = smem + warp * C::WARPB;
    uint64_t* myBar = bar + warp * 2;
    // keys of this warp's tile i: 16 consecutive rows, tiles of the 4 warps interleaved
    auto tile_k0 = [&](int i) { return lo + split * kSplit + (i * kWarps + warp) * kTileKeys; };
    auto tile_nk = [&](int i) { return max(0, min(kTileKeys, hi - tile_k0(i))); };
    auto issue = [&](int i) {
        const int k0 = tile_k0(i), nk = tile_nk(i);
        if (lane == 0 && nk > 0) {
            unsigned char* st = myS + (i & 1) * C::STAGEB;
            const uint32_t bytes = (uint32_t)nk * C::ROWB;
            mbar_arrive_expect_tx(&myBar[i & 1], 2 * bytes);
            bulk_copy_g2s(st, Kg + (head_row0 + k0) * D, bytes, &myBar[i & 1]);
            bulk_copy_g2s(st + C::HALF, Vg + (head_row0 + k0) * D, bytes, &myBar[i & 1]);
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

    // the query of the G heads, rotated at t = len - 1, times log2(e)/sqrt(d)
    {
        const int t = len - 1;
        for (int idx = threadIdx.x; idx < G * D / 2; idx += blockDim.x) {
            const int h = idx / (D / 2), i = idx % (D / 2);
            const size_t off = ((size_t)b * a.Hq + (size_t)kvh * G + h) * D + 2 * i;
            const float x0 = ld_elem(a.q, off, 1), x1 = ld_elem(a.q, off + 1, 1);
            float y0 = x0, y1 = x1;
            if (a.rope) rope_pair(x0, x1, a.rope[(size_t)t * (D / 2) + i], y0, y1);
            sQ[h * D + 2 * i] = y0 * a.scale_log2;
            sQ[h * D + 2 * i + 1] = y1 * a.scale_log2;
        }
    }
    __syncthreads();
    const int r = lane % C::LPR, grp = lane / C::LPR;
    const int r2 = lane % C::LPR2, grp2 = lane / C::LPR2;
    float q[G][C::QD];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < C::QD; e += 4) {
            const int dim = (r + (e / 8) * C::LPR) * 8 + (e % 8);
            const float4 f = *reinterpret_cast<const float4*>(sQ + h * D + dim);
            q[h][e] = f.x; q[h][e + 1] = f.y; q[h][e + 2] = f.z; q[h][e + 3] = f.w;
        }

    float* myP = sP + warp * kTileKeys * G;
    float m_w[G], l_w[G], acc[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m_w[h] = -INFINITY; l_w[h] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
    }
    bool ok = true;
    for (int i = 0; i < kTilesPerWarp && ok; ++i) {
        const int nk = tile_nk(i);
        if (nk == 0) break;                       // later tiles of this warp are empty too
        const unsigned char* tK = myS + (i & 1) * C::STAGEB;
        const unsigned char* tV = tK + C::HALF;
        ok = mbar_wait(&myBar[i & 1], (uint32_t)((i >> 1) & 1));
        if (!ok) {
            if (lane == 0) atomicOr(a.hdr, kErrWait);
            mbar_wait(&myBar[i & 1], (uint32_t)((i >> 1) & 1));
            break;
        }
        // ---- scores of the tile
#pragma unroll
        for (int kb = 0; kb < C::KPG; kb += C::KB) {
            float part[C::M];
#pragma unroll
            for (int k = 0; k < C::KB; ++k) {
                const int t = grp * C::KPG + kb + k;
                float x[C::QD];
#pragma unroll
                for (int e = 0; e < C::QD; e += 8) {
                    const uint4 u = *reinterpret_cast<const uint4*>(tK + t * C::ROWB + (r + (e / 8) * C::LPR) * 16);
                    bf16x8_to_f32(u, x + e);
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < C::QD; e += 2)
                        s2 = __ffma2_rn(make_float2(q[h][e], q[h][e + 1]), make_float2(x[e], x[e + 1]), s2);
                    part[k * G + h] = s2.x + s2.y;
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
                myP[t * G + (o % G)] = (t < nk) ? part[j] : -INFINITY;
            }
        }
        __syncwarp();
        // ---- online softmax, two heads per pass: lane = (key lane & 15, head + lane >> 4)
        float alpha[G];
#pragma unroll
        for (int h = 0; h < G; h += 2) {
            const int hh = h + (lane >> 4), t = lane & 15;
            const float s = myP[t * G + hh];
            float mx = s;
#pragma unroll
            for (int o = 8; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_lo = __shfl_sync(0xffffffffu, mx, 0), m_hi = __shfl_sync(0xffffffffu, mx, 16);
            const float mn0 = fmaxf(m_w[h], m_lo), mn1 = fmaxf(m_w[h + 1], m_hi);
            const float mn = (lane >> 4) ? mn1 : mn0;
            const float p = exp2f(s - mn);                // masked keys: 2^-inf = 0
            myP[t * G + hh] = p;
            float ls = p;
#pragma unroll
            for (int o = 8; o; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
            const float l_lo = __shfl_sync(0xffffffffu, ls, 0), l_hi = __shfl_sync(0xffffffffu, ls, 16);
            alpha[h] = exp2f(m_w[h] - mn0);               // 0 while the maximum was -inf
            alpha[h + 1] = exp2f(m_w[h + 1] - mn1);
            l_w[h] = l_w[h] * alpha[h] + l_lo;
            l_w[h + 1] = l_w[h + 1] * alpha[h + 1] + l_hi;
            m_w[h] = mn0;
            m_w[h + 1] = mn1;
        }
        __syncwarp();
        // ---- P.V, after rescaling the accumulators to the new maxima
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[h][e] *= alpha[h];
        for (int t = grp2; t < nk; t += C::RPP2) {
            const uint4 u = *reinterpret_cast<const uint4*>(tV + t * C::ROWB + r2 * 16);
            float x[8];
            bf16x8_to_f32(u, x);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float pv = myP[t * G + h];
                const float2 pp = make_float2(pv, pv);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float2 rr = __ffma2_rn(pp, make_float2(x[e], x[e + 1]), make_float2(acc[h][e], acc[h][e + 1]));
                    acc[h][e] = rr.x;
                    acc[h][e + 1] = rr.y;
                }
            }
        }
        // this stage is free once every lane is past its reads: refill it
        __syncwarp();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (i + 2 < kTilesPerWarp) issue(i + 2);
    }
#pragma unroll
    for (int mask = C::LPR2; mask < 32; mask <<= 1)
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], mask);

    // ---- this warp's partial into its own stage buffers (the copies it issued are
    // complete: every issued tile was waited for, except after a timeout)
    __syncwarp();
    float* part_w = reinterpret_cast<float*>(myS);        // [G][2 + D]
    if (grp2 == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int e = 0; e < 8; ++e) part_w[h * (D + 2) + 2 + r2 * 8 + e] = acc[h][e];
            if (r2 == 0) { part_w[h * (D + 2)] = m_w[h]; part_w[h * (D + 2) + 1] = l_w[h]; }
        }
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
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t st) {
    using C = GqaCfg<D, G>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(decode_gqa_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    decode_gqa_kernel<D, G><<<dim3(a.max_splits, a.Hkv, a.B), kWarps * 32, C::SMEM, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool gqa_decode_supported(int d, int g) { return (d == 64 || d == 128) && (g == 4 || g == 8); }

cudaError_t launch_decode_gqa(const DecodeArgs& a, cudaStream_t st) {
#define KVC_CASE(D, G) \
    if (a.d == D && a.g == G) return launch_t<D, G>(a, st);
    KVC_CASE(128, 4) KVC_CASE(128, 8) KVC_CASE(64, 4) KVC_CASE(64, 8)
#undef KVC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kvc
