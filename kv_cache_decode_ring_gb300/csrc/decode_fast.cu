// decode_fast.cu -- split-K decode attention for bf16 caches, head_dim 64 or 128,
// 1..8 query heads per KV head, on sm_103a.
//
// Same mathematics as decode.cu ([LOOP] §三 step; [LEAN] §2.1): per split of
// kSplit keys and per query head, (m, l, acc[d]) with m in the log2 domain; the
// combine kernel merges the splits.
//
// Design (HBM-bound: every K/V byte is read once per KV head, and each byte
// feeds the g query heads of its group from shared memory):
//  * CTA = 4 warps = one split of 4 x 32 keys of one (request, KV head); a
//    grid-stride loop over splits keeps the launch valid for any length.
//  * Each warp copies its 32 K rows and 32 V rows (contiguous in the cache:
//    8 KB each for d = 128) with two cp.async.bulk copies completing on one
//    mbarrier; all copies of the CTA are issued before any wait, so three
//    resident CTAs keep up to 192 KB per SM in flight.
//  * Scores: lane = (16-byte chunk of the row, key group).  Each lane forms the
//    8-dim partial dot products of a batch of keys for all g heads, and a
//    reduce-scatter across the lanes of a row (log2(d/8) shuffle steps, halving
//    the values each step) leaves every lane with finished scores, instead of
//    an all-reduce per score.
//  * Softmax within the warp's 32 keys, then P.V with lanes owning 8 output
//    dims of every head; the warps' partials merge in shared memory.
//  * Waits on mbarriers are bounded (1 s of %globaltimer); on expiry the kernel
//    sets the device error word and leaves.
#include "kvc_internal.h"
#include "async_copy.h"

namespace kvc {
namespace {

constexpr int kWarps = 4;
constexpr int kTile = 32;                   // keys per warp
constexpr int kSplitKeys = kWarps * kTile;  // keys per CTA split

template <int D, int G>
struct Cfg {
    // scores: a lane holds QD dims of a key row for all G heads (16 for G <= 4, else 8,
    // bounding the query registers at 64), as the 16-byte chunks r, r + LPR, ... of the
    // row, so that the LPR lanes of a row read one contiguous 16*LPR-byte run per load
    static constexpr int QD = G <= 4 ? 16 : 8;
    static constexpr int LPR = D / QD;                // score lanes per row
    static constexpr int RPP = 32 / LPR;              // key groups per warp
    static constexpr int KPG = kTile / RPP;           // keys per group per tile
    static constexpr int KB0 = 2 * LPR / G;
    static constexpr int KB = KB0 < KPG ? (KB0 < 1 ? 1 : KB0) : KPG;  // keys per reduce batch
    static constexpr int M = KB * G;                  // partial sums per lane per batch
    static constexpr int OUT = M / LPR;               // finished scores per lane per batch
    // P.V: a lane holds 8 output dims of every head
    static constexpr int LPR2 = D / 8;
    static constexpr int RPP2 = 32 / LPR2;
    static constexpr int ROWB = D * 2;
    static constexpr int TILEB = kTile * ROWB;        // bytes of one warp's K (or V) tile
    static constexpr int PARTB = G * (D + 2) * 4;     // one warp's partial (m, l, acc)
    static_assert(M % LPR == 0 && OUT >= 1, "batch shape");
    static_assert(PARTB <= TILEB, "partial must fit in the warp's K tile");
    static constexpr int OFF_P = 2 * kWarps * TILEB;                    // scores [warp][kTile][G]
    static constexpr int OFF_Q = OFF_P + kWarps * kTile * G * 4;        // rotated scaled query [G][D]
    static constexpr int OFF_BAR = OFF_Q + G * D * 4;
    static constexpr size_t SMEM = OFF_BAR + kWarps * 8 + 128;
};

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32, 3) decode_fast_kernel(const DecodeArgs a) {
    using C = Cfg<D, G>;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* sK = smem;                                   // [warp][kTile][D] bf16
    unsigned char* sV = smem + kWarps * C::TILEB;               // [warp][kTile][D] bf16
    float* sP = reinterpret_cast<float*>(smem + C::OFF_P);     // [warp][kTile][G]
    float* sQ = reinterpret_cast<float*>(smem + C::OFF_Q);     // [G][D]
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, kvh = blockIdx.y;
    dep_wait();                              // launched dependent: see launch_dep
    dep_release();
    const int len = a.next_pos[b];
    int lo, hi;
    key_range(len, a.S, a.W, a.ring, lo, hi);
    const int nsplit = (hi - lo + kSplitKeys - 1) / kSplitKeys;
    if ((int)blockIdx.x >= nsplit) return;

    const int warp_ = threadIdx.x >> 5;
    const size_t head_row0 = ((size_t)b * a.Hkv + kvh) * a.S;
    const __nv_bfloat16* Kg = static_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* Vg = static_cast<const __nv_bfloat16*>(a.v);
    unsigned char* myK = sK + warp_ * C::TILEB;
    unsigned char* myV = sV + warp_ * C::TILEB;
    // paged: lane 0 loads the page numbers of its warp's tile of a split one split ahead
    // of the copies, so the block table's latency passes while the current split computes
    constexpr int kRuns = kTile / kPage + 1;              // pages a tile can touch
    int pf[kRuns];
    auto fetch_pages = [&](int split) {
        const int k0 = lo + split * kSplitKeys + warp_ * kTile;
        const int nk = max(0, min(kTile, hi - k0));
        const int32_t* trow = a.table + (size_t)b * (a.S / kPage);
#pragma unroll
        for (int j = 0; j < kRuns; ++j)
            pf[j] = (nk > 0 && (k0 / kPage + j) * kPage < k0 + nk) ? trow[k0 / kPage + j] : 0;
    };
    // lane 0 of each warp: copy its K/V rows of `split` (paged: from the pages in pf)
    auto issue = [&](int split) {
        const int k0 = lo + split * kSplitKeys + warp_ * kTile;
        const int nk = max(0, min(kTile, hi - k0));
        if ((threadIdx.x & 31) == 0 && nk > 0) {
            const uint32_t bytes = (uint32_t)nk * C::ROWB;
            mbar_arrive_expect_tx(&bar[warp_], 2 * bytes);
            if (!a.table) {
                bulk_copy_g2s(myK, Kg + (head_row0 + k0) * D, bytes, &bar[warp_]);
                bulk_copy_g2s(myV, Vg + (head_row0 + k0) * D, bytes, &bar[warp_]);
            } else {
                // one copy per run of rows inside one page
#pragma unroll
                for (int j = 0, r = 0; j < kRuns; ++j) {
                    if (r >= nk) break;
                    const int run = min(nk - r, kPage - (k0 + r) % kPage);
                    const int page = pf[j] < 0 ? 0 : pf[j];    // never taken: every slot read is mapped
                    const size_t row = ((size_t)page * a.Hkv + kvh) * kPage + (k0 + r) % kPage;
                    bulk_copy_g2s(myK + r * C::ROWB, Kg + row * D, (uint32_t)run * C::ROWB, &bar[warp_]);
                    bulk_copy_g2s(myV + r * C::ROWB, Vg + row * D, (uint32_t)run * C::ROWB, &bar[warp_]);
                    r += run;
                }
            }
        }
    };
    if ((threadIdx.x & 31) == 0) {
        mbar_init(&bar[warp_], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const bool pager = a.table && (threadIdx.x & 31) == 0;
    if (pager) fetch_pages(blockIdx.x);
    issue(blockIdx.x);                       // the first split's rows start moving at once
    if (pager && (int)(blockIdx.x + gridDim.x) < nsplit) fetch_pages(blockIdx.x + gridDim.x);

    // Query of the G heads, rotated at t = len - 1, fp32, times log2(e)/sqrt(d): once per CTA
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

    const int r = lane % C::LPR, grp = lane / C::LPR;          // score mapping
    const int r2 = lane % C::LPR2, grp2 = lane / C::LPR2;      // P.V mapping
    float q[G][C::QD];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < C::QD; e += 4) {
            const int dim = (r + (e / 8) * C::LPR) * 8 + (e % 8);
            const float4 f = *reinterpret_cast<const float4*>(sQ + h * D + dim);
            q[h][e] = f.x; q[h][e + 1] = f.y; q[h][e + 2] = f.z; q[h][e + 3] = f.w;
        }

    float* myP = sP + warp * kTile * G;
    uint32_t phase = 0;

    for (int split = blockIdx.x; split < nsplit; split += gridDim.x) {
        const int k0 = lo + split * kSplitKeys + warp * kTile;
        const int nk = max(0, min(kTile, hi - k0));
        float m_w[G], l_w[G], acc[G][8];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m_w[h] = -INFINITY; l_w[h] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
        }
        bool ok = true;
        if (nk > 0) {
            ok = mbar_wait(&bar[warp], phase);
            if (!ok) {
                // flag the error, give the copies in flight one more bounded wait, and
                // skip this split's arithmetic
                if (lane == 0) atomicOr(a.hdr, kErrWait);
                mbar_wait(&bar[warp], phase);
            }
            phase ^= 1u;                      // this warp's barrier completed one phase
        }
        if (nk > 0 && ok) {
            // ---- scores: batches of KB keys per group, reduce-scatter over the LPR lanes of a row
#pragma unroll
            for (int kb = 0; kb < C::KPG; kb += C::KB) {
                float part[C::M];
#pragma unroll
                for (int k = 0; k < C::KB; ++k) {
                    const int t = grp * C::KPG + kb + k;
                    float x[C::QD];
#pragma unroll
                    for (int e = 0; e < C::QD; e += 8) {
                        const uint4 u = *reinterpret_cast<const uint4*>(myK + t * C::ROWB + (r + (e / 8) * C::LPR) * 16);
                        bf16x8_to_f32(u, x + e);
                    }
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < C::QD; e += 2)
                            s2 = ffma2(make_float2(q[h][e], q[h][e + 1]), make_float2(x[e], x[e + 1]), s2);
                        part[k * G + h] = s2.x + s2.y;
                    }
                }
                // reduce-scatter: after the step with mask m, lanes with that bit set keep the
                // upper half of the remaining values; lane r ends with outputs [r*OUT, (r+1)*OUT)
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
            // ---- softmax over the warp's keys: lane = key
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float s = myP[lane * G + h];
                float mx = s;
#pragma unroll
                for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float p = exp2f(s - mx);           // masked keys: 2^-inf = 0
                myP[lane * G + h] = p;
                float l = p;
#pragma unroll
                for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
                m_w[h] = mx;
                l_w[h] = l;
            }
            __syncwarp();
            // ---- P.V: lane owns dims [8 r2, 8 r2 + 8) of every head for keys of its group
            for (int t = grp2; t < nk; t += C::RPP2) {
                const uint4 u = *reinterpret_cast<const uint4*>(myV + t * C::ROWB + r2 * 16);
                float x[8];
                bf16x8_to_f32(u, x);
                float pv[G];
#pragma unroll
                for (int h = 0; h < G; ++h) pv[h] = myP[t * G + h];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float2 pp = make_float2(pv[h], pv[h]);
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const float2 rr = ffma2(pp, make_float2(x[e], x[e + 1]), make_float2(acc[h][e], acc[h][e + 1]));
                        acc[h][e] = rr.x;
                        acc[h][e + 1] = rr.y;
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
        // ---- this warp's partial into its own K tile (done with K)
        __syncwarp();
        float* part_w = reinterpret_cast<float*>(myK);       // [G][2 + D]
        if (grp2 == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
#pragma unroll
                for (int e = 0; e < 8; ++e) part_w[h * (D + 2) + 2 + r2 * 8 + e] = acc[h][e];
                if (r2 == 0) { part_w[h * (D + 2)] = m_w[h]; part_w[h * (D + 2) + 1] = l_w[h]; }
            }
        }
        __syncthreads();
        // ---- merge the warps' partials and write the split's partial
        for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
            const int h = idx / D, i = idx % D;
            float mx = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w)
                mx = fmaxf(mx, reinterpret_cast<const float*>(sK + w * C::TILEB)[h * (D + 2)]);
            float l = 0.f, sacc = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float* pw = reinterpret_cast<const float*>(sK + w * C::TILEB) + h * (D + 2);
                const float f = pw[0] == -INFINITY ? 0.f : exp2f(pw[0] - mx);
                l += pw[1] * f;
                sacc += pw[2 + i] * f;
            }
            const size_t row = ((size_t)b * a.Hq + (size_t)kvh * G + h) * a.max_splits + split;
            a.part_acc[row * D + i] = sacc;
            if (i == 0) a.part_ml[row] = make_float2(mx, l);
        }
        // shared memory is rewritten by the next split's copies: order these generic
        // accesses before the async-proxy writes
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (split + (int)gridDim.x < nsplit) {
            issue(split + gridDim.x);
            if (pager && split + 2 * (int)gridDim.x < nsplit) fetch_pages(split + 2 * gridDim.x);
        }
    }
}

template <int D, int G>
cudaError_t launch_t(const DecodeArgs& a, int grid_x, cudaStream_t st) {
    using C = Cfg<D, G>;
    if (cudaError_t e = allow_smem(reinterpret_cast<const void*>(decode_fast_kernel<D, G>), C::SMEM)) return e;
    dim3 grid(grid_x, a.Hkv, a.B);
    return launch_dep(decode_fast_kernel<D, G>, grid, dim3(kWarps * 32), C::SMEM, st, a);
}

}  // namespace

bool fast_decode_supported(const DecodeArgs& a) {
    return (a.d == 64 || a.d == 128) && (a.g == 1 || a.g == 2 || a.g == 4 || a.g == 8) &&
           a.split == kSplitKeys;
}

cudaError_t launch_decode_fast(const DecodeArgs& a, cudaStream_t st) {
    // grid.x covers the longest window the cache can hold; CTAs beyond a request's
    // splits exit at once, and the grid-stride loop keeps any length covered
    const int grid_x = a.max_splits;
#define KVC_CASE(D, G) \
    if (a.d == D && a.g == G) return launch_t<D, G>(a, grid_x, st);
    KVC_CASE(128, 1) KVC_CASE(128, 2) KVC_CASE(128, 4) KVC_CASE(128, 8)
    KVC_CASE(64, 1) KVC_CASE(64, 2) KVC_CASE(64, 4) KVC_CASE(64, 8)
#undef KVC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kvc
