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
    static constexpr int LPR = D / 8;                 // lanes per row (one 16-B chunk each)
    static constexpr int RPP = 32 / LPR;              // rows (key groups) per warp
    static constexpr int KPG = kTile / RPP;           // keys per group per tile
    static constexpr int KB0 = 2 * LPR / G;
    static constexpr int KB = KB0 < KPG ? (KB0 < 1 ? 1 : KB0) : KPG;  // keys per reduce batch
    static constexpr int M = KB * G;                  // partial sums per lane per batch
    static constexpr int OUT = M / LPR;               // finished scores per lane per batch
    static constexpr int ROWB = D * 2;
    static constexpr int TILEB = kTile * ROWB;        // bytes of one warp's K (or V) tile
    static constexpr int PARTB = G * (D + 2) * 4;     // one warp's partial (m, l, acc)
    static_assert(M % LPR == 0 && OUT >= 1, "batch shape");
    static_assert(PARTB <= TILEB, "partial must fit in the warp's K tile");
    static constexpr size_t SMEM = 2 * (size_t)kWarps * TILEB + (size_t)kWarps * kTile * G * 4 + kWarps * 8 + 128;
};

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32, 3) decode_fast_kernel(const DecodeArgs a) {
    using C = Cfg<D, G>;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* sK = smem;                                   // [warp][kTile][D] bf16
    unsigned char* sV = smem + kWarps * C::TILEB;               // [warp][kTile][D] bf16
    float* sP = reinterpret_cast<float*>(smem + 2 * kWarps * C::TILEB);   // [warp][kTile][G]
    uint64_t* bar = reinterpret_cast<uint64_t*>(sP + kWarps * kTile * G);  // [warp]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, kvh = blockIdx.y;
    const int len = a.next_pos[b];
    int lo, hi;
    key_range(len, a.S, a.W, a.ring, lo, hi);
    const int nsplit = (hi - lo + kSplitKeys - 1) / kSplitKeys;
    if ((int)blockIdx.x >= nsplit) return;

    if (threadIdx.x < kWarps) mbar_init(&bar[threadIdx.x], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();

    // Query chunk of this lane for all G heads, rotated at t = len - 1, fp32,
    // pre-multiplied by log2(e)/sqrt(d).
    const int r = lane % C::LPR, grp = lane / C::LPR;
    float q[G][8];
    {
        const int t = len - 1;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const size_t off = ((size_t)b * a.Hq + (size_t)kvh * G + h) * D + r * 8;
            const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + off);
            float x[8];
            bf16x8_to_f32(u, x);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float y0 = x[2 * j], y1 = x[2 * j + 1];
                if (a.rope) rope_pair(x[2 * j], x[2 * j + 1], a.rope[(size_t)t * (D / 2) + r * 4 + j], y0, y1);
                q[h][2 * j] = y0 * a.scale_log2;
                q[h][2 * j + 1] = y1 * a.scale_log2;
            }
        }
    }

    const size_t head_row0 = ((size_t)b * a.Hkv + kvh) * a.S;
    const __nv_bfloat16* Kg = static_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* Vg = static_cast<const __nv_bfloat16*>(a.v);
    unsigned char* myK = sK + warp * C::TILEB;
    unsigned char* myV = sV + warp * C::TILEB;
    float* myP = sP + warp * kTile * G;
    uint32_t phase = 0;

    for (int split = blockIdx.x; split < nsplit; split += gridDim.x) {
        const int k0 = lo + split * kSplitKeys + warp * kTile;
        const int nk = max(0, min(kTile, hi - k0));

        // ---- issue this warp's copies
        if (lane == 0 && nk > 0) {
            const uint32_t bytes = (uint32_t)nk * C::ROWB;
            mbar_arrive_expect_tx(&bar[warp], 2 * bytes);
            bulk_copy_g2s(myK, Kg + (head_row0 + k0) * D, bytes, &bar[warp]);
            bulk_copy_g2s(myV, Vg + (head_row0 + k0) * D, bytes, &bar[warp]);
        }
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
                    const uint4 u = *reinterpret_cast<const uint4*>(myK + t * C::ROWB + r * 16);
                    float x[8];
                    bf16x8_to_f32(u, x);
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
            // ---- P.V: lane owns dims [8r, 8r+8) of every head for keys of its group
            for (int t = grp; t < nk; t += C::RPP) {
                const uint4 u = *reinterpret_cast<const uint4*>(myV + t * C::ROWB + r * 16);
                float x[8];
                bf16x8_to_f32(u, x);
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
        // ---- this warp's partial into its own K tile (done with K)
        __syncwarp();
        float* part_w = reinterpret_cast<float*>(myK);       // [G][2 + D]
        if (grp == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
#pragma unroll
                for (int e = 0; e < 8; ++e) part_w[h * (D + 2) + 2 + r * 8 + e] = acc[h][e];
                if (r == 0) { part_w[h * (D + 2)] = m_w[h]; part_w[h * (D + 2) + 1] = l_w[h]; }
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
            float l = 0.f, s = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float* pw = reinterpret_cast<const float*>(sK + w * C::TILEB) + h * (D + 2);
                const float f = pw[0] == -INFINITY ? 0.f : exp2f(pw[0] - mx);
                l += pw[1] * f;
                s += pw[2 + i] * f;
            }
            const size_t row = ((size_t)b * a.Hq + (size_t)kvh * G + h) * a.max_splits + split;
            a.part_acc[row * D + i] = s;
            if (i == 0) a.part_ml[row] = make_float2(mx, l);
        }
        // shared memory is rewritten by the next split's copies: order these generic
        // accesses before the async-proxy writes
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
    }
}

template <int D, int G>
cudaError_t launch_t(const DecodeArgs& a, int grid_x, cudaStream_t st) {
    using C = Cfg<D, G>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(decode_fast_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 grid(grid_x, a.Hkv, a.B);
    decode_fast_kernel<D, G><<<grid, kWarps * 32, C::SMEM, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool fast_decode_supported(const DecodeArgs& a) {
    return (a.d == 64 || a.d == 128) && (a.g == 1 || a.g == 2 || a.g == 4 || a.g == 8) &&
           a.split == kSplitKeys;
}

int fast_split_keys() { return kSplitKeys; }

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
