// decode.cu -- split-K decode attention for one new query per request, and the
// cross-split combine.
//
// out = softmax(q . K^T / sqrt(d)) . V over the cached window of the newest
// token ([LOOP] §三 step; [LEAN] §2.1 with the window mask).  The key range of
// request b is split into chunks of `split` keys; each chunk yields, per query
// head, (m, l, acc[d]) with m the chunk's maximum logit (log2 domain), l the
// sum of 2^(logit - m) and acc the correspondingly weighted sum of values.  The
// combine rescales the chunks to a common maximum:
//     m* = max m_s,  out = sum_s 2^(m_s - m*) acc_s / sum_s 2^(m_s - m*) l_s.
// GQA: the g query heads of a KV head are served by the same CTA, so every K/V
// row is read from memory once per KV head.  Single-query decode needs no
// causal mask: every cached row precedes the query ([LOOP] §六).
#include "kvc_internal.h"

namespace kvc {

cudaError_t launch_decode_fast(const DecodeArgs& a, cudaStream_t st);  // decode_fast.cu
bool fast_decode_supported(const DecodeArgs& a);

namespace {

constexpr int kThreads = 128;

// Rotated query of KV head `kvh` of request b (g heads) into shared memory, fp32.
__device__ void load_query(const DecodeArgs& a, int b, int kvh, int t, int bf16, float* q) {
    const int d = a.d, half = d / 2;
    for (int idx = threadIdx.x; idx < a.g * half; idx += blockDim.x) {
        const int hh = idx / half, i = idx % half;
        const size_t off = ((size_t)b * a.Hq + (size_t)kvh * a.g + hh) * d;
        const float x0 = ld_elem(a.q, off + 2 * i, bf16), x1 = ld_elem(a.q, off + 2 * i + 1, bf16);
        float y0 = x0, y1 = x1;
        if (a.rope) rope_pair(x0, x1, a.rope[(size_t)t * half + i], y0, y1);
        q[hh * d + 2 * i] = y0;
        q[hh * d + 2 * i + 1] = y1;
    }
}

// Generic kernel: any dtype, any even d <= 256, any group size.  CTA =
// (chunk of kGenericSplit keys, KV head, request).  Straightforward two-pass
// evaluation of its chunk in shared memory.
template <int BF16>
__global__ void __launch_bounds__(kThreads) decode_generic_kernel(const DecodeArgs a) {
    extern __shared__ float smem[];
    const int b = blockIdx.z, kvh = blockIdx.y, chunk = blockIdx.x;
    const int len = a.next_pos[b];
    int lo, hi;
    key_range(len, a.S, a.W, a.ring, lo, hi);
    const int k0 = lo + chunk * a.split;
    if (k0 >= hi) return;
    const int nk = min(hi - k0, a.split);
    const int d = a.d, g = a.g;
    float* q = smem;               // [g][d]
    float* s = smem + g * d;       // [g][split]
    load_query(a, b, kvh, len - 1, BF16, q);
    __syncthreads();
    for (int idx = threadIdx.x; idx < g * nk; idx += blockDim.x) {
        const int hh = idx / nk, j = idx % nk;
        const size_t row = kv_row(a.table, b, kvh, k0 + j, a.Hkv, a.S) * d;
        float acc = 0.f;
        for (int i = 0; i < d; ++i) acc = fmaf(q[hh * d + i], ld_elem(a.k, row + i, BF16), acc);
        s[hh * a.split + j] = acc * a.scale_log2;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int hh = warp; hh < g; hh += nw) {
        float m = -INFINITY;
        for (int j = lane; j < nk; j += 32) m = fmaxf(m, s[hh * a.split + j]);
        for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        for (int j = lane; j < nk; j += 32) {
            const float p = exp2f(s[hh * a.split + j] - m);
            s[hh * a.split + j] = p;
            l += p;
        }
        for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0)
            a.part_ml[((size_t)b * a.Hq + (size_t)kvh * g + hh) * a.max_splits + chunk] = make_float2(m, l);
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < g * d; idx += blockDim.x) {
        const int hh = idx / d, i = idx % d;
        float acc = 0.f;
        for (int j = 0; j < nk; ++j)
            acc = fmaf(s[hh * a.split + j], ld_elem(a.v, kv_row(a.table, b, kvh, k0 + j, a.Hkv, a.S) * d + i, BF16), acc);
        a.part_acc[(((size_t)b * a.Hq + (size_t)kvh * g + hh) * a.max_splits + chunk) * d + i] = acc;
    }
}

// Combine: WPR warps per (request, query head) row, 8 / WPR rows per CTA.  One pass over
// the splits: warp w takes the splits w, w + WPR, ..., kU at a time with every load of a
// round issued together, and keeps a running maximum, denominator and weighted sum (lanes
// over 4-dim groups), rescaled when a round raises the maximum; the WPR warps' (m, l, acc)
// meet in shared memory once.  One warp per row when rows have few splits (more rows in
// flight), eight when rows are few and long, four otherwise.
constexpr int kCombineThreads = 256;
constexpr int kCombineU = 4;            // splits a warp loads per round

template <int WPR>
__global__ void __launch_bounds__(kCombineThreads) combine_rows_kernel(const CombineArgs c) {
    constexpr int kWarpsPerRow = WPR;
    constexpr int kRowsPerCta = kCombineThreads / 32 / WPR;
    __shared__ float4 sacc[kRowsPerCta][kWarpsPerRow][64];          // d <= 256
    __shared__ float2 sml[kRowsPerCta][kWarpsPerRow];               // each warp's (m, l)
    dep_wait();                                                      // launched dependent: see launch_dep
    dep_release();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = warp / kWarpsPerRow, w = warp % kWarpsPerRow;
    const size_t row = (size_t)blockIdx.x * kRowsPerCta + r;
    const bool valid = row < (size_t)c.B * c.Hq;
    const bool vec = c.d % 4 == 0;
    int ns = 0;
    const float2* ml = c.part_ml + row * c.max_splits;
    const float* pa = c.part_acc + row * c.max_splits * c.d;
    if (valid) {
        const int b = (int)(row / c.Hq);
        const int len = c.next_pos[b];
        int lo, hi;
        key_range(len, c.S, c.W, c.ring, lo, hi);
        if (c.align_lo) lo &= ~(kPage - 1);         // the paged GQA decode's split origin
        ns = (hi - lo + c.split - 1) / c.split;
    }
    if (valid && vec) {
        float m = -INFINITY, l = 0.f;
        float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
        for (int s0 = w; s0 < ns; s0 += kWarpsPerRow * kCombineU) {
            float2 v[kCombineU];
            float4 x[kCombineU][2];
#pragma unroll
            for (int u = 0; u < kCombineU; ++u) {
                const int s = s0 + u * kWarpsPerRow;
                v[u] = s < ns ? __ldg(ml + s) : make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int i0 = 4 * lane + 128 * k;
                    x[u][k] = (s < ns && i0 < c.d) ? __ldg(reinterpret_cast<const float4*>(pa + (size_t)s * c.d + i0))
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            float mn = m;
#pragma unroll
            for (int u = 0; u < kCombineU; ++u) mn = fmaxf(mn, v[u].x);
            if (mn == -INFINITY) continue;                      // no keys in any split so far
            const float sc = exp2f(m - mn);                     // 0 while m was -inf
            l *= sc;
#pragma unroll
            for (int k = 0; k < 2; ++k) { acc[k].x *= sc; acc[k].y *= sc; acc[k].z *= sc; acc[k].w *= sc; }
#pragma unroll
            for (int u = 0; u < kCombineU; ++u) {
                const float f = exp2f(v[u].x - mn);               // 0 for an empty split
                l = fmaf(v[u].y, f, l);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    acc[k].x = fmaf(x[u][k].x, f, acc[k].x); acc[k].y = fmaf(x[u][k].y, f, acc[k].y);
                    acc[k].z = fmaf(x[u][k].z, f, acc[k].z); acc[k].w = fmaf(x[u][k].w, f, acc[k].w);
                }
            }
            m = mn;
        }
        if (lane == 0) sml[r][w] = make_float2(m, l);
#pragma unroll
        for (int k = 0; k < 2; ++k)
            if (4 * lane + 128 * k < c.d) sacc[r][w][lane + 32 * k] = acc[k];
    }
    __syncthreads();
    if (!valid || w != 0) return;
    if (vec) {
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < kWarpsPerRow; ++k) M = fmaxf(M, sml[r][k].x);
        float f[kWarpsPerRow], L = 0.f;
#pragma unroll
        for (int k = 0; k < kWarpsPerRow; ++k) {
            f[k] = sml[r][k].x == -INFINITY ? 0.f : exp2f(sml[r][k].x - M);
            L = fmaf(sml[r][k].y, f[k], L);
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int i0 = 4 * lane; i0 < c.d; i0 += 128) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kWarpsPerRow; ++k) {
                const float4 x = sacc[r][k][i0 / 4];
                acc.x = fmaf(x.x, f[k], acc.x); acc.y = fmaf(x.y, f[k], acc.y);
                acc.z = fmaf(x.z, f[k], acc.z); acc.w = fmaf(x.w, f[k], acc.w);
            }
            const float o[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (c.bf16) static_cast<__nv_bfloat16*>(c.out)[row * c.d + i0 + e] = __float2bfloat16_rn(o[e]);
                else static_cast<float*>(c.out)[row * c.d + i0 + e] = o[e];
            }
        }
    } else {
        // head dims not a multiple of 4 (small shapes): the row's first warp alone, two passes
        float mx = -INFINITY;
        for (int s = lane; s < ns; s += 32) mx = fmaxf(mx, __ldg(ml + s).x);
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float L = 0.f;
        for (int s = lane; s < ns; s += 32) {
            const float2 v = __ldg(ml + s);
            L += v.y * exp2f(v.x - mx);
        }
        for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int i = lane; i < c.d; i += 32) {
            float acc = 0.f;
            for (int s = 0; s < ns; ++s) acc = fmaf(__ldg(pa + (size_t)s * c.d + i), exp2f(__ldg(ml + s).x - mx), acc);
            if (c.bf16) static_cast<__nv_bfloat16*>(c.out)[row * c.d + i] = __float2bfloat16_rn(acc * inv);
            else static_cast<float*>(c.out)[row * c.d + i] = acc * inv;
        }
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, const CombineArgs& c, bool fast, const KvMaps* maps, cudaStream_t st) {
    if (a.gqa) {
        if (!maps) return cudaErrorInvalidValue;
        cudaError_t e = launch_decode_gqa(a, *maps, st);
        if (e != cudaSuccess) return e;
    } else if (fast) {
        cudaError_t e = launch_decode_fast(a, st);
        if (e != cudaSuccess) return e;
    } else {
        dim3 grid(a.max_splits, a.Hkv, a.B);
        const size_t smem = (size_t)a.g * (a.d + a.split) * sizeof(float);
        // (the grant is always the largest, so shapes of different sizes never narrow it)
        const void* k = a.bf16 ? reinterpret_cast<const void*>(decode_generic_kernel<1>)
                               : reinterpret_cast<const void*>(decode_generic_kernel<0>);
        if (smem > 48 * 1024)
            if (cudaError_t e = allow_smem(k, kMaxSmemPerBlock)) return e;
        if (a.bf16) decode_generic_kernel<1><<<grid, kThreads, smem, st>>>(a);
        else decode_generic_kernel<0><<<grid, kThreads, smem, st>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const size_t rows = (size_t)a.B * a.Hq;
    if (a.max_splits <= 8)
        return launch_dep(combine_rows_kernel<1>, dim3((unsigned)((rows + 7) / 8)), dim3(kCombineThreads), 0, st, c);
    if (rows < 1024) return launch_dep(combine_rows_kernel<8>, dim3((unsigned)rows), dim3(kCombineThreads), 0, st, c);
    return launch_dep(combine_rows_kernel<4>, dim3((unsigned)((rows + 1) / 2)), dim3(kCombineThreads), 0, st, c);
}

}  // namespace kvc
