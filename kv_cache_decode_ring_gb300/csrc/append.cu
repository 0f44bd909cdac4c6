// append.cu -- cache writes: append one token or many rows, trim, INT8 block
// quantization with residual witnesses.
//
// [LOOP] §三 "KVCacheManager.step": write k_t, v_t at cache[:, :, pos]; pos < max_seq_len.
// [LEAN] §3.3 step / §3.4 ringToList: a ring of W slots, slot = position mod W,
//        each slot keeps its absolute position (§3.2 KV Cell).
// [PREFIX] "哪些東西必須一起裁剪": trim keeps rows [:cut] and sets next_position = cut.
// [WITCERT] "频带酉性与双层证书": per-token, per-band residual norms w_{t,b} (16 x fp16);
//        "SGLang 生产级落地与闭环门控修复": per-block scales; the write kernel
//        quantizes and records the band norms.
#include <algorithm>
#include <cstring>
#include <vector>

#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxGroup = 1024;  // requests per launch when per-request values ride in params

struct Group {
    int32_t val[kMaxGroup];  // counts (append) or cuts (trim)
    int b0, nb;
};

__device__ __forceinline__ void flag(uint32_t* hdr, uint32_t bit) { atomicOr(hdr, bit); }

__device__ __forceinline__ bool position_ok(const AppendArgs& a, long long p) {
    if (p < 0 || p > 0x7fffffffLL) return false;
    if (!a.ring && p >= a.S) return false;
    if (a.rope && p >= a.P) return false;
    return true;
}

// Stored value of element pair (2i, 2i+1) of a key row at position p.
__device__ __forceinline__ void key_pair(const AppendArgs& a, const void* src, size_t off, int i,
                                         int p, float& y0, float& y1) {
    float x0 = ld_elem(src, off + 2 * i, a.bf16), x1 = ld_elem(src, off + 2 * i + 1, a.bf16);
    if (a.rope) {
        rope_pair(x0, x1, a.rope[(size_t)p * (a.d / 2) + i], y0, y1);
    } else {
        y0 = x0; y1 = x1;
    }
}

__device__ __forceinline__ void store_pair(void* dst, size_t off, float y0, float y1, int bf16) {
    if (bf16) {
        __nv_bfloat162 t;
        t.x = __float2bfloat16_rn(y0);
        t.y = __float2bfloat16_rn(y1);
        *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(dst) + off) = t;
    } else {
        *reinterpret_cast<float2*>(static_cast<float*>(dst) + off) = make_float2(y0, y1);
    }
}

// ---------------------------------------------------------------------------
// INT8: quantize one 16-row block held in shared memory (fp32 copies of the
// exact bf16 values) and write codes, scales and witnesses.  All threads of the
// CTA take part.  s = amax/127 (IEEE division); code = clamp(rint(x/s), +-127);
// residual r = x - code*s is exact in fp32 (|r| <= s/2 on the grid of s), so one
// fma computes it exactly; band norms are summed in index order with every
// operation rounded toward +inf and stored as fp16 rounded up, so the witness
// is never below the true residual norm.
// Tier B ([WITCERT] subtractive dither): key code = clamp(rint(x/s + u)), u = r/256 - 1/2
// from the block's Philox calls (one per thread, bytes staged in shared memory; channel
// c takes byte c mod 16 of group c/16); values keep the plain quantizer; no witnesses.
// ---------------------------------------------------------------------------
// `blk` is the absolute block number (it keys the dither counters); the block is stored
// in block slot blk (contiguous) or blk mod S/16 (ring).
__device__ void quantize_block(const AppendArgs& a, const float* sK, const float* sV, float* red,
                               int b, int h, int blk) {
    const int pblk = a.ring ? blk % (a.S / kQBlock) : blk;
    const int d = a.d, n = kQBlock * d;
    uint8_t* du = reinterpret_cast<uint8_t*>(red + 64);        // [16][d] key dither bytes (Tier B)
    if (a.dither) {
        const int kg = d / 16;
        const uint32_t c2 = (uint32_t)h + a.layer_ctr, c3 = a.req_id[b];
        for (int i = threadIdx.x; i < kQBlock * kg; i += blockDim.x) {
            const int t = i / kg, j = i % kg;
            const uint4 r = philox4x32_10(make_uint4((uint32_t)(blk * kQBlock + t), (uint32_t)j, c2, c3), a.key0,
                                          a.key1);
            const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int e = 0; e < 16; ++e) du[t * d + 16 * j + e] = (uint8_t)(w[e >> 2] >> (8 * (e & 3)));
        }
    }
    float mk = 0.f, mv = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        mk = fmaxf(mk, fabsf(sK[i]));
        mv = fmaxf(mv, fabsf(sV[i]));
    }
    for (int o = 16; o; o >>= 1) {
        mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
        mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0) { red[warp] = mk; red[32 + warp] = mv; }
    __syncthreads();
    mk = 0.f; mv = 0.f;
    for (int w = 0; w < nw; ++w) { mk = fmaxf(mk, red[w]); mv = fmaxf(mv, red[32 + w]); }
    const float s_k = __fdiv_rn(mk, 127.0f), s_v = __fdiv_rn(mv, 127.0f);
    const size_t lin = int8_block(a.table, b, h, pblk, a.Hkv, a.S);
    const size_t row0 = lin * kQBlock;
    if (threadIdx.x == 0) {
        a.sk[lin] = s_k;
        a.sv[lin] = s_v;
    }
    // codes stored biased (c + 128) at the block positions kq_offset / vq_offset
    uint8_t* kb = reinterpret_cast<uint8_t*>(a.kq) + row0 * d;
    uint8_t* vb = reinterpret_cast<uint8_t*>(a.vq) + row0 * d;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int ck = 0, cv = 0;
        float yk = s_k != 0.f ? __fdiv_rn(sK[i], s_k) : 0.f;
        float yv = s_v != 0.f ? __fdiv_rn(sV[i], s_v) : 0.f;
        if (a.dither) yk = __fadd_rn(yk, __fmaf_rn((float)du[i], 0.00390625f, -0.5f));   // u = r/256 - 1/2, exact
        if (s_k != 0.f) ck = max(-127, min(127, __float2int_rn(yk)));
        if (s_v != 0.f) cv = max(-127, min(127, __float2int_rn(yv)));
        const int t = i / d, dim = i % d;
        kb[kq_offset(d, t, dim)] = (uint8_t)(ck + 128);
        vb[vq_offset(d, t, dim)] = (uint8_t)(cv + 128);
    }
    if (a.dither) return;                                // Tier B keeps no witnesses
    // witnesses: one thread per (row, band)
    const int bw = d / kBands;
    for (int rb = threadIdx.x; rb < kQBlock * kBands; rb += blockDim.x) {
        const int r = rb / kBands, band = rb % kBands;
        float acc = 0.f;
        for (int j = band * bw; j < (band + 1) * bw; ++j) {
            const float x = sK[r * d + j];
            int c = 0;
            if (s_k != 0.f) c = max(-127, min(127, __float2int_rn(__fdiv_rn(x, s_k))));
            const float res = __fmaf_rn(-(float)c, s_k, x);   // exact
            acc = __fadd_ru(acc, __fmul_ru(res, res));
        }
        a.wit[(row0 + r) * kBands + band] = __float2half_ru(__fsqrt_ru(acc));
    }
}

// One token per request.  CTA (b, y) writes KV heads [y hpc, (y + 1) hpc) of request b
// (and, for the INT8 tiers, quantizes their blocks when the row completes one).  Every
// CTA of the request reads next_position[b] first; the last of them to finish (an
// arrival counter, reset by that CTA) writes positions[slot] and advances
// next_position[b], so no CTA can read the advanced value.
__global__ void __launch_bounds__(kThreads) append_token_kernel(const AppendArgs a) {
    extern __shared__ float smem[];
    dep_wait();                                        // launched dependent: see launch_dep
    dep_release();
    const int b = blockIdx.x;
    const int p = a.next_pos[b];
    if (!position_ok(a, p)) {                          // (every CTA of the request returns here)
        if (threadIdx.x == 0 && blockIdx.y == 0) flag(a.hdr, kErrPosition);
        return;
    }
    const int h0 = blockIdx.y * a.hpc;
    const int nh = min(a.Hkv - h0, a.hpc);             // KV heads of this CTA (>= 1)
    const int d = a.d, half = d / 2;
    const int slot = a.ring ? p % a.S : p;
    const int tslot = p % kQBlock;                     // INT8: the row's place in the exact tail
    if (a.bf16 && d % 8 == 0) {
        // 8 elements (16 bytes) per item, kU items per thread with every load issued
        // before any arithmetic: one round trip for the whole row set.  The rows go to
        // the cache (bf16) or to the exact tail (INT8 tier).
        constexpr int kU = 4;
        const int vec = d / 8, n = nh * vec;
        const uint4* K = static_cast<const uint4*>(a.k);
        const uint4* V = static_cast<const uint4*>(a.v);
        __nv_bfloat16* kdst = a.int8 ? a.ktail : static_cast<__nv_bfloat16*>(a.kc);
        __nv_bfloat16* vdst = a.int8 ? a.vtail : static_cast<__nv_bfloat16*>(a.vc);
        for (int base = threadIdx.x; base < n; base += kU * blockDim.x) {
            uint4 kx[kU], vx[kU];
            float4 cs[kU][2];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int idx = base + u * blockDim.x;
                if (idx >= n) continue;
                const int h = h0 + idx / vec, c = idx % vec;
                kx[u] = __ldg(K + ((size_t)b * a.Hkv + h) * vec + c);
                vx[u] = __ldg(V + ((size_t)b * a.Hkv + h) * vec + c);
                if (a.rope) {
                    const float4* r = reinterpret_cast<const float4*>(a.rope + (size_t)p * half + 4 * c);
                    cs[u][0] = __ldg(r);
                    cs[u][1] = __ldg(r + 1);
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int idx = base + u * blockDim.x;
                if (idx >= n) continue;
                const int h = h0 + idx / vec, c = idx % vec;
                const size_t dst = (a.int8 ? (((size_t)b * a.Hkv + h) * kQBlock + tslot)
                                           : kv_row(a.table, b, h, slot, a.Hkv, a.S)) * d + 8 * c;
                uint4 ko = kx[u];
                if (a.rope) {
                    uint32_t w[4] = {kx[u].x, kx[u].y, kx[u].z, kx[u].w};
                    const float2 r[4] = {make_float2(cs[u][0].x, cs[u][0].y), make_float2(cs[u][0].z, cs[u][0].w),
                                         make_float2(cs[u][1].x, cs[u][1].y), make_float2(cs[u][1].z, cs[u][1].w)};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __nv_bfloat162 x2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
                        float y0, y1;
                        rope_pair(__low2float(x2), __high2float(x2), r[e], y0, y1);
                        const __nv_bfloat162 o2 = __floats2bfloat162_rn(y0, y1);
                        w[e] = *reinterpret_cast<const uint32_t*>(&o2);
                    }
                    ko = make_uint4(w[0], w[1], w[2], w[3]);
                }
                *reinterpret_cast<uint4*>(kdst + dst) = ko;
                *reinterpret_cast<uint4*>(vdst + dst) = vx[u];
            }
        }
        if (a.int8 && tslot == kQBlock - 1) {
            // the 16th row completes the block: every KV head quantizes its 16 tail rows
            float* sK = smem;
            float* sV = smem + kQBlock * d;
            float* red = smem + 2 * kQBlock * d;
            __threadfence_block();
            for (int h = h0; h < h0 + nh; ++h) {
                const size_t tail = ((size_t)b * a.Hkv + h) * kQBlock * d;
                __syncthreads();                       // the tail rows written; smem free
                for (int i = threadIdx.x; i < kQBlock * d; i += blockDim.x) {
                    sK[i] = __bfloat162float(a.ktail[tail + i]);
                    sV[i] = __bfloat162float(a.vtail[tail + i]);
                }
                __syncthreads();
                quantize_block(a, sK, sV, red, b, h, p / kQBlock);
            }
        }
    } else {
        // fp32 caches and other head sizes (never INT8: that tier is bf16 with d % 16 == 0)
        for (int idx = threadIdx.x; idx < nh * half; idx += blockDim.x) {
            const int h = h0 + idx / half, i = idx % half;
            const size_t src = ((size_t)b * a.Hkv + h) * d;
            const size_t dst = kv_row(a.table, b, h, slot, a.Hkv, a.S) * d;
            float y0, y1;
            key_pair(a, a.k, src, i, p, y0, y1);
            store_pair(a.kc, dst + 2 * i, y0, y1, a.bf16);
            store_pair(a.vc, dst + 2 * i, ld_elem(a.v, src + 2 * i, a.bf16),
                       ld_elem(a.v, src + 2 * i + 1, a.bf16), a.bf16);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        bool last = gridDim.y == 1;
        if (!last) {
            __threadfence();                            // this CTA's rows, before its arrival
            last = atomicAdd(&a.arrive[b], 1) == (int)gridDim.y - 1;
            if (last) {
                a.arrive[b] = 0;
                __threadfence();
            }
        }
        if (last) {
            a.pos[(size_t)b * a.S + slot] = p;
            a.next_pos[b] = p + 1;
        }
    }
}

// Many rows per request (non-INT8).  CTA (row tile, KV head, request) writes
// rows; next_position is only read here and advanced by advance_kernel.
__global__ void __launch_bounds__(kThreads) append_rows_kernel(const AppendArgs a, const Group g) {
    const int bi = blockIdx.z, b = g.b0 + bi, h = blockIdx.y;
    const int cnt = g.val[bi];
    const int np = a.next_pos[b];
    const int d = a.d, half = d / 2;
    const int rows_per_cta = kThreads / half > 0 ? kThreads / half : 1;
    const int r = blockIdx.x * rows_per_cta + threadIdx.x / half;
    const int i = threadIdx.x % half;
    if (threadIdx.x >= rows_per_cta * half || r >= cnt) return;
    if (a.ring && r < cnt - a.S) return;            // overwritten later in this call
    const long long p = (long long)np + r;
    if (!position_ok(a, p)) {
        flag(a.hdr, kErrPosition);
        return;
    }
    const int slot = a.ring ? (int)(p % a.S) : (int)p;
    const size_t src = (size_t)b * a.sb + (size_t)h * a.sh + (size_t)r * a.sr;
    const size_t dst = kv_row(a.table, b, h, slot, a.Hkv, a.S) * d;
    float y0, y1;
    key_pair(a, a.k, src, i, (int)p, y0, y1);
    store_pair(a.kc, dst + 2 * i, y0, y1, a.bf16);
    store_pair(a.vc, dst + 2 * i, ld_elem(a.v, src + 2 * i, a.bf16), ld_elem(a.v, src + 2 * i + 1, a.bf16),
               a.bf16);
    if (h == 0 && i == 0) a.pos[(size_t)b * a.S + slot] = (int)p;
}

// Many bf16 rows per request, 16 bytes (8 elements) per thread: d/8 threads per row.
// Same per-pair arithmetic and rounding as append_rows_kernel (RoPE in fp32, one bf16
// rounding per element; values copied bit for bit); the inputs are 16-byte aligned.
__global__ void __launch_bounds__(kThreads) append_rows_vec_kernel(const AppendArgs a, const Group g) {
    const int bi = blockIdx.z, b = g.b0 + bi, h = blockIdx.y;
    const int cnt = g.val[bi];
    const int np = a.next_pos[b];
    const int vec = a.d / 8;
    const int rows_per_cta = kThreads / vec;
    const int r = blockIdx.x * rows_per_cta + threadIdx.x / vec;
    const int c = threadIdx.x % vec;
    if (threadIdx.x >= rows_per_cta * vec || r >= cnt) return;
    if (a.ring && r < cnt - a.S) return;            // overwritten later in this call
    const long long p = (long long)np + r;
    if (!position_ok(a, p)) {
        flag(a.hdr, kErrPosition);
        return;
    }
    const int slot = a.ring ? (int)(p % a.S) : (int)p;
    const size_t src = (size_t)b * a.sb + (size_t)h * a.sh + (size_t)r * a.sr + 8 * (size_t)c;
    const uint4 kx = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.k) + src));
    const uint4 vx = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.v) + src));
    uint4 ko = kx;
    if (a.rope) {
        const float4* rp = reinterpret_cast<const float4*>(a.rope + (size_t)p * (a.d / 2) + 4 * c);
        const float4 c0 = __ldg(rp), c1 = __ldg(rp + 1);
        uint32_t w[4] = {kx.x, kx.y, kx.z, kx.w};
        const float2 cs[4] = {make_float2(c0.x, c0.y), make_float2(c0.z, c0.w),
                              make_float2(c1.x, c1.y), make_float2(c1.z, c1.w)};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 x2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
            float y0, y1;
            rope_pair(__low2float(x2), __high2float(x2), cs[e], y0, y1);
            const __nv_bfloat162 o2 = __floats2bfloat162_rn(y0, y1);
            w[e] = *reinterpret_cast<const uint32_t*>(&o2);
        }
        ko = make_uint4(w[0], w[1], w[2], w[3]);
    }
    const size_t dst = kv_row(a.table, b, h, slot, a.Hkv, a.S) * a.d + 8 * (size_t)c;
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.kc) + dst) = ko;
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.vc) + dst) = vx;
    if (h == 0 && c == 0) a.pos[(size_t)b * a.S + slot] = (int)p;
}

// INT8 rows, phase 1: every 16-position block that the new rows complete.
// CTA (block index from floor(np/16), KV head, request).  Rows below np come
// from the tail, the rest from the input.  Phase 2 (tail_kernel) writes the
// rows of a still-incomplete last block after this kernel has read the tail.
__global__ void __launch_bounds__(kThreads) quantize_rows_kernel(const AppendArgs a, const Group g) {
    extern __shared__ float smem[];
    const int bi = blockIdx.z, b = g.b0 + bi, h = blockIdx.y;
    const int cnt = g.val[bi];
    const int np = a.next_pos[b];
    const int blk = np / kQBlock + blockIdx.x;
    const int p0 = blk * kQBlock;
    if (p0 + kQBlock > np + cnt) return;             // block not completed by this call
    // a ring keeps the newest S/16 complete blocks: one overwritten later in this call is skipped
    if (a.ring && p0 < ((np + cnt) / kQBlock) * kQBlock - a.S) return;
    if (!position_ok(a, (long long)p0 + kQBlock - 1)) {
        if (threadIdx.x == 0) flag(a.hdr, kErrPosition);
        return;
    }
    const int d = a.d, half = d / 2;
    float* sK = smem;
    float* sV = smem + kQBlock * d;
    float* red = smem + 2 * kQBlock * d;
    const size_t tail = ((size_t)b * a.Hkv + h) * kQBlock * d;
    for (int idx = threadIdx.x; idx < kQBlock * half; idx += blockDim.x) {
        const int r = idx / half, i = idx % half, p = p0 + r;
        float k0, k1, v0, v1;
        if (p < np) {
            k0 = __bfloat162float(a.ktail[tail + (size_t)r * d + 2 * i]);
            k1 = __bfloat162float(a.ktail[tail + (size_t)r * d + 2 * i + 1]);
            v0 = __bfloat162float(a.vtail[tail + (size_t)r * d + 2 * i]);
            v1 = __bfloat162float(a.vtail[tail + (size_t)r * d + 2 * i + 1]);
        } else {
            const size_t src = (size_t)b * a.sb + (size_t)h * a.sh + (size_t)(p - np) * a.sr;
            key_pair(a, a.k, src, i, p, k0, k1);
            k0 = __bfloat162float(__float2bfloat16_rn(k0));
            k1 = __bfloat162float(__float2bfloat16_rn(k1));
            v0 = ld_elem(a.v, src + 2 * i, 1);
            v1 = ld_elem(a.v, src + 2 * i + 1, 1);
        }
        sK[r * d + 2 * i] = k0; sK[r * d + 2 * i + 1] = k1;
        sV[r * d + 2 * i] = v0; sV[r * d + 2 * i + 1] = v1;
    }
    __syncthreads();
    quantize_block(a, sK, sV, red, b, h, blk);
    if (h == 0)
        for (int r = threadIdx.x; r < kQBlock; r += blockDim.x)
            a.pos[(size_t)b * a.S + (a.ring ? (p0 + r) % a.S : p0 + r)] = p0 + r;
}

// INT8 rows, phase 2 (one CTA per request): rows of the last, incomplete block
// go to the exact tail; then next_position advances.
__global__ void __launch_bounds__(kThreads) tail_kernel(const AppendArgs a, const Group g) {
    const int bi = blockIdx.x, b = g.b0 + bi;
    const int cnt = g.val[bi];
    const int np = a.next_pos[b];
    const int end = np + cnt;
    const int first = max(np, (end / kQBlock) * kQBlock);   // rows of the incomplete block
    const int d = a.d, half = d / 2;
    for (int idx = threadIdx.x; idx < a.Hkv * (end - first) * half; idx += blockDim.x) {
        const int h = idx / ((end - first) * half);
        const int rem = idx % ((end - first) * half);
        const int p = first + rem / half, i = rem % half;
        if (!position_ok(a, p)) { flag(a.hdr, kErrPosition); continue; }
        const size_t src = (size_t)b * a.sb + (size_t)h * a.sh + (size_t)(p - np) * a.sr;
        const size_t tail = (((size_t)b * a.Hkv + h) * kQBlock + p % kQBlock) * d;
        float k0, k1;
        key_pair(a, a.k, src, i, p, k0, k1);
        a.ktail[tail + 2 * i] = __float2bfloat16_rn(k0);
        a.ktail[tail + 2 * i + 1] = __float2bfloat16_rn(k1);
        a.vtail[tail + 2 * i] = __float2bfloat16_rn(ld_elem(a.v, src + 2 * i, 1));
        a.vtail[tail + 2 * i + 1] = __float2bfloat16_rn(ld_elem(a.v, src + 2 * i + 1, 1));
        if (h == 0 && i == 0 && (a.ring || p < a.S)) a.pos[(size_t)b * a.S + (a.ring ? p % a.S : p)] = p;
    }
    __syncthreads();
    if (threadIdx.x == 0) a.next_pos[b] = end;
}

__global__ void advance_kernel(int32_t* next_pos, const Group g) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < g.nb) next_pos[g.b0 + i] += g.val[i];
}

// Trim: CTA per request.  Contiguous: slots [cut, old next_position) become
// empty.  Ring: every slot holding a position >= cut becomes empty.
__global__ void trim_kernel(int32_t* next_pos, int32_t* pos, const Group g, int S, int ring) {
    const int bi = blockIdx.x, b = g.b0 + bi;
    const int cut = g.val[bi];
    const int np = next_pos[b];
    int32_t* pb = pos + (size_t)b * S;
    if (ring) {
        for (int s = threadIdx.x; s < S; s += blockDim.x)
            if (pb[s] >= cut) pb[s] = -1;
    } else {
        for (int s = cut + threadIdx.x; s < np && s < S; s += blockDim.x) pb[s] = -1;
    }
    __syncthreads();
    if (threadIdx.x == 0) next_pos[b] = cut;
}

// rows of K and V in fp32, the reduction slots, and the key dither bytes of Tier B
size_t quant_smem(int d) { return (size_t)(2 * kQBlock * d + 64) * sizeof(float) + kQBlock * d; }

// ---- paged caches: the block table ------------------------------------------
constexpr int kTableBatch = 256;

struct TableUpdates {
    int n;
    int2 e[kTableBatch];                  // (table index, physical page)
};

__global__ void table_update_kernel(const TableUpdates u, int32_t* table) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < u.n) table[u.e[i].x] = u.e[i].y;
}

}  // namespace

// Map the pages that slots [from[b], to[b]) of every request b need (a ring's slots
// wrap modulo S), from the host free list; the device table follows on `st`.  On
// exhaustion nothing is mapped and *status = KVC_ERR_CAPACITY.
cudaError_t map_pages(kvc_handle* h, const std::vector<int>& from, const std::vector<int>& to, cudaStream_t st,
                      int* status) {
    const Shape& s = h->sh;
    const int np = s.S / kPage;
    std::vector<int> need;                 // table indices to map, in request and page order
    for (int b = 0; b < s.B; ++b) {
        const long long lo = from[b], hi = to[b];
        if (hi <= lo) continue;
        for (int lp = 0; lp < np; ++lp) {
            const size_t idx = (size_t)b * np + lp;
            if (h->table_h[idx] >= 0) continue;
            if (page_touched(s, lp, lo, hi)) need.push_back((int)idx);
        }
    }
    *status = KVC_OK;
    if (need.empty()) return cudaSuccess;
    if (need.size() > h->page_free.size()) { *status = KVC_ERR_CAPACITY; return cudaSuccess; }
    std::vector<int2> upd;
    for (int idx : need) {
        const int page = h->page_free.back();
        h->page_free.pop_back();
        h->table_h[idx] = page;
        upd.push_back(make_int2(idx, page));
    }
    int32_t* table = reinterpret_cast<int32_t*>(h->state + h->L.table);
    if (upd.size() > 4 * (size_t)kTableBatch)      // a large prefill: the whole table at once
        return cudaMemcpyAsync(table, h->table_h.data(), h->table_h.size() * 4, cudaMemcpyHostToDevice, st);
    for (size_t i0 = 0; i0 < upd.size(); i0 += kTableBatch) {
        TableUpdates u;
        u.n = (int)std::min<size_t>(kTableBatch, upd.size() - i0);
        std::memcpy(u.e, upd.data() + i0, u.n * sizeof(int2));
        table_update_kernel<<<1, kTableBatch, 0, st>>>(u, table);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_append_token(const AppendArgs& a, cudaStream_t st) {
    const size_t smem = a.int8 ? quant_smem(a.d) : 0;
    return launch_dep(append_token_kernel, dim3(a.B, (a.Hkv + a.hpc - 1) / a.hpc), dim3(kThreads), smem, st, a);
}

cudaError_t launch_append_rows_group(const AppendArgs& a, const Group& g, cudaStream_t st) {
    if (!a.int8) {
        const bool vec = a.bf16 && a.d % 8 == 0 && a.d / 8 <= kThreads &&
                         reinterpret_cast<uintptr_t>(a.k) % 16 == 0 && reinterpret_cast<uintptr_t>(a.v) % 16 == 0 &&
                         a.sb % 8 == 0 && a.sh % 8 == 0 && a.sr % 8 == 0;
        if (vec) {
            const int rows_per_cta = kThreads / (a.d / 8);
            dim3 grid((a.n + rows_per_cta - 1) / rows_per_cta, a.Hkv, g.nb);
            append_rows_vec_kernel<<<grid, kThreads, 0, st>>>(a, g);
        } else {
            const int half = a.d / 2;
            const int rows_per_cta = kThreads / half > 0 ? kThreads / half : 1;
            dim3 grid((a.n + rows_per_cta - 1) / rows_per_cta, a.Hkv, g.nb);
            append_rows_kernel<<<grid, kThreads, 0, st>>>(a, g);
        }
        advance_kernel<<<(g.nb + 255) / 256, 256, 0, st>>>(a.next_pos, g);
    } else {
        dim3 grid((a.n + kQBlock - 1) / kQBlock + 1, a.Hkv, g.nb);
        quantize_rows_kernel<<<grid, kThreads, quant_smem(a.d), st>>>(a, g);
        tail_kernel<<<g.nb, kThreads, 0, st>>>(a, g);
    }
    return cudaGetLastError();
}

}  // namespace kvc

namespace kvc {

// Host side of the grouped launches: per-request values travel in kernel
// parameters (no staging copies), kMaxGroup requests per launch.
cudaError_t launch_append_rows_counts(const AppendArgs& a, const int32_t* counts, cudaStream_t st) {
    for (int b0 = 0; b0 < a.B; b0 += kMaxGroup) {
        Group g;
        g.b0 = b0;
        g.nb = a.B - b0 < kMaxGroup ? a.B - b0 : kMaxGroup;
        for (int i = 0; i < g.nb; ++i) g.val[i] = counts[b0 + i];
        cudaError_t e = launch_append_rows_group(a, g, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_trim_cuts(int32_t* next_pos, int32_t* pos, const int32_t* cuts, int B, int S,
                             int ring, cudaStream_t st) {
    for (int b0 = 0; b0 < B; b0 += kMaxGroup) {
        Group g;
        g.b0 = b0;
        g.nb = B - b0 < kMaxGroup ? B - b0 : kMaxGroup;
        for (int i = 0; i < g.nb; ++i) g.val[i] = cuts[b0 + i];
        trim_kernel<<<g.nb, 256, 0, st>>>(next_pos, pos, g, S, ring);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace kvc
