// int8_gate.cu -- gated fallback of the INT8 tier.
//
// [WITCERT] "SGLang 生产级落地与闭环门控修复": once the risk of a head or of a block
// crosses the water line, the lossless block is swapped in from the full-precision
// backing store and its witness stub is zeroed; in the saturated zone blocks are
// ranked by risk score and truncated.  Here:
//  * the risk of a complete block is the largest c_t of its 16 tokens over the query
//    heads of its KV head (from a decode's per-token bound);
//  * the gate picks every block with tanh(risk) > tau, highest risk first, up to a
//    budget (host);
//  * a restored block's 16 K and V rows go, bf16 and unchanged, to a pool entry in the
//    state buffer; its witnesses become 0, the block map points at the entry and the
//    block joins its head's list; the quantized decode skips it and the exact-block
//    decode (int8_exact.cu) serves its tokens exactly (c_t = 0).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "kvc_internal.h"

namespace kvc {
namespace {

// one warp per block: max over g heads x 16 tokens of c_t
__global__ void __launch_bounds__(256) block_risk_kernel(const float* ct, float* risk, const int32_t* next_pos,
                                                         int Hq, int Hkv, int g, int S) {
    const int b = blockIdx.z, h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nblk = S / kQBlock;
    const int blk = blockIdx.x * 8 + warp;
    if (blk >= nblk) return;
    const int nfull = next_pos[b] & ~(kQBlock - 1);
    float r = 0.f;
    if ((blk + 1) * kQBlock <= nfull) {
        for (int idx = lane; idx < g * kQBlock; idx += 32) {
            const int hh = idx / kQBlock, t = idx % kQBlock;
            r = fmaxf(r, ct[((size_t)b * Hq + (size_t)h * g + hh) * S + (size_t)blk * kQBlock + t]);
        }
        for (int o = 16; o; o >>= 1) r = fmaxf(r, __shfl_xor_sync(0xffffffffu, r, o));
    }
    if (lane == 0) risk[((size_t)b * Hkv + h) * nblk + blk] = r;
}

constexpr int kRestoreBatch = 256;        // blocks per launch (kernel parameter space)

struct RestoreList {
    int n;
    int4 e[kRestoreBatch];                // (request, KV head, block, pool entry)
    int slot[kRestoreBatch];              // position in the head's list of restored blocks
};

// CTA per block: the 16 K and V rows, bf16 and unchanged, into the pool entry in the
// exact-block decode's order; witnesses to 0; block map and list entries
__global__ void __launch_bounds__(256) restore_kernel(const RestoreList L, const __nv_bfloat16* kfull,
                                                      const __nv_bfloat16* vfull, __nv_bfloat16* xpool,
                                                      __half* wit, int32_t* xmap, int32_t* xn, int32_t* xlist,
                                                      int32_t* xent, int Hkv, int S, int d) {
    if ((int)blockIdx.x >= L.n) return;
    const int4 e = L.e[blockIdx.x];
    const size_t row0 = ((size_t)e.x * Hkv + e.y) * S + (size_t)e.z * kQBlock;
    unsigned char* kd = reinterpret_cast<unsigned char*>(xpool + (size_t)e.w * 2 * kQBlock * d);
    unsigned char* vd = kd + kQBlock * d * 2;
    for (int i = threadIdx.x; i < kQBlock * d; i += blockDim.x) {
        const int t = i / d, x = i % d;
        *reinterpret_cast<__nv_bfloat16*>(kd + xk_offset(d, t, x)) = kfull[row0 * d + i];
        *reinterpret_cast<__nv_bfloat16*>(vd + xv_offset(d, t, x)) = vfull[row0 * d + i];
    }
    for (int i = threadIdx.x; i < kQBlock * kBands; i += blockDim.x) wit[row0 * kBands + i] = __float2half(0.f);
    if (threadIdx.x == 0) {
        const size_t head = (size_t)e.x * Hkv + e.y;
        xmap[head * (S / kQBlock) + e.z] = e.w;
        xlist[head * kMaxRestored + L.slot[blockIdx.x]] = e.z;
        xent[head * kMaxRestored + L.slot[blockIdx.x]] = e.w;
        atomicAdd(&xn[head], 1);
    }
}

}  // namespace

cudaError_t int8_drop_restored(kvc_handle* h, const int32_t* h_cut, cudaStream_t st) {
    const Shape& s = h->sh;
    const int nblk = s.S / kQBlock;
    int32_t* xmap = reinterpret_cast<int32_t*>(h->state + h->L.xmap);
    bool changed = false;
    for (int b = 0; b < s.B; ++b)
        for (int hh = 0; hh < s.Hkv; ++hh) {
            const size_t head = (size_t)b * s.Hkv + hh;
            bool head_changed = false;
            for (int blk = 0; blk < nblk; ++blk) {
                const size_t i = head * nblk + blk;
                if (h->xmap_h[i] < 0 || (blk + 1) * kQBlock <= h_cut[b]) continue;
                h->xfree.push_back(h->xmap_h[i]);
                h->xmap_h[i] = -1;
                h->xn_h[head] -= 1;
                cudaError_t e = cudaMemsetAsync(xmap + i, 0xff, 4, st);
                if (e != cudaSuccess) return e;
                head_changed = true;
            }
            if (!head_changed) continue;
            // the head's list keeps its surviving blocks, in their order
            int n = 0;
            for (int j = 0; j < kMaxRestored && n < h->xn_h[head]; ++j) {
                const int32_t blk = h->xlist_h[head * kMaxRestored + j];
                if (h->xmap_h[head * nblk + blk] != h->xent_h[head * kMaxRestored + j]) continue;
                h->xlist_h[head * kMaxRestored + n] = blk;
                h->xent_h[head * kMaxRestored + n] = h->xent_h[head * kMaxRestored + j];
                ++n;
            }
            for (const auto& pr : {std::make_pair(h->L.xlist, &h->xlist_h), std::make_pair(h->L.xent, &h->xent_h)}) {
                cudaError_t e = cudaMemcpyAsync(h->state + pr.first + head * kMaxRestored * 4,
                                                pr.second->data() + head * kMaxRestored, (size_t)n * 4,
                                                cudaMemcpyHostToDevice, st);
                if (e != cudaSuccess) return e;
            }
            changed = true;
        }
    if (!changed) return cudaSuccess;
    return cudaMemcpyAsync(h->state + h->L.xn, h->xn_h.data(), h->xn_h.size() * 4, cudaMemcpyHostToDevice, st);
}

}  // namespace kvc

using namespace kvc;

extern "C" int kvc_int8_block_risk(kvc_t h, const float* d_ct, float* d_risk, kvc_stream_t stream) {
    if (!h || !on_device(h) || !d_ct || !d_risk || !h->sh.int8) return KVC_ERR_ARG;
    if (h->sh.dither) return KVC_ERR_UNSUPPORTED;          // Tier B has no per-token bound
    // the gate restores blocks of contiguous caches that attend to their whole history
    if (h->sh.ring || h->sh.W > 0) return KVC_ERR_UNSUPPORTED;
    const Shape& s = h->sh;
    const int nblk = s.S / kQBlock;
    block_risk_kernel<<<dim3((nblk + 7) / 8, s.Hkv, s.B), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        d_ct, d_risk, reinterpret_cast<const int32_t*>(h->state + h->L.next_pos), s.Hq, s.Hkv, s.g, s.S);
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

extern "C" int kvc_int8_gate(const float* h_risk, int32_t B, int32_t Hkv, int32_t nblk, double tau,
                             int32_t max_blocks, int32_t* h_sel, int32_t* h_n_sel) {
    if (!h_risk || !h_n_sel || B < 1 || Hkv < 1 || nblk < 0 || max_blocks < 0 || (max_blocks > 0 && !h_sel))
        return KVC_ERR_ARG;
    struct Cand { float r; int32_t b, h, k; size_t idx; };
    std::vector<Cand> c;
    for (int32_t b = 0; b < B; ++b)
        for (int32_t hh = 0; hh < Hkv; ++hh)
            for (int32_t k = 0; k < nblk; ++k) {
                const float r = h_risk[((size_t)b * Hkv + hh) * nblk + k];
                if (std::tanh((double)r) > tau) c.push_back({r, b, hh, k, 0});
            }
    // highest risk first; ties in (request, head, block) order, the order of c
    for (size_t i = 0; i < c.size(); ++i) c[i].idx = i;
    const int32_t n = (int32_t)std::min<size_t>(c.size(), (size_t)max_blocks);
    std::partial_sort(c.begin(), c.begin() + n, c.end(),
                      [](const Cand& x, const Cand& y) { return x.r > y.r || (x.r == y.r && x.idx < y.idx); });
    for (int32_t i = 0; i < n; ++i) {
        h_sel[3 * i] = c[i].b;
        h_sel[3 * i + 1] = c[i].h;
        h_sel[3 * i + 2] = c[i].k;
    }
    *h_n_sel = n;
    return KVC_OK;
}

extern "C" int kvc_int8_restore(kvc_t h, const int32_t* h_blocks, int32_t n, const void* d_k_full,
                                const void* d_v_full, kvc_stream_t stream) {
    if (!h || !on_device(h) || n < 0 || (n > 0 && (!h_blocks || !d_k_full || !d_v_full)) || !h->sh.int8)
        return KVC_ERR_ARG;
    if (h->sh.dither) return KVC_ERR_UNSUPPORTED;
    const Shape& s = h->sh;
    const int nblk = s.S / kQBlock;
    // validate everything first: nothing is restored on error
    std::vector<int4> todo;
    std::vector<size_t> seen;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t b = h_blocks[3 * i], hh = h_blocks[3 * i + 1], k = h_blocks[3 * i + 2];
        if (b < 0 || b >= s.B || hh < 0 || hh >= s.Hkv || k < 0 || k >= nblk) return KVC_ERR_ARG;
        if ((k + 1) * kQBlock > (h->np[b] / kQBlock) * kQBlock) return KVC_ERR_ARG;   // not a complete block
        const size_t idx = ((size_t)b * s.Hkv + hh) * nblk + k;
        if (h->xmap_h[idx] >= 0 || std::find(seen.begin(), seen.end(), idx) != seen.end()) continue;
        seen.push_back(idx);
        todo.push_back(make_int4(b, hh, k, -1));
    }
    if (todo.size() > h->xfree.size()) return KVC_ERR_CAPACITY;
    {
        // the exact-rows split of the decode serves at most kMaxRestored blocks per head
        std::vector<int32_t> per(h->xn_h);
        for (const auto& e : todo)
            if (++per[(size_t)e.x * s.Hkv + e.y] > kMaxRestored) return KVC_ERR_CAPACITY;
    }
    std::vector<int> slots(todo.size());
    for (size_t i = 0; i < todo.size(); ++i) {
        int4& e = todo[i];
        const size_t head = (size_t)e.x * s.Hkv + e.y;
        e.w = h->xfree.back();
        h->xfree.pop_back();
        h->xmap_h[head * nblk + e.z] = e.w;
        slots[i] = h->xn_h[head];
        h->xlist_h[head * kMaxRestored + slots[i]] = e.z;
        h->xent_h[head * kMaxRestored + slots[i]] = e.w;
        h->xn_h[head] += 1;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (size_t i0 = 0; i0 < todo.size(); i0 += kRestoreBatch) {
        RestoreList L;
        L.n = (int)std::min<size_t>(kRestoreBatch, todo.size() - i0);
        std::memcpy(L.e, todo.data() + i0, L.n * sizeof(int4));
        std::memcpy(L.slot, slots.data() + i0, L.n * sizeof(int));
        restore_kernel<<<L.n, 256, 0, st>>>(
            L, static_cast<const __nv_bfloat16*>(d_k_full), static_cast<const __nv_bfloat16*>(d_v_full),
            reinterpret_cast<__nv_bfloat16*>(h->state + h->L.xpool), reinterpret_cast<__half*>(h->state + h->L.wit),
            reinterpret_cast<int32_t*>(h->state + h->L.xmap), reinterpret_cast<int32_t*>(h->state + h->L.xn),
            reinterpret_cast<int32_t*>(h->state + h->L.xlist), reinterpret_cast<int32_t*>(h->state + h->L.xent),
            s.Hkv, s.S, s.d);
        if (cudaGetLastError() != cudaSuccess) return KVC_ERR_CUDA;
    }
    return KVC_OK;
}
