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
// Layout read per (request, KV head): per 16-token block 16*d K code bytes and
// 16*d V code bytes (biased, in the block orders of kq_offset / vq_offset),
// fp16 witnesses [S][16], fp32 scales [S/16]; exact bf16 tail [16][d] for the
// rows of the incomplete block.
//
// Kernel shape: CTA = 4 warps = a split of 1024 tokens (64 blocks; 2048 for caches
// of 16384 slots or more; any multiple of 64 in between if configured); each warp
// streams its 16 to 32 blocks through two or three shared-memory stages (codes and
// witnesses by bulk copy on the stage's mbarrier; two where four CTAs fit on an SM),
// so copies overlap arithmetic; online softmax over the warp's blocks, warps merged
// at the end.  One extra split handles the exact tail rows of the incomplete block
// (c_t = 0 there).  Blocks restored to full precision by the gated fallback are
// skipped here and served by the exact-block decode (int8_exact.cu), whose splits
// follow.
//
// Both contractions of a block run on the tensor cores as fp16 MMAs with fp32
// accumulation (m16n8k16), operands built in registers:
//  * codes -> fp16 exactly: a byte permute makes 1024 + u from the biased byte
//    u = c + 128 and one half2 add subtracts 1152;
//  * scores, transposed: S^T[16 tokens][cols] = K[16][d] . Q^T[d][cols] where the
//    columns are (head, hi) and (head, lo): the rotated query, scaled by a power
//    of two, split into two fp16 parts (about 22 significant bits).  The result
//    fragment leaves lane L the whole scores of head L%4 for tokens L/4 and
//    L/4 + 8, so the block maximum is a 3-step shuffle among 8 lanes;
//  * P.V, transposed: O^T[d][cols] += V^T[d][16] . P^T[16][cols], P = the block's
//    softmax weights times s_V / (the warp's largest s_V), again as fp16 hi + lo.
//    Lane L accumulates the output of the same head L%4, so the online-softmax
//    rescale is local to the lane.  The reference maximum moves only when a
//    block exceeds it by more than 2^8 (log2 domain), so weights stay <= 2^8 and
//    the accumulators are rescaled rarely; the weights carry a 2^7 scale, which
//    keeps them normal fp16 numbers below 2^15.
// The bound is evaluated in fp32 from the fp32 query with every operation
// rounded toward +inf (band norms, products with the witnesses, their sums, an
// upward 1/sqrt(d)); tanh gets two ulps of headroom over CUDA tanhf's documented
// error.  Query and weight splits change the output by about 2^-22 relative.
#include <cmath>

#include "async_copy.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kWarps = 4;
// one 16-token block per tile; a warp takes split / (kWarps * 16) tiles (16 to 32)
constexpr float kLazyMax = 8.f;            // log2-domain headroom of the reference maximum
static_assert(kInt8Split % (kWarps * kQBlock) == 0 && kInt8SplitLong % (kWarps * kQBlock) == 0, "split shape");
static_assert(kInt8SplitLong / (kWarps * kQBlock) <= 32, "one tile's scales per lane");

struct Int8Args {
    const void* q;
    const int8_t* kq;
    const int8_t* vq;
    const float* sk;
    const float* sv;
    const __half* wit;
    const __nv_bfloat16* ktail;
    const __nv_bfloat16* vtail;
    const int32_t* xmap;            // [B][Hkv][S/16] pool entry of a restored block, -1 = quantized
    const int32_t* xn;              // [B][Hkv] restored blocks
    const __nv_bfloat16* xpool;     // [entry][2][16][d] K and V rows of restored blocks
    const int32_t* next_pos;
    const float2* rope;
    float2* part_ml;
    float* part_acc;
    float* part_c;
    float* ct;          // nullable: c_t per token [B][Hq][S]
    uint32_t* hdr;
    const uint32_t* req_id;         // Tier B: request IDs of the dither counters
    const int32_t* table;           // paged caches: the block table (a page is one block)
    uint32_t layer_ctr;             // Tier B: 65536 * layer
    uint32_t rk[20];                // Tier B: Philox round keys (k0 + r W0, k1 + r W1), r = 0..9
    int B, Hq, Hkv, d, S, max_splits;
    int W, ring;        // attention window (0 = all; a ring's is its size) and layout
    int split;          // tokens per quantized split
    int grid;           // grid columns: quantized splits + the exact-tail split
    float scale_log2;   // log2(e)/sqrt(d)
    float inv_sqrt_d_up;
};

struct Int8CombineArgs {
    const float2* part_ml;
    const float* part_acc;
    const float* part_c;
    const int32_t* next_pos;
    const int32_t* xn;              // [B][Hkv] restored blocks (they join the exact-rows split)
    void* out;
    float* cmax;        // nullable
    float* tanh_out;    // nullable
    int B, Hq, Hkv, d, S, max_splits, out_bf16;
    int W, ring;
    int split;          // tokens per quantized split
};

// D (16x8, fp32) += A (16x16, fp16, row) . B (16x8, fp16, col)
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four biased code bytes u = c + 128 -> two half2 words holding the exact codes:
// lo = (c0, c1), hi = (c2, c3).  0x64 above a byte u is the fp16 1024 + u.
__device__ __forceinline__ void codes_to_half2(uint32_t u, uint32_t& lo, uint32_t& hi) {
    uint32_t x, y;
    asm("prmt.b32 %0, %1, 0x64646464, 0x5140;" : "=r"(x) : "r"(u));
    asm("prmt.b32 %0, %1, 0x64646464, 0x7362;" : "=r"(y) : "r"(u));
    const __half2 off = __halves2half2(__ushort_as_half(0xE480), __ushort_as_half(0xE480));  // -1152
    const __half2 a = __hadd2(*reinterpret_cast<const __half2*>(&x), off);
    const __half2 b = __hadd2(*reinterpret_cast<const __half2*>(&y), off);
    lo = *reinterpret_cast<const uint32_t*>(&a);
    hi = *reinterpret_cast<const uint32_t*>(&b);
}

// Tier B: four dither bytes r -> two half2 words of -u = (128 - r)/256, exact in
// fp16: the byte permute makes 1024 + r, and one fma gives (1024 + r)(-1/256) + 4.5.
__device__ __forceinline__ void dither_to_half2(uint32_t r, uint32_t& lo, uint32_t& hi) {
    uint32_t x, y;
    asm("prmt.b32 %0, %1, 0x64646464, 0x5140;" : "=r"(x) : "r"(r));
    asm("prmt.b32 %0, %1, 0x64646464, 0x7362;" : "=r"(y) : "r"(r));
    const __half2 m = __halves2half2(__ushort_as_half(0x9C00), __ushort_as_half(0x9C00));   // -1/256
    const __half2 c = __halves2half2(__ushort_as_half(0x4480), __ushort_as_half(0x4480));   // 4.5
    const __half2 a = __hfma2(*reinterpret_cast<const __half2*>(&x), m, c);
    const __half2 b = __hfma2(*reinterpret_cast<const __half2*>(&y), m, c);
    lo = *reinterpret_cast<const uint32_t*>(&a);
    hi = *reinterpret_cast<const uint32_t*>(&b);
}

// Philox4x32-10 with the round keys precomputed on the host (kernel parameters, so
// each key xor folds into the three-input xor of its round).
// One 32 x 32 -> 64-bit product per multiplier, as the round defines it.
__device__ __forceinline__ uint4 philox_rk(uint4 c, const uint32_t (&rk)[20]) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        uint64_t p0, p1;
        asm("mul.wide.u32 %0, %1, 0xD2511F53;" : "=l"(p0) : "r"(c.x));
        asm("mul.wide.u32 %0, %1, 0xCD9E8D57;" : "=l"(p1) : "r"(c.z));
        c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ rk[2 * r], (uint32_t)p1,
                       (uint32_t)(p0 >> 32) ^ c.w ^ rk[2 * r + 1], (uint32_t)p0);
    }
    return c;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int w) {
    return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

// 2^x with the hardware approximation (relative error about 2^-22; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// x = hi + lo with hi = fp16(x) and lo = fp16(x - hi)
__device__ __forceinline__ void split_half(float x, __half& hi, __half& lo) {
    hi = __float2half_rn(x);
    lo = __float2half_rn(x - __half2float(hi));
}

template <int D, int G, bool DITHER = false>
struct I8 {
    static constexpr int KS = D / 16;               // k-steps of the score MMA (= m-tiles of P.V)
    static constexpr int NT = (2 * G + 7) / 8;      // 8-column tiles of (head, hi|lo) columns
    static constexpr int HPL = NT;                  // heads per lane (L%4, and 4 + L%4)
    static constexpr int KW = D / 16;               // K code words per lane per row (= KS)
    static constexpr int VW = D / 8;                // V code words per lane
    static constexpr int CB = kQBlock * D;          // bytes of one block's codes (K or V)
    static constexpr int WB = DITHER ? 0 : kQBlock * kBands * 2;     // witnesses (none in Tier B)
    static constexpr int STAGEB = 2 * CB + WB;
    // copy stages per warp: two at d = 128 with up to 4 heads per KV head (four CTAs per SM
    // then fit in registers and shared memory: more warps in flight), else three
    static constexpr int STAGES = (D == 128 && G <= 4) ? 2 : 3;
    static constexpr int WARPB = STAGES * STAGEB;
    static constexpr int PARTF = G * (D + 3);       // floats of one warp's partial (m, l, c, acc)
    static_assert(PARTF * 4 <= WARPB, "partial must fit in the warp's stages");
    // P^T staging per warp and column tile: 8 rows of 16 fp16 tokens; row n at
    // 32 n + 16 (n >= 4) bytes, so the lanes' stores and 8-byte loads are free of
    // bank conflicts
    static constexpr int PROWB = 288;
    // after the warps' stages: P^T staging [warp][NT] (the fp32 query during
    // preparation), fp16 query [2G][D], band norms [G][20], score factors [G],
    // barriers [warp][STAGES]
    static constexpr int OFF_P = kWarps * WARPB;
    static constexpr int PBYTES = (kWarps * NT * PROWB > G * D * 4 ? kWarps * NT * PROWB : G * D * 4);
    static constexpr int OFF_QH = OFF_P + ((PBYTES + 15) / 16) * 16;
    static constexpr int OFF_NQ = OFF_QH + 2 * G * D * 2;
    static constexpr int OFF_F = OFF_NQ + G * 20 * 4;       // norms padded to 20 floats a head
    static constexpr int OFF_BAR = OFF_F + ((G * 4 + 15) / 16) * 16;
    static constexpr size_t SMEM = OFF_BAR + kWarps * STAGES * 8 + 128;
};

__device__ __forceinline__ int prow(int n) { return 32 * n + (n >= 4 ? 16 : 0); }

// DITHER: Tier B ([WITCERT] subtractive dither on the keys).  Each lane regenerates,
// with Philox, exactly the dithers of the key codes it holds: rows g and g + 8 of the
// block over the dims qd (D/4) .. + D/4 - 1, i.e. D/64 whole groups of 16 channels
// per row.  The -u terms enter the score contraction as a second fp16 MMA into the
// same accumulator ((code - u) s = s code + s (-u)); values are plain codes.  No
// witnesses are read and no bound is formed.
// At most 4 heads per KV head (or d = 64) fit 4 CTAs per SM (at most 128 registers).
// GEN: a windowed, ring or paged cache (block slots from int8_window, blocks through the
// table, the first block masked before the window start); without it the kernel serves
// a contiguous cache attending to its whole history with none of that arithmetic.
template <int D, int G, bool DITHER, bool GEN>
__global__ void __launch_bounds__(kWarps * 32, (D < 128 || G <= 4) ? 4 : 3)
int8_decode_kernel(const Int8Args a) {
    using C = I8<D, G, DITHER>;
    constexpr int kStages = C::STAGES;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* sPm = smem + C::OFF_P;                                // [warp][NT] P^T staging
    __half* sQh = reinterpret_cast<__half*>(smem + C::OFF_QH);          // [2G][D]: row 2h hi, 2h + 1 lo
    float* sNQ = reinterpret_cast<float*>(smem + C::OFF_NQ);            // [G][20] band norms
    float* sF = reinterpret_cast<float*>(smem + C::OFF_F);              // [G] score factors
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);     // [warp][kStages]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
    dep_wait();                                                          // launched dependent: see launch_dep
    dep_release();
    const int len = a.next_pos[b];
    const int nfull = len & ~(kQBlock - 1);
    // the window's complete blocks: physical block slots [blo, bhi) (see int8_window)
    const Int8Window iw = GEN ? int8_window(len, a.S, a.W, a.ring)
                              : Int8Window{0, len / kQBlock, 0, len / kQBlock, a.S / kQBlock};
    const int bps = a.split / kQBlock;                        // blocks per split
    const int nsq = (iw.bhi - iw.blo + bps - 1) / bps;
    const int tpw = a.split / (kWarps * kQBlock);             // tiles per warp
    const bool tail_split = split == nsq;
    if (split > nsq || (tail_split && len == nfull && a.xn[(size_t)b * a.Hkv + kvh] == 0)) return;
    const int t_q = len - 1;
    const size_t rowq0 = (size_t)b * a.Hq + (size_t)kvh * G;    // first query row of the group

    if (tail_split) {
        // ---- exact tail rows [nfull, len), served in bf16 with c_t = 0.  Warp 0, 32 rows
        // at a time, online softmax over the chunks; lane = row for the scores, lane =
        // dims for P.V.  With no tail rows (a head with restored blocks) it writes the
        // empty partial, so the combine reads contiguous splits.
        if (warp != 0) return;
        const size_t bh = (size_t)b * a.Hkv + kvh;
        const int nt = len - nfull;
        float* qs = reinterpret_cast<float*>(smem);          // [G][D] scaled query
        float* pt = qs + G * D;                              // [32][G] weights of a chunk
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
        const size_t tail0 = bh * kQBlock * D;
        const int total = nt;
        auto row_ptr = [&](int r, bool v) { return (v ? a.vtail : a.ktail) + tail0 + (size_t)r * D; };
        auto row_pos = [&](int r) { return nfull + r; };
        float m[G], l[G], acc[G][D / 32];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m[h] = -INFINITY; l[h] = 0.f;
#pragma unroll
            for (int e = 0; e < D / 32; ++e) acc[h][e] = 0.f;
        }
        for (int r0 = 0; r0 < total; r0 += 32) {
            const int r = r0 + lane;
            const bool valid = r < total && (!GEN || nfull + r >= iw.lo);   // rows before the window: masked
            float s[G];
#pragma unroll
            for (int h = 0; h < G; ++h) s[h] = -INFINITY;
            if (valid) {
                const __nv_bfloat16* kr = row_ptr(r, false);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float x = 0.f;
                    for (int i = 0; i < D; ++i) x = fmaf(qs[h * D + i], __bfloat162float(kr[i]), x);
                    s[h] = x;
                }
                if (a.ct) {
                    const int p = row_pos(r);
                    const int slot = (GEN && a.ring) ? p % a.S : p;   // a ring's slot of position p
#pragma unroll
                    for (int h = 0; h < G; ++h) a.ct[(rowq0 + h) * a.S + slot] = 0.f;
                }
            }
            float alpha[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float mx = s[h];
                for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float mn = fmaxf(m[h], mx);                 // finite: the chunk holds the newest row
                alpha[h] = exp2f(m[h] - mn);                      // 0 on the first chunk
                const float p = valid ? exp2f(s[h] - mn) : 0.f;
                float ls = p;
                for (int o = 16; o; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
                l[h] = l[h] * alpha[h] + ls;
                m[h] = mn;
                pt[lane * G + h] = p;
            }
            __syncwarp();
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < D / 32; ++e) acc[h][e] *= alpha[h];
            const int nrow = min(32, total - r0);
            for (int j = 0; j < nrow; ++j) {
                const __nv_bfloat16* vr = row_ptr(r0 + j, true);
#pragma unroll
                for (int e = 0; e < D / 32; ++e) {
                    const float v = __bfloat162float(vr[lane + 32 * e]);
#pragma unroll
                    for (int h = 0; h < G; ++h) acc[h][e] = fmaf(pt[j * G + h], v, acc[h][e]);
                }
            }
            __syncwarp();
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const size_t row = (rowq0 + h) * a.max_splits + split;
            if (lane == 0) { a.part_ml[row] = make_float2(m[h], l[h]); a.part_c[row] = 0.f; }
#pragma unroll
            for (int e = 0; e < D / 32; ++e) a.part_acc[row * D + lane + 32 * e] = acc[h][e];
        }
        return;
    }

    // ---- quantized split ----------------------------------------------------
    const size_t bh = (size_t)b * a.Hkv + kvh;
    unsigned char* myS = smem + warp * C::WARPB;
    uint64_t* myBar = bar + warp * kStages;
    // block of this warp's tile i (tiles of the 4 warps interleaved)
    auto tile_blk = [&](int i) { return iw.blo + split * bps + i * kWarps + warp; };
    auto tile_ok = [&](int i) { return tile_blk(i) < iw.bhi; };
    auto issue = [&](int i) {
        if (lane == 0 && tile_ok(i)) {
            const size_t r0 = (GEN ? int8_block(a.table, b, kvh, tile_blk(i), a.Hkv, a.S)
                                   : bh * (a.S / kQBlock) + tile_blk(i)) * kQBlock;   // its first row
            const int sg = i % kStages;
            unsigned char* st = myS + sg * C::STAGEB;
            mbar_arrive_expect_tx(&myBar[sg], (uint32_t)C::STAGEB);
            bulk_copy_g2s(st, a.kq + r0 * D, C::CB, &myBar[sg]);
            bulk_copy_g2s(st + C::CB, a.vq + r0 * D, C::CB, &myBar[sg]);
            if (!DITHER) bulk_copy_g2s(st + 2 * C::CB, a.wit + r0 * kBands, C::WB, &myBar[sg]);
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

    // block scales of this warp's tiles: lane i < 16 holds tile i's s_K and its s_V
    // relative to the warp's largest s_V, times 2^7
    float skv = 0.f, rvv = 0.f;
    int xmv = -1;                                     // >= 0: restored, served by the exact split
    if (lane < tpw && tile_ok(lane)) {
        const size_t lin = GEN ? int8_block(a.table, b, kvh, tile_blk(lane), a.Hkv, a.S)
                               : bh * (a.S / kQBlock) + tile_blk(lane);
        skv = a.sk[lin];
        rvv = a.sv[lin];
        xmv = a.xmap[bh * (a.S / kQBlock) + tile_blk(lane)];
    }
    float svmax = rvv;
#pragma unroll
    for (int o = 16; o; o >>= 1) svmax = fmaxf(svmax, __shfl_xor_sync(0xffffffffu, svmax, o));
    rvv = svmax > 0.f ? rvv / svmax * 128.f : 0.f;

    // ---- query preparation, once per CTA while the copies fly: rotated fp32
    // query; per head a power-of-two scale 2^e putting max|q| in [2^14, 2^15),
    // the scaled query as fp16 hi + lo, and the band norms of the fp32 query,
    // rounded up, for the bound
    float* qf = reinterpret_cast<float*>(sPm);                 // [G][D] until the P staging uses it
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
        int ex = 0;
        frexpf(amax, &ex);                                    // amax = m 2^ex, m in [1/2, 1)
        const int e = max(-126, min(126, 15 - ex));
        const float up = __int_as_float((127 + e) << 23), down = __int_as_float((127 - e) << 23);
        for (int i = lane; i < D; i += 32) {
            __half hi, lo;
            split_half(qf[h * D + i] * up, hi, lo);
            sQh[(2 * h) * D + i] = hi;
            sQh[(2 * h + 1) * D + i] = lo;
        }
        if (lane < kBands) {
            float ss = 0.f;
            for (int e2 = lane * (D / kBands); e2 < (lane + 1) * (D / kBands); ++e2)
                ss = __fadd_ru(ss, __fmul_ru(qf[h * D + e2], qf[h * D + e2]));
            sNQ[h * 20 + lane] = __fsqrt_ru(ss);
        }
        if (lane == 0) sF[h] = (amax > 0.f ? down : 0.f) * a.scale_log2;
    }
    __syncthreads();

    // ---- per-lane fragments: g = L/4 (MMA group), qd = L%4
    const int g = lane >> 2, qd = lane & 3;
    // Tier B counter words: KV head + 65536 layer, request ID
    const uint32_t dc2 = (uint32_t)kvh + a.layer_ctr;
    const uint32_t dc3 = DITHER ? a.req_id[b] : 0u;
    // score B operand (Q^T): column n = 8 nt + g = (head n/2, hi|lo n%2); k-step s
    // covers the dims qd (D/4) + 4 s .. + 3 in the lane's registers
    uint32_t qb[C::NT][C::KS][2];
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
        const int n = 8 * nt + g;
#pragma unroll
        for (int s = 0; s < C::KS; ++s) {
            uint2 v = make_uint2(0u, 0u);
            if (n < 2 * G) v = *reinterpret_cast<const uint2*>(sQh + n * D + qd * (D / 4) + 4 * s);
            qb[nt][s][0] = v.x;
            qb[nt][s][1] = v.y;
        }
    }
    // the lane's heads (4 nt + qd; those >= G only carry dummy values)
    float fq[C::HPL];
#pragma unroll
    for (int nt = 0; nt < C::HPL; ++nt) fq[nt] = sF[min(4 * nt + qd, G - 1)];

    unsigned char* myPm = sPm + warp * C::NT * C::PROWB;
    float m_w[C::HPL], l_w[C::HPL], c_w[C::HPL];
    float acc[C::KS][C::NT][4];
#pragma unroll
    for (int nt = 0; nt < C::HPL; ++nt) { m_w[nt] = -INFINITY; l_w[nt] = 0.f; c_w[nt] = 0.f; }
#pragma unroll
    for (int mt = 0; mt < C::KS; ++mt)
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;

    for (int i = 0; i < tpw; ++i) {
        if (!tile_ok(i)) break;                   // later tiles of this warp are empty too
        const int sg = i % kStages;
        const uint32_t par = (uint32_t)((i / kStages) & 1);
        const unsigned char* tK = myS + sg * C::STAGEB;
        const unsigned char* tV = tK + C::CB;
        const uint4* tW = reinterpret_cast<const uint4*>(tK + 2 * C::CB);
        const int p0 = tile_blk(i) * kQBlock;                          // first slot of the block
        const int pa = GEN ? int8_abs_block(iw, tile_blk(i), a.ring) * kQBlock : p0;   // its first position
        // tokens g and g + 8 of the block before the window start are masked (first block only)
        const bool vis0 = !GEN || pa + g >= iw.lo, vis1 = !GEN || pa + g + 8 >= iw.lo;
        if (!mbar_wait(&myBar[sg], par)) {
            // give up: flag it, and let this stage's copy and the later stages'
            // (if issued) land before the stages are reused for the partial
            if (lane == 0) atomicOr(a.hdr, kErrWait);
            mbar_wait(&myBar[sg], par);
            for (int j = i + 1; j < i + kStages && j < tpw; ++j)
                if (tile_ok(j)) mbar_wait(&myBar[j % kStages], (uint32_t)((j / kStages) & 1));
            break;
        }
        const float s_k = __shfl_sync(0xffffffffu, skv, i);
        const float r_v = __shfl_sync(0xffffffffu, rvv, i);

        // a block restored by the gated fallback is served by the exact-rows split
        if (__shfl_sync(0xffffffffu, xmv, i) < 0) {
            // ---- scores S^T = K Q^T: rows g and g + 8 of the block, D/64 16-byte
            // chunks each (at d = 128 odd rows hold their chunk pairs swapped)
            uint32_t kw0[C::KW], kw1[C::KW];
    #pragma unroll
            for (int j = 0; j < C::KW / 4; ++j) {
                const int ch = (C::KW / 4) * qd + (D == 128 ? (j ^ (g & 1)) : j);
                const uint4 u0 = *reinterpret_cast<const uint4*>(tK + g * D + ch * 16);
                const uint4 u1 = *reinterpret_cast<const uint4*>(tK + (g + 8) * D + ch * 16);
                kw0[4 * j] = u0.x; kw0[4 * j + 1] = u0.y; kw0[4 * j + 2] = u0.z; kw0[4 * j + 3] = u0.w;
                kw1[4 * j] = u1.x; kw1[4 * j + 1] = u1.y; kw1[4 * j + 2] = u1.z; kw1[4 * j + 3] = u1.w;
            }
            float sacc[C::NT][4];
    #pragma unroll
            for (int nt = 0; nt < C::NT; ++nt)
    #pragma unroll
                for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
    #pragma unroll
            for (int s = 0; s < C::KS; ++s) {
                uint32_t a0, a1, a2, a3;
                codes_to_half2(kw0[s], a0, a2);
                codes_to_half2(kw1[s], a1, a3);
    #pragma unroll
                for (int nt = 0; nt < C::NT; ++nt) mma_f16(sacc[nt], a0, a1, a2, a3, qb[nt][s][0], qb[nt][s][1]);
            }
            if constexpr (DITHER) {
                // key group qd (D/64) + j of rows g and g + 8: words s = 4 j .. 4 j + 3
    #pragma unroll
                for (int j = 0; j < D / 64; ++j) {
                    const uint32_t grp = (uint32_t)(qd * (D / 64) + j);
                    const uint4 r0 = philox_rk(make_uint4((uint32_t)(pa + g), grp, dc2, dc3), a.rk);
                    const uint4 r1 = philox_rk(make_uint4((uint32_t)(pa + g + 8), grp, dc2, dc3), a.rk);
    #pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        uint32_t a0, a1, a2, a3;
                        dither_to_half2(word_of(r0, w), a0, a2);
                        dither_to_half2(word_of(r1, w), a1, a3);
    #pragma unroll
                        for (int nt = 0; nt < C::NT; ++nt)
                            mma_f16(sacc[nt], a0, a1, a2, a3, qb[nt][4 * j + w][0], qb[nt][4 * j + w][1]);
                    }
                }
            }

            // ---- online softmax of the lane's head over tokens g, g + 8; weights
            // times r_v into the P^T staging as fp16 hi + lo; and the bound
            float alpha[C::HPL];
            bool rescale = false;
    #pragma unroll
            for (int nt = 0; nt < C::HPL; ++nt) {
                const float f = fq[nt] * s_k;
                const float s0 = vis0 ? (sacc[nt][0] + sacc[nt][1]) * f : -INFINITY;
                const float s1 = vis1 ? (sacc[nt][2] + sacc[nt][3]) * f : -INFINITY;
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
                __half h0, l0, h1, l1;
                split_half(e0 * r_v, h0, l0);
                split_half(e1 * r_v, h1, l1);
                unsigned char* pt = myPm + nt * C::PROWB;
                *reinterpret_cast<__half*>(pt + prow(2 * qd) + 2 * g) = h0;
                *reinterpret_cast<__half*>(pt + prow(2 * qd + 1) + 2 * g) = l0;
                *reinterpret_cast<__half*>(pt + prow(2 * qd) + 2 * (g + 8)) = h1;
                *reinterpret_cast<__half*>(pt + prow(2 * qd + 1) + 2 * (g + 8)) = l1;

                if constexpr (DITHER) continue;                  // Tier B: no bound
                // bound of tokens g, g + 8 for head hq, every operation rounded up
                const int hq = 4 * nt + qd;
                const float4* nq = reinterpret_cast<const float4*>(sNQ + min(hq, G - 1) * 20);
                float cb[2];
    #pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    float2 c2 = make_float2(0.f, 0.f);
    #pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint4 u = tW[(g + 8 * tt) * 2 + c];
                        const float4 na = nq[2 * c], nb = nq[2 * c + 1];
                        c2 = __ffma2_ru(make_float2(na.x, na.y), __half22float2(*reinterpret_cast<const __half2*>(&u.x)), c2);
                        c2 = __ffma2_ru(make_float2(na.z, na.w), __half22float2(*reinterpret_cast<const __half2*>(&u.y)), c2);
                        c2 = __ffma2_ru(make_float2(nb.x, nb.y), __half22float2(*reinterpret_cast<const __half2*>(&u.z)), c2);
                        c2 = __ffma2_ru(make_float2(nb.z, nb.w), __half22float2(*reinterpret_cast<const __half2*>(&u.w)), c2);
                    }
                    cb[tt] = __fmul_ru(__fadd_ru(c2.x, c2.y), a.inv_sqrt_d_up);
                }
                cb[0] = vis0 ? cb[0] : 0.f;                     // outside the window: no bound
                cb[1] = vis1 ? cb[1] : 0.f;
                c_w[nt] = fmaxf(c_w[nt], fmaxf(cb[0], cb[1]));
                if (a.ct && hq < G) {
                    a.ct[(rowq0 + hq) * a.S + p0 + g] = cb[0];
                    a.ct[(rowq0 + hq) * a.S + p0 + g + 8] = cb[1];
                }
            }
            if (__any_sync(0xffffffffu, rescale) && i > 0) {     // at i = 0 the accumulators are 0
    #pragma unroll
                for (int mt = 0; mt < C::KS; ++mt)
    #pragma unroll
                    for (int nt = 0; nt < C::NT; ++nt)
    #pragma unroll
                        for (int e = 0; e < 4; ++e) acc[mt][nt][e] *= alpha[nt];
            }
            __syncwarp();

            // ---- P.V: O^T += V^T P^T; B operand = P^T column g, tokens 4 qd .. + 3
            uint2 pb[C::NT];
    #pragma unroll
            for (int nt = 0; nt < C::NT; ++nt)
                pb[nt] = *reinterpret_cast<const uint2*>(myPm + nt * C::PROWB + prow(g) + 8 * qd);
            constexpr int CPR = D / 32;                  // 16-byte chunks of the lane's V run
            const int swz = (lane / (8 / CPR)) % CPR;
            uint32_t vw[C::VW];
    #pragma unroll
            for (int j = 0; j < CPR; ++j) {
                const uint4 u = *reinterpret_cast<const uint4*>(tV + lane * (D / 2) + ((j ^ swz) << 4));
                vw[4 * j] = u.x; vw[4 * j + 1] = u.y; vw[4 * j + 2] = u.z; vw[4 * j + 3] = u.w;
            }
    #pragma unroll
            for (int mt = 0; mt < C::KS; ++mt) {
                uint32_t a0, a1, a2, a3;
                codes_to_half2(vw[2 * mt], a0, a2);           // dim 16 mt + g
                codes_to_half2(vw[2 * mt + 1], a1, a3);       // dim 16 mt + 8 + g
    #pragma unroll
                for (int nt = 0; nt < C::NT; ++nt) mma_f16(acc[mt][nt], a0, a1, a2, a3, pb[nt].x, pb[nt].y);
            }
        }
        // this stage and the staging are free once every lane is past its reads
        __syncwarp();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (i + kStages < tpw) issue(i + kStages);
    }

    // ---- this warp's partial into its stage buffers (all issued copies were awaited):
    // l and the bound's maximum over the 8 lanes of a head; output = (hi + lo) columns
    __syncwarp();
    float* part_w = reinterpret_cast<float*>(myS);             // [G][3 + D]
    const float oscale = svmax * (1.f / 128.f);
#pragma unroll
    for (int nt = 0; nt < C::HPL; ++nt) {
        float l = l_w[nt], c = c_w[nt];
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l += __shfl_xor_sync(0xffffffffu, l, o);
            c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, o));
        }
        const int hq = 4 * nt + qd;
        if (hq < G) {
#pragma unroll
            for (int mt = 0; mt < C::KS; ++mt) {
                part_w[hq * (D + 3) + 3 + 16 * mt + g] = (acc[mt][nt][0] + acc[mt][nt][1]) * oscale;
                part_w[hq * (D + 3) + 3 + 16 * mt + 8 + g] = (acc[mt][nt][2] + acc[mt][nt][3]) * oscale;
            }
            if (g == 0) {
                part_w[hq * (D + 3)] = m_w[nt];
                part_w[hq * (D + 3) + 1] = l;
                part_w[hq * (D + 3) + 2] = c;
            }
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

// Combine: WPR warps per (request, query head) row, 8 / WPR rows per CTA (the design of
// the bf16 combine): one pass over the splits, warp w taking the splits w, w + WPR, ...,
// kU at a time with every load of a round issued together, keeping a running maximum,
// denominator, weighted sum (lanes over 4-dim groups) and bound maximum; the WPR warps'
// results meet in shared memory once.
constexpr int kCombineThreads = 256;
constexpr int kCombineU = 4;            // splits a warp loads per round

template <int WPR>
__global__ void __launch_bounds__(kCombineThreads) int8_combine_kernel(const Int8CombineArgs c) {
    constexpr int kRows = kCombineThreads / 32 / WPR;
    __shared__ float4 sacc[kRows][WPR][32];                       // d <= 128
    __shared__ float4 sml[kRows][WPR];                            // each warp's (m, l, max c)
    dep_wait();                                                    // launched dependent: see launch_dep
    dep_release();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = warp / WPR, w = warp % WPR;
    const size_t row = (size_t)blockIdx.x * kRows + r;
    const bool valid = row < (size_t)c.B * c.Hq;
    if (valid) {
        const int b = (int)(row / c.Hq), hq = (int)(row % c.Hq);
        const int len = c.next_pos[b];
        const int nfull = len & ~(kQBlock - 1);
        const int kvh = hq / (c.Hq / c.Hkv);
        const int nx = c.xn[(size_t)b * c.Hkv + kvh];
        const Int8Window iw = int8_window(len, c.S, c.W, c.ring);
        const int bps = c.split / kQBlock;
        // quantized splits, the exact-rows split (if it ran), the exact-block splits
        const int ns = (iw.bhi - iw.blo + bps - 1) / bps + (len > nfull || nx > 0 ? 1 : 0) +
                       (nx + kExactBlocksPerCta - 1) / kExactBlocksPerCta;
        const float2* ml = c.part_ml + row * c.max_splits;
        const float* pc = c.part_c + row * c.max_splits;
        const float* pa = c.part_acc + row * c.max_splits * c.d;
        const int i0 = 4 * lane;                                  // (d <= 128: one 4-dim group a lane)
        float m = -INFINITY, l = 0.f, cm = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = w; s0 < ns; s0 += WPR * kCombineU) {
            float2 v[kCombineU];
            float4 x[kCombineU];
#pragma unroll
            for (int u = 0; u < kCombineU; ++u) {
                const int s = s0 + u * WPR;
                v[u] = s < ns ? __ldg(ml + s) : make_float2(-INFINITY, 0.f);
                cm = fmaxf(cm, s < ns ? __ldg(pc + s) : 0.f);
                x[u] = (s < ns && i0 < c.d) ? __ldg(reinterpret_cast<const float4*>(pa + (size_t)s * c.d + i0))
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float mn = m;
#pragma unroll
            for (int u = 0; u < kCombineU; ++u) mn = fmaxf(mn, v[u].x);
            if (mn == -INFINITY) continue;                      // no keys in any split so far
            const float sc = exp2f(m - mn);                     // 0 while m was -inf
            l *= sc;
            acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
#pragma unroll
            for (int u = 0; u < kCombineU; ++u) {
                const float f = exp2f(v[u].x - mn);               // 0 for an empty split
                l = fmaf(v[u].y, f, l);
                acc.x = fmaf(x[u].x, f, acc.x); acc.y = fmaf(x[u].y, f, acc.y);
                acc.z = fmaf(x[u].z, f, acc.z); acc.w = fmaf(x[u].w, f, acc.w);
            }
            m = mn;
        }
        if (lane == 0) sml[r][w] = make_float4(m, l, cm, 0.f);
        if (i0 < c.d) sacc[r][w][lane] = acc;
    }
    __syncthreads();
    if (!valid || w != 0) return;
    float M = -INFINITY, cm = 0.f;
#pragma unroll
    for (int k = 0; k < WPR; ++k) { M = fmaxf(M, sml[r][k].x); cm = fmaxf(cm, sml[r][k].z); }
    float f[WPR], L = 0.f;
#pragma unroll
    for (int k = 0; k < WPR; ++k) {
        f[k] = sml[r][k].x == -INFINITY ? 0.f : exp2f(sml[r][k].x - M);
        L = fmaf(sml[r][k].y, f[k], L);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int i0 = 4 * lane; i0 < c.d; i0 += 128) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < WPR; ++k) {
            const float4 x = sacc[r][k][i0 / 4];
            acc.x = fmaf(x.x, f[k], acc.x); acc.y = fmaf(x.y, f[k], acc.y);
            acc.z = fmaf(x.z, f[k], acc.z); acc.w = fmaf(x.w, f[k], acc.w);
        }
        const float o[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (c.out_bf16) static_cast<__nv_bfloat16*>(c.out)[row * c.d + i0 + e] = __float2bfloat16_rn(o[e]);
            else static_cast<float*>(c.out)[row * c.d + i0 + e] = o[e];
        }
    }
    if (lane == 0) {
        if (c.cmax) c.cmax[row] = cm;
        if (c.tanh_out) c.tanh_out[row] = tanh_up(cm);
    }
}

template <int D, int G, bool DITHER, bool GEN>
cudaError_t launch_t(const Int8Args& a, cudaStream_t st) {
    using C = I8<D, G, DITHER>;
    const void* k = reinterpret_cast<const void*>(int8_decode_kernel<D, G, DITHER, GEN>);
    if (cudaError_t e = allow_smem(k, C::SMEM)) return e;
    return launch_dep(int8_decode_kernel<D, G, DITHER, GEN>, dim3(a.grid, a.Hkv, a.B), dim3(kWarps * 32),
                      C::SMEM, st, a);
}

template <int D, int G>
cudaError_t launch_dg(const Int8Args& a, bool dither, bool gen, cudaStream_t st) {
    if (dither) return gen ? launch_t<D, G, true, true>(a, st) : launch_t<D, G, true, false>(a, st);
    return gen ? launch_t<D, G, false, true>(a, st) : launch_t<D, G, false, false>(a, st);
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
    a.wit = s.dither ? nullptr : reinterpret_cast<const __half*>(h->state + h->L.wit);
    a.req_id = reinterpret_cast<const uint32_t*>(h->state + h->L.req_id);
    a.table = s.pages ? reinterpret_cast<const int32_t*>(h->state + h->L.table) : nullptr;
    a.layer_ctr = 65536u * (uint32_t)h->cfg.layer_index;
    for (int r = 0; r < 10; ++r) {
        a.rk[2 * r] = h->cfg.dither_key_lo + (uint32_t)r * 0x9E3779B9u;
        a.rk[2 * r + 1] = h->cfg.dither_key_hi + (uint32_t)r * 0xBB67AE85u;
    }
    a.ktail = reinterpret_cast<const __nv_bfloat16*>(h->state + h->L.ktail);
    a.vtail = reinterpret_cast<const __nv_bfloat16*>(h->state + h->L.vtail);
    a.xmap = reinterpret_cast<const int32_t*>(h->state + h->L.xmap);
    a.xn = reinterpret_cast<const int32_t*>(h->state + h->L.xn);
    a.xpool = reinterpret_cast<const __nv_bfloat16*>(h->state + h->L.xpool);
    a.next_pos = reinterpret_cast<const int32_t*>(h->state + h->L.next_pos);
    a.rope = s.rope ? reinterpret_cast<const float2*>(h->state + h->L.rope) : nullptr;
    a.part_ml = reinterpret_cast<float2*>(h->state + h->L.part_ml);
    a.part_acc = reinterpret_cast<float*>(h->state + h->L.part_acc);
    a.part_c = reinterpret_cast<float*>(h->state + h->L.part_c);
    a.ct = ct;
    a.hdr = reinterpret_cast<uint32_t*>(h->state + h->L.hdr);
    a.B = s.B; a.Hq = s.Hq; a.Hkv = s.Hkv; a.d = s.d; a.S = s.S; a.max_splits = s.max_splits;
    a.W = s.W; a.ring = s.ring;
    a.split = s.split;
    a.grid = int8_grid(s);
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.d));
    a.inv_sqrt_d_up = std::nextafter((float)(1.0 / std::sqrt((double)s.d)), 1.0f);
    cudaError_t e = cudaErrorInvalidValue;
    const bool gen = s.W > 0 || s.ring || s.pages > 0;
#define KVC_CASE(D, G) \
    if (s.d == D && s.g == G) e = launch_dg<D, G>(a, s.dither, gen, st);
    KVC_CASE(128, 1) KVC_CASE(128, 2) KVC_CASE(128, 4) KVC_CASE(128, 8)
    KVC_CASE(64, 1) KVC_CASE(64, 2) KVC_CASE(64, 4) KVC_CASE(64, 8)
#undef KVC_CASE
    if (e != cudaSuccess) return e;
    if (s.xpool > 0 && (e = launch_int8_exact(h, q, ct, st)) != cudaSuccess) return e;
    Int8CombineArgs c{};
    c.part_ml = a.part_ml; c.part_acc = a.part_acc; c.part_c = a.part_c; c.next_pos = a.next_pos; c.xn = a.xn;
    c.out = out; c.cmax = cmax; c.tanh_out = tanh_out;
    c.B = s.B; c.Hq = s.Hq; c.Hkv = s.Hkv; c.d = s.d; c.S = s.S; c.max_splits = s.max_splits;
    c.out_bf16 = s.out_bf16; c.W = s.W; c.ring = s.ring;
    c.split = s.split;
    const size_t rows = (size_t)s.B * s.Hq;
    if (s.max_splits <= 8)
        e = launch_dep(int8_combine_kernel<1>, dim3((unsigned)((rows + 7) / 8)), dim3(kCombineThreads), 0, st, c);
    else if (rows < 1024)
        e = launch_dep(int8_combine_kernel<8>, dim3((unsigned)rows), dim3(kCombineThreads), 0, st, c);
    else
        e = launch_dep(int8_combine_kernel<4>, dim3((unsigned)((rows + 1) / 2)), dim3(kCombineThreads), 0, st, c);
    return e;
}

}  // namespace kvc
