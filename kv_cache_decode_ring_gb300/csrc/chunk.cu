// chunk.cu -- chunked causal (or sliding-window) suffix attention on tcgen05.
//
// [PREFIX] "哪些東西必須一起裁剪": after the cache is trimmed to `cut`, the
// suffix tokens[cut:] are computed in one chunk from next_position = cut:
// suffix query i sits at position p = cut + i and attends to cached positions
// [max(0, p - W + 1), p] (W = 0: all), exactly what a one-token decode at p
// would see ([LEAN] §2.1 masks).  The suffix K/V rows are appended to the
// contiguous cache first, so every key a query needs lies in one contiguous
// run of cache rows.
//
// This is a dense contraction, so it runs on the 5th-generation tensor cores:
//  * CTA = 128 query rows of one query head (4 warps, thread = row);
//  * Q, K, V tiles arrive by TMA (128-byte swizzle), K/V double-buffered;
//  * S = Q K^T and O += P V are tcgen05.mma (bf16 in, fp32 accumulate) issued
//    by one thread into tensor memory (S: 128 columns, O: 128 columns);
//  * each thread reads its S row from tensor memory, applies the causal and
//    window masks by absolute position, runs the online softmax in fp32 (log2
//    domain), rescales its O row in tensor memory when its running maximum
//    grows, and writes its P row to shared memory for the next MMA;
//  * the rotated query and P are not exact in bf16, so each enters its MMA as
//    two bf16 terms (hi, lo) accumulated in fp32 (about 16 significant bits);
//  * K/V tiles are walked backwards from the diagonal;
//  * tcgen05.ld/st are warp-collective: every lane of a warp issues them.
// Every mbarrier wait is bounded; on expiry the kernel flags the device error
// word, skips the remaining work and still frees its tensor memory.
#include <cuda.h>

#include <cmath>
#include <mutex>

#include "async_copy.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kBM = 128;          // query rows per CTA
constexpr int kBN = 128;          // keys per tile
constexpr int kD = 128;           // head dim of this kernel
constexpr int kThreads = 128;
constexpr int kTile = kBM * kD * 2;   // 32 KB: two 64-column halves of [128 rows][128 B]
constexpr int kHalf = kTile / 2;
// Operands that are not exact bf16 (the rotated query and the softmax weights)
// enter the MMAs as two bf16 terms, hi = bf16(x) and lo = bf16(x - hi), both
// accumulated in fp32: about 16 significant bits instead of 8.  P_hi reuses the
// K stage of its tile (free once S is computed, refilled only after P V completes).
constexpr int OFF_Q = 0;                   // Q hi
constexpr int OFF_QLO = OFF_Q + kTile;     // Q lo
constexpr int OFF_K = OFF_QLO + kTile;     // 2 stages (stage j%2 also holds P hi of tile j)
constexpr int OFF_V = OFF_K + 2 * kTile;   // 2 stages
constexpr int OFF_P = OFF_V + 2 * kTile;   // P lo
constexpr int OFF_BAR = OFF_P + kTile;     // q, kv[2], s, o
constexpr int OFF_MISC = OFF_BAR + 64;     // tensor memory base, abort flag
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;
constexpr uint32_t kTmemCols = 256;        // S: [0, 128), O: [128, 256)

struct ChunkArgs {
    const int32_t* next_pos;   // after the append: cut + n
    void* out;                 // [B][n][Hq][d]
    uint32_t* hdr;
    int B, Hq, Hkv, g, S, W, n, out_bf16;
    float scale_log2;
};

// ---- tcgen05 wrappers -------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle, sm_100 format:
// start address >> 4 (bits 0-13), leading-dimension byte offset >> 4 (16-29),
// stride-dimension byte offset >> 4 (32-45), version 1 (46-47), layout 2 =
// SWIZZLE_128B (61-63).  K-major operands: 8-row groups 1024 B apart (SBO).
// MN-major operands additionally step `lbo` bytes to the next 64 MN elements.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(1024u >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: D fp32 (bit 4), A and B bf16 (bits 7, 10),
// B MN-major when b_mn (bit 16), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, int acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's tensor-memory lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
          "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
          "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
          "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
          "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
          "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
          "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
          "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
          "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
          "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
          "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
}

// All threads wait on the same barrier phase; if any of them gave up, all of them know.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, uint32_t* hdr) {
    const bool ok = mbar_wait(bar, parity);
    if (!ok && (threadIdx.x & 31) == 0) atomicOr(hdr, kErrWait);
    return __syncthreads_and(ok ? 1 : 0) != 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    chunk_attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQlo,
                      const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const ChunkArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* sQ = smem + OFF_Q;
    unsigned char* sQlo = smem + OFF_QLO;
    unsigned char* sK = smem + OFF_K;
    unsigned char* sV = smem + OFF_V;
    unsigned char* sP = smem + OFF_P;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + OFF_BAR);   // [0] q, [1..2] kv, [3] s, [4] o
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int b = blockIdx.z, hq = blockIdx.y, i0 = blockIdx.x * kBM;
    const int kvh = hq / a.g;
    const int np = a.next_pos[b];
    const int cut = np - a.n;
    const int rows = min(kBM, a.n - i0);
    const int p_first = cut + i0, p_last = cut + i0 + rows - 1;
    const int lo = a.W > 0 ? max(0, p_first - a.W + 1) : 0;
    const int ntiles = (p_last + 1 - lo + kBN - 1) / kBN;
    const int head_row0 = (b * a.Hkv + kvh) * a.S;

    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(&bar[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tO = tmem + 128;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

    // ---- loads: Q once, the first two K/V tiles
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], 2 * kTile);
        tma_load_3d(sQ, &tmQ, 0, hq, b * a.n + i0, &bar[0]);
        tma_load_3d(sQ + kHalf, &tmQ, 64, hq, b * a.n + i0, &bar[0]);
        tma_load_3d(sQlo, &tmQlo, 0, hq, b * a.n + i0, &bar[0]);
        tma_load_3d(sQlo + kHalf, &tmQlo, 64, hq, b * a.n + i0, &bar[0]);
        for (int j = 0; j < 2 && j < ntiles; ++j) {
            const int kbase = p_last + 1 - kBN * (j + 1);
            mbar_arrive_expect_tx(&bar[1 + j], 2 * kTile);
            tma_load_2d(sK + j * kTile, &tmK, 0, head_row0 + kbase, &bar[1 + j]);
            tma_load_2d(sK + j * kTile + kHalf, &tmK, 64, head_row0 + kbase, &bar[1 + j]);
            tma_load_2d(sV + j * kTile, &tmV, 0, head_row0 + kbase, &bar[1 + j]);
            tma_load_2d(sV + j * kTile + kHalf, &tmV, 64, head_row0 + kbase, &bar[1 + j]);
        }
    }
    bool ok = wait_all(&bar[0], 0, a.hdr);

    const int row = tid;                       // query row of this thread = tensor-memory lane
    const int p = cut + i0 + row;              // its absolute position
    const bool row_valid = row < rows;
    const int key_lo = a.W > 0 ? max(0, p - a.W + 1) : 0;
    float m = -INFINITY, l = 0.f;
    constexpr uint32_t idesc_qk = instr_desc(kBM, kBN, false);
    constexpr uint32_t idesc_pv = instr_desc(kBM, kD, true);

    for (int j = 0; j < ntiles && ok; ++j) {
        const int st = j & 1;
        const int kbase = p_last + 1 - kBN * (j + 1);
        // ---- S = Q K^T
        if (tid == 0) {
            ok = mbar_wait(&bar[1 + st], (uint32_t)((j >> 1) & 1));
            if (ok) {
                fence_after();
                const uint32_t q0 = smem_u32(sQ), q1 = smem_u32(sQlo), k0 = smem_u32(sK + st * kTile);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s) {
                    const uint32_t off = (s >> 2) * kHalf + (s & 3) * 32;
                    mma_bf16(tS, smem_desc(q0 + off, 16), smem_desc(k0 + off, 16), idesc_qk, s > 0);
                }
#pragma unroll
                for (int s = 0; s < kD / 16; ++s) {
                    const uint32_t off = (s >> 2) * kHalf + (s & 3) * 32;
                    mma_bf16(tS, smem_desc(q1 + off, 16), smem_desc(k0 + off, 16), idesc_qk, 1);
                }
                mma_commit(&bar[3]);
            } else {
                atomicOr(a.hdr, kErrWait);
            }
        }
        if (!__syncthreads_and(ok ? 1 : 0)) { ok = false; break; }
        ok = wait_all(&bar[3], (uint32_t)(j & 1), a.hdr);
        if (!ok) break;
        fence_after();
        // ---- softmax on this thread's row
        float s[kBN];
#pragma unroll
        for (int c = 0; c < kBN; c += 32) tmem_ld32(tS + lane_off + c, s + c);
        float mx = m;
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
            const int key = kbase + c;
            const bool vis = row_valid && key >= key_lo && key <= p;
            s[c] = vis ? s[c] * a.scale_log2 : -INFINITY;
            mx = fmaxf(mx, s[c]);
        }
        const float base = mx == -INFINITY ? 0.f : mx;
        const float alpha = exp2f(m - base);          // 0 when m = -inf
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
            s[c] = exp2f(s[c] - base);
            rs += s[c];
        }
        l = l * alpha + rs;
        // O holds the previous tiles at the old maximum: rescale the rows whose maximum
        // grew.  tcgen05.ld/st are warp-collective (.sync.aligned), so the whole warp
        // takes part whenever any of its rows needs it; the others scale by 1.
        const bool grow = j > 0 && alpha != 1.f;
        if (__any_sync(0xffffffffu, grow)) {
            const float f = grow ? alpha : 1.f;
#pragma unroll
            for (int c = 0; c < kD; c += 32) {
                float o[32];
                tmem_ld32(tO + lane_off + c, o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] *= f;
                tmem_st32(tO + lane_off + c, o);
            }
        }
        m = mx;
        // P row -> shared memory as hi and lo bf16 terms, K-major 128-byte swizzle
        unsigned char* sPhi = sK + st * kTile;
#pragma unroll
        for (int c = 0; c < kBN / 8; ++c) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(s[8 * c + 2 * e], s[8 * c + 2 * e + 1]);
                const float2 hf = __bfloat1622float2(h2);
                hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
                lo[e] = pack_bf16(s[8 * c + 2 * e] - hf.x, s[8 * c + 2 * e + 1] - hf.y);
            }
            const int off = (c >> 3) * kHalf + row * 128 + (((c & 7) ^ (row & 7)) * 16);
            *reinterpret_cast<uint4*>(sPhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(sP + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        fence_before();
        __syncthreads();
        // ---- O += P V
        if (tid == 0) {
            fence_after();
            const uint32_t ph = smem_u32(sK + st * kTile), pl = smem_u32(sP), v0 = smem_u32(sV + st * kTile);
#pragma unroll
            for (int s2 = 0; s2 < kBN / 16; ++s2) {
                const uint32_t aoff = (s2 >> 2) * kHalf + (s2 & 3) * 32;
                mma_bf16(tO, smem_desc(ph + aoff, 16), smem_desc(v0 + s2 * 2048, kHalf), idesc_pv, (j > 0 || s2 > 0));
            }
#pragma unroll
            for (int s2 = 0; s2 < kBN / 16; ++s2) {
                const uint32_t aoff = (s2 >> 2) * kHalf + (s2 & 3) * 32;
                mma_bf16(tO, smem_desc(pl + aoff, 16), smem_desc(v0 + s2 * 2048, kHalf), idesc_pv, 1);
            }
            mma_commit(&bar[4]);
        }
        ok = wait_all(&bar[4], (uint32_t)(j & 1), a.hdr);
        if (!ok) break;
        fence_after();
        // ---- refill this stage with tile j + 2
        if (tid == 0 && j + 2 < ntiles) {
            const int kb2 = p_last + 1 - kBN * (j + 3);
            mbar_arrive_expect_tx(&bar[1 + st], 2 * kTile);
            tma_load_2d(sK + st * kTile, &tmK, 0, head_row0 + kb2, &bar[1 + st]);
            tma_load_2d(sK + st * kTile + kHalf, &tmK, 64, head_row0 + kb2, &bar[1 + st]);
            tma_load_2d(sV + st * kTile, &tmV, 0, head_row0 + kb2, &bar[1 + st]);
            tma_load_2d(sV + st * kTile + kHalf, &tmV, 64, head_row0 + kb2, &bar[1 + st]);
        }
    }

    // ---- epilogue: O / l; every lane reads (warp-collective), valid rows store
    if (ok) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const size_t orow = (((size_t)b * a.n + i0 + row) * a.Hq + hq) * kD;
#pragma unroll
        for (int c = 0; c < kD; c += 32) {
            float o[32];
            tmem_ld32(tO + lane_off + c, o);
            if (!row_valid) continue;
            if (a.out_bf16) {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow + c);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint4 u;
                    u.x = pack_bf16(o[8 * e + 0] * inv, o[8 * e + 1] * inv);
                    u.y = pack_bf16(o[8 * e + 2] * inv, o[8 * e + 3] * inv);
                    u.z = pack_bf16(o[8 * e + 4] * inv, o[8 * e + 5] * inv);
                    u.w = pack_bf16(o[8 * e + 6] * inv, o[8 * e + 7] * inv);
                    dst[e] = u;
                }
            } else {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow + c);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    dst[e] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv, o[4 * e + 3] * inv);
            }
        }
    } else if (!ok) {
        // make sure no tensor-core operation still targets our columns before freeing them
        if (tid == 0) {
            mbar_wait(&bar[3], 0);
            mbar_wait(&bar[4], 0);
        }
    }
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// Query rows rotated at their positions (fp32 rule of the cache keys), split into
// bf16 hi = bf16(y) and lo = bf16(y - hi).
__global__ void rope_q_kernel(const __nv_bfloat16* q, __nv_bfloat16* qr, __nv_bfloat16* qlo,
                              const int32_t* next_pos, const float2* rope, int n, int Hq, int d) {
    const int b = blockIdx.y;
    const int cut = next_pos[b] - n;
    const size_t per_b = (size_t)n * Hq * (d / 2);
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < per_b; idx += (size_t)gridDim.x * blockDim.x) {
        const int i = (int)(idx / ((size_t)Hq * (d / 2)));
        const int pr = (int)(idx % (d / 2));
        const size_t off = (size_t)b * n * Hq * d + idx * 2;
        const float x0 = __bfloat162float(q[off]), x1 = __bfloat162float(q[off + 1]);
        float y0 = x0, y1 = x1;
        if (rope) rope_pair(x0, x1, rope[(size_t)(cut + i) * (d / 2) + pr], y0, y1);
        const __nv_bfloat16 h0 = __float2bfloat16_rn(y0), h1 = __float2bfloat16_rn(y1);
        qr[off] = h0;
        qr[off + 1] = h1;
        qlo[off] = __float2bfloat16_rn(y0 - __bfloat162float(h0));
        qlo[off + 1] = __float2bfloat16_rn(y1 - __bfloat162float(h1));
    }
}

// ---- tensor maps -----------------------------------------------------------
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

}  // namespace

bool make_tensor_map_bf16(CUtensorMap* tm, void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                          const cuuint32_t* box) {
    EncodeTiled enc = encoder();
    if (!enc) return false;
    cuuint32_t es[3] = {1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool chunk_supported(const Shape& s) { return s.bf16 && !s.int8 && !s.ring && s.d == kD; }

cudaError_t launch_chunk(kvc_handle* h, const void* q, void* out, int n, cudaStream_t st) {
    const Shape& s = h->sh;
    __nv_bfloat16* qr = reinterpret_cast<__nv_bfloat16*>(h->state + h->L.qrot);
    __nv_bfloat16* qlo = qr + (size_t)s.B * s.max_chunk * s.Hq * s.d;
    const int32_t* np = reinterpret_cast<const int32_t*>(h->state + h->L.next_pos);
    const float2* rope = s.rope ? reinterpret_cast<const float2*>(h->state + h->L.rope) : nullptr;
    rope_q_kernel<<<dim3(128, s.B), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(q), qr, qlo, np, rope, n, s.Hq,
                                                  s.d);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    CUtensorMap tq, tql, tk, tv;
    const cuuint64_t qdims[3] = {(cuuint64_t)s.d, (cuuint64_t)s.Hq, (cuuint64_t)s.B * n};
    const cuuint64_t qstr[2] = {(cuuint64_t)s.d * 2, (cuuint64_t)s.Hq * s.d * 2};
    const cuuint32_t qbox[3] = {64, 1, kBM};
    const cuuint64_t kdims[2] = {(cuuint64_t)s.d, (cuuint64_t)s.B * s.Hkv * s.S};
    const cuuint64_t kstr[1] = {(cuuint64_t)s.d * 2};
    const cuuint32_t kbox[2] = {64, kBN};
    if (!make_tensor_map_bf16(&tq, qr, 3, qdims, qstr, qbox) || !make_tensor_map_bf16(&tql, qlo, 3, qdims, qstr, qbox) ||
        !make_tensor_map_bf16(&tk, h->state + h->L.k, 2, kdims, kstr, kbox) ||
        !make_tensor_map_bf16(&tv, h->state + h->L.v, 2, kdims, kstr, kbox))
        return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        e = cudaFuncSetAttribute(chunk_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    ChunkArgs a{};
    a.next_pos = np; a.out = out; a.hdr = reinterpret_cast<uint32_t*>(h->state + h->L.hdr);
    a.B = s.B; a.Hq = s.Hq; a.Hkv = s.Hkv; a.g = s.g; a.S = s.S; a.W = s.W; a.n = n; a.out_bf16 = s.out_bf16;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.d));
    chunk_attn_kernel<<<dim3((n + kBM - 1) / kBM, s.Hq, s.B), kThreads, SMEM_BYTES, st>>>(tq, tql, tk, tv, a);
    return cudaGetLastError();
}

}  // namespace kvc
