/*
 * kvc.h -- C ABI of libkvc, a single-GPU (GB300, sm_103a) library for one
 * autoregressive decode step over a KV cache.
 *
 * Sources of the operations, cited by page title and section:
 *   [LEAN]    "用Lean4形式化验证滑动窗口KV Cache的正确性" (framerc.cn/news/4505248)
 *   [PREFIX]  "LLM 機制實驗（五）：改了歷史，能否只重算變化的後綴？"
 *             (huhohoo.com/zh-TW/docs/llm/longest-prefix-reuse)
 *   [LOOP]    "KV Cache 自回归生成推理（增量更新与状态拼接）" (airsota.com/?p=549)
 *   [WITCERT] "WitCert: Sound Runtime Risk Observability and Gating for
 *             KV-Cache Quantization" (agifrontier.github.io tutorial)
 *
 * Conventions
 *  - Ownership: the caller owns every device buffer (the cache state, inputs,
 *    outputs) and the stream.  The library owns only the small host handle.
 *    kvc_create() and kvc_destroy() neither allocate nor free device memory.
 *  - Pointers named d_* are device pointers, h_* host pointers.  Device
 *    inputs must be 16-byte aligned and densely packed in the stated layout.
 *  - Devices: a handle lives on the device that was current at kvc_create();
 *    every later call on it that touches the device must run with that device
 *    current, else it returns KVC_ERR_ARG and enqueues nothing.
 *  - Streams: kvc_stream_t is a cudaStream_t (NULL = the legacy default
 *    stream).  Compute calls only enqueue work and return; none waits for the
 *    GPU, except kvc_create (uploads tables), kvc_export and
 *    kvc_device_status (read back).  One handle serves one stream at a time:
 *    calls on one handle from different streams race on its state.  The
 *    decode-path kernels (append, decode, combine) start as programmatic
 *    dependent launches.  They may be scheduled while the previous kernel on the
 *    stream drains, but they wait for it to complete before touching memory.
 *    So the order of work on a stream, and CUDA graph capture, behave as with
 *    ordinary launches.
 *  - Element types: KVC_F32 = IEEE fp32, KVC_BF16 = bfloat16.  q, k and v
 *    use the cache dtype; outputs use kvc_config.out_dtype (default: the
 *    cache dtype).
 *  - Positions are absolute, 0-based, signed 32-bit; -1 marks an empty slot.
 *  - Errors: every entry point returns a KVC_* status.  Arguments are checked
 *    on the host before anything is enqueued; a failed call changes nothing.
 *    Kernels also check their own bounds and set a sticky device error word
 *    (read by kvc_device_status) instead of writing out of bounds.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kvc_handle* kvc_t;
typedef void* kvc_stream_t; /* a cudaStream_t */

/* ---- status codes ---------------------------------------------------- */
#define KVC_OK 0
#define KVC_ERR_ARG 1          /* null pointer, bad shape/dtype/size, call out of order */
#define KVC_ERR_CAPACITY 2     /* contiguous cache full: position >= max_seq_len
                                  ([LOOP] §三 "assert pos < max_seq_len"), or a
                                  position beyond the RoPE table */
#define KVC_ERR_EVICTED 3      /* trim needs rows the cache no longer holds exactly:
                                  evicted from a ring ([PREFIX] "為什麼滑窗部分命中必須回退")
                                  or already folded into an INT8 block */
#define KVC_ERR_CUDA 4         /* a CUDA runtime call failed */
#define KVC_ERR_UNSUPPORTED 5  /* valid request this build does not implement */
#define KVC_ERR_DEVICE 6       /* a kernel flagged an error (see kvc_device_status) */

/* ---- configuration --------------------------------------------------- */
enum { KVC_F32 = 0, KVC_BF16 = 1 };
enum { KVC_CONTIGUOUS = 0, KVC_RING = 1 };
enum { KVC_QUANT_NONE = 0, KVC_QUANT_INT8 = 1, KVC_QUANT_INT8_DITHER = 2 };

typedef struct {
    int32_t dtype;        /* KVC_F32 or KVC_BF16 */
    int32_t layout;       /* KVC_CONTIGUOUS: slot = position, capacity = max_seq_len
                             ([LOOP] §三, preallocated (B, H, max_S, D) buffers);
                             KVC_RING: slot = position mod W, capacity = W
                             ([LEAN] §3.4 ring buffer, §2.3 lastWindow) */
    int32_t kv_quant;     /* KVC_QUANT_NONE, KVC_QUANT_INT8_DITHER (Tier B, see
                             dither_key_lo below) or KVC_QUANT_INT8 ([WITCERT]; bf16
                             caches, contiguous with any window or a ring.  Blocks are
                             16 positions; a ring of W slots, W % 16 == 0, keeps block n
                             in block slot n mod W/16 and holds the newest W/16
                             complete blocks plus the exact rows of the incomplete
                             one, which covers its window [LEAN] §3.4) */
    int32_t batch;        /* B >= 1 requests */
    int32_t n_q_heads;    /* Hq >= 1 */
    int32_t n_kv_heads;   /* Hkv >= 1, Hq % Hkv == 0; query head h reads KV head h / (Hq/Hkv).
                             Shapes served by the generic decode (fp32 caches; bf16 with d
                             other than 64/128 or more than 8 query heads per KV head)
                             need g (d + 64) 4 <= 232448 bytes of shared memory, g = Hq/Hkv */
    int32_t head_dim;     /* d: even, 2..256; INT8 needs d % 16 == 0 */
    int32_t capacity;     /* slots per (request, KV head); INT8 needs capacity % 16 == 0 */
    int32_t window;       /* attention window W: 0 = full history (contiguous only);
                             a ring must use 0 or its capacity.  The query at
                             position t sees positions [max(0, t-W+1), t] ([LEAN] §2.1). */
    int32_t max_position; /* RoPE table length; every position must stay below it.
                             0 = capacity (contiguous).  Required for a ring with RoPE. */
    float rope_base;      /* rotary base (e.g. 10000); 0 = keys and queries not rotated */
    int32_t max_chunk;    /* largest n for kvc_chunk_attn (sizes a ring's staging rows) */
    int32_t out_dtype;    /* attention outputs: 0 = the cache dtype, else KVC_F32 or
                             KVC_BF16 (+1 is added so that 0 keeps the default):
                             pass KVC_F32 + 1 or KVC_BF16 + 1 */
    int32_t int8_exact_blocks; /* INT8 only: capacity of the pool of blocks restored
                             to full precision by kvc_int8_restore (0 = none).
                             Contiguous caches with window 0 only. */
    int32_t page_pool;    /* paged K/V storage ([LEAN] §6.1 block table; [LOOP] §八 Q1,
                             16-token pages mapped on demand): 0 = each
                             request owns `capacity` slots; > 0 = K and V live in a pool
                             of page_pool pages of 16 slots (all KV heads of one request)
                             mapped by a per-request block table, allocated on append and
                             freed by trim; capacity (the per-request logical
                             slots) must be a multiple of 16.  With INT8 a page holds
                             one quantization block of every KV head (codes, scales,
                             witnesses); the exact tail stays per request; no gate pool. */
    int32_t store_slots;  /* device slots for saved prefills (kvc_store_save /
                             kvc_store_load), each holding one request's K, V and
                             positions; 0 = none.  Not with INT8. */
    int32_t layer_index;  /* KVC_QUANT_INT8_DITHER: the layer in the dither counter */
    uint32_t dither_key_lo, dither_key_hi;
                          /* KVC_QUANT_INT8_DITHER (Tier B, [WITCERT] subtractive-
                             dither paragraph; counter from "SGLang 生产级落地与闭环门控修复"):
                             the Philox4x32-10 key.  Same shapes and limits as
                             KVC_QUANT_INT8, without witnesses: key element (token t,
                             channel c) of a block is stored as
                               code = clamp(rint(x/s + u), -127, 127), read as (code - u) s,
                             u = r/256 - 1/2 with r byte c mod 16 of the call
                               Philox4x32-10(counter = (t, c/16,
                                                       kv_head + 65536 layer_index,
                                                       request ID), key)
                             (byte i = bits 8(i mod 4) .. of word i/4); values keep the
                             plain block quantizer.  The request ID is b unless set by
                             kvc_set_request_id. */
    int32_t int8_split;   /* INT8 tiers: positions per quantized split of the decode (a
                             CTA's share of one request and KV head), a multiple of 64
                             in [1024, 2048]; 0 = 2048 when the cache (or a contiguous
                             cache's window + 32) spans 16384 slots or more, else 1024.
                             A tuning knob only: results do not depend on it beyond
                             fp32 rounding order.  Must be 0 without INT8. */
} kvc_config;

/* Bytes of the device state buffer for `cfg` (cache rows, positions,
 * next_position, RoPE table, INT8 arrays, split-K workspace).
 * Returns KVC_ERR_ARG for an invalid configuration. */
int kvc_state_bytes(const kvc_config* cfg, size_t* bytes);

/* Bind a handle to a caller-allocated device buffer of at least
 * kvc_state_bytes() bytes (256-byte aligned) on the current device.  Sets
 * every position to -1 and every next_position to 0, and uploads the RoPE
 * table; waits for `stream`.  The buffer must outlive the handle. */
int kvc_create(const kvc_config* cfg, void* d_state, size_t bytes, kvc_stream_t stream,
               kvc_t* out);

/* Release the host handle (the device buffer stays the caller's). */
int kvc_destroy(kvc_t h);

/* Append one token to every request ([LOOP] §三 step: write cache[pos];
 * [LEAN] §3.3 step).  d_k, d_v: [B][Hkv][d], keys not yet rotated.  For each
 * request: pos = next_position; the key is rotated at pos (if RoPE) and
 * rounded to the cache dtype; k, v go to slot pos (contiguous) or pos mod W
 * (ring); positions[slot] = pos; next_position = pos + 1.  INT8: the row goes
 * to the request's exact tail block; the 16th row of a block quantizes the
 * block and writes its witnesses.  KVC_ERR_CAPACITY if a contiguous cache is
 * full (nothing is written). */
int kvc_append(kvc_t h, const void* d_k, const void* d_v, kvc_stream_t stream);

/* Append up to n tokens per request, in order, from d_k, d_v [B][Hkv][n][d]
 * (prefill).  h_counts (host, B entries, NULL = n for all) limits request b to
 * its first h_counts[b] rows.  Same per-row semantics as kvc_append; on a ring
 * only the rows that stay resident are written. */
int kvc_append_rows(kvc_t h, const void* d_k, const void* d_v, int32_t n,
                    const int32_t* h_counts, kvc_stream_t stream);

/* Decode attention for the newest token of every request ([LOOP] §三 step;
 * [LEAN] §2.1).  d_q: [B][Hq][d] not yet rotated; the query sits at
 * t = next_position - 1, is rotated at t (if RoPE) in fp32, and attends to the
 * cached positions [max(0, t-W+1), t]:
 *     out = softmax(q . K^T / sqrt(d)) . V            d_out: [B][Hq][d]
 * evaluated as split-K flash decoding with an online softmax and a cross-split
 * combine, fp32 accumulation, rounded once to the output dtype.  Needs at least
 * one cached token per request, and on a ring an append after any trim.
 * INT8 caches also return, per (request, query head), the witness bound
 * ([WITCERT] "频带酉性与双层证书"):
 *     c_t = (1/sqrt d) sum_b ||q_b|| w_{t,b}   for every cached token in the window,
 *     d_cmax[b][h] = max_t c_t,  d_tanh[b][h] >= tanh(max_t c_t),
 * computed with upward rounding so that c_t >= |q . r_t| / sqrt(d) for the
 * stored residual r_t, hence attention total variation <= d_tanh
 * ([WITCERT] "为什么在线监控 KV 误差如此困难？").  d_ct (nullable) receives c_t
 * as [B][Hq][capacity] indexed by slot: the tokens of the window, and 0 for the
 * tokens before the window start that share its first block; other slots are not
 * written.  With a window (or a ring), max_t runs over the window only.
 * For non-quantized caches d_cmax/d_tanh (nullable) receive 0 and d_ct must
 * be NULL. */
int kvc_decode_attn(kvc_t h, const void* d_q, void* d_out, float* d_cmax, float* d_tanh,
                    float* d_ct, kvc_stream_t stream);
/* Tier B (KVC_QUANT_INT8_DITHER) caches regenerate every dither from its counter,
 * attend over the rows (code - u) s and the exact tail, and return no bound: the
 * tier's probabilistic certificate needs a per-request failure budget and a
 * concentration formula that the page does not give.  d_cmax, d_tanh and d_ct
 * must be NULL (KVC_ERR_ARG otherwise). */

/* Tier B: the request ID of request b in the dither counters, so that a
 * request's stream does not depend on its batch slot.  Only while request b holds
 * no rows (KVC_ERR_ARG otherwise, and for other tiers). */
int kvc_set_request_id(kvc_t h, int32_t b, uint32_t request_id, kvc_stream_t stream);

/* Decode attention that allocates nothing (the pages have no counterpart; this
 * is a deployment variant of kvc_decode_attn).
 *
 * Who it is for: callers that cannot call cudaMalloc while they decode. Examples:
 *   - a serving engine that reserved all device memory for its KV pool;
 *   - a runtime whose own allocator owns every device buffer;
 *   - host code that must not wait on the allocator's device synchronisation.
 *
 * What it does: the same computation and result as kvc_decode_attn (out
 * only; bf16/fp32 caches, not INT8).  The split-K partials go to a fixed
 * array of KVC_NOALLOC_SCRATCH_BYTES inside the library, not to the state
 * buffer's workspace.  The caller passes q and out; the cache is the handle's.
 *
 * The fixed array:
 *   - Every GPU that loads the library holds it until the process exits.
 *   - The first call on a device looks up the array's device address with that
 *     device current.  Make that first call before any stream capture.
 *   - Every call shares the array and overwrites it.  Each call writes every
 *     partial it reads, so nothing has to start at zero.
 *   - Calls that overlap on the GPU race on the array, even on different
 *     handles or streams: serialise them.
 *   - The looked-up address is kept for the life of the process.  A device
 *     reset (cudaDeviceReset, or the primary context torn down and made again)
 *     unloads the array, so this entry point must not be called after one.
 *
 * Errors:
 *   - KVC_ERR_CAPACITY if the problem needs more than the array holds, that is
 *     if B*Hq*splits*(8 + 4*d) bytes (+ 256 bytes of alignment) exceed
 *     KVC_NOALLOC_SCRATCH_BYTES, with
 *       splits = ceil(min(capacity, window) / split) + (page_pool > 0 ? 1 : 0)
 *     (window 0 = capacity), where split is the decode kernel's keys per split:
 *       1024, or 2048 when min(capacity, window) >= 16384, for bf16 caches with
 *         d = 64 or 128 and 4 or 8 query heads per KV head;
 *       128 for the other bf16 caches with d = 64 or 128 and at most 8 query
 *         heads per KV head;
 *       64 otherwise.
 *   - KVC_ERR_ARG for the cases kvc_decode_attn refuses, or if the current device
 *     is not the handle's.
 *   - KVC_ERR_UNSUPPORTED for an INT8 cache.
 * It calls no cudaMalloc, cudaFree or other allocating routine. */
#define KVC_NOALLOC_SCRATCH_BYTES (64u << 20)
/* See the comment above KVC_NOALLOC_SCRATCH_BYTES: d_q, d_out as for kvc_decode_attn. */
int kvc_decode_attn_noalloc(kvc_t h, const void* d_q, void* d_out, kvc_stream_t stream);

/* Continue every request from next_position = h_cut[b] ([PREFIX]
 * "哪些東西必須一起裁剪": keep k[:cut], v[:cut], positions[:cut]; next_position
 * = cut).  h_cut: host, B entries, 0 <= cut <= next_position.  Rows at
 * positions >= cut are dropped (positions set to -1).  A ring accepts the cut
 * only if every position the next query needs is still resident, i.e. with
 * lo = max(0, cut-W+1): lo == cut or lo >= max(0, next_position-W); an INT8
 * cache only if no quantized block is split (cut % 16 == 0 or cut within the
 * exact tail).  Otherwise KVC_ERR_EVICTED and nothing changes. */
int kvc_trim(kvc_t h, const int32_t* h_cut, kvc_stream_t stream);

/* Chunked causal suffix attention after a trim ([PREFIX] model.chunk(tokens[cut:],
 * cache)).  Appends n rows per request at positions cut .. cut+n-1 (as
 * kvc_append_rows) and answers every suffix query i at p = cut + i over
 * positions [max(0, p-W+1), p]:
 *     d_q [B][n][Hq][d], d_k, d_v [B][n][Hkv][d]  ->  d_out [B][n][Hq][d].
 * Row i equals what kvc_decode_attn returns for that query after appending
 * rows 0..i.  bf16 caches with head_dim 128, without INT8: contiguous, or a ring
 * whose size W is a multiple of 16 (paged or not); n <= max_chunk.  On a ring the
 * suffix may be longer than W: appending it first would evict rows that early
 * suffix queries need ([LEAN] §3.4), so the call stages the rotated suffix rows
 * in the state buffer (sized by max_chunk), attends, and then appends them; the
 * ring ends as n one-token appends would leave it.
 * The tensor-core products take fp16 operands: the query (rotated, times
 * log2(e)/sqrt(d)), the softmax weights and the K and V rows.  Every K and V row
 * of the keys the call reads, and every scaled query, must be below 65520 in
 * magnitude (the fp16 range); otherwise bit 2 of the device error word is set and
 * the output is not valid.  Nothing else is lost: K and V values in
 * [2^-14, 65504] are exact in fp16, smaller ones keep an absolute error of at
 * most 2^-25. */
int kvc_chunk_attn(kvc_t h, const void* d_q, const void* d_k, const void* d_v, int32_t n,
                   void* d_out, kvc_stream_t stream);

/* ---- gated fallback of the INT8 tier ----------------------------------
 * [WITCERT] "SGLang 生产级落地与闭环门控修复": once the risk of a head or a block
 * crosses the water line, the lossless block is swapped in from the full-precision
 * backing store and its witness is zeroed; in the saturated zone blocks are ranked by
 * risk and truncated.  Three steps, each usable alone:
 *   kvc_int8_block_risk  (device) the risk of every complete block from a decode's c_t;
 *   kvc_int8_gate        (host)   which blocks to restore;
 *   kvc_int8_restore     (device) restore them.
 * A restored block is served exactly (bf16) from a pool inside the state buffer
 * (kvc_config.int8_exact_blocks entries); its tokens get c_t = 0 from then on.  A
 * trim that drops a restored block returns its pool entry. */

/* d_risk[b][h][k] = max over the query heads of KV head h and the 16 tokens of block
 * k of d_ct[b][hq][t] (the per-token bound of the last kvc_decode_attn on this cache,
 * [B][Hq][capacity] fp32), for every complete block of request b; 0 elsewhere.
 * d_risk: fp32 [B][Hkv][capacity/16], device.  Async on `stream`.
 * KVC_ERR_ARG: not an INT8 cache, or a null pointer.  KVC_ERR_UNSUPPORTED: Tier B,
 * a ring or a window (the gated fallback serves contiguous caches that attend to
 * their whole history). */
int kvc_int8_block_risk(kvc_t h, const float* d_ct, float* d_risk, kvc_stream_t stream);

/* Host only.  Every (request, KV head, block) of h_risk ([B][Hkv][nblk] fp32, host)
 * with tanh(risk) > tau (both in double), highest risk first, ties broken by the smaller
 * (request, head, block); at most max_blocks of them into h_sel ([max_blocks][3]
 * int32 triples); their number into *h_n_sel.  KVC_ERR_ARG: bad sizes or pointers. */
int kvc_int8_gate(const float* h_risk, int32_t B, int32_t Hkv, int32_t nblk, double tau, int32_t max_blocks,
                  int32_t* h_sel, int32_t* h_n_sel);

/* Restore the n blocks listed in h_blocks ([n][3] int32 (request, KV head, block),
 * host): copy each block's 16 rows of K and V from the full-precision backing store
 * d_k_full / d_v_full (bf16 [B][Hkv][capacity][d], device: the rows an exact cache
 * holds, keys rotated) into the pool, zero the block's witnesses, and serve its
 * tokens from the pool in every later decode.  Blocks already restored are skipped.
 * KVC_ERR_ARG: not an INT8 cache, null pointer, or a block that is not complete;
 * KVC_ERR_CAPACITY: the pool has too few free entries, or a (request, KV head) would
 * hold more than 1024 restored blocks (nothing is restored then). */
int kvc_int8_restore(kvc_t h, const int32_t* h_blocks, int32_t n, const void* d_k_full, const void* d_v_full,
                     kvc_stream_t stream);

/* Bit-exact readback of one state array for tests and debug asserts
 * ([LEAN] §6.3: export the cache and compare it with the specification).
 * Copies into h_dst (exactly kvc_export_bytes() bytes) and waits for `stream`. */
enum {
    KVC_EXPORT_K = 0,             /* [B][Hkv][capacity][d] cache dtype (non-INT8) */
    KVC_EXPORT_V = 1,
    KVC_EXPORT_POSITIONS = 2,     /* int32 [B][capacity] */
    KVC_EXPORT_NEXT_POSITION = 3, /* int32 [B] */
    KVC_EXPORT_KQ = 4,            /* int8 [B][Hkv][capacity][d] signed codes (INT8; stored
                                     biased and in the decode's block order, converted here) */
    KVC_EXPORT_VQ = 5,            /* int8 [B][Hkv][capacity][d], as KQ */
    KVC_EXPORT_SK = 6,            /* fp32 [B][Hkv][capacity/16]           (INT8) */
    KVC_EXPORT_SV = 7,
    KVC_EXPORT_WITNESS = 8,       /* fp16 [B][Hkv][capacity][16]          (INT8) */
    KVC_EXPORT_KTAIL = 9,         /* bf16 [B][Hkv][16][d] exact tail rows (INT8) */
    KVC_EXPORT_VTAIL = 10,
    KVC_EXPORT_XMAP = 11,         /* int32 [B][Hkv][capacity/16]: pool entry of a restored
                                     block, -1 = quantized (INT8) */
    KVC_EXPORT_PAGE_TABLE = 12    /* int32 [B][capacity/16]: physical page of each logical
                                     page, -1 = none (paged caches; K and V exports are
                                     gathered through it into [B][Hkv][capacity][d]) */
};
/* *bytes = the size of export `which` for this handle.  KVC_ERR_ARG for a null
 * pointer or an export the cache does not hold (K/V of an INT8 cache, INT8 arrays
 * of a bf16/fp32 cache, the page table of an unpaged cache). */
int kvc_export_bytes(kvc_t h, int32_t which, size_t* bytes);
/* Copy export `which` into h_dst (host, `bytes` = kvc_export_bytes exactly, else
 * KVC_ERR_ARG), after the work already queued on `stream`; returns when the copy
 * is complete. */
int kvc_export(kvc_t h, int32_t which, void* h_dst, size_t bytes, kvc_stream_t stream);

/* Host mirror of next_position (B entries), kept by the handle.  Enqueued but
 * unexecuted work is already counted. */
int kvc_next_positions(kvc_t h, int32_t* h_out);

/* Waits for `stream`, then returns the device error word (0 = none; bit 0: a
 * kernel met a position outside the cache or RoPE table; bit 1: a bounded wait
 * gave up; bit 2: kvc_chunk_attn met an operand beyond the fp16 range) and
 * clears it. */
int kvc_device_status(kvc_t h, kvc_stream_t stream, int32_t* h_status);

/* Health check of the failure path: enqueues one CTA that waits, with the same
 * bounded wait the kernels use for their copies, on a barrier that nothing
 * signals.  The wait gives up after its bound (about one second), sets bit 1 of
 * the device error word and returns; nothing faults and the context stays
 * usable.  A following kvc_device_status reports the bit (and clears it). */
int kvc_check_wait_path(kvc_t h, kvc_stream_t stream);

/* Host only.  Rows of a stored prefill that a new query can reuse ([PREFIX]
 * "先看一次歷史編輯", "查詢流程與快取所有權", "為什麼滑窗部分命中必須回退"):
 * cut = length of the longest contiguous common prefix of old and new IDs,
 * at most n_new - 1 (the last query token is always recomputed).  With ring != 0
 * only a full match of the cached prefix followed by new tokens is reused
 * (cut = n_old), otherwise cut = 0.  KVC_ERR_ARG if n_new < 1, n_old < 0 or a
 * pointer is NULL where its count is positive. */
int kvc_prefix_cut(const int64_t* h_old_ids, int32_t n_old, const int64_t* h_new_ids,
                   int32_t n_new, int32_t ring, int32_t* h_cut);

/* ---- prefix store ([PREFIX] "查詢流程與快取所有權") -------------------------
 * Policy and data are split.  A kvc_pstore_t (host only, no GPU needed) decides
 * which stored prefill a query reuses and how many of its rows; the rows
 * themselves live in the store slots of a handle's state (kvc_config.store_slots)
 * and move with kvc_store_save / kvc_store_load.  A pstore slot index names the
 * handle's store slot that holds that entry's rows. */
typedef struct kvc_pstore* kvc_pstore_t;

/* Host only.  A store of at most `capacity` prefills of caches configured as
 * `cfg` ([PREFIX]: at most two).  The configuration (dtype, layout, window, head
 * shape, RoPE base) is part of every entry's computation signature; a ring
 * layout selects the sliding-window reuse rule.  KVC_ERR_ARG for capacity < 1 or
 * an invalid cfg. */
int kvc_pstore_create(const kvc_config* cfg, int32_t capacity, kvc_pstore_t* out);
/* Host only.  Frees the store (its entries' IDs, scopes and signatures); the rows
 * in the handle's store slots are untouched.  KVC_ERR_ARG for NULL. */
int kvc_pstore_destroy(kvc_pstore_t ps);

/* Host only.  Records a prefill of the n_ids >= 1 token IDs h_ids under the
 * application scope `scope` (NUL-terminated, compared byte for byte) and the
 * caller's part of the computation signature (sig_bytes bytes at h_sig, e.g. a
 * hash of the weights and of the implementation; h_sig may be NULL when
 * sig_bytes is 0).  *h_slot = the slot used: the lowest free one, else the slot
 * of the oldest entry, which is replaced (the page is silent on eviction). */
int kvc_pstore_insert(kvc_pstore_t ps, const int64_t* h_ids, int32_t n_ids, const char* scope,
                      const void* h_sig, int32_t sig_bytes, int32_t* h_slot);

/* Host only.  Lookup of a query of n_ids >= 1 token IDs, in the page's order:
 * entries with the same scope and signature are eligible; each offers the cut
 * of kvc_prefix_cut (longest contiguous common prefix, at most n_ids - 1; on a
 * ring only a whole-prefix match); the largest cut wins, ties going to the most
 * recently inserted entry.  *h_slot = that entry's slot and *h_cut its cut, or
 * -1 and 0 when no entry offers a row. */
int kvc_pstore_lookup(kvc_pstore_t ps, const int64_t* h_ids, int32_t n_ids, const char* scope,
                      const void* h_sig, int32_t sig_bytes, int32_t* h_slot, int32_t* h_cut);

/* Copies request b's cache into store slot `slot` of the state: K and V rows
 * and positions (every slot of a ring).  n must equal request b's next_position
 * (the prefill's length, n >= 1).  KVC_ERR_UNSUPPORTED without store slots. */
int kvc_store_save(kvc_t h, int32_t slot, int32_t b, int32_t n, kvc_stream_t stream);

/* Request b continues from rows [0, cut) of store slot `slot` ([PREFIX] step 4:
 * the kept K, V and positions are copied out of the store, which keeps its
 * own): the slot's rows at positions below cut are copied into request b,
 * every other slot of b is emptied, and next_position[b] = cut.  slot = -1 with
 * cut = 0 empties request b.  Other requests are untouched.  KVC_ERR_ARG if the
 * slot holds nothing or cut exceeds its length; KVC_ERR_EVICTED if a ring slot no
 * longer holds rows that the token at `cut` would attend to (the kvc_trim rule);
 * KVC_ERR_CAPACITY if a paged cache lacks pages (nothing changes).  On a ring, as
 * after kvc_trim, the next call on the handle must append. */
int kvc_store_load(kvc_t h, int32_t slot, int32_t b, int32_t cut, kvc_stream_t stream);

/* kvc_store_load for n requests at once (h_slots, h_b, h_cuts: host arrays of n
 * entries; the requests distinct), in one launch per 64 requests.  Every entry
 * is checked before anything changes; the statuses are those of kvc_store_load. */
int kvc_store_load_batch(kvc_t h, int32_t n, const int32_t* h_slots, const int32_t* h_b,
                         const int32_t* h_cuts, kvc_stream_t stream);

/* Static description of a status code. */
const char* kvc_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* KVC_H */
