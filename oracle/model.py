"""Whole decode-step oracle: per request the full history, attention by definition.

TEST INFRASTRUCTURE (see the package docstring).

The model keeps, for every request, the *full history* of stored rows (row j =
absolute position j) -- never a ring -- and answers every query by masked
attention over that history ([LEAN] §2.1).  The physical cache the GPU should
hold is derived separately: slot = position for a contiguous cache ([LOOP] §三,
``cache[:, :, pos]``), and for a ring the :class:`~oracle.listmodel.RingBuffer`
head/count model ([LEAN] §3.4), whose ``ringToList`` must equal ``lastWindow``.

Stored rows: keys are RoPE-rotated at their position when a rotary base is set
(fp32 arithmetic, see ``oracle.c``) and then rounded to the cache dtype; values
are stored as given.  The query is rotated the same way and kept in fp32.

INT8 tier ([WITCERT] "频带酉性与双层证书" and "SGLang 生产级落地与闭环门控修复"):
complete 16-position blocks of a contiguous cache hold INT8 codes with one fp32
scale for K and one for V plus 16 fp16 witnesses per key row; the rows of the
incomplete last block stay exact (bf16) with witness 0.  A block restored by the
gated fallback ("SGLang 生产级落地与闭环门控修复": swap in the lossless block
from the full-precision backing store, zero its witnesses) is held exact as
well, with residual 0 and witness 0.

Tier B ([WITCERT], the subtractive-dither paragraph, and "SGLang 生产级落地与闭环门控修复"
for the counter): key codes rint(x/s + u) with a Philox dither u per element, read
back as (code - u) s; values keep the plain quantizer; no witnesses.  The probabilistic certificate of this tier needs a
failure budget and a concentration formula the page does not give, so the oracle
states no bound for it.

[LEAN]    "用Lean4形式化验证滑动窗口KV Cache的正确性" (framerc.cn/news/4505248)
[PREFIX]  "LLM 機制實驗（五）：改了歷史，能否只重算變化的後綴？" (huhohoo.com)
[LOOP]    "KV Cache 自回归生成推理（增量更新与状态拼接）" (airsota.com/?p=549)
[WITCERT] "WitCert: Sound Runtime Risk Observability and Gating for KV-Cache Quantization"
"""
from __future__ import annotations

import copy
import math
from typing import List

import numpy as np

from . import numerics as nm
from .listmodel import Cell, RingBuffer, last_window, ring_trim_allowed

QBLOCK = 16      # tokens per quantization block
NBANDS = 16      # witness bands per key row


class OracleError(Exception):
    def __init__(self, code: str, msg: str = ""):
        super().__init__(code + (": " + msg if msg else ""))
        self.code = code


def as_f32(x, dtype: str) -> np.ndarray:
    """Input values as fp32 (exact): ``x`` holds fp32 values or bf16 bit patterns."""
    x = np.asarray(x)
    if dtype == "bf16":
        return nm.bf16_to_f32(x.astype(np.uint16))
    return x.astype(np.float32)


class DecodeOracle:
    """Reference model of a KV cache for B requests of one layer.

    layout: "contiguous" (capacity = max_seq_len) or "ring" (capacity = window W).
    window: attention window (0 = full history; a ring always attends to W).
    dtype: "f32" or "bf16" (inputs and stored rows).  quant: None or "int8".
    """

    def __init__(self, B, Hq, Hkv, d, layout="contiguous", capacity=0, window=0,
                 rope_base=0.0, dtype="f32", quant=None, dither_key=(0, 0), layer=0):
        assert Hq % Hkv == 0
        self.B, self.Hq, self.Hkv, self.d = B, Hq, Hkv, d
        self.g = Hq // Hkv
        self.layout, self.capacity = layout, capacity
        self.window = capacity if layout == "ring" else window
        self.rope_base, self.dtype, self.quant = rope_base, dtype, quant
        # Tier B (quant "int8-dither"): the Philox key, the layer and each request's ID
        self.dither_key, self.layer = tuple(dither_key), layer
        self.request_ids = list(range(B))
        # full history of stored rows per request: lists of [Hkv, d] fp32 arrays
        self.hk: List[List[np.ndarray]] = [[] for _ in range(B)]
        self.hv: List[List[np.ndarray]] = [[] for _ in range(B)]
        self.rings = [RingBuffer(capacity) for _ in range(B)] if layout == "ring" else None
        # INT8 blocks restored to full precision: restored[b][kv_head] = set of block indices
        self.restored = [[set() for _ in range(Hkv)] for _ in range(B)]

    # ------------------------------------------------------------ rows
    def stored_rows(self, x, positions) -> np.ndarray:
        """Rows as the cache stores them: rotated (keys, if RoPE) and rounded to the dtype."""
        xf = as_f32(x, self.dtype)
        if self.rope_base:
            xf = nm.rope_rotate(xf, positions, self.rope_base)
            if self.dtype == "bf16":
                xf = nm.bf16_to_f32(nm.f32_to_bf16(xf))
        return xf

    def query_rows(self, q, positions) -> np.ndarray:
        """The query as attention sees it: rotated at its position (if RoPE), kept in fp32."""
        qf = as_f32(q, self.dtype)
        if self.rope_base:
            qf = nm.rope_rotate(qf, positions, self.rope_base)
        return qf

    def length(self, b) -> int:
        return len(self.hk[b])

    # ------------------------------------------------------------ mutations
    def append(self, k, v, active=None):
        """One new token per request: k, v [B, Hkv, d] (pre-RoPE).  ``active`` masks requests."""
        for b in range(self.B):
            if active is not None and not active[b]:
                continue
            pos = self.length(b)
            if self.layout == "contiguous" and pos >= self.capacity:
                raise OracleError("capacity", "position %d >= max_seq_len %d" % (pos, self.capacity))
            kb = self.stored_rows(np.asarray(k)[b], np.full(self.Hkv, pos))
            vb = as_f32(np.asarray(v)[b], self.dtype)
            self.hk[b].append(kb)
            self.hv[b].append(vb)
            if self.rings is not None:
                self.rings[b].push(Cell(pos, kb, vb))

    def append_rows(self, k, v, counts):
        """counts[b] tokens per request from k, v [B, Hkv, n, d], in order."""
        for r in range(int(max(counts)) if len(counts) else 0):
            act = [r < c for c in counts]
            self.append(np.asarray(k)[:, :, r], np.asarray(v)[:, :, r], active=act)

    def trim(self, cuts):
        """Continue every request from ``next_position = cut`` ([PREFIX] "哪些東西必須一起裁剪").

        Rows at positions >= cut leave the history.  A ring accepts the cut only
        if every row the next query needs is resident
        (:func:`~oracle.listmodel.ring_trim_allowed`); an INT8 cache only if no
        already-quantized block has to be split.  Nothing changes on error.
        """
        for b, cut in enumerate(cuts):
            n = self.length(b)
            if cut < 0 or cut > n:
                raise OracleError("arg", "cut %d outside [0, %d]" % (cut, n))
            if self.rings is not None and not ring_trim_allowed(cut, n, self.capacity):
                raise OracleError("evicted", "request %d: rows needed after cut %d are gone" % (b, cut))
            if self.quant in ("int8", "int8-dither") and cut % QBLOCK and cut < (n // QBLOCK) * QBLOCK:
                raise OracleError("evicted", "request %d: cut %d splits a quantized block" % (b, cut))
        for b, cut in enumerate(cuts):
            n = self.length(b)
            del self.hk[b][cut:]
            del self.hv[b][cut:]
            if self.rings is not None:
                self.rings[b].truncate(n - cut, cut % self.capacity)
            for h in range(self.Hkv):          # restored blocks past the cut leave with their rows
                self.restored[b][h] = {blk for blk in self.restored[b][h] if (blk + 1) * QBLOCK <= cut}

    def snapshot(self, b):
        """Request b's stored rows, ring state and restored blocks, as a private copy."""
        ring = self.rings[b] if self.rings is not None else None
        return copy.deepcopy((self.hk[b], self.hv[b], ring, self.restored[b]))

    def load(self, b, snap, cut):
        """Request b continues from rows [0, cut) of a snapshot (None = an empty request).

        The same as putting the snapshot's state back and trimming request b to ``cut``
        ([PREFIX] "查詢流程與快取所有權", step 4: the kept rows are copied out of the
        store, which keeps its own).  A ring refuses a cut whose rows were evicted
        before the snapshot was taken.  Nothing changes on error.
        """
        if snap is None:
            if cut != 0:
                raise OracleError("arg", "an empty request continues from 0")
            snap = ([], [], RingBuffer(self.capacity) if self.rings is not None else None,
                    [set() for _ in range(self.Hkv)])
        hk, hv, ring, restored = copy.deepcopy(snap)
        n = len(hk)
        if cut < 0 or cut > n:
            raise OracleError("arg", "cut %d outside [0, %d]" % (cut, n))
        if ring is not None and not ring_trim_allowed(cut, n, self.capacity):
            raise OracleError("evicted", "rows needed after cut %d were evicted" % cut)
        self.hk[b], self.hv[b], self.restored[b] = hk, hv, restored
        if self.rings is not None:
            self.rings[b] = ring
        cuts = [self.length(x) for x in range(self.B)]
        cuts[b] = cut
        self.trim(cuts)

    # ------------------------------------------------------------ attention
    def _history(self, b, kv_head, lo=0, hi=None):
        hi = self.length(b) if hi is None else hi
        K = np.stack([r[kv_head] for r in self.hk[b][lo:hi]]) if hi > lo else np.zeros((0, self.d), np.float32)
        V = np.stack([r[kv_head] for r in self.hv[b][lo:hi]]) if hi > lo else np.zeros((0, self.d), np.float32)
        return K, V

    def decode(self, q, nthreads=1, full_history=True) -> np.ndarray:
        """Attention of the newest token's query: q [B, Hq, d] -> fp64 [B, Hq, d].

        The query sits at position t = length - 1 and sees positions
        [max(0, t - W + 1), t] of the full history (W = window; 0 = all).
        With ``full_history=False`` only rows from the window start on are passed
        (the masked rows carry zero weight, so the result is the same).
        """
        out = np.zeros((self.B, self.Hq, self.d))
        qs, ks, vs, ts, p0s, idx = [], [], [], [], [], []
        for b in range(self.B):
            t = self.length(b) - 1
            if t < 0:
                continue
            qr = self.query_rows(np.asarray(q)[b], np.full(self.Hq, t)).astype(np.float64)
            lo = 0 if full_history or not self.window else max(0, t - self.window + 1)
            for h in range(self.Hkv):
                K, V = self._history(b, h, lo)
                qs.append(qr[h * self.g:(h + 1) * self.g])
                ks.append(K); vs.append(V); ts.append(t); p0s.append(lo); idx.append((b, h))
        res = nm.attend_many(qs, ks, vs, ts, self.window, p0s, nthreads=nthreads)
        for (b, h), o in zip(idx, res):
            out[b, h * self.g:(h + 1) * self.g] = o
        return out

    def chunk(self, q, k, v) -> np.ndarray:
        """Append n suffix rows and answer each suffix query ([PREFIX] ``model.chunk``).

        q [B, n, Hq, d], k/v [B, n, Hkv, d].  Suffix query i sits at position
        cut + i and sees exactly what a one-token decode at that position sees.
        """
        q, k, v = np.asarray(q), np.asarray(k), np.asarray(v)
        n = q.shape[1]
        out = np.zeros((self.B, n, self.Hq, self.d))
        for i in range(n):
            self.append(k[:, i], v[:, i])
            out[:, i] = self.decode(q[:, i])
        return out

    # ------------------------------------------------------------ physical state
    def expected_positions(self) -> np.ndarray:
        """positions[b][slot] (int32, -1 = empty) the GPU cache must hold."""
        S = self.capacity
        pos = np.full((self.B, S), -1, dtype=np.int32)
        for b in range(self.B):
            if self.rings is None:
                pos[b, :self.length(b)] = np.arange(self.length(b))
            else:
                ring = self.rings[b]
                for i in range(ring.count):
                    slot = (ring.head + i) % ring.w
                    pos[b, slot] = ring.buf[slot].pos
        return pos

    def expected_rows(self, b, which="k") -> dict:
        """{slot: stored row [Hkv, d] fp32} for every live slot of request b."""
        rows = {}
        if self.rings is None:
            src = self.hk[b] if which == "k" else self.hv[b]
            for s, r in enumerate(src):
                rows[s] = r
        else:
            ring = self.rings[b]
            for i in range(ring.count):
                slot = (ring.head + i) % ring.w
                cell = ring.buf[slot]
                rows[slot] = cell.key if which == "k" else cell.val
        return rows

    def logical_window(self, b) -> list:
        """lastWindow(W, history) as cells ([LEAN] §2.3); W = capacity of a ring."""
        cells = [Cell(p, self.hk[b][p], self.hv[b][p]) for p in range(self.length(b))]
        return last_window(self.window if self.window else len(cells), cells)

    # ------------------------------------------------------------ INT8 tier
    def set_request_id(self, b, rid):
        """Tier B: the request ID in the dither counters; only while request b is empty."""
        if self.length(b):
            raise OracleError("arg", "request %d holds rows" % b)
        self.request_ids[b] = int(rid) & 0xFFFFFFFF

    def dither(self, b, h):
        """Tier B: u(p0, n) -> [n, d] fp32 key dithers of (request b, KV head h), else None."""
        if self.quant != "int8-dither":
            return None
        key, rid, layer, d = self.dither_key, self.request_ids[b], self.layer, self.d

        def u(p0, n):
            return nm.dither_values(nm.dither_rows(key, rid, layer, h, p0, n, d))
        return u

    def quantized_block(self, b, h, blk):
        """(sK, codesK [16,d], sV, codesV, wit bits [16,16]) of one complete block
        (Tier B: dithered key codes, plain value codes, no witnesses: None)."""
        lo = blk * QBLOCK
        K = np.stack([self.hk[b][p][h] for p in range(lo, lo + QBLOCK)])
        V = np.stack([self.hv[b][p][h] for p in range(lo, lo + QBLOCK)])
        u = self.dither(b, h)
        if u is not None:
            sK, cK = nm.quantize_block_dither(K, u(lo, QBLOCK))
            sV, cV = nm.quantize_block(V)
            return sK, cK, sV, cV, None
        sK, cK = nm.quantize_block(K)
        sV, cV = nm.quantize_block(V)
        wit = np.stack([nm.witness_row(K[r], cK[r], sK, NBANDS) for r in range(QBLOCK)])
        return sK, cK, sV, cV, wit

    def int8_view(self, b, h, lo=0, hi=None):
        """Rows [lo, hi) of (b, h) as attention sees them in the INT8 tier (see :func:`int8_rows`)."""
        n = self.length(b)
        hi = n if hi is None else hi
        K = np.stack([self.hk[b][p][h] for p in range(lo, hi)]) if hi > lo else np.zeros((0, self.d), np.float32)
        V = np.stack([self.hv[b][p][h] for p in range(lo, hi)]) if hi > lo else np.zeros((0, self.d), np.float32)
        return int8_rows(K, V, lo, (n // QBLOCK) * QBLOCK, self.restored[b][h], self.dither(b, h))

    def restore(self, blocks):
        """Gated fallback ("SGLang 生产级落地与闭环门控修复"): hold the listed complete
        blocks, (request, KV head, block index) triples, exact again from then on."""
        for b, h, blk in blocks:
            if (blk + 1) * QBLOCK > (self.length(b) // QBLOCK) * QBLOCK:
                raise OracleError("arg", "block %d of request %d is not complete" % (blk, b))
            self.restored[b][h].add(blk)

    def decode_int8(self, q, heads=None):
        """INT8-tier decode of the newest token for the listed (b, query head) pairs
        (all by default); see :func:`int8_decode_one` for the returned fields."""
        res = {}
        if heads is None:
            heads = [(b, hq) for b in range(self.B) for hq in range(self.Hq)]
        for (b, hq) in heads:
            t = self.length(b) - 1
            qf = self.query_rows(np.asarray(q)[b, hq:hq + 1], np.full(1, t))[0]
            lo = 0 if not self.window else max(0, t - self.window + 1)
            lo_blk = (lo // QBLOCK) * QBLOCK
            h = hq // self.g
            K = np.stack([self.hk[b][p][h] for p in range(lo_blk, t + 1)])
            V = np.stack([self.hv[b][p][h] for p in range(lo_blk, t + 1)])
            res[(b, hq)] = int8_decode_one(qf, K, V, lo_blk, t, self.window, (self.length(b) // QBLOCK) * QBLOCK,
                                           self.restored[b][h], self.dither(b, h))
        return res


def int8_rows(K, V, p0, nfull, restored=(), dither=None):
    """Rows at positions p0.. of one (request, KV head) as the INT8 tier holds them.

    ``K``, ``V``: [n, d] exact stored rows (fp32 values of the bf16 cache); ``p0`` a
    block boundary; positions below ``nfull`` lie in complete blocks; ``restored``
    holds the block indices (position // 16) brought back to full precision by the
    gated fallback.  Returns (K_deq, V_deq, K_exact, resid, wit_values), all fp64:
    complete blocks dequantized (code * s, exact in fp64) with their key residuals
    and witness values; the exact tail rows and restored blocks with residual 0 and
    witness 0 ([WITCERT] "频带酉性与双层证书"; "SGLang 生产级落地与闭环门控修复").

    Tier B ([WITCERT], the subtractive-dither paragraph): ``dither(p0, n)`` gives the
    fp32 key dithers u of n rows from position p0; key codes are rint(x/s + u) and the
    keys read back as (code - u) s, exact in fp64; values keep the plain quantizer.
    There are no witnesses then (the returned witness values are None).
    """
    n, d = K.shape
    assert p0 % QBLOCK == 0
    Kd = K.astype(np.float64).copy()
    Vd = V.astype(np.float64).copy()
    R = np.zeros((n, d))
    Wt = np.zeros((n, NBANDS))
    for r0 in range(0, n, QBLOCK):
        if p0 + r0 + QBLOCK > nfull or r0 + QBLOCK > n:
            break
        if (p0 + r0) // QBLOCK in restored:
            continue
        sl = slice(r0, r0 + QBLOCK)
        if dither is not None:
            uK = dither(p0 + r0, QBLOCK)
            sK, cK = nm.quantize_block_dither(K[sl], uK)
            sV, cV = nm.quantize_block(V[sl])
            Kd[sl] = (cK.astype(np.float64) - uK.astype(np.float64)) * np.float64(sK)
            Vd[sl] = cV.astype(np.float64) * np.float64(sV)
            R[sl] = K[sl].astype(np.float64) - Kd[sl]
            continue
        sK, cK = nm.quantize_block(K[sl])
        sV, cV = nm.quantize_block(V[sl])
        Kd[sl] = cK.astype(np.float64) * np.float64(sK)
        Vd[sl] = cV.astype(np.float64) * np.float64(sV)
        R[sl] = K[sl].astype(np.float64) - Kd[sl]
        Wt[sl] = np.stack([nm.f16_values(nm.witness_row(K[r0 + i], cK[i], sK, NBANDS)) for i in range(QBLOCK)])
    return Kd, Vd, K.astype(np.float64), R, (None if dither is not None else Wt)


def int8_decode_one(qf, K, V, p0, t, window, nfull, restored=(), dither=None):
    """INT8-tier decode of one query row over rows p0..t of one KV head, fp64.

    Returns {"out": attention over the dequantized rows, "out_exact": over the
    exact bf16 rows, "c": c_t per key in the window, "eps": |q . r_t| / sqrt(d),
    "tv": total variation between the exact and the dequantized softmax,
    "cmax": max_t c_t, "q": the fp32 query}.  c_t = (1/sqrt d) sum_b ||q_b|| w_{t,b}
    ([WITCERT] "频带酉性与双层证书") from the fp32 query and the stored witnesses.
    Tier B (``dither``, see :func:`int8_rows`): no witnesses, so "c" is None and
    "cmax" 0.
    """
    d = K.shape[1]
    bw = d // NBANDS
    q64 = np.asarray(qf, dtype=np.float64)
    Kd, Vd, Kx, R, W = int8_rows(K, V, p0, nfull, restored, dither)
    Vx = V.astype(np.float64)
    out = nm.attend(q64, Kd, Vd, t, window, p0=p0)[0]
    out_exact = nm.attend(q64, Kx, Vx, t, window, p0=p0)[0]
    p_deq = nm.softmax_weights(q64, Kd, t, window, p0=p0)
    p_ex = nm.softmax_weights(q64, Kx, t, window, p0=p0)
    eps = np.abs(R @ q64) / math.sqrt(d)
    lo = 0 if not window else max(0, t - window + 1)
    vis = slice(lo - p0, None)
    if W is None:
        return {"out": out, "out_exact": out_exact, "c": None, "eps": eps[vis],
                "tv": 0.5 * np.abs(p_ex - p_deq).sum(), "cmax": 0.0, "q": qf}
    qn = np.sqrt((q64.reshape(NBANDS, bw) ** 2).sum(axis=1))
    c = (W * qn[None, :]).sum(axis=1) / math.sqrt(d)
    return {"out": out, "out_exact": out_exact, "c": c[vis], "eps": eps[vis],
            "tv": 0.5 * np.abs(p_ex - p_deq).sum(), "cmax": float(c[vis].max()) if c[vis].size else 0.0,
            "q": qf}


# ---------------------------------------------------------------------- gated fallback
def block_risk(c_heads, nfull):
    """Risk of every complete block of one (request, KV head): the largest c_t of its
    16 tokens over the KV head's query heads ("SGLang 生产级落地与闭环门控修复": a
    block whose accumulated risk crosses the water line is swapped back in).

    ``c_heads``: [g, n] c_t of positions 0..n-1 for the g query heads; returns
    [nfull // 16] floats.
    """
    c = np.asarray(c_heads, dtype=np.float64)
    nb = nfull // QBLOCK
    return np.array([c[:, blk * QBLOCK:(blk + 1) * QBLOCK].max() if c.size else 0.0 for blk in range(nb)])


def gate_select(risk, tau, budget=None):
    """Blocks to restore: every (request, KV head, block) whose risk gives
    tanh(risk) > tau, highest risk first (ties: smaller (request, head, block)),
    cut to ``budget`` blocks ("SGLang 生产级落地与闭环门控修复": triggered by the
    certificate, ranked by risk score and truncated).

    ``risk``: {(b, h): [nblk] array}.
    """
    cand = []
    for (b, h), r in sorted(risk.items()):
        for blk, x in enumerate(np.asarray(r, dtype=np.float64)):
            if math.tanh(x) > tau:
                cand.append((-x, b, h, blk))
    cand.sort()
    if budget is not None:
        cand = cand[:budget]
    return [(b, h, blk) for _, b, h, blk in cand]
