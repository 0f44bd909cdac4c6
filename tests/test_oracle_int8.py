"""Pins of the oracle's INT8 tier: quantizer, residual, witness, bound (CPU only).

[WITCERT] "WitCert: Sound Runtime Risk Observability and Gating for KV-Cache Quantization"
  "为什么在线监控 KV 误差如此困难？": TV <= tanh(max |eps|)
  "频带酉性与双层证书": ||(R_n x)_b|| = ||x_b||; w_{t,b} = ||r_{t,b}||; |eps_t| = |q.r_t|/sqrt(d)
      <= (1/sqrt d) sum_b ||q_b|| w_{t,b} = c_t; 16 bands, 32 B per token and head
  "SGLang 生产级落地与闭环门控修复": per-block scale factors
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import numerics as nm
from oracle.model import NBANDS, QBLOCK, DecodeOracle


def _block(rng, outliers=False, scale=1.0):
    x = rng.standard_normal((QBLOCK, 128)).astype(np.float32) * np.float32(scale)
    if outliers:
        x[:, [3, 40, 77, 120]] *= np.float32(20.0)
    return nm.bf16_to_f32(nm.f32_to_bf16(x))          # cache values are bf16


@pytest.mark.parametrize("outliers", [False, True])
def test_quantizer_against_numpy_and_exact_nearest(outliers):
    rng = np.random.default_rng(11 + outliers)
    for _ in range(20):
        x = _block(rng, outliers, scale=float(rng.choice([1e-3, 1.0, 300.0])))
        s, codes = nm.quantize_block(x)
        amax = np.float32(np.abs(x).max())
        assert s == amax / np.float32(127.0)                    # one fp32 division (numpy)
        ref = np.clip(np.rint(x / s), -127, 127).astype(np.int8)  # numpy fp32 divide + rint (half even)
        assert np.array_equal(codes, ref)
        assert np.abs(codes).max() == 127                        # the amax element maps to +-127
        assert np.abs(codes.astype(np.int64)).max() <= 127
        # exact arithmetic: each code is a nearest integer to x/s unless x/s is within fp32
        # rounding of a half-integer
        S = Fraction(float(s))
        for v, c in zip(x.reshape(-1)[::37], codes.reshape(-1)[::37]):
            y = Fraction(float(v)) / S
            if abs(abs(y - math.floor(y)) - Fraction(1, 2)) < Fraction(1, 1 << 20):
                continue
            assert c == max(-127, min(127, round(y)))


def test_quantizer_zero_block():
    s, codes = nm.quantize_block(np.zeros((QBLOCK, 128), np.float32))
    assert s == 0.0 and not codes.any()


def test_residual_is_exact_in_fp32():
    rng = np.random.default_rng(12)
    for trial in range(30):
        x = _block(rng, outliers=trial % 2 == 1, scale=float(10.0 ** rng.uniform(-6, 4)))
        x[0, :5] = np.float32(1e-30)                            # tiny entries next to large ones
        s, codes = nm.quantize_block(x)
        for r in range(QBLOCK):
            res = nm.residual_row(x[r], codes[r], s)
            exact = [Fraction(float(a)) - int(c) * Fraction(float(s)) for a, c in zip(x[r], codes[r])]
            assert all(Fraction(float(a)) == e for a, e in zip(res, exact))
            # |r| <= s (1/2 + 127 * 2^-24): x/s is one fp32 division, rounded before rint
            assert max(abs(e) for e in exact) <= Fraction(float(s)) * (Fraction(1, 2) + Fraction(127, 1 << 24))
            nm.witness_row(x[r], codes[r], s)                     # raises if a residual were inexact


def _f16(bits):
    return Fraction(float(np.array(bits, np.uint16).view(np.float16)))


@pytest.mark.parametrize("outliers", [False, True])
def test_witness_is_a_tight_upper_bound_exactly(outliers):
    # exact rational arithmetic: w^2 >= sum r_i^2 over the band, and the next smaller fp16
    # value is below the norm times (1 + 2^-18) (the fp32 round-up chain adds < 2^-18).
    rng = np.random.default_rng(13 + outliers)
    bw = 128 // NBANDS
    for _ in range(6):
        x = _block(rng, outliers)
        s, codes = nm.quantize_block(x)
        for r in range(0, QBLOCK, 3):
            w = nm.witness_row(x[r], codes[r], s)
            res = [Fraction(float(a)) - int(c) * Fraction(float(s)) for a, c in zip(x[r], codes[r])]
            for b in range(NBANDS):
                sq = sum(v * v for v in res[b * bw:(b + 1) * bw])
                wb = _f16(w[b])
                assert wb * wb >= sq
                if w[b] > 0:
                    prev = _f16(int(w[b]) - 1)
                    assert prev * prev < sq * Fraction((1 << 18) + 1, 1 << 18) ** 2


def test_witness_special_cases():
    s = np.float32(0.5)
    # zero residual -> witness 0
    codes = np.arange(-64, 64, dtype=np.int8)
    x = (codes.astype(np.float32) * s).astype(np.float32)
    assert not nm.witness_row(x, codes, s).any()
    # one nonzero residual per band with an exact square root: w = that magnitude
    x2 = x.copy()
    x2[::8] += np.float32(0.125)                                # residual 0.125 in every band
    w = nm.witness_row(x2, codes, s)
    assert all(float(np.array(b, np.uint16).view(np.float16)) == 0.125 for b in w)
    # 32 bytes of witness per token and head ([WITCERT]: 16 bands x fp16)
    assert w.nbytes == 32


def _int8_model(rng, T=70, outliers=True, window=0):
    B, Hq, Hkv, d = 1, 4, 2, 128
    m = DecodeOracle(B, Hq, Hkv, d, "contiguous", 256, window, 10000.0, "bf16", "int8")
    for t in range(T):
        k = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        if outliers:
            k[:, :, [5, 17, 64, 99]] *= 20.0
        v = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        m.append(nm.f32_to_bf16(k), nm.f32_to_bf16(v))
    return m


@pytest.mark.parametrize("outliers", [False, True])
def test_bound_soundness(outliers):
    # |eps_t| <= c_t for every cached token (Cauchy-Schwarz per band), and the attention total
    # variation between exact and dequantized keys is <= tanh(max_t c_t); it is in fact
    # <= tanh(max_t |eps_t| / 2), the tight form of the same inequality.
    rng = np.random.default_rng(14 + outliers)
    m = _int8_model(rng, outliers=outliers)
    for trial in range(5):
        q = nm.f32_to_bf16(rng.standard_normal((1, 4, 128)).astype(np.float32) * (1 + 3 * trial))
        res = m.decode_int8(q)
        for key, r in res.items():
            assert np.all(r["eps"] <= r["c"] * (1 + 1e-12))
            assert r["tv"] <= math.tanh(r["cmax"])
            assert r["tv"] <= math.tanh(r["eps"].max() / 2) * (1 + 1e-9) + 1e-15
            # the tail block (rows 64..69) is exact: c_t = 0 there
            assert np.all(r["c"][64:] == 0) and np.all(r["eps"][64:] == 0)


def test_bound_tv_extremes():
    # Two keys, logits perturbed by +E and -E: the TV equals tanh(E/2) at the worst mass split,
    # and tanh(E) >= it.  Checks the TV evaluation against the closed form.
    for E in (0.01, 0.3, 2.0):
        a = 1.0 / (math.exp(E) + 1.0)                       # optimal mass on the +E key
        p = np.array([a, 1 - a])
        logits = np.log(p)
        ph = np.exp(logits + np.array([E, -E])); ph /= ph.sum()
        tv = 0.5 * np.abs(p - ph).sum()
        assert abs(tv - math.tanh(E / 2)) < 1e-12 and tv <= math.tanh(E)


def test_zero_residual_cache_has_zero_bound():
    # keys that are exact multiples of their block scale: residual 0, c = 0, TV = 0
    B, Hq, Hkv, d = 1, 2, 1, 128
    m = DecodeOracle(B, Hq, Hkv, d, "contiguous", 64, 0, 0.0, "bf16", "int8")
    rng = np.random.default_rng(15)
    for t in range(32):
        c = rng.integers(-126, 127, (1, 1, d)).astype(np.float32)
        c[0, 0, 0] = 127.0                                   # amax = 127 * 2^-4 -> s = 2^-4
        k = c * np.float32(1.0 / 16)
        cv = rng.integers(-127, 128, (1, 1, d)).astype(np.float32)
        cv[0, 0, 1] = -127.0                                 # values exact on their grid too
        m.append(nm.f32_to_bf16(k), nm.f32_to_bf16(cv * np.float32(0.25)))
    res = m.decode_int8(nm.f32_to_bf16(rng.standard_normal((1, 2, d)).astype(np.float32)))
    for r in res.values():
        assert r["cmax"] == 0.0 and r["tv"] == 0.0
        assert np.array_equal(r["out"], r["out_exact"])


def test_int8_trim_rules():
    rng = np.random.default_rng(16)
    m = _int8_model(rng, T=40, outliers=False)               # blocks 0, 1 quantized; tail 32..39
    from oracle.model import OracleError
    with pytest.raises(OracleError):
        m.trim([20])                                          # would split quantized block 1
    m.trim([35])                                              # only tail rows go
    assert m.length(0) == 35
    m.trim([16])                                              # block boundary
    assert m.length(0) == 16


# ---- the window of the INT8 tier (max_t c_t over the window; [LEAN] §2.1 masks) ----------
def _hand_window(m, q_bits, t, lo, h_q):
    """Attention of query head h_q of request 0 over positions [lo, t] assembled by hand:
    complete blocks dequantized with the block quantizer, tail rows exact, plain fp64
    softmax; c_t from the witnesses and the query's band norms."""
    g = m.Hq // m.Hkv
    h = h_q // g
    nfull = (m.length(0) // QBLOCK) * QBLOCK
    qf = m.query_rows(np.asarray(q_bits)[0, h_q:h_q + 1], np.full(1, t))[0].astype(np.float64)
    K, V, C = [], [], []
    qn = np.sqrt((qf.reshape(NBANDS, -1) ** 2).sum(axis=1))
    for p in range(lo, t + 1):
        if p < nfull:
            b0 = (p // QBLOCK) * QBLOCK
            Kb = np.stack([m.hk[0][x][h] for x in range(b0, b0 + QBLOCK)])
            Vb = np.stack([m.hv[0][x][h] for x in range(b0, b0 + QBLOCK)])
            sK, cK = nm.quantize_block(Kb)
            sV, cV = nm.quantize_block(Vb)
            r = p - b0
            K.append(cK[r].astype(np.float64) * np.float64(sK))
            V.append(cV[r].astype(np.float64) * np.float64(sV))
            w = nm.f16_values(nm.witness_row(Kb[r], cK[r], sK, NBANDS)).astype(np.float64)
            C.append((w * qn).sum() / math.sqrt(m.d))
        else:
            K.append(m.hk[0][p][h].astype(np.float64))
            V.append(m.hv[0][p][h].astype(np.float64))
            C.append(0.0)
    K, V = np.stack(K), np.stack(V)
    s = K @ qf / math.sqrt(m.d)
    e = np.exp(s - s.max())
    return (e @ V) / e.sum(), np.array(C)


@pytest.mark.parametrize("window,T", [(20, 70), (16, 64), (5, 70), (40, 37)])
def test_windowed_decode_by_hand(window, T):
    # the window starts inside a block, on a block boundary, inside the exact tail, and
    # before position 0 (all rows visible)
    rng = np.random.default_rng(40 + window)
    m = _int8_model(rng, T=T, outliers=True, window=window)
    q = nm.f32_to_bf16(rng.standard_normal((1, 4, 128)).astype(np.float32))
    res = m.decode_int8(q)
    t = T - 1
    lo = max(0, t - window + 1)
    for (b, hq), r in res.items():
        out, c = _hand_window(m, q, t, lo, hq)
        assert np.allclose(r["out"], out, rtol=1e-12, atol=1e-12)
        assert np.allclose(r["c"], c, rtol=1e-12, atol=0) and r["c"].shape == (t + 1 - lo,)
        assert r["cmax"] == pytest.approx(c.max(), rel=1e-12)
        assert np.all(r["eps"] <= r["c"] * (1 + 1e-12)) and r["tv"] <= math.tanh(r["cmax"])


def test_window_reductions():
    rng = np.random.default_rng(50)
    full = _int8_model(rng, T=70, window=0)
    rng = np.random.default_rng(50)
    wide = _int8_model(rng, T=70, window=1000)
    rng = np.random.default_rng(50)
    one = _int8_model(rng, T=70, window=1)
    q = nm.f32_to_bf16(np.random.default_rng(51).standard_normal((1, 4, 128)).astype(np.float32))
    a, b, c = full.decode_int8(q), wide.decode_int8(q), one.decode_int8(q)
    for key in a:
        # a window covering every position is the unwindowed tier
        assert np.array_equal(a[key]["out"], b[key]["out"]) and a[key]["cmax"] == b[key]["cmax"]
        # one visible key (position 69, in the exact tail): its value row, exactly; no bound
        h = key[1] // 2
        assert np.array_equal(c[key]["out"], one.hv[0][69][h].astype(np.float64))
        assert c[key]["cmax"] == 0.0 and c[key]["tv"] == 0.0


def test_window_max_ignores_tokens_before_the_window():
    # a token with a large residual just before the window start raises the unwindowed
    # bound but not the windowed one
    B, Hq, Hkv, d = 1, 2, 1, 128
    rng = np.random.default_rng(52)
    rows = [rng.standard_normal((1, 1, d)).astype(np.float32) for _ in range(48)]
    rows[10][0, 0, 3] = 3000.0                       # block 0: huge scale, large residuals elsewhere
    def build(window):
        m = DecodeOracle(B, Hq, Hkv, d, "contiguous", 64, window, 0.0, "bf16", "int8")
        for k in rows:
            m.append(nm.f32_to_bf16(k), nm.f32_to_bf16(k))
        return m
    q = nm.f32_to_bf16(np.ones((1, 2, d), np.float32))
    allw = build(0).decode_int8(q)
    win = build(30).decode_int8(q)                   # positions 18..47: blocks 1 and 2 only
    for key in allw:
        assert win[key]["cmax"] < allw[key]["cmax"] / 10


def test_ring_int8_equals_windowed_contiguous():
    # a ring of W slots attends to the same window as a contiguous cache with window W
    W, T = 32, 90
    rng = np.random.default_rng(53)
    ring = DecodeOracle(1, 4, 2, 128, "ring", W, 0, 10000.0, "bf16", "int8")
    cont = DecodeOracle(1, 4, 2, 128, "contiguous", 256, W, 10000.0, "bf16", "int8")
    for t in range(T):
        k = nm.f32_to_bf16(rng.standard_normal((1, 2, 128)).astype(np.float32))
        v = nm.f32_to_bf16(rng.standard_normal((1, 2, 128)).astype(np.float32))
        ring.append(k, v)
        cont.append(k, v)
        if t in (3, 31, 32, 47, 89):
            q = nm.f32_to_bf16(rng.standard_normal((1, 4, 128)).astype(np.float32))
            a, b = ring.decode_int8(q), cont.decode_int8(q)
            for key in a:
                assert np.array_equal(a[key]["out"], b[key]["out"]) and np.array_equal(a[key]["c"], b[key]["c"])
