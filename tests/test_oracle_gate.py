"""Pins of the oracle's gated fallback (CPU only).

[WITCERT] "WitCert: Sound Runtime Risk Observability and Gating for KV-Cache Quantization"
  "SGLang 生产级落地与闭环门控修复": once a head's or block's risk crosses the water line,
      the lossless block is swapped in from the full-precision backing store and its
      witness is zeroed; in the saturated zone blocks are ranked by risk and truncated.
  "为什么在线监控 KV 误差如此困难？": TV <= tanh(max |eps|); tau = 0.2 as the usual threshold.
"""
import math

import numpy as np
import pytest

from oracle import numerics as nm
from oracle.model import QBLOCK, DecodeOracle, block_risk, gate_select


def _risks(rng, B=3, H=2, nblk=7):
    # a mix of blocks below, at and above atanh(0.2) = 0.2027, with repeated values for ties
    pool = np.array([0.01, 0.1, 0.2, math.atanh(0.2), 0.21, 0.5, 0.5, 1.3, 4.0])
    return {(b, h): rng.choice(pool, nblk) for b in range(B) for h in range(H)}


@pytest.mark.parametrize("seed", range(6))
def test_gate_selection_invariants(seed):
    rng = np.random.default_rng(seed)
    risk = _risks(rng)
    tau = 0.2
    qualifying = {(b, h, k) for (b, h), r in risk.items() for k, x in enumerate(r) if math.tanh(x) > tau}
    full = gate_select(risk, tau)
    assert set(full) == qualifying and len(full) == len(qualifying)      # every qualifying block, once
    vals = [risk[(b, h)][k] for b, h, k in full]
    assert vals == sorted(vals, reverse=True)                              # highest risk first
    for i in range(len(full) - 1):                                         # ties: smaller index first
        if vals[i] == vals[i + 1]:
            assert full[i] < full[i + 1]
    # atanh(0.2) itself does not qualify: tanh(x) > tau is strict
    assert all(math.tanh(risk[(b, h)][k]) > tau for b, h, k in full)
    for budget in (0, 1, 3, len(full) + 5):
        part = gate_select(risk, tau, budget)
        assert part == full[:budget]                                       # truncation of the ranking
        if part and len(part) < len(full):
            worst = min(risk[(b, h)][k] for b, h, k in part)
            assert all(risk[(b, h)][k] <= worst for b, h, k in full[len(part):])


def test_block_risk_is_the_block_maximum_over_group_heads():
    rng = np.random.default_rng(3)
    c = rng.random((4, 70))
    r = block_risk(c, 64)
    assert r.shape == (4,)                                               # only complete blocks
    for blk in range(4):
        assert r[blk] == max(c[h, t] for h in range(4) for t in range(16 * blk, 16 * blk + 16))


def _int8_model(seed=13, n=200, tau_outliers=20.0):
    from kv_cache_decode_ring_gb300 import workloads as wl
    w = wl.small("gate", B=2, Hq=8, Hkv=2, d=128, capacity=256, rope_base=10000.0, quant="int8",
                 seed=seed, outliers=(4, tau_outliers))
    m = DecodeOracle(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, "contiguous", w.capacity, 0,
                     w.rope_base, "bf16", "int8")
    k, v = w.prefill_chunk(0, n)
    m.append_rows(wl.as_numpy(k), wl.as_numpy(v), [n, n - 37])
    q = wl.as_numpy(w.step_qkv(0)[0])
    return w, m, q


def _risk_of(m, res):
    risk = {}
    for b in range(m.B):
        nfull = m.length(b) // QBLOCK * QBLOCK
        for h in range(m.Hkv):
            c = np.stack([res[(b, hq)]["c"] for hq in range(h * m.g, (h + 1) * m.g)])
            risk[(b, h)] = block_risk(c, nfull)
    return risk


def test_restoring_the_gated_blocks_brings_every_head_under_tau():
    w, m, q = _int8_model()
    res = m.decode_int8(q)
    tau = 0.2
    assert max(math.tanh(r["cmax"]) for r in res.values()) > tau    # the outliers make it risky
    sel = gate_select(_risk_of(m, res), tau)
    assert sel
    m.restore(sel)
    after = m.decode_int8(q)
    for (b, hq), r in after.items():
        assert math.tanh(r["cmax"]) <= tau, (b, hq)
        assert r["tv"] <= math.tanh(r["cmax"]) + 1e-15               # the bound still holds
        assert np.all(r["eps"] <= r["c"] * (1 + 1e-12) + 1e-300)
        h = hq // m.g
        for blk in m.restored[b][h]:                                  # restored tokens: exact
            sl = slice(blk * QBLOCK, (blk + 1) * QBLOCK)
            assert np.all(r["c"][sl] == 0.0) and np.all(r["eps"][sl] == 0.0)
    # outputs move toward exact attention: every head's error to the exact output does not grow
    for key in res:
        e0 = np.abs(res[key]["out"] - res[key]["out_exact"]).max()
        e1 = np.abs(after[key]["out"] - after[key]["out_exact"]).max()
        assert e1 <= e0 + 1e-12


def test_restored_block_equals_exact_rows_in_the_attention():
    w, m, q = _int8_model(seed=5, n=96)
    m.restore([(0, 1, 2), (1, 0, 0)])
    res = m.decode_int8(q, heads=[(0, 4), (1, 0)])
    for (b, hq), r in res.items():
        h = hq // m.g
        t = m.length(b) - 1
        K = np.stack([m.hk[b][p][h] for p in range(t + 1)]).astype(np.float64)
        V = np.stack([m.hv[b][p][h] for p in range(t + 1)]).astype(np.float64)
        nfull = m.length(b) // QBLOCK * QBLOCK
        for blk in range(nfull // QBLOCK):                           # dequantize the others by hand
            if blk in m.restored[b][h]:
                continue
            sl = slice(blk * QBLOCK, (blk + 1) * QBLOCK)
            sK, cK = nm.quantize_block(K[sl].astype(np.float32))
            sV, cV = nm.quantize_block(V[sl].astype(np.float32))
            K[sl] = cK * np.float64(sK)
            V[sl] = cV * np.float64(sV)
        qf = r["q"].astype(np.float64)
        lg = K @ qf / math.sqrt(m.d)
        p = np.exp(lg - lg.max())
        ref = (p[:, None] * V).sum(0) / p.sum()
        assert np.allclose(r["out"], ref, rtol=1e-12, atol=1e-12)


def test_restore_nothing_is_identity_and_trim_drops_restored_blocks():
    w, m, q = _int8_model(seed=9, n=130)
    before = m.decode_int8(q)
    m.restore([])
    same = m.decode_int8(q)
    for key in before:
        assert np.array_equal(before[key]["out"], same[key]["out"])
    m.restore([(0, 0, 1), (0, 0, 6), (1, 1, 3)])
    m.trim([96, 64])
    assert m.restored[0][0] == {1} and m.restored[1][1] == {3}
    with pytest.raises(Exception):
        m.restore([(1, 0, 4)])                                        # block 4 of request 1 is gone
