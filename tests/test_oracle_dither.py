"""Pins of the oracle's Tier B: Philox dither streams and the subtractive-dither INT8
quantizer (CPU only).

[WITCERT] "WitCert: Sound Runtime Risk Observability and Gating for KV-Cache Quantization",
paragraph on Tier B (为了进一步压榨显存极限): a uniform pseudo-random dither is added at
write time and cancelled at read time from the same Philox stream; the residual is then
uniform and independent of the data.  "SGLang 生产级落地与闭环门控修复": the Philox counter
is the self-contained five-tuple (request, layer, KV head, token, channel), so the stream
does not depend on batch order.
"""
import math
import os

import numpy as np
import pytest

from oracle import numerics as nm
from oracle.model import QBLOCK, DecodeOracle, int8_decode_one

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _kat():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                ctr, key, out = [[int(x, 16) for x in part.split()] for part in line.split("|")]
                rows.append((ctr, key, out))
    return rows


@pytest.mark.parametrize("case", _kat())
def test_philox_known_answers(case):
    ctr, key, out = case
    assert [int(x) for x in nm.philox4x32_10(ctr, key)] == out


def test_dither_rows_state_the_mapping():
    key = (0x12345678, 0x9abcdef0)
    for d in (64, 128):
        rows = nm.dither_rows(key, 7, 3, 5, 1000, 6, d)
        for r in range(6):
            assert np.array_equal(rows[r], nm.dither_bytes(key, 7, 3, 5, 1000 + r, d))
    # byte i of the call for (token 42, group 1, KV head 5 of layer 3, request 7) is channel 16 + i
    w = nm.philox4x32_10([42, 1, 5 + 65536 * 3, 7], key).view(np.uint8)
    assert np.array_equal(nm.dither_bytes(key, 7, 3, 5, 42, 128)[16:32], w)


def test_dither_streams_are_distinct_and_uniform():
    key = (1, 2)
    base = nm.dither_rows(key, 0, 0, 0, 0, 64, 128)
    # every field of the five-tuple (and the key) selects another stream
    for other in (nm.dither_rows(key, 1, 0, 0, 0, 64, 128), nm.dither_rows(key, 0, 1, 0, 0, 64, 128),
                  nm.dither_rows(key, 0, 0, 1, 0, 64, 128), nm.dither_rows(key, 0, 0, 0, 1, 64, 128),
                  nm.dither_rows((1, 3), 0, 0, 0, 0, 64, 128)):
        assert (other != base).mean() > 0.99 - 1 / 256 - 0.01
    big = nm.dither_rows(key, 9, 0, 2, 0, 2048, 128).reshape(-1)           # 262144 bytes
    hist = np.bincount(big, minlength=256)
    chi2 = ((hist - big.size / 256) ** 2 / (big.size / 256)).sum()
    assert chi2 < 255 + 6 * math.sqrt(2 * 255)                              # about 6 sigma
    u = nm.dither_values(big)
    assert u.min() == -0.5 and u.max() == 0.5 - 1 / 256


def test_zero_dither_is_the_plain_quantizer():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((16, 128)) * 3).astype(np.float32)
    s0, c0 = nm.quantize_block(x)
    s1, c1 = nm.quantize_block_dither(x, np.zeros_like(x))
    assert s0 == s1 and np.array_equal(c0, c1)
    s2, c2 = nm.quantize_block_dither(np.zeros_like(x), nm.dither_values(rng.integers(0, 256, x.shape)))
    assert s2 == 0 and not c2.any()


def test_subtractive_dither_error_is_bounded_uniform_and_data_independent():
    """Reconstruction x_hat = (code - u) s: |x_hat - x| <= s/2, and over many dithers the
    error is uniform on one step (mean 0, variance s^2/12) whatever the data's offset from
    the grid; without subtracting u the variance would depend on that offset."""
    rng = np.random.default_rng(7)
    key = (3, 4)
    for frac in (0.0, 0.1, 0.3, 0.5):
        errs, errs_nosub = [], []
        for blk in range(48):
            k = rng.integers(-100, 100, (16, 128)).astype(np.float32)
            k[0, 0] = 127.0                                   # amax = 127 s with s = 1/8
            x = ((k + np.float32(frac)) / np.float32(8.0)).astype(np.float32)
            x[0, 0] = np.float32(127.0 / 8.0)
            u = nm.dither_values(nm.dither_rows(key, blk, 0, 0, 16 * blk, 16, 128))
            s, c = nm.quantize_block_dither(x, u)
            assert s == np.float32(127.0 / 8.0) / np.float32(127.0)
            xh = (c.astype(np.float64) - u.astype(np.float64)) * np.float64(s)
            e = (xh - x.astype(np.float64)) / np.float64(s)
            assert np.abs(e).max() <= 0.5 + 1e-5
            errs.append(e.reshape(-1)[1:])
            errs_nosub.append(((c.astype(np.float64) * np.float64(s) - x) / np.float64(s)).reshape(-1)[1:])
        e = np.concatenate(errs)
        assert abs(e.mean()) < 0.01 and abs(e.var() - 1 / 12) < 0.005, (frac, e.mean(), e.var())
        n = np.concatenate(errs_nosub)
        want = frac * (1 - frac)            # non-subtractive: rint(f + u) - f is 1 - f or -f
        assert abs(n.var() - want) < 0.01, (frac, n.var())


def test_tier_b_decode_is_attention_over_dequantized_rows():
    rng = np.random.default_rng(5)
    d, n = 128, 70
    K = (rng.standard_normal((n, d)) * 2).astype(np.float32)
    V = rng.standard_normal((n, d)).astype(np.float32)
    q = rng.standard_normal(d).astype(np.float32)
    key, rid, layer, h = (11, 12), 4, 2, 1

    def u(p0, m):
        return nm.dither_values(nm.dither_rows(key, rid, layer, h, p0, m, d))
    res = int8_decode_one(q, K, V, 0, n - 1, 0, (n // QBLOCK) * QBLOCK, (), u)
    Kd, Vd = K.astype(np.float64).copy(), V.astype(np.float64).copy()
    for blk in range(n // QBLOCK):
        sl = slice(blk * QBLOCK, (blk + 1) * QBLOCK)
        sK, cK = nm.quantize_block_dither(K[sl], u(blk * QBLOCK, QBLOCK))
        sV, cV = nm.quantize_block(V[sl])                  # values: the plain quantizer
        Kd[sl] = (cK - u(blk * QBLOCK, QBLOCK).astype(np.float64)) * float(sK)
        Vd[sl] = cV * float(sV)
    lg = Kd @ q.astype(np.float64) / math.sqrt(d)
    p = np.exp(lg - lg.max())
    assert np.allclose(res["out"], (p[:, None] * Vd).sum(0) / p.sum(), rtol=1e-12, atol=1e-12)
    assert res["c"] is None and res["tv"] < 0.05
    # the model draws the same streams from its key, layer and request IDs
    m = DecodeOracle(1, 1, 1, d, "contiguous", 128, 0, 0.0, "bf16", "int8-dither", dither_key=key, layer=layer)
    m.set_request_id(0, rid)
    assert m.request_ids[0] == rid
    m.append(np.zeros((1, 1, d), np.uint16), np.zeros((1, 1, d), np.uint16))
    with pytest.raises(Exception):
        m.set_request_id(0, rid + 1)                     # the stored codes depend on the ID
