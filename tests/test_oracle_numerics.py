"""Pins of the oracle's number formats, RoPE and masked attention (CPU only).

Each check compares the oracle with something other than itself: a library
routine (torch/numpy rounding, torch SDPA), high-precision math (mpmath),
closed forms, or invariants the pages state.

[LEAN]    "用Lean4形式化验证滑动窗口KV Cache的正确性" (framerc.cn/news/4505248)
[LOOP]    "KV Cache 自回归生成推理（增量更新与状态拼接）" (airsota.com/?p=549)
[WITCERT] "WitCert: Sound Runtime Risk Observability and Gating for KV-Cache Quantization"
"""
import math

import numpy as np
import pytest
import torch

from oracle import numerics as nm

mpmath = pytest.importorskip("mpmath")


# ------------------------------------------------------------------ bf16 / fp16

def _special_f32():
    rng = np.random.default_rng(1)
    a = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    u = a.view(np.uint32)
    ties = ((u & 0xFFFF0000) | 0x8000).view(np.float32)            # exact halfway cases
    near = ((u & 0xFFFF0000) | 0x7FFF).view(np.float32)
    sub = np.array([1e-40, -1e-40, 1.1754942e-38, 0.0, -0.0], dtype=np.float32)
    big = np.array([3.3895314e38, 3.4028235e38, -3.4028235e38, np.inf, -np.inf], dtype=np.float32)
    return np.concatenate([a, ties, near, sub, big])


def test_bf16_rounding_matches_torch():
    x = _special_f32()
    ours = nm.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # widening back is exact
    assert np.array_equal(nm.bf16_to_f32(ours), torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_bf16_nan_stays_nan():
    assert np.isnan(nm.bf16_to_f32(nm.f32_to_bf16(np.array([np.nan], np.float32))))[0]


def _f16_up_numpy(x):
    """Smallest fp16 >= x by numpy: nearest fp16, stepped up once if it fell below x."""
    h = np.float16(np.float32(x))
    if float(h) < float(np.float32(x)):
        h = np.nextafter(h, np.float16(np.inf))
    return int(np.array(h, dtype=np.float16).view(np.uint16))


def test_f16_round_up_matches_numpy_rule():
    rng = np.random.default_rng(2)
    xs = list(rng.exponential(1.0, 3000).astype(np.float32)) + list(rng.uniform(0, 70000, 500).astype(np.float32))
    xs += [0.0, 1e-9, 5.96e-8, 6e-8, 6.1e-5, 65504.0, 65504.01, 65519.0, 65520.0, 1e6]
    for x in xs:
        assert nm.f32_to_f16_up(x) == _f16_up_numpy(x), x


def test_f16_values_are_fixed_points_and_next_up():
    for bits in range(0, 0x7C00, 7):
        v = np.array(bits, dtype=np.uint16).view(np.float16)
        assert nm.f32_to_f16_up(float(v)) == bits
        assert nm.f16_value(bits) == float(v)
        above = np.nextafter(np.float32(v), np.float32(np.inf))
        if bits < 0x7BFF:
            assert nm.f32_to_f16_up(float(above)) == bits + 1


# ------------------------------------------------------------------ RoPE

@pytest.mark.parametrize("d,base", [(128, 10000.0), (64, 10000.0), (4, 10000.0), (128, 500000.0)])
def test_rope_table_is_rounded_exact_cos_sin(d, base):
    # cos/sin of the double angle p*theta_i, each rounded once to fp32.  theta_i and the angle
    # come from libm pow and one double multiply; mpmath evaluates cos/sin of that double
    # exactly enough to round; cases within 1e-25 of a rounding boundary are skipped.
    mpmath.mp.dps = 40
    rng = np.random.default_rng(3)
    positions = [0, 1, 2, 3, 4095, 4096, 8191, 32767, 131071] + list(rng.integers(0, 131088, 20))
    for p in positions:
        cs = nm.rope_cos_sin(base, d, int(p), 1)[0]
        for i in range(d // 2):
            theta = math.pow(base, (-2 * i) / d)
            exact_theta = mpmath.power(mpmath.mpf(base), mpmath.mpf(-2 * i) / d)
            assert abs(theta - float(exact_theta)) <= 2 * math.ulp(theta)
            ang = float(p) * theta
            for j, fn in ((0, mpmath.cos), (1, mpmath.sin)):
                ex = fn(mpmath.mpf(ang))
                f = np.float32(float(ex))
                lo = np.nextafter(f, np.float32(-np.inf))
                hi = np.nextafter(f, np.float32(np.inf))
                # correctly rounded unless ex is (almost) exactly halfway between neighbours
                halfway = min(abs(ex - (mpmath.mpf(float(f)) + mpmath.mpf(float(lo))) / 2),
                              abs(ex - (mpmath.mpf(float(f)) + mpmath.mpf(float(hi))) / 2))
                if halfway < mpmath.mpf(10) ** -25:
                    continue
                assert cs[i, j] == f, (p, i, j)


def test_rope_rotation_pins():
    rng = np.random.default_rng(4)
    d, base = 128, 10000.0
    x = rng.standard_normal((50, d)).astype(np.float32)
    pos = rng.integers(0, 40000, 50)
    y = nm.rope_rotate(x, pos, base)
    # (1) the fp32 formula evaluated independently with numpy float32 (one rounding per op)
    cs = np.stack([nm.rope_cos_sin(base, d, int(p), 1)[0] for p in pos])
    c, s = cs[..., 0], cs[..., 1]
    x0, x1 = x[:, 0::2], x[:, 1::2]
    ref = np.empty_like(x)
    ref[:, 0::2] = (x0 * c) - (x1 * s)
    ref[:, 1::2] = (x1 * c) + (x0 * s)
    assert ref.dtype == np.float32 and np.array_equal(y, ref)
    # (2) a rotation: close to the fp64 complex product with exact angles
    ang = pos[:, None].astype(np.float64) * (base ** (-(2.0 * np.arange(d // 2)) / d))[None, :]
    z = (x0.astype(np.float64) + 1j * x1.astype(np.float64)) * np.exp(1j * ang)
    assert np.allclose(y[:, 0::2], z.real, atol=2e-6, rtol=1e-5)
    assert np.allclose(y[:, 1::2], z.imag, atol=2e-6, rtol=1e-5)
    # (3) position 0 is the identity exactly
    assert np.array_equal(nm.rope_rotate(x, np.zeros(50, np.int64), base), x)
    # (4) each pair keeps its norm ([WITCERT] band unitarity), up to fp32 rounding
    n0 = x0.astype(np.float64) ** 2 + x1.astype(np.float64) ** 2
    n1 = y[:, 0::2].astype(np.float64) ** 2 + y[:, 1::2].astype(np.float64) ** 2
    assert np.allclose(n0, n1, rtol=1e-5, atol=1e-6)


def test_rope_dot_product_depends_on_relative_position():
    rng = np.random.default_rng(5)
    d, base = 64, 10000.0
    q = rng.standard_normal(d).astype(np.float32)
    k = rng.standard_normal(d).astype(np.float32)
    for (p, pk, shift) in [(10, 3, 100), (4000, 2, 7), (500, 499, 30000)]:
        a = nm.rope_rotate(q, [p], base).astype(np.float64) @ nm.rope_rotate(k, [pk], base).astype(np.float64)
        b = nm.rope_rotate(q, [p + shift], base).astype(np.float64) @ nm.rope_rotate(k, [pk + shift], base).astype(np.float64)
        assert abs(a - b) < 2e-3 * (1 + abs(a))


# ------------------------------------------------------------------ attention

def _sdpa(q, K, V, t, window, p0=0):
    """torch SDPA in fp64 with an explicit boolean mask (a library evaluation)."""
    n = K.shape[0]
    pos = p0 + torch.arange(n)
    mask = pos <= t
    if window > 0:
        mask &= pos >= t - window + 1
    o = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, None], torch.from_numpy(K)[None, None], torch.from_numpy(V)[None, None],
        attn_mask=mask[None, None, None, :])
    return o[0, 0].numpy()


@pytest.mark.parametrize("d", [4, 64, 128])
@pytest.mark.parametrize("window", [0, 1, 3, 16, 1000])
def test_attention_matches_sdpa(d, window):
    rng = np.random.default_rng(6 + d + window)
    for n in (1, 2, 17, 130):
        K = rng.standard_normal((n, d))
        V = rng.standard_normal((n, d))
        q = rng.standard_normal((3, d))
        for t in sorted({0, n // 2, n - 1}):
            out = nm.attend(q, K, V, t, window)
            ref = _sdpa(q, K, V, t, window)
            assert np.allclose(out, ref, atol=1e-12, rtol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(7)
    d = 8
    K = rng.standard_normal((20, d)).astype(np.float32)
    V = rng.standard_normal((20, d)).astype(np.float32)
    q = rng.standard_normal((1, d))
    # one visible key: the output is that value exactly
    assert np.array_equal(nm.attend(q, K, V, 0)[0], V[0].astype(np.float64))
    assert np.array_equal(nm.attend(q, K, V, 9, window=1)[0], V[9].astype(np.float64))
    # equal logits: the mean of the visible values
    Kc = np.tile(K[:1], (20, 1))
    assert np.allclose(nm.attend(q, Kc, V, 19, window=5)[0], V[15:20].astype(np.float64).mean(0), atol=1e-14)
    # a window at least as long as the history is full attention
    assert np.array_equal(nm.attend(q, K, V, 19, window=20), nm.attend(q, K, V, 19, window=0))
    # masked rows (future and outside the window) do not matter
    K2, V2 = K.copy(), V.copy()
    K2[15:] = 99.0; V2[15:] = -99.0; K2[:5] = 7.0; V2[:5] = 3.0
    assert np.array_equal(nm.attend(q, K, V, 14, window=10), nm.attend(q, K2, V2, 14, window=10))
    # order of the visible rows does not matter (up to rounding)
    perm = np.r_[np.arange(5), rng.permutation(np.arange(5, 15)), np.arange(15, 20)]
    assert np.allclose(nm.attend(q, K, V, 14, window=10), nm.attend(q, K[perm], V[perm], 14, window=10,), atol=1e-14)


def test_attention_kinds_agree():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((30, 16)).astype(np.float32)
    bits = nm.f32_to_bf16(x)
    xb = nm.bf16_to_f32(bits)
    q = rng.standard_normal((2, 16))
    a = nm.attend(q, bits, bits, 29)
    b = nm.attend(q, xb, xb, 29)
    c = nm.attend(q, xb.astype(np.float64), xb.astype(np.float64), 29)
    assert np.array_equal(a, b) and np.array_equal(b, c)


def test_ring_attention_equals_full_history_masked():
    # [LEAN] §4.2 corollary: attention over the ring's contents equals full-history attention
    # with the window mask, at every step through the three ring phases.
    from oracle.listmodel import Cell, RingBuffer
    rng = np.random.default_rng(9)
    W, d = 4, 4
    K = rng.standard_normal((40, d)); V = rng.standard_normal((40, d)); Q = rng.standard_normal((40, 1, d))
    ring = RingBuffer(W)
    for t in range(40):
        ring.push(Cell(t, K[t], V[t]))
        live = ring.as_list()
        Kr = np.stack([c.key for c in live]); Vr = np.stack([c.val for c in live])
        ring_out = nm.attend(Q[t], Kr, Vr, t, window=0, p0=live[0].pos)
        full_out = nm.attend(Q[t], K[:t + 1], V[:t + 1], t, window=W)
        assert np.allclose(ring_out, full_out, atol=1e-15)


def test_loop_unit_test_shapes():
    # [LOOP] §四: three steps, B=1, H=2, D=4, max_seq_len=10 -> out (1,2,1,4), current_len == 3.
    from oracle.model import DecodeOracle
    rng = np.random.default_rng(10)
    m = DecodeOracle(1, 2, 2, 4, "contiguous", 10)
    for t in range(3):
        q, k, v = (rng.standard_normal((1, 2, 4)).astype(np.float32) for _ in range(3))
        m.append(k, v)
        out = m.decode(q)
        assert out.reshape(1, 2, 1, 4).shape == (1, 2, 1, 4)
    assert m.length(0) == 3
