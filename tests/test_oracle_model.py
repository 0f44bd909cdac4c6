"""Pins of the whole decode-step oracle on the toy fp32 workload (CPU only).

Toy workload: B=1, H=2, head_dim=4, q/k/v ~ N(0,1) fp32 from seed 7, 64 decode
steps; a full cache (max_seq_len 64), a ring W=4, and a trim of an 8-token
history at cut=4 continued with 8 new tokens.

[LEAN]   "用Lean4形式化验证滑动窗口KV Cache的正确性" (framerc.cn/news/4505248)
[PREFIX] "LLM 機制實驗（五）：改了歷史，能否只重算變化的後綴？" (huhohoo.com)
[LOOP]   "KV Cache 自回归生成推理（增量更新与状态拼接）" (airsota.com/?p=549)
"""
import numpy as np
import pytest
import torch

from kv_cache_decode_ring_gb300 import workloads as wl
from oracle import numerics as nm
from oracle.listmodel import last_window, position_invariant
from oracle.model import DecodeOracle, OracleError

TOL_F32 = 1e-5


def _sdpa_step(q, K, V, t, window):
    """torch SDPA (fp64) of one query over rows 0..t with a window mask."""
    pos = torch.arange(K.shape[0])
    mask = pos <= t
    if window:
        mask &= pos >= t - window + 1
    o = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q.astype(np.float64))[None], torch.from_numpy(K.astype(np.float64))[None],
        torch.from_numpy(V.astype(np.float64))[None], attn_mask=mask[None, None, :])
    return o[0].numpy()


def _toy_inputs(w, steps=64):
    qs, ks, vs = [], [], []
    for s in range(steps):
        q, k, v = w.step_qkv(s)
        qs.append(q.numpy()); ks.append(k.numpy()); vs.append(v.numpy())
    return np.stack(qs), np.stack(ks), np.stack(vs)


@pytest.mark.parametrize("variant", ["full", "ring"])
def test_toy_decode_against_sdpa_and_cache_model(variant):
    w = wl.toy(variant)
    Q, Kin, Vin = _toy_inputs(w)
    m = DecodeOracle(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.layout, w.capacity, w.window,
                     w.rope_base, w.dtype)
    W = w.capacity if w.layout == "ring" else 0
    for t in range(64):
        m.append(Kin[t], Vin[t])
        out = m.decode(Q[t])
        for h in range(2):
            ref = _sdpa_step(Q[t, 0, h][None], Kin[:t + 1, 0, h], Vin[:t + 1, 0, h], t, W)
            assert np.allclose(out[0, h], ref[0], atol=1e-13)
        if t == 0:
            assert np.array_equal(out[0], Vin[0, 0].astype(np.float64))   # one key: v_0 exactly
        pos = m.expected_positions()[0]
        if variant == "full":
            assert np.array_equal(pos[:t + 1], np.arange(t + 1)) and np.all(pos[t + 1:] == -1)
        else:
            # slot s holds the newest position congruent to s mod W; empty while not full
            for s in range(4):
                want = max((p for p in range(t + 1) if p % 4 == s), default=-1)
                assert pos[s] == want
            window = m.logical_window(0)
            assert [c.pos for c in window] == [c.pos for c in last_window(4, list(m.logical_window(0)))]
            assert position_invariant(window) and window[0].pos == max(0, t - 3)
            ring = m.rings[0].as_list()
            assert [c.pos for c in ring] == [c.pos for c in window]
            assert all(np.array_equal(a.key, b.key) for a, b in zip(ring, window))


def _stale_outputs(hist_k, hist_v, cut, old_len, suf_q, suf_k, suf_v, base, window=0):
    """Planted mistake: K/V trimmed to ``cut`` rows but the suffix encoded from the OLD next
    position ([PREFIX] "哪些東西必須一起裁剪", negative control).  Rows keep their order; the
    suffix row i and query i are rotated at old_len + i instead of cut + i.
    Shapes: hist [cut, H, d], suffix [n, H, d] (one query head per KV head)."""
    rot = (lambda x, p: nm.rope_rotate(x, p, base)) if base else (lambda x, p: x)
    n, H = suf_q.shape[0], suf_q.shape[1]
    out = np.zeros((n, H, suf_q.shape[2]))
    for h in range(H):
        K = [rot(hist_k[j, h], [j]) for j in range(cut)]
        V = [hist_v[j, h] for j in range(cut)]
        for i in range(n):
            K.append(rot(suf_k[i, h], [old_len + i])); V.append(suf_v[i, h])
            q = rot(suf_q[i, h], [old_len + i]).astype(np.float64)
            out[i, h] = nm.attend(q[None], np.stack(K).astype(np.float64), np.stack(V).astype(np.float64),
                                  t=len(K) - 1, window=window)[0]
    return out


@pytest.mark.parametrize("rope_base", [0.0, 10000.0])
def test_toy_trim_continue_equals_recompute_and_stale_diverges(rope_base):
    w = wl.toy("trim")
    hist, cut, n = w.extra["history"], w.extra["cut"], w.extra["suffix"]
    Q, Kin, Vin = _toy_inputs(w, steps=hist + n)
    def model():
        return DecodeOracle(1, 2, 2, 4, "contiguous", 64, 0, rope_base, "f32")
    # trimmed: 8 history tokens, trim to cut, continue with n new tokens
    a = model()
    for t in range(hist):
        a.append(Kin[t], Vin[t])
    a.trim([cut])
    assert a.length(0) == cut and np.array_equal(a.expected_positions()[0][:cut], np.arange(cut))
    suf = slice(hist, hist + n)
    sq, sk, sv = (x[suf].transpose(1, 0, 2, 3) for x in (Q, Kin, Vin))   # [B, n, H, d]
    out_a = a.chunk(sq, sk, sv)
    # full recompute: the first cut history tokens, then the same suffix
    b = model()
    for t in range(cut):
        b.append(Kin[t], Vin[t])
    out_b = b.chunk(sq, sk, sv)
    assert np.array_equal(out_a, out_b)
    assert np.array_equal(a.expected_positions(), b.expected_positions())
    assert np.array_equal(a.expected_positions()[0][:cut + n], np.arange(cut + n))
    # negative control: keep the stale next_position (= 8)
    stale = _stale_outputs(Kin[:cut, 0], Vin[:cut, 0], cut, hist, Q[suf, 0], Kin[suf, 0], Vin[suf, 0], rope_base)
    stale_pos = np.r_[np.arange(cut), hist + np.arange(n)]
    assert not position_invariant([type("C", (), {"pos": int(p)})() for p in stale_pos])
    if rope_base:
        # positions enter the logits: the stale path must exceed the fp32 tolerance
        err = np.abs(stale - out_a[0]).max()
        assert err > 100 * TOL_F32, err
    else:
        # without RoPE the logits ignore positions; the divergence shows in the positions only
        assert np.allclose(stale, out_a[0], atol=1e-12)


def test_ring_trim_evicted_and_allowed():
    m = DecodeOracle(1, 2, 2, 4, "ring", 4, 4, 0.0, "f32")
    rng = np.random.default_rng(17)
    for t in range(10):
        m.append(rng.standard_normal((1, 2, 4)).astype(np.float32), rng.standard_normal((1, 2, 4)).astype(np.float32))
    with pytest.raises(OracleError) as e:
        m.trim([4])                       # [PREFIX]: rows 0..3 long gone from a W=4 ring
    assert e.value.code == "evicted"
    m.trim([9])                           # needs positions 6..8: resident
    assert m.expected_positions()[0].tolist() == [8, -1, 6, 7]
    m.append(rng.standard_normal((1, 2, 4)).astype(np.float32), rng.standard_normal((1, 2, 4)).astype(np.float32))
    assert m.expected_positions()[0].tolist() == [8, 9, 6, 7]
    assert [c.pos for c in m.rings[0].as_list()] == [6, 7, 8, 9]


def test_capacity_error():
    m = DecodeOracle(1, 2, 2, 4, "contiguous", 3)
    z = np.zeros((1, 2, 4), np.float32)
    for _ in range(3):
        m.append(z, z)
    with pytest.raises(OracleError) as e:
        m.append(z, z)                    # [LOOP] §三: assert pos < max_seq_len
    assert e.value.code == "capacity"


def test_bf16_rope_rows_and_gqa_grouping():
    rng = np.random.default_rng(18)
    m = DecodeOracle(1, 4, 2, 64, "contiguous", 16, 0, 10000.0, "bf16")
    ks = []
    for t in range(5):
        k = nm.f32_to_bf16(rng.standard_normal((1, 2, 64)).astype(np.float32))
        v = nm.f32_to_bf16(rng.standard_normal((1, 2, 64)).astype(np.float32))
        m.append(k, v); ks.append(k)
    rows = m.expected_rows(0, "k")
    for t in range(5):
        want = nm.bf16_to_f32(nm.f32_to_bf16(nm.rope_rotate(nm.bf16_to_f32(ks[t][0]), [t, t], 10000.0)))
        assert np.array_equal(rows[t], want)
    # query heads 0,1 read KV head 0; heads 2,3 read KV head 1
    q = nm.f32_to_bf16(rng.standard_normal((1, 4, 64)).astype(np.float32))
    out = m.decode(q)
    qr = m.query_rows(q[0], np.full(4, 4)).astype(np.float64)
    for h in range(4):
        K = np.stack([rows[t][h // 2] for t in range(5)])
        V = np.stack([m.hv[0][t][h // 2] for t in range(5)])
        assert np.allclose(out[0, h], _sdpa_step(qr[h][None], K, V, 4, 0)[0], atol=1e-13)
