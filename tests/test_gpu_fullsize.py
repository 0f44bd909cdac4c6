"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

The bf16 decodes are checked at every (request, head) of their checked steps; the
INT8 and chunk workloads, whose oracle is slower, at sampled heads.  References are
fp64 attention over the generator's own rows (never the GPU cache), plus closed-form
checks of positions that hold at any size.

Full-cache MHA decode: B=32, H=32, d=128, contiguous 8192, context 4096 + 128 steps;
contiguous rows, or 16-slot pages behind a block table (as the paged bench lines).
Sliding-window GQA decode: B=64, Hq=32, Hkv=8, d=128, ring W=4096, RoPE 10000,
per-request lengths L_b uniform in [1, 32768]; and one request run from
position 0 to 32767 through the not-full, exactly-full and first-replacement steps.
INT8 with witnesses (before and after one gated fallback), and Tier B: B=8, Hq=32,
Hkv=8, d=128, context 131072 + 16 steps.
"""
import numpy as np
import pytest
import torch

from kv_cache_decode_ring_gb300 import kvc
from kv_cache_decode_ring_gb300 import workloads as wl
from oracle import numerics as nm

from _parity import assert_close, host, oracle_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_decode_ring_gb300 import build
    build.build()


def _rows(model, x_np, positions):
    return model.stored_rows(x_np, positions).astype(np.float64)


def _threads():
    import os
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


@pytest.mark.parametrize("paged", [False, True], ids=["contiguous", "paged"])
def test_full_cache_mha_every_head(paged):
    # every (request, head) of the checked steps against fp64 attention (no RoPE: the cache
    # rows are the generator's bf16 values, kept on the host as bit patterns)
    w = wl.full_cache_mha()
    ctx = w.extra["context"]
    B, H, d = w.batch, w.n_q_heads, w.head_dim
    # paged: exactly the 16-slot pages the 128 steps need, as many as the bench's pool per step
    cache = kvc.Cache.from_workload(w, page_pool=B * -(-(ctx + 128) // 16) if paged else 0)
    k, v = w.prefill_chunk(0, ctx, device="cuda")
    cache.append_rows(k, v)
    hK = np.empty((B, H, ctx + 128, d), dtype=np.uint16)
    hV = np.empty_like(hK)
    hK[:, :, :ctx] = host(k)
    hV[:, :, :ctx] = host(v)
    del k, v
    check_at = {0, 1, 63, 127}
    for s in range(128):
        q, k1, v1 = w.step_qkv(s, device="cuda")
        cache.append(k1, v1)
        out = cache.decode(q)
        hK[:, :, ctx + s] = host(k1)
        hV[:, :, ctx + s] = host(v1)
        if s not in check_at:
            continue
        t = ctx + s
        qf = nm.bf16_to_f32(host(q)).astype(np.float64)                 # [B, H, d]
        probs = [(b, h) for b in range(B) for h in range(H)]
        ref = nm.attend_many([qf[b, h][None] for b, h in probs], [hK[b, h, :t + 1] for b, h in probs],
                             [hV[b, h, :t + 1] for b, h in probs], [t] * len(probs), 0, None,
                             nthreads=_threads())
        ref = np.stack(ref).reshape(B, H, d)
        assert_close(out.cpu(), ref, "bf16", "full-cache step %d, every (request, head)" % s)
    # positions after 128 steps: slot p holds p for p < ctx + 128 (closed form, every request)
    pos = cache.export(kvc.KVC_EXPORT_POSITIONS)
    want = np.where(np.arange(w.capacity) < ctx + 128, np.arange(w.capacity), -1)
    assert np.array_equal(pos, np.broadcast_to(want, pos.shape))
    assert cache.device_status() == 0


def _ring_positions_ok(pos_row, length, W):
    """Slot s holds the largest p < length with p = s mod W (or -1)."""
    s = np.arange(W)
    last = length - 1
    want = last - ((last - s) % W)
    want = np.where(want >= 0, want, -1)
    return np.array_equal(pos_row, want)


@pytest.mark.parametrize("paged", [False, True], ids=["ring", "paged-ring"])
def test_sliding_window_gqa_every_head(paged):
    # every request and every query head at the decode step, against fp64 attention over the
    # window rows as the oracle stores them (rotated at their positions, rounded to bf16)
    w = wl.sliding_window_gqa()
    W, Lmax = w.capacity, w.extra["max_len"]
    B, Hq, Hkv, d = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
    lengths = w.extra["lengths"]                   # current token at L_b - 1
    cache = kvc.Cache.from_workload(w, max_position=Lmax, page_pool=B * (W // 16) if paged else 0)
    model = oracle_for(w)
    # the generator's rows of every request's window (bf16 bit patterns, [Hkv, n, d])
    keep_k, keep_v = [[] for _ in range(B)], [[] for _ in range(B)]
    chunk = 4096
    for c in range((Lmax + chunk - 1) // chunk):
        counts = [int(min(max(L - 1 - c * chunk, 0), chunk)) for L in lengths]
        if not any(counts):
            continue
        k, v = w.prefill_chunk(c, chunk, device="cuda")
        cache.append_rows(k, v, counts=counts)
        hk, hv = host(k), host(v)
        for b in range(B):
            lo = max(0, lengths[b] - W) - c * chunk   # first window row inside this chunk
            a_, z_ = max(0, lo), counts[b]
            if z_ > a_:
                keep_k[b].append(hk[b, :, a_:z_])
                keep_v[b].append(hv[b, :, a_:z_])
        del k, v, hk, hv
    q, k1, v1 = w.step_qkv(0, device="cuda")
    cache.append(k1, v1)
    out = cache.decode(q).cpu()                 # bf16: its own rounding allowed
    g = Hq // Hkv
    pos = cache.export(kvc.KVC_EXPORT_POSITIONS)
    for b in range(B):
        assert _ring_positions_ok(pos[b], lengths[b], W), b
    hq, hk1, hv1 = host(q), host(k1), host(v1)
    ref = np.empty((B, Hq, d))
    for b in range(B):
        t = lengths[b] - 1
        lo = max(0, t - W + 1)
        Kin = np.concatenate(keep_k[b] + [hk1[b][:, None]], axis=1)       # [Hkv, n, d]
        Vin = np.concatenate(keep_v[b] + [hv1[b][:, None]], axis=1)
        assert Kin.shape[1] == t + 1 - lo
        K = _rows(model, Kin, np.broadcast_to(np.arange(lo, t + 1), Kin.shape[:2]))
        V = nm.bf16_to_f32(Vin).astype(np.float64)
        qr = model.query_rows(hq[b], np.full(Hq, t)).astype(np.float64)   # [Hq, d]
        r = nm.attend_many([qr[h * g:(h + 1) * g] for h in range(Hkv)], [K[h] for h in range(Hkv)],
                           [V[h] for h in range(Hkv)], [t] * Hkv, W, [lo] * Hkv, nthreads=_threads())
        ref[b] = np.concatenate(r)
        keep_k[b] = keep_v[b] = None
    assert_close(out, ref, "bf16", "sliding window, every (request, head)")
    assert cache.device_status() == 0


def test_one_request_through_the_ring_phases():
    base = wl.sliding_window_gqa()
    W = base.capacity
    w = wl.small("ring-long", B=1, Hq=32, Hkv=8, d=128, layout="ring", capacity=W, window=W,
                 rope_base=10000.0, seed=29)
    cache = kvc.Cache.from_workload(w, max_position=32768)
    model = oracle_for(w)
    check = {0, W - 2, W - 1, W, W + 1, 2 * W, 32767}
    hist_k, hist_v = [], []
    for t in range(32768):
        q, k1, v1 = w.step_qkv(t, device="cuda")
        cache.append(k1, v1)
        hist_k.append(host(k1[0])); hist_v.append(host(v1[0]))
        if t not in check:
            continue
        out = cache.decode(q).cpu()
        lo = max(0, t - W + 1)
        for h in (0, 5):
            Kin = np.stack([x[h] for x in hist_k[lo:t + 1]])
            K = _rows(model, Kin, np.arange(lo, t + 1))
            V = nm.bf16_to_f32(np.stack([x[h] for x in hist_v[lo:t + 1]])).astype(np.float64)
            qr = model.query_rows(host(q[0, h * 4:(h + 1) * 4]), np.full(4, t)).astype(np.float64)
            ref = nm.attend(qr, K, V, t, W, p0=lo)
            assert_close(out[0, h * 4:(h + 1) * 4], ref, "bf16", "ring t=%d h=%d" % (t, h))
        pos = cache.export(kvc.KVC_EXPORT_POSITIONS)[0]
        assert _ring_positions_ok(pos, t + 1, W), t
    assert cache.device_status() == 0


def test_int8_witness_sampled():
    # INT8 KV with witnesses: B=8, Hq=32, Hkv=8, d=128, context 131072 prefilled through the
    # block quantizer, then 16 one-token steps (the last completes a block)
    import math
    from oracle.model import QBLOCK, int8_decode_one
    w = wl.int8_witness()
    ctx = w.extra["context"]
    cache = kvc.Cache.from_workload(w)
    model = oracle_for(w)
    g = w.n_q_heads // w.n_kv_heads
    sample = [(0, 0), (5, 6)]
    keep = {bh: ([], []) for bh in sample}
    chunk = 8192
    for c in range(ctx // chunk):
        k, v = w.prefill_chunk(c, chunk, device="cuda")
        cache.append_rows(k, v)
        for (b, h) in sample:
            keep[(b, h)][0].append(host(k[b, h])); keep[(b, h)][1].append(host(v[b, h]))
        del k, v
    cmax = torch.empty((w.batch, w.n_q_heads), device="cuda")
    th = torch.empty((w.batch, w.n_q_heads), device="cuda")
    for s in range(16):
        q, k1, v1 = w.step_qkv(s, device="cuda")
        cache.append(k1, v1)
        out = cache.decode(q, None, cmax, th)
        for (b, h) in sample:
            keep[(b, h)][0].append(host(k1[b, h])[None]); keep[(b, h)][1].append(host(v1[b, h])[None])
        if s not in (0, 15):
            continue
        t = ctx + s
        nfull = (t + 1) // QBLOCK * QBLOCK
        o, cm, tc = out.cpu(), cmax.cpu().numpy(), th.cpu().numpy()       # o in bf16: its own rounding allowed
        for (b, h) in sample:
            Kin = np.concatenate(keep[(b, h)][0]); Vin = np.concatenate(keep[(b, h)][1])
            K = model.stored_rows(Kin, np.arange(t + 1))
            V = nm.bf16_to_f32(Vin)
            for hq in (h * g, h * g + g - 1):
                qr = model.query_rows(host(q[b, hq])[None], [t])[0]
                r = int8_decode_one(qr, K, V, 0, t, 0, nfull)
                assert_close(o[b, hq][None], r["out"][None], "bf16", "int8 full s=%d b=%d h=%d" % (s, b, hq))
                assert cm[b, hq] >= r["cmax"] * (1 - 1e-12) and cm[b, hq] <= r["cmax"] * (1 + 1e-5)
                assert tc[b, hq] >= math.tanh(cm[b, hq]) * (1 - 1e-7) and r["tv"] <= tc[b, hq]
                assert np.all(r["eps"] <= r["c"] * (1 + 1e-12))
    # a sample of blocks bit-exact: codes, scales, witnesses
    from oracle import numerics as onm
    KQ = cache.export(kvc.KVC_EXPORT_KQ); SK = cache.export(kvc.KVC_EXPORT_SK)
    WT = cache.export(kvc.KVC_EXPORT_WITNESS)
    for (b, h) in sample:
        Kin = np.concatenate(keep[(b, h)][0])
        n = Kin.shape[0]
        for blk in (0, 1, 4095, 8191, n // QBLOCK - 1):
            pos = np.arange(blk * QBLOCK, (blk + 1) * QBLOCK)
            Kb = model.stored_rows(Kin[pos], pos)
            sK, cK = onm.quantize_block(Kb)
            assert SK[b, h, blk] == sK and np.array_equal(KQ[b, h, pos], cK), (b, h, blk)
            wit = np.stack([onm.witness_row(Kb[i], cK[i], sK) for i in range(QBLOCK)])
            assert np.array_equal(WT[b, h, pos], wit), (b, h, blk)
    assert cache.device_status() == 0


def test_int8_witness_ring_sampled():
    # INT8 + witness on a ring of 32768 slots at the INT8 workload's shape (the bench's
    # int8-witness-ring line): 131072 positions streamed through the ring, then 16 steps;
    # sampled heads against the oracle over the window, and a sample of ring block slots
    # bit-exact (block n in slot n mod 2048)
    import math
    from oracle.model import QBLOCK, int8_decode_one
    w = wl.int8_witness_ring()
    ctx, W = w.extra["context"], w.capacity
    cache = kvc.Cache.from_workload(w, max_position=ctx + 64)
    model = oracle_for(w)
    g = w.n_q_heads // w.n_kv_heads
    sample = [(0, 0), (6, 5)]
    keep = {bh: ([], []) for bh in sample}          # rows from position ctx - W - 16 on
    chunk, first = 8192, ctx - W - 16
    for c in range(ctx // chunk):
        k, v = w.prefill_chunk(c, chunk, device="cuda")
        cache.append_rows(k, v)
        a_ = max(0, first - c * chunk)
        if a_ < chunk:
            for (b, h) in sample:
                keep[(b, h)][0].append(host(k[b, h, a_:])); keep[(b, h)][1].append(host(v[b, h, a_:]))
        del k, v
    cmax = torch.empty((w.batch, w.n_q_heads), device="cuda")
    th = torch.empty((w.batch, w.n_q_heads), device="cuda")
    for s in range(16):
        q, k1, v1 = w.step_qkv(s, device="cuda")
        cache.append(k1, v1)
        out = cache.decode(q, None, cmax, th)
        for (b, h) in sample:
            keep[(b, h)][0].append(host(k1[b, h])[None]); keep[(b, h)][1].append(host(v1[b, h])[None])
        if s not in (0, 15):
            continue
        t = ctx + s
        nfull = (t + 1) // QBLOCK * QBLOCK
        lo = t - W + 1
        p0 = lo // QBLOCK * QBLOCK
        o, cm, tc = out.cpu(), cmax.cpu().numpy(), th.cpu().numpy()
        for (b, h) in sample:
            Kin = np.concatenate(keep[(b, h)][0]); Vin = np.concatenate(keep[(b, h)][1])
            Kin, Vin = Kin[p0 - first:], Vin[p0 - first:]
            K = model.stored_rows(Kin, np.arange(p0, t + 1))
            V = nm.bf16_to_f32(Vin)
            for hq in (h * g, h * g + g - 1):
                qr = model.query_rows(host(q[b, hq])[None], [t])[0]
                r = int8_decode_one(qr, K, V, p0, t, W, nfull)
                assert_close(o[b, hq][None], r["out"][None], "bf16", "int8 ring s=%d b=%d h=%d" % (s, b, hq))
                assert cm[b, hq] >= r["cmax"] * (1 - 1e-12) and cm[b, hq] <= r["cmax"] * (1 + 1e-5)
                assert tc[b, hq] >= math.tanh(cm[b, hq]) * (1 - 1e-7) and r["tv"] <= tc[b, hq]
    from oracle import numerics as onm
    KQ = cache.export(kvc.KVC_EXPORT_KQ); SK = cache.export(kvc.KVC_EXPORT_SK)
    WT = cache.export(kvc.KVC_EXPORT_WITNESS)
    nfb = (ctx + 16) // QBLOCK
    for (b, h) in sample:
        Kin = np.concatenate(keep[(b, h)][0])
        for blk in (nfb - W // QBLOCK, nfb - 1000, nfb - 1):
            pos = np.arange(blk * QBLOCK, (blk + 1) * QBLOCK)
            Kb = model.stored_rows(Kin[pos - first], pos)
            sK, cK = onm.quantize_block(Kb)
            slot = blk % (W // QBLOCK)
            sl = slice(slot * QBLOCK, (slot + 1) * QBLOCK)
            assert SK[b, h, slot] == sK and np.array_equal(KQ[b, h, sl], cK), (b, h, blk)
            wit = np.stack([onm.witness_row(Kb[i], cK[i], sK) for i in range(QBLOCK)])
            assert np.array_equal(WT[b, h, sl], wit), (b, h, blk)
    assert cache.device_status() == 0


def test_int8_gated_sampled():
    # The INT8 workload after one gated fallback, as the gated bench line runs it: a decode
    # with per-token c_t, the block risk, the gate at tau = 0.2 with a budget of 1 % of the
    # complete blocks, the restore from a bf16 backing store of the same rows; then decode
    # steps with the restored blocks served exactly.  Risk (a max) and the selection are
    # checked exactly, the outputs of the heads with the most and the fewest restored blocks
    # against the oracle.
    import copy
    from oracle.model import QBLOCK, int8_decode_one, block_risk, gate_select
    w = wl.int8_witness()
    ctx, chunk = w.extra["context"], 8192
    B, Hq, Hkv = w.batch, w.n_q_heads, w.n_kv_heads
    g = Hq // Hkv
    budget = int(0.01 * B * Hkv * (ctx // QBLOCK))
    cache = kvc.Cache.from_workload(w, int8_exact_blocks=budget)
    wb = copy.copy(w)
    wb.quant = None
    full = kvc.Cache.from_workload(wb)
    for c in range(ctx // chunk):
        k, v = w.prefill_chunk(c, chunk, device="cuda")
        cache.append_rows(k, v)
        full.append_rows(k, v)
        del k, v
    kf = torch.from_numpy(full.export(kvc.KVC_EXPORT_K).view(np.int16)).view(torch.bfloat16).cuda()
    vf = torch.from_numpy(full.export(kvc.KVC_EXPORT_V).view(np.int16)).view(torch.bfloat16).cuda()
    full.close()
    steps = [w.step_qkv(s, device="cuda") for s in range(4)]
    q, k1, v1 = steps[0]
    cache.append(k1, v1)
    S = cache.S
    ct = torch.zeros((B, Hq, S), device="cuda")
    cmax = torch.empty((B, Hq), device="cuda")
    th = torch.empty((B, Hq), device="cuda")
    cache.decode(q, None, cmax, th, ct)
    risk = cache.block_risk(ct).cpu().numpy()
    ct_h = ct.cpu().numpy()
    del ct
    t = ctx
    for b in range(B):
        for h in range(Hkv):
            want = block_risk(ct_h[b, h * g:(h + 1) * g, :t + 1], t + 1)
            assert np.array_equal(risk[b, h, :len(want)], want.astype(np.float32)), (b, h)
            assert not risk[b, h, len(want):].any(), (b, h)           # incomplete blocks: no risk
    sel = kvc.kvc_int8_gate(risk, 0.2, budget)
    want = gate_select({(b, h): risk[b, h].astype(np.float64) for b in range(B) for h in range(Hkv)}, 0.2, budget)
    assert [tuple(int(x) for x in r) for r in sel] == want
    cache.restore(sel, kf, vf)
    del kf, vf
    torch.cuda.empty_cache()
    restored = {(b, h): set() for b in range(B) for h in range(Hkv)}
    for b, h, blk in want:
        restored[(b, h)].add(blk)
    counts = sorted(restored, key=lambda bh: (len(restored[bh]), bh))
    sample = [counts[-1], counts[0]]
    assert len(restored[sample[0]]) > 0
    # the sampled heads' rows, regenerated from the workload's generator
    Kin = {bh: [] for bh in sample}
    Vin = {bh: [] for bh in sample}
    for c in range(ctx // chunk):
        k, v = w.prefill_chunk(c, chunk, device="cuda")
        for (b, h) in sample:
            Kin[(b, h)].append(host(k[b, h])); Vin[(b, h)].append(host(v[b, h]))
        del k, v
    model = oracle_for(w)
    for s in range(4):
        q, k1, v1 = steps[s]
        if s:
            cache.append(k1, v1)
        out = cache.decode(q, None, cmax, th).cpu()             # bf16: its own rounding allowed
        cm = cmax.cpu().numpy()
        for (b, h) in sample:
            Kin[(b, h)].append(host(k1[b, h])[None]); Vin[(b, h)].append(host(v1[b, h])[None])
        if s not in (0, 3):
            continue
        t = ctx + s
        nfull = (t + 1) // QBLOCK * QBLOCK
        for (b, h) in sample:
            K = model.stored_rows(np.concatenate(Kin[(b, h)]), np.arange(t + 1))
            V = nm.bf16_to_f32(np.concatenate(Vin[(b, h)]))
            for hq in (h * g, h * g + g - 1):
                qr = model.query_rows(host(q[b, hq])[None], [t])[0]
                r = int8_decode_one(qr, K, V, 0, t, 0, nfull, restored[(b, h)])
                assert_close(out[b, hq][None], r["out"][None], "bf16", "gated s=%d b=%d h=%d" % (s, b, hq))
                assert cm[b, hq] >= r["cmax"] * (1 - 1e-12) and cm[b, hq] <= r["cmax"] * (1 + 1e-5)
    assert cache.device_status() == 0


def test_int8_dither_sampled():
    # Tier B at the INT8 workload's shape: the same tokens, keys quantized with the
    # subtractive dither of the (position, channel group, KV head + 65536 layer, request ID)
    # Philox counter, values plain, no witnesses; context 131072, then 16 one-token steps
    from oracle.model import QBLOCK, int8_decode_one
    w = wl.int8_dither()
    ctx = w.extra["context"]
    cache = kvc.Cache.from_workload(w)
    model = oracle_for(w)
    g = w.n_q_heads // w.n_kv_heads
    sample = [(0, 0), (3, 7), (7, 2)]
    keep = {bh: ([], []) for bh in sample}
    chunk = 8192
    for c in range(ctx // chunk):
        k, v = w.prefill_chunk(c, chunk, device="cuda")
        cache.append_rows(k, v)
        for (b, h) in sample:
            keep[(b, h)][0].append(host(k[b, h])); keep[(b, h)][1].append(host(v[b, h]))
        del k, v
    for s in range(16):
        q, k1, v1 = w.step_qkv(s, device="cuda")
        cache.append(k1, v1)
        out = cache.decode(q)
        for (b, h) in sample:
            keep[(b, h)][0].append(host(k1[b, h])[None]); keep[(b, h)][1].append(host(v1[b, h])[None])
        if s not in (0, 15):
            continue
        t = ctx + s
        nfull = (t + 1) // QBLOCK * QBLOCK
        o = out.cpu()                                            # bf16: its own rounding allowed
        for (b, h) in sample:
            Kin = np.concatenate(keep[(b, h)][0]); Vin = np.concatenate(keep[(b, h)][1])
            K = model.stored_rows(Kin, np.arange(t + 1))
            V = nm.bf16_to_f32(Vin)
            for hq in (h * g, h * g + g - 1):
                qr = model.query_rows(host(q[b, hq])[None], [t])[0]
                r = int8_decode_one(qr, K, V, 0, t, 0, nfull, dither=model.dither(b, h))
                assert r["c"] is None
                assert_close(o[b, hq][None], r["out"][None], "bf16", "tier B full s=%d b=%d h=%d" % (s, b, hq))
    # a sample of blocks bit-exact: dithered key codes, plain value codes, scales
    KQ = cache.export(kvc.KVC_EXPORT_KQ); SK = cache.export(kvc.KVC_EXPORT_SK)
    VQ = cache.export(kvc.KVC_EXPORT_VQ); SV = cache.export(kvc.KVC_EXPORT_SV)
    for (b, h) in sample:
        Kin = np.concatenate(keep[(b, h)][0]); Vin = np.concatenate(keep[(b, h)][1])
        u = model.dither(b, h)
        n = Kin.shape[0]
        for blk in (0, 1, 4095, 8191, n // QBLOCK - 1):
            pos = np.arange(blk * QBLOCK, (blk + 1) * QBLOCK)
            sK, cK = nm.quantize_block_dither(model.stored_rows(Kin[pos], pos), u(blk * QBLOCK, QBLOCK))
            sV, cV = nm.quantize_block(nm.bf16_to_f32(Vin[pos]))
            assert SK[b, h, blk] == sK and np.array_equal(KQ[b, h, pos], cK), (b, h, blk)
            assert SV[b, h, blk] == sV and np.array_equal(VQ[b, h, pos], cV), (b, h, blk)
    assert cache.device_status() == 0


@pytest.mark.parametrize("windowed,via", [(False, "trim"), (True, "trim"), (False, "store")],
                         ids=["full", "w4096", "full-store"])
def test_prefix_reuse_sampled(windowed, via):
    # 16 requests with an 8192-token prefix (Hq=32, Hkv=8, d=128, RoPE 10000), cut at seeded
    # points in [0, 8191], then a 512-token suffix by kvc_chunk_attn; sampled rows against the oracle,
    # and the stale-next_position control (planted on the CPU) must exceed the tolerance.
    # via "trim": kvc_trim; via "store": every prefill saved under its token IDs, the requests
    # then refilled with other rows, and each cut taken back by a host lookup and one batched
    # load, as the store bench line runs it
    w = wl.prefix_reuse(windowed)
    n, pre, W = w.extra["suffix"], w.extra["prefix"], w.window
    cuts = w.extra["cuts"]
    cache = kvc.Cache.from_workload(w, max_chunk=n, store_slots=w.batch if via == "store" else 0)
    model = oracle_for(w)
    g = w.n_q_heads // w.n_kv_heads
    reqs = [int(np.argmin(cuts)), int(np.argmax(cuts)), 3, 11]
    hs = [0, 7]                                        # KV heads sampled
    keep = {(r, h): [] for r in reqs for h in hs}
    for c in range(pre // 2048):
        k = w.keys((w.batch, w.n_kv_heads, 2048, w.head_dim), "prefix%d" % c, "cuda")
        v = w.values((w.batch, w.n_kv_heads, 2048, w.head_dim), "prefix%d" % c, "cuda")
        cache.append_rows(k, v)
        for (r, h) in keep:
            keep[(r, h)].append((host(k[r, h]), host(v[r, h])))
        del k, v
    if via == "trim":
        cache.trim(cuts)
    else:
        store = kvc.PrefixStore(cache.cfg, w.batch)
        rng = np.random.default_rng(w.seed)
        queries = []
        for r in range(w.batch):
            ids = rng.integers(0, 1 << 31, pre, dtype=np.int64)
            assert cache.save_prefix(store, r, ids, "test", b"prefix-reuse") == r
            queries.append(np.concatenate([ids[:cuts[r]], rng.integers(1 << 32, 1 << 33, n, dtype=np.int64)]))
        cache.trim([0] * w.batch)
        k = w.keys((w.batch, w.n_kv_heads, 2048, w.head_dim), "other", "cuda")
        v = w.values((w.batch, w.n_kv_heads, 2048, w.head_dim), "other", "cuda")
        cache.append_rows(k, v)
        del k, v
        found = [store.lookup(x, "test", b"prefix-reuse") for x in queries]
        assert [f[0] for f in found] == list(range(w.batch)) and [f[1] for f in found] == list(cuts)
        cache.store_load_batch([f[0] for f in found], list(range(w.batch)), [f[1] for f in found])
        assert np.array_equal(cache.export(kvc.KVC_EXPORT_NEXT_POSITION), np.asarray(cuts))
        store.close()
    q = w.queries((w.batch, n, w.n_q_heads, w.head_dim), "suffix", "cuda")
    k = w.keys((w.batch, n, w.n_kv_heads, w.head_dim), "suffix", "cuda")
    v = w.values((w.batch, n, w.n_kv_heads, w.head_dim), "suffix", "cuda")
    out = cache.chunk(q, k, v).float().cpu().numpy().astype(np.float64)
    hq_, hk_, hv_ = host(q), host(k), host(v)
    for (r, h) in keep:
        cut = cuts[r]
        Kpre = np.concatenate([a for a, _ in keep[(r, h)]])[:cut]
        Vpre = np.concatenate([b for _, b in keep[(r, h)]])[:cut]
        Kall = np.concatenate([Kpre, hk_[r, :, h]])
        Vall = np.concatenate([Vpre, hv_[r, :, h]])
        K = model.stored_rows(Kall, np.arange(cut + n)).astype(np.float64)
        V = nm.bf16_to_f32(Vall).astype(np.float64)
        Kst = np.concatenate([K[:cut], model.stored_rows(hk_[r, :, h], pre + np.arange(n)).astype(np.float64)])
        worst_stale = -np.inf
        for i in (0, 1, 127, 128, 255, 511):
            p = cut + i
            qr = model.query_rows(hq_[r, i, h * g:(h + 1) * g], np.full(g, p)).astype(np.float64)
            ref = nm.attend(qr, K[:p + 1], V[:p + 1], p, W)
            got = out[r, i, h * g:(h + 1) * g]
            err = np.abs(got - ref) - (2e-3 + 2e-3 * np.abs(ref) + np.ldexp(1.0, np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))).astype(int) - 8))
            assert err.max() <= 0, (r, h, i, err.max())
            # stale next_position: same rows, suffix encoded from the old length `pre`
            qs = model.query_rows(hq_[r, i, h * g:(h + 1) * g], np.full(g, pre + i)).astype(np.float64)
            stale = nm.attend(qs, Kst[:p + 1], V[:p + 1], p, W)
            worst_stale = max(worst_stale, (np.abs(stale - got) - (2e-3 + 2e-3 * np.abs(got))).max())
        if cut > 0:
            assert worst_stale > 0, ("stale control within tolerance", r, h, cut)
    assert cache.device_status() == 0
