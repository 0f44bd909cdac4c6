"""GPU parity of the INT8 tier: block quantizer and witnesses bit-exact, fused decode
within tolerance of attention over the dequantized cache, and the bound sound.

[WITCERT] "WitCert: Sound Runtime Risk Observability and Gating for KV-Cache Quantization"
  "频带酉性与双层证书": w_{t,b} = ||r_{t,b}||, c_t = (1/sqrt d) sum_b ||q_b|| w_{t,b} >= |q.r_t|/sqrt d
  "为什么在线监控 KV 误差如此困难？": TV <= tanh(max |eps|)
"""
import math

import numpy as np
import pytest
import torch

from kv_cache_decode_ring_gb300 import kvc
from kv_cache_decode_ring_gb300 import workloads as wl
from oracle import numerics as nm
from oracle.model import NBANDS, QBLOCK, DecodeOracle

from _parity import assert_close, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_decode_ring_gb300 import build
    build.build()


def _oracle(w):
    return DecodeOracle(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, "contiguous", w.capacity, 0,
                        w.rope_base, "bf16", "int8")


def check_int8_state(cache, model, requests=None):
    """Codes, scales, witnesses of every complete block and the exact tail rows, bit-exact."""
    KQ = cache.export(kvc.KVC_EXPORT_KQ); VQ = cache.export(kvc.KVC_EXPORT_VQ)
    SK = cache.export(kvc.KVC_EXPORT_SK); SV = cache.export(kvc.KVC_EXPORT_SV)
    WT = cache.export(kvc.KVC_EXPORT_WITNESS)
    KT = cache.export(kvc.KVC_EXPORT_KTAIL); VT = cache.export(kvc.KVC_EXPORT_VTAIL)
    pos = cache.export(kvc.KVC_EXPORT_POSITIONS)
    assert np.array_equal(pos, model.expected_positions())
    for b in (range(model.B) if requests is None else requests):
        n = model.length(b)
        nfull = n // QBLOCK * QBLOCK
        for h in range(model.Hkv):
            for blk in range(nfull // QBLOCK):
                sK, cK, sV, cV, wit = model.quantized_block(b, h, blk)
                sl = slice(blk * QBLOCK, (blk + 1) * QBLOCK)
                assert SK[b, h, blk] == sK and SV[b, h, blk] == sV, (b, h, blk)
                assert np.array_equal(KQ[b, h, sl], cK) and np.array_equal(VQ[b, h, sl], cV), (b, h, blk)
                if blk in model.restored[b][h]:
                    assert not WT[b, h, sl].any(), (b, h, blk)     # the gated fallback zeroed them
                else:
                    assert np.array_equal(WT[b, h, sl], wit), (b, h, blk)
            for p in range(nfull, n):
                assert np.array_equal(KT[b, h, p % QBLOCK], nm.f32_to_bf16(model.hk[b][p][h])), (b, h, p)
                assert np.array_equal(VT[b, h, p % QBLOCK], nm.f32_to_bf16(model.hv[b][p][h])), (b, h, p)


def check_decode(cache, model, q, heads=None):
    B, Hq = model.B, model.Hq
    out = torch.empty((B, Hq, model.d), dtype=torch.float32, device="cuda")
    cmax = torch.full((B, Hq), -1.0, device="cuda")
    th = torch.full((B, Hq), -1.0, device="cuda")
    ct = torch.full((B, Hq, cache.S), -7.0, device="cuda")
    kvc.kvc_decode_attn(cache.h, q.cuda(), out, cmax, th, ct)
    res = model.decode_int8(host(q), heads)
    cm, tc, ctn = cmax.cpu().numpy(), th.cpu().numpy(), ct.cpu().numpy()
    for (b, hq), r in res.items():
        assert_close(out[b, hq][None], r["out"][None], "bf16", "int8 decode b=%d h=%d" % (b, hq))
        n = model.length(b)
        c_gpu = ctn[b, hq, :n].astype(np.float64)
        # the bound on every token: sound (>= |q.r|/sqrt d and >= the exact c_t) and tight
        assert np.all(c_gpu >= r["eps"]), (b, hq)
        assert np.all(c_gpu >= r["c"] * (1 - 1e-12)), (b, hq)
        assert np.all(c_gpu <= r["c"] * (1 + 1e-5) + 1e-30), (b, hq)
        assert cm[b, hq] >= r["cmax"] * (1 - 1e-12) and cm[b, hq] <= r["cmax"] * (1 + 1e-5) + 1e-30
        assert tc[b, hq] >= math.tanh(cm[b, hq]) * (1 - 1e-7) and tc[b, hq] <= 1.0
        assert r["tv"] <= tc[b, hq], (b, hq, r["tv"], tc[b, hq])
    return out


# every group size the fused kernel instantiates (1, 2, 4, 8), at both head dims
@pytest.mark.parametrize("d,Hq,Hkv", [(128, 8, 2), (64, 8, 1), (128, 4, 4), (64, 4, 4), (128, 4, 2),
                                      (64, 4, 2), (128, 16, 2), (64, 8, 2)])
def test_int8_prefill_decode_parity(d, Hq, Hkv):
    w = wl.small("int8-%d-%d-%d" % (d, Hq, Hkv), B=3, Hq=Hq, Hkv=Hkv, d=d, capacity=512, rope_base=10000.0,
                 quant="int8", seed=19, outliers=(4, 20.0))
    cache = kvc.Cache.from_workload(w, out_dtype="f32")
    model = _oracle(w)
    lengths = [1, 37, 300]
    k, v = w.prefill_chunk(0, max(lengths))
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    check_int8_state(cache, model)
    for s in range(20):                          # crosses block completions on single appends
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        if s % 4 == 3 or s == 0:
            check_int8_state(cache, model)
        check_decode(cache, model, q)
    assert cache.device_status() == 0


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 8, 2), (64, 8, 1)])
def test_int8_multi_split_parity(d, Hq, Hkv):
    # several 1024-token splits, warps with fewer blocks than tiles, a request of exactly
    # one block (no exact tail) and one whose last split holds a single block
    w = wl.small("int8-long-%d" % d, B=4, Hq=Hq, Hkv=Hkv, d=d, capacity=2624, rope_base=10000.0,
                 quant="int8", seed=29, outliers=(4, 20.0))
    cache = kvc.Cache.from_workload(w, out_dtype="f32")
    model = _oracle(w)
    lengths = [1030, 2500, 16, 2064]
    k, v = w.prefill_chunk(0, max(lengths))
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    check_int8_state(cache, model, requests=[0, 2])
    for s in range(2):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        check_decode(cache, model, q)
    assert cache.device_status() == 0


def test_int8_long_split_parity():
    # 2048-token splits: lengths around one and several of them, and a request of a
    # single block
    w = wl.small("int8-long-split", B=3, Hq=8, Hkv=2, d=128, capacity=16400, rope_base=10000.0,
                 quant="int8", seed=37, outliers=(4, 20.0))
    cache = kvc.Cache.from_workload(w, out_dtype="f32", int8_split=2048)
    model = _oracle(w)
    lengths = [2047, 6150, 16]
    k, v = w.prefill_chunk(0, max(lengths))
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    check_int8_state(cache, model, requests=[0, 2])
    for s in range(2):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        check_decode(cache, model, q)
    assert cache.device_status() == 0


@pytest.mark.parametrize("layout", ["contiguous", "window", "ring"])
@pytest.mark.parametrize("split", [1088, 1600, 1984])
def test_int8_split_lengths(split, layout):
    # the decode's split length is a multiple of 64 positions between 1024 and 2048 (chosen
    # per device unless configured): odd numbers of tiles per warp, requests ending inside,
    # at and just past a split, a window starting inside a split, a ring past its wrap
    ring = layout == "ring"
    cap = 4096 if ring else 6160
    w = wl.small("int8-split-%d-%s" % (split, layout), B=4, Hq=8, Hkv=2, d=128, layout="ring" if ring else "contiguous",
                 capacity=cap, window=cap if ring else (2500 if layout == "window" else 0), rope_base=10000.0,
                 quant="int8", seed=41, outliers=(4, 20.0))
    cache = kvc.Cache.from_workload(w, max_position=8192 if ring else 0, out_dtype="f32", int8_split=split)
    model = _oracle_layout(w)
    lengths = [split - 1, 2 * split + 17, 16, cap + split + 33] if ring else [split - 1, 2 * split + 17, 16, 3 * split]
    k, v = w.prefill_chunk(0, max(lengths))
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    for s in range(2):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        check_decode_window(cache, model, q, ring=ring)
    if ring:
        check_int8_ring_state(cache, model)
    assert cache.device_status() == 0


def test_int8_trim_rules_and_continue():
    w = wl.small("int8-trim", B=2, Hq=4, Hkv=2, d=128, capacity=256, rope_base=10000.0, quant="int8", seed=5)
    cache = kvc.Cache.from_workload(w, out_dtype="f32")
    model = _oracle(w)
    k, v = w.prefill_chunk(0, 100)
    cache.append_rows(k.cuda(), v.cuda(), counts=[100, 70])
    model.append_rows(host(k), host(v), [100, 70])
    with pytest.raises(kvc.KvcError) as e:
        cache.trim([90, 70])                     # 90 splits the quantized block 80..95
    assert e.value.code == kvc.KVC_ERR_EVICTED
    cache.trim([98, 64])                         # 98: inside the exact tail; 64: a block boundary
    model.trim([98, 64])
    check_int8_state(cache, model)
    for s in range(20):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        check_decode(cache, model, q)
    check_int8_state(cache, model)


def test_int8_zero_residual_gives_zero_bound():
    # keys on their blocks' quantization grid: residual 0, witnesses 0, bound 0
    w = wl.small("int8-exact", B=1, Hq=2, Hkv=1, d=128, capacity=64, rope_base=0.0, quant="int8", seed=2)
    cache = kvc.Cache.from_workload(w, out_dtype="f32")
    model = _oracle(w)
    rng = np.random.default_rng(4)
    c = rng.integers(-126, 127, (1, 1, 48, 128)).astype(np.float32)
    c[..., 0] = 127.0
    k = torch.from_numpy(c / 16).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((1, 1, 48, 128)).astype(np.float32)).to(torch.bfloat16)
    cache.append_rows(k.cuda(), v.cuda())
    model.append_rows(host(k), host(v), [48])
    assert not cache.export(kvc.KVC_EXPORT_WITNESS).any()
    q = w.queries((1, 2, 128), "zero-residual")
    check_decode(cache, model, q)


def _backing_store(w, k, v, lengths, extra):
    """Full-precision rows of the same tokens: a bf16 cache fed the same appends (the
    caller's backing store), exported and put back on the device."""
    import copy
    wb = copy.copy(w)
    wb.quant = None
    full = kvc.Cache.from_workload(wb)
    full.append_rows(k.cuda(), v.cuda(), counts=lengths)
    for k1, v1 in extra:
        full.append(k1.cuda(), v1.cuda())
    kf = torch.from_numpy(full.export(kvc.KVC_EXPORT_K).view(np.int16)).view(torch.bfloat16).cuda()
    vf = torch.from_numpy(full.export(kvc.KVC_EXPORT_V).view(np.int16)).view(torch.bfloat16).cuda()
    return kf, vf


@pytest.mark.parametrize("cap,lengths,split,pool,cuts", [
    (512, [300, 263], 0, 96, [160, 64]),
    (2624, [2500, 1100], 1088, 512, [1600, 64]),     # several quantized splits before the exact-block ones
], ids=["one-split", "split-1088"])
def test_int8_gated_fallback(cap, lengths, split, pool, cuts):
    # [WITCERT] "SGLang 生产级落地与闭环门控修复": risk from the decode's c_t, gate at tau,
    # restore the chosen blocks from the backing store; their tokens become exact (c_t = 0)
    # and every head's tanh(max c_t) drops to tau or below
    tau = 0.2
    w = wl.small("int8-gate", B=2, Hq=8, Hkv=2, d=128, capacity=cap, rope_base=10000.0, quant="int8",
                 seed=13, outliers=(4, 20.0))
    cache = kvc.Cache.from_workload(w, out_dtype="f32", int8_exact_blocks=pool, int8_split=split)
    model = _oracle(w)
    k, v = w.prefill_chunk(0, max(lengths))
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    q, k1, v1 = w.step_qkv(0)
    cache.append(k1.cuda(), v1.cuda())
    model.append(host(k1), host(v1))
    B, Hq, S = w.batch, w.n_q_heads, cache.S
    out = torch.empty((B, Hq, w.head_dim), dtype=torch.float32, device="cuda")
    cmax = torch.empty((B, Hq), device="cuda")
    th = torch.empty((B, Hq), device="cuda")
    ct = torch.zeros((B, Hq, S), device="cuda")
    kvc.kvc_decode_attn(cache.h, q.cuda(), out, cmax, th, ct)
    assert th.max().item() > tau                                   # the outlier channels make it risky
    # block risk: the block maximum of the decode's own c_t, bit-exact
    risk = cache.block_risk(ct).cpu().numpy()
    ctn = ct.cpu().numpy()
    g = Hq // w.n_kv_heads
    for b in range(B):
        nfull = model.length(b) // QBLOCK * QBLOCK
        for h in range(w.n_kv_heads):
            for blk in range(S // QBLOCK):
                want = ctn[b, h * g:(h + 1) * g, blk * 16:blk * 16 + 16].max() if (blk + 1) * 16 <= nfull else 0.0
                assert risk[b, h, blk] == want, (b, h, blk)
    sel = kvc.kvc_int8_gate(risk, tau, 1000)
    assert 0 < len(sel) <= pool
    top = kvc.kvc_int8_gate(risk, tau, 5)                           # a budget keeps the riskiest
    assert np.array_equal(top, sel[:5])
    kf, vf = _backing_store(w, k, v, lengths, [(k1, v1)])
    cache.restore(sel, kf, vf)
    model.restore([tuple(x) for x in sel])
    xm = cache.export(kvc.KVC_EXPORT_XMAP)
    ent = [xm[b, h, blk] for b, h, blk in sel]
    assert min(ent) >= 0 and len(set(ent)) == len(ent) and (xm >= 0).sum() == len(sel)
    check_int8_state(cache, model)
    # the same query again: restored tokens are exact with c_t = 0; every head under tau
    res = model.decode_int8(host(q))
    ct2 = torch.full((B, Hq, S), -7.0, device="cuda")
    kvc.kvc_decode_attn(cache.h, q.cuda(), out, cmax, th, ct2)
    ctn2 = ct2.cpu().numpy()
    assert np.all(th.cpu().numpy() <= tau)
    for b, h, blk in sel:
        assert np.all(ctn2[b, h * g:(h + 1) * g, blk * 16:blk * 16 + 16] == 0.0)
    for (b, hq), r in res.items():
        assert_close(out[b, hq][None], r["out"][None], "bf16", "gated decode b=%d h=%d" % (b, hq))
    check_decode(cache, model, q)
    # later steps, then a trim that drops the restored blocks past the cut
    steps = [(k1, v1)]
    for s in range(1, 4):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        check_decode(cache, model, q)
    cache.trim(cuts)
    model.trim(cuts)
    xm = cache.export(kvc.KVC_EXPORT_XMAP)
    for b in range(B):
        for h in range(w.n_kv_heads):
            live = {blk for blk in range(S // 16) if xm[b, h, blk] >= 0}
            assert live == model.restored[b][h], (b, h)
    check_int8_state(cache, model)
    for s in range(4, 8):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        check_decode(cache, model, q)
    assert cache.device_status() == 0


def test_int8_restore_errors():
    w = wl.small("int8-gate-err", B=1, Hq=4, Hkv=1, d=64, capacity=128, rope_base=0.0, quant="int8", seed=3)
    cache = kvc.Cache.from_workload(w, out_dtype="f32", int8_exact_blocks=2)
    k, v = w.prefill_chunk(0, 70)
    cache.append_rows(k.cuda(), v.cuda())
    kf, vf = _backing_store(w, k, v, None, [])
    with pytest.raises(kvc.KvcError) as e:
        cache.restore([(0, 0, 4)], kf, vf)                 # block 4 = positions 64..79: incomplete
    assert e.value.code == kvc.KVC_ERR_ARG
    with pytest.raises(kvc.KvcError) as e:
        cache.restore([(0, 0, 0), (0, 0, 1), (0, 0, 2)], kf, vf)     # pool of 2
    assert e.value.code == kvc.KVC_ERR_CAPACITY
    assert (cache.export(kvc.KVC_EXPORT_XMAP) < 0).all()            # nothing restored
    cache.restore([(0, 0, 1), (0, 0, 1)], kf, vf)                    # duplicates count once
    cache.restore([(0, 0, 1), (0, 0, 3)], kf, vf)                    # already restored: skipped
    assert (cache.export(kvc.KVC_EXPORT_XMAP) >= 0).sum() == 2


# ---- windowed and ring INT8 caches ------------------------------------------------------
def _oracle_layout(w):
    return DecodeOracle(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.layout, w.capacity,
                        0 if w.layout == "ring" else w.window, w.rope_base, "bf16", w.quant,
                        dither_key=w.extra.get("dither_key", (0, 0)), layer=w.extra.get("layer", 0))


def check_int8_ring_state(cache, model):
    """A ring of S slots keeps block n in block slot n mod S/16: the newest S/16 complete
    blocks, their codes, scales and witnesses bit-exact, and the exact tail rows."""
    KQ = cache.export(kvc.KVC_EXPORT_KQ); VQ = cache.export(kvc.KVC_EXPORT_VQ)
    SK = cache.export(kvc.KVC_EXPORT_SK); SV = cache.export(kvc.KVC_EXPORT_SV)
    WT = cache.export(kvc.KVC_EXPORT_WITNESS) if model.quant == "int8" else None
    KT = cache.export(kvc.KVC_EXPORT_KTAIL)
    assert np.array_equal(cache.export(kvc.KVC_EXPORT_POSITIONS), model.expected_positions())
    nbk = model.capacity // QBLOCK
    for b in range(model.B):
        n = model.length(b)
        nfb = n // QBLOCK
        for h in range(model.Hkv):
            for blk in range(max(0, nfb - nbk), nfb):
                sK, cK, sV, cV, wit = model.quantized_block(b, h, blk)
                k = blk % nbk
                sl = slice(k * QBLOCK, (k + 1) * QBLOCK)
                assert SK[b, h, k] == sK and SV[b, h, k] == sV, (b, h, blk)
                assert np.array_equal(KQ[b, h, sl], cK) and np.array_equal(VQ[b, h, sl], cV), (b, h, blk)
                if WT is not None:
                    assert np.array_equal(WT[b, h, sl], wit), (b, h, blk)
            for p in range(nfb * QBLOCK, n):
                assert np.array_equal(KT[b, h, p % QBLOCK], nm.f32_to_bf16(model.hk[b][p][h])), (b, h, p)


def check_decode_window(cache, model, q, ring):
    """Outputs against attention over the dequantized window; c_t of every token in the
    window (slot = position, or position mod S on a ring) sound and tight; max_t c_t over
    the window; TV <= tanh(max c_t)."""
    B, Hq, S = model.B, model.Hq, model.capacity
    out = torch.empty((B, Hq, model.d), dtype=torch.float32, device="cuda")
    bound = model.quant == "int8"
    cmax = torch.full((B, Hq), -1.0, device="cuda") if bound else None
    th = torch.full((B, Hq), -1.0, device="cuda") if bound else None
    ct = torch.full((B, Hq, S), -7.0, device="cuda") if bound else None
    kvc.kvc_decode_attn(cache.h, q.cuda(), out, cmax, th, ct)
    res = model.decode_int8(host(q))
    for (b, hq), r in res.items():
        assert_close(out[b, hq][None], r["out"][None], "bf16", "int8 window decode b=%d h=%d" % (b, hq))
        if not bound:
            continue
        t = model.length(b) - 1
        lo = max(0, t - model.window + 1) if model.window else 0
        slots = np.arange(lo, t + 1) % S if ring else np.arange(lo, t + 1)
        c_gpu = ct[b, hq].cpu().numpy().astype(np.float64)[slots]
        assert c_gpu.shape == r["c"].shape
        assert np.all(c_gpu >= r["eps"]), (b, hq)
        assert np.all(c_gpu >= r["c"] * (1 - 1e-12)), (b, hq)
        assert np.all(c_gpu <= r["c"] * (1 + 1e-5) + 1e-30), (b, hq)
        cm, tc = float(cmax[b, hq]), float(th[b, hq])
        assert cm >= r["cmax"] * (1 - 1e-12) and cm <= r["cmax"] * (1 + 1e-5) + 1e-30, (b, hq)
        assert tc >= math.tanh(cm) * (1 - 1e-7) and tc <= 1.0
        assert r["tv"] <= tc, (b, hq, r["tv"], tc)


@pytest.mark.parametrize("window", [8, 100, 1000], ids=["w8-inside-a-block", "w100", "w1000"])
def test_int8_windowed_contiguous(window):
    # blocks wholly before the window are skipped, the first block is masked per token,
    # and a window shorter than a block sits in the exact tail
    w = wl.small("int8-w%d" % window, B=3, Hq=8, Hkv=2, d=128, capacity=1536, window=window,
                 rope_base=10000.0, quant="int8", seed=23, outliers=(4, 20.0))
    cache = kvc.Cache.from_workload(w, out_dtype="f32")
    model = _oracle_layout(w)
    lengths = [1, 250, 1300]
    k, v = w.prefill_chunk(0, max(lengths))
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    check_int8_state(cache, model)
    for s in range(18):                                  # crosses a block completion
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        check_decode_window(cache, model, q, ring=False)
    check_int8_state(cache, model)
    assert cache.device_status() == 0


@pytest.mark.parametrize("quant", ["int8", "int8-dither"])
def test_int8_ring_through_first_replacement(quant):
    # W = 64 slots (4 blocks): the not-full phase, the first block overwritten, the window
    # cutting into the oldest block; a prefill longer than the ring (its early blocks are
    # never stored) and one-token appends
    extra = {"outliers": (4, 20.0)}
    if quant == "int8-dither":
        extra.update(dither_key=(0x243F6A88, 0x85A308D3), layer=0)
    w = wl.small("int8-ring-" + quant, B=3, Hq=8, Hkv=2, d=128, layout="ring", capacity=64, window=64,
                 rope_base=10000.0, quant=quant, seed=31, **extra)
    cache = kvc.Cache.from_workload(w, max_position=512, out_dtype="f32")
    model = _oracle_layout(w)
    lengths = [3, 70, 150]
    k, v = w.prefill_chunk(0, max(lengths))
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    check_int8_ring_state(cache, model)
    for s in range(90):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        if s % 5 == 0 or s < 20:
            check_decode_window(cache, model, q, ring=True)
        if s % 15 == 14:
            check_int8_ring_state(cache, model)
    assert cache.device_status() == 0


def test_int8_ring_trim_rules():
    # a ring trim must keep what the next query needs; an INT8 trim must not split a block
    w = wl.small("int8-ring-trim", B=2, Hq=4, Hkv=1, d=128, layout="ring", capacity=64, window=64,
                 rope_base=10000.0, quant="int8", seed=37)
    cache = kvc.Cache.from_workload(w, max_position=512, out_dtype="f32")
    model = _oracle_layout(w)
    k, v = w.prefill_chunk(0, 40)
    cache.append_rows(k.cuda(), v.cuda())
    model.append_rows(host(k), host(v), [40, 40])
    with pytest.raises(kvc.KvcError) as e:
        cache.trim([20, 40])                           # splits a quantized block
    assert e.value.code == kvc.KVC_ERR_EVICTED
    cache.trim([32, 39])                               # a block boundary; inside the exact tail
    model.trim([32, 39])
    check_int8_ring_state(cache, model)
    for s in range(40):                                # wrap the ring after the trim
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        check_decode_window(cache, model, q, ring=True)
    check_int8_ring_state(cache, model)
    assert cache.device_status() == 0



@pytest.mark.parametrize("layout,quant", [("contiguous", "int8"), ("ring", "int8"), ("ring", "int8-dither")])
def test_int8_paged(layout, quant):
    # a 16-slot page holds one quantization block of every KV head: codes, scales and
    # witnesses gathered through the block table equal the unpaged layout's, bit for bit
    extra = {"outliers": (4, 20.0)}
    if quant == "int8-dither":
        extra.update(dither_key=(0x243F6A88, 0x85A308D3), layer=0)
    W = 128
    w = wl.small("int8-paged-%s-%s" % (layout, quant), B=3, Hq=8, Hkv=2, d=128, layout=layout,
                 capacity=512 if layout == "contiguous" else W, window=0 if layout == "contiguous" else W,
                 rope_base=10000.0, quant=quant, seed=47, **extra)
    cap = w.capacity
    cache = kvc.Cache.from_workload(w, out_dtype="f32", page_pool=3 * cap // 16,
                                    max_position=1024 if layout == "ring" else 0)
    model = _oracle_layout(w)
    lengths = [3, 200, 300] if layout == "ring" else [3, 200, 400]
    k, v = w.prefill_chunk(0, max(lengths))
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    check = check_int8_ring_state if layout == "ring" else check_int8_state
    check(cache, model)
    for s in range(20):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        check_decode_window(cache, model, q, ring=layout == "ring")
    check(cache, model)
    if layout == "contiguous":
        cache.trim([0, 192, 400])                       # block boundaries: pages past the cut return
        model.trim([0, 192, 400])
        tab = cache.export(kvc.KVC_EXPORT_PAGE_TABLE)
        assert (tab[0] < 0).all() and (tab[1, :12] >= 0).all() and (tab[1, 12:] < 0).all()
        q, k1, v1 = w.step_qkv(50)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        check_decode_window(cache, model, q, ring=False)
        check(cache, model)
    assert cache.device_status() == 0
