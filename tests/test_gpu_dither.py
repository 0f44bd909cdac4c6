"""GPU parity of Tier B: subtractive-dither INT8 codes bit-exact, and the decode, which
regenerates every dither from its Philox counter, within tolerance of attention over
the rows (code - u) s.

[WITCERT] "WitCert: Sound Runtime Risk Observability and Gating for KV-Cache Quantization",
the Tier B paragraph (为了进一步压榨显存极限): dither added at write, cancelled at read from
the same Philox stream, no witness stored; "SGLang 生产级落地与闭环门控修复": the counter is
(request ID, layer, KV head, token, channel), independent of batch order.
"""
import numpy as np
import pytest
import torch

from kv_cache_decode_ring_gb300 import kvc
from kv_cache_decode_ring_gb300 import workloads as wl
from oracle import numerics as nm
from oracle.model import QBLOCK

from _parity import assert_close, host, oracle_for

pytestmark = pytest.mark.gpu
KEY = (0x243F6A88, 0x85A308D3)


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_decode_ring_gb300 import build
    build.build()


def _w(name, **kw):
    kw.setdefault("layer", 3)
    kw.setdefault("dither_key", KEY)
    return wl.small(name, quant="int8-dither", **kw)


def check_state(cache, model, requests=None):
    """Codes and scales of every complete block and the exact tail rows, bit-exact."""
    KQ = cache.export(kvc.KVC_EXPORT_KQ); VQ = cache.export(kvc.KVC_EXPORT_VQ)
    SK = cache.export(kvc.KVC_EXPORT_SK); SV = cache.export(kvc.KVC_EXPORT_SV)
    KT = cache.export(kvc.KVC_EXPORT_KTAIL); VT = cache.export(kvc.KVC_EXPORT_VTAIL)
    assert np.array_equal(cache.export(kvc.KVC_EXPORT_POSITIONS), model.expected_positions())
    for b in (range(model.B) if requests is None else requests):
        n = model.length(b)
        nfull = n // QBLOCK * QBLOCK
        for h in range(model.Hkv):
            for blk in range(nfull // QBLOCK):
                sK, cK, sV, cV, wit = model.quantized_block(b, h, blk)
                assert wit is None
                sl = slice(blk * QBLOCK, (blk + 1) * QBLOCK)
                assert SK[b, h, blk] == sK and SV[b, h, blk] == sV, (b, h, blk)
                assert np.array_equal(KQ[b, h, sl], cK), ("K codes", b, h, blk)
                assert np.array_equal(VQ[b, h, sl], cV), ("V codes", b, h, blk)
            for p in range(nfull, n):
                assert np.array_equal(KT[b, h, p % QBLOCK], nm.f32_to_bf16(model.hk[b][p][h])), (b, h, p)
                assert np.array_equal(VT[b, h, p % QBLOCK], nm.f32_to_bf16(model.hv[b][p][h])), (b, h, p)


def check_decode(cache, model, q):
    out = torch.empty((model.B, model.Hq, model.d), dtype=torch.float32, device="cuda")
    kvc.kvc_decode_attn(cache.h, q.cuda(), out)
    res = model.decode_int8(host(q))
    for (b, hq), r in res.items():
        assert_close(out[b, hq][None], r["out"][None], "bf16", "dither decode b=%d h=%d" % (b, hq))
    return out


@pytest.mark.parametrize("d,Hq,Hkv,cap", [(128, 8, 2, 1104), (128, 4, 4, 1104), (128, 16, 2, 1104),
                                           (64, 8, 2, 1104), (64, 2, 1, 1104), (128, 2, 1, 1104),
                                           (128, 8, 2, 16400)])      # the last: 2048-token splits
def test_dither_parity(d, Hq, Hkv, cap):
    w = _w("dither-%d-%d-%d-%d" % (d, Hq, Hkv, cap), B=3, Hq=Hq, Hkv=Hkv, d=d, capacity=cap, rope_base=10000.0,
           seed=31, outliers=(4, 20.0))
    cache = kvc.Cache.from_workload(w, out_dtype="f32")
    model = oracle_for(w)
    lengths = [1060, 47, 16] if cap < 16384 else [4150, 2047, 16]
    k, v = w.prefill_chunk(0, max(lengths))
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    check_state(cache, model)
    for s in range(18):                               # single appends complete blocks
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        if s in (0, 16, 17):
            check_state(cache, model)
        check_decode(cache, model, q)
    assert cache.device_status() == 0


def test_dither_stream_follows_the_request_id_not_the_slot():
    """Request ID r in slot 0 of one cache and in slot 1 of another: identical codes."""
    w = _w("dither-id", B=2, Hq=4, Hkv=2, d=128, capacity=64, rope_base=10000.0, seed=3)
    a, b = kvc.Cache.from_workload(w, out_dtype="f32"), kvc.Cache.from_workload(w, out_dtype="f32")
    a.set_request_id(0, 777); a.set_request_id(1, 5)
    b.set_request_id(0, 5); b.set_request_id(1, 777)
    k, v = w.prefill_chunk(0, 48)
    a.append_rows(k.cuda(), v.cuda())
    b.append_rows(k.flip(0).contiguous().cuda(), v.flip(0).contiguous().cuda())   # the rows swap slots too
    ka, kb = a.export(kvc.KVC_EXPORT_KQ), b.export(kvc.KVC_EXPORT_KQ)
    assert np.array_equal(ka[0], kb[1]) and np.array_equal(ka[1], kb[0])
    model = oracle_for(w)
    model.set_request_id(0, 777); model.set_request_id(1, 5)
    model.append_rows(host(k), host(v), [48, 48])
    check_state(a, model)
    with pytest.raises(kvc.KvcError) as e:
        a.set_request_id(0, 1)                         # request 0 holds rows
    assert e.value.code == kvc.KVC_ERR_ARG
    q = w.step_qkv(0)[0]
    a.append(*(t.cuda() for t in w.step_qkv(0)[1:]))
    model.append(*(host(t) for t in w.step_qkv(0)[1:]))
    check_decode(a, model, q)


def test_dither_trim_and_refusals():
    w = _w("dither-trim", B=2, Hq=4, Hkv=2, d=128, capacity=256, rope_base=10000.0, seed=8)
    cache = kvc.Cache.from_workload(w, out_dtype="f32")
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, 150)
    cache.append_rows(k.cuda(), v.cuda(), counts=[150, 70])
    model.append_rows(host(k), host(v), [150, 70])
    with pytest.raises(kvc.KvcError) as e:
        cache.trim([140, 70])                          # splits a quantized block
    assert e.value.code == kvc.KVC_ERR_EVICTED
    cache.trim([128, 66])
    model.trim([128, 66])
    for s in range(20):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        check_decode(cache, model, q)
    check_state(cache, model)
    q = w.step_qkv(99)[0].cuda()
    out = torch.empty((2, 4, 128), dtype=torch.float32, device="cuda")
    cm = torch.empty((2, 4), device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_decode_attn(cache.h, q, out, cm)       # no bound in Tier B
    assert e.value.code == kvc.KVC_ERR_ARG
    with pytest.raises(kvc.KvcError) as e:
        cache.export(kvc.KVC_EXPORT_WITNESS)
    assert e.value.code == kvc.KVC_ERR_ARG
    ct = torch.zeros((2, 4, 256), device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        cache.block_risk(ct)
    assert e.value.code == kvc.KVC_ERR_UNSUPPORTED
    assert cache.device_status() == 0
