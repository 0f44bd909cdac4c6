"""GPU parity of kvc_chunk_attn (trim, then chunked causal/windowed suffix attention).

[PREFIX] "LLM 機制實驗（五）：改了歷史，能否只重算變化的後綴？": trim K/V/positions to
`cut`, continue from next_position = cut with model.chunk(tokens[cut:]); the result
must equal a full recompute, and keeping the stale next_position must diverge.
"""
import numpy as np
import pytest
import torch

from kv_cache_decode_ring_gb300 import kvc
from kv_cache_decode_ring_gb300 import workloads as wl
from oracle import numerics as nm

from _parity import assert_close, check_state, host, oracle_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_decode_ring_gb300 import build
    build.build()


def _prefilled(w, lengths, cuts, max_chunk, out_dtype=None, page_pool=0):
    cache = kvc.Cache.from_workload(w, max_chunk=max_chunk, out_dtype=out_dtype, page_pool=page_pool)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, max(lengths))
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    cache.trim(cuts)
    model.trim(cuts)
    return cache, model


def _suffix(w, n, tag="suffix"):
    B, Hq, Hkv, d = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
    return (w.queries((B, n, Hq, d), tag), w.keys((B, n, Hkv, d), tag), w.values((B, n, Hkv, d), tag))


CHUNK_CASES = [
    # name, Hq, Hkv, capacity, window, paged
    ("gqa4", 8, 2, 1024, 0, False),
    ("gqa4-w100", 8, 2, 1024, 100, False),
    ("gqa3-odd-pair", 6, 2, 1000, 0, False),      # a CTA's second head slot idle; capacity not a multiple of 16
    ("mha-w300", 3, 3, 1024, 300, False),
    ("gqa4-paged", 8, 2, 1024, 0, True),
    ("gqa4-w100-paged", 8, 2, 1024, 100, True),
]


@pytest.mark.parametrize("case", CHUNK_CASES, ids=lambda c: c[0])
def test_chunk_matches_recompute(case):
    name, Hq, Hkv, cap, window, paged = case
    w = wl.small("chunk-" + name, B=3, Hq=Hq, Hkv=Hkv, d=128, capacity=cap, window=window,
                 rope_base=10000.0, seed=17)
    lengths, cuts, n = [600, 300, 40], [413, 0, 40], 200
    cache, model = _prefilled(w, lengths, cuts, n, out_dtype="f32", page_pool=3 * (cap // 16) if paged else 0)
    q, k, v = _suffix(w, n)
    out = cache.chunk(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    ref = model.chunk(host(q), host(k), host(v))
    err = np.abs(out.double().cpu().numpy() - ref)
    print("chunk max abs err %.3e, max rel excess %.3f" % (err.max(), (err / (2e-3 + 2e-3 * np.abs(ref))).max()))
    assert_close(out, ref, "bf16", "chunk %s" % name)
    check_state(cache, model, w)
    assert list(cache.next_positions()) == [c + n for c in cuts]
    assert cache.device_status() == 0


def test_chunk_rows_equal_one_token_decodes():
    # row i of the chunk equals a decode of the same query at position cut + i
    w = wl.small("chunk-vs-decode", B=2, Hq=8, Hkv=2, d=128, capacity=512, rope_base=10000.0, seed=3)
    lengths, cuts, n = [300, 129], [257, 129], 130
    a, _ = _prefilled(w, lengths, cuts, n, out_dtype="f32")
    b, _ = _prefilled(w, lengths, cuts, n, out_dtype="f32")
    q, k, v = _suffix(w, n)
    out = a.chunk(q.cuda(), k.cuda(), v.cuda()).cpu()
    for i in range(n):
        b.append(k[:, i].contiguous().cuda(), v[:, i].contiguous().cuda())
        if i % 13 == 0 or i == n - 1:
            d = b.decode(q[:, i].contiguous().cuda()).cpu()
            assert_close(out[:, i], d.double().numpy(), "bf16", "chunk row %d vs decode" % i)


def test_stale_next_position_diverges():
    # planted on the CPU: the same trimmed rows, suffix rotated from the old length
    w = wl.small("chunk-stale", B=2, Hq=4, Hkv=1, d=128, capacity=512, rope_base=10000.0, seed=9)
    lengths, cuts, n = [300, 300], [120, 0], 64
    cache, model = _prefilled(w, lengths, cuts, n, out_dtype="f32")
    q, k, v = _suffix(w, n)
    out = cache.chunk(q.cuda(), k.cuda(), v.cuda()).double().cpu().numpy()
    hk, hv = host(k), host(v)
    # the prefix rows of request 0 as stored, plus the suffix encoded at positions 300 + i
    K = [model.hk[0][p][0] for p in range(cuts[0])]
    V = [model.hv[0][p][0] for p in range(cuts[0])]
    stale = np.zeros((n, 4, 128))
    for i in range(n):
        K.append(model.stored_rows(hk[0, i], [lengths[0] + i])[0])
        V.append(nm.bf16_to_f32(hv[0, i])[0])
        qr = model.query_rows(host(q)[0, i], np.full(4, lengths[0] + i)).astype(np.float64)
        stale[i] = nm.attend(qr, np.stack(K).astype(np.float64), np.stack(V).astype(np.float64), len(K) - 1)
    excess = np.abs(stale - out[0]) - (2e-3 + 2e-3 * np.abs(out[0]))
    assert excess.max() > 0, "the stale-position control must exceed the tolerance"


def test_chunk_rejects_bad_shapes():
    w = wl.small("chunk-bad", B=1, Hq=2, Hkv=1, d=64, capacity=128, rope_base=0.0)
    cache = kvc.Cache.from_workload(w, max_chunk=16)
    q, k, v = _suffix(w, 8)
    with pytest.raises(kvc.KvcError) as e:
        cache.chunk(q.cuda(), k.cuda(), v.cuda())   # d=64: not built for the tensor-core path
    assert e.value.code == kvc.KVC_ERR_UNSUPPORTED
    w2 = wl.small("chunk-big", B=1, Hq=2, Hkv=1, d=128, capacity=128, rope_base=0.0)
    c2 = kvc.Cache.from_workload(w2, max_chunk=16)
    q, k, v = _suffix(w2, 32)
    with pytest.raises(kvc.KvcError) as e:
        c2.chunk(q.cuda(), k.cuda(), v.cuda())      # n > max_chunk
    assert e.value.code == kvc.KVC_ERR_ARG


def test_chunk_bf16_outputs_and_longer_prefix():
    # bf16 outputs (the bench's format) over a prefix of several thousand keys, cuts
    # on and off 16-key and 128-key boundaries
    w = wl.small("chunk-long", B=4, Hq=8, Hkv=2, d=128, capacity=4096, rope_base=10000.0, seed=29)
    lengths, cuts, n = [3000, 2500, 4000, 1000], [2048, 1999, 3456, 1], 300
    cache, model = _prefilled(w, lengths, cuts, n)
    q, k, v = _suffix(w, n)
    out = cache.chunk(q.cuda(), k.cuda(), v.cuda())
    assert out.dtype == torch.bfloat16
    ref = model.chunk(host(q), host(k), host(v))
    assert_close(out, ref, "bf16", "chunk bf16 out")
    assert cache.device_status() == 0


def test_chunk_flags_values_beyond_fp16_range():
    # the products take fp16 operands: a value row beyond 65504 is reported in the
    # device error word (bit 2), not silently rounded
    w = wl.small("chunk-range", B=1, Hq=4, Hkv=2, d=128, capacity=256, rope_base=10000.0, seed=5)
    cache, model = _prefilled(w, [64], [64], 32)
    q, k, v = _suffix(w, 32)
    v = v.clone()
    v[0, 5, 1, 7] = 1.0e6
    cache.chunk(q.cuda(), k.cuda(), v.cuda())
    assert cache.device_status() == 4
    assert cache.device_status() == 0          # read and cleared


RING_CASES = [
    # name, capacity W, lengths before, cuts (None = no trim), n, paged
    ("ring-wrapped-no-trim", 256, [600, 300, 257], None, 200, False),
    ("ring-not-full-trim", 256, [200, 130, 40], [77, 130, 0], 300, False),   # the suffix wraps the ring
    ("ring-suffix-longer-than-w", 128, [100, 5, 300], None, 300, False),
    ("ring-paged", 256, [600, 300, 257], None, 200, True),
]


@pytest.mark.parametrize("case", RING_CASES, ids=lambda c: c[0])
def test_ring_chunk_matches_recompute(case):
    # on a ring the suffix rows are staged, attended beside the resident rows, then
    # appended: outputs against the oracle's one-token-at-a-time continuation, and the
    # ring's slots and positions afterwards bit-exact
    name, W, lengths, cuts, n, paged = case
    w = wl.small("chunk-" + name, B=3, Hq=8, Hkv=2, d=128, layout="ring", capacity=W, window=W,
                 rope_base=10000.0, seed=43)
    cache = kvc.Cache.from_workload(w, max_chunk=n, max_position=4096, out_dtype="f32",
                                    page_pool=3 * (W // 16) if paged else 0)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, max(lengths))
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    if cuts is not None:
        cache.trim(cuts)
        model.trim(cuts)
    q, ks, vs = _suffix(w, n)
    out = cache.chunk(q.cuda(), ks.cuda(), vs.cuda())
    ref = model.chunk(host(q), host(ks), host(vs))
    assert_close(out, ref, "bf16", "ring chunk %s" % name)
    check_state(cache, model, w)
    # and the ring keeps decoding from there
    q1, k1, v1 = w.step_qkv(0)
    cache.append(k1.cuda(), v1.cuda())
    model.append(host(k1), host(v1))
    assert_close(cache.decode(q1.cuda()), model.decode(host(q1)), "bf16", "decode after the ring chunk")
    assert cache.device_status() == 0
