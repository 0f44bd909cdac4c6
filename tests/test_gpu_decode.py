"""GPU parity of append, decode attention and trim through the C ABI against the oracle.

Cache contents, positions and next_position are compared bit-exact after every
mutation; attention outputs within 1e-5 (fp32) or 2e-3 (bf16), relative and absolute.
"""
import numpy as np
import pytest
import torch

from kv_cache_decode_ring_gb300 import kvc
from kv_cache_decode_ring_gb300 import workloads as wl

from _parity import assert_close, check_state, host, oracle_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_decode_ring_gb300 import build
    build.build()
    torch.cuda.init()


def _step(cache, model, w, q, k, v, check=True):
    cache.append(k.cuda(), v.cuda())
    model.append(host(k), host(v))
    out = cache.decode(q.cuda())
    ref = model.decode(host(q))
    assert_close(out, ref, w.dtype, "decode")
    if check:
        check_state(cache, model, w)
    return out


@pytest.mark.parametrize("variant", ["full", "ring"])
def test_toy_fp32_every_step(variant):
    # toy workload: B=1, H=2, d=4, fp32, seed 7, 64 steps; full cache or ring W=4 through
    # the not-full, exactly-full and first-replacement phases
    w = wl.toy(variant)
    cache = kvc.Cache.from_workload(w)
    model = oracle_for(w)
    for s in range(64):
        q, k, v = w.step_qkv(s)
        out = _step(cache, model, w, q, k, v)
        if s == 0:
            assert torch.equal(out.cpu()[0], v[0])            # one key: the output is v_0
    assert cache.device_status() == 0


def test_toy_fp32_trim_and_continue():
    # 8-token history, trim at cut=4, continue with 8 new tokens from next_position=4
    w = wl.toy("trim")
    hist, cut, n = w.extra["history"], w.extra["cut"], w.extra["suffix"]
    cache = kvc.Cache.from_workload(w)
    model = oracle_for(w)
    for s in range(hist):
        _step(cache, model, w, *w.step_qkv(s))
    cache.trim([cut])
    model.trim([cut])
    check_state(cache, model, w)
    assert cache.next_positions()[0] == cut
    for s in range(hist, hist + n):
        _step(cache, model, w, *w.step_qkv(s))
    pos = cache.export(kvc.KVC_EXPORT_POSITIONS)[0]
    assert np.array_equal(pos[:cut + n], np.arange(cut + n)) and np.all(pos[cut + n:] == -1)


CASES = [
    # name, Hq, Hkv, d, layout, capacity, window, rope
    ("mha-d128", 4, 4, 128, "contiguous", 1024, 0, 0.0),
    ("gqa4-d128-rope", 8, 2, 128, "contiguous", 1024, 0, 10000.0),
    ("gqa4-d128-window", 8, 2, 128, "contiguous", 1024, 100, 10000.0),
    ("gqa8-d64", 8, 1, 64, "contiguous", 700, 0, 0.0),
    ("ring-gqa4-d128", 8, 2, 128, "ring", 128, 128, 10000.0),
    ("ring-mha-d64", 2, 2, 64, "ring", 300, 300, 10000.0),
    ("gqa2-d96-generic", 4, 2, 96, "contiguous", 600, 0, 500.0),
    ("f32-gqa4-d128", 8, 2, 128, "contiguous", 600, 0, 10000.0),
]

# GQA decode splits of 1024 keys (2048 once a request may attend to 16384 keys): lengths
# that span several splits and end inside one, and a window that starts inside a split
LONG_CASES = [
    # name, Hq, Hkv, d, capacity, window, lengths
    ("gqa4-d128-3splits", 8, 2, 128, 3200, 0, [1, 1023, 1025, 3100]),
    ("gqa8-d64-window", 8, 1, 64, 3200, 1500, [700, 3000, 2049, 1500]),
    ("gqa4-d128-long-split", 8, 2, 128, 16400, 0, [2047, 2049, 6000, 16390]),
]


@pytest.mark.parametrize("case", LONG_CASES, ids=lambda c: c[0])
def test_gqa_split_parity(case):
    name, Hq, Hkv, d, cap, window, lengths = case
    w = wl.small(name, B=4, Hq=Hq, Hkv=Hkv, d=d, capacity=cap, window=window, rope_base=10000.0, seed=41)
    cache = kvc.Cache.from_workload(w)
    model = oracle_for(w)
    for c0 in range(0, max(lengths), 4096):                  # prefill in chunks
        n = min(4096, max(lengths) - c0)
        k, v = w.prefill_chunk(c0 // 4096, n)
        counts = [max(0, min(n, x - c0)) for x in lengths]
        cache.append_rows(k.cuda(), v.cuda(), counts=counts)
        model.append_rows(host(k), host(v), counts)
    for s in range(2):
        _step(cache, model, w, *w.step_qkv(s))
    check_state(cache, model, w)
    assert cache.device_status() == 0


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_small_parity(case):
    name, Hq, Hkv, d, layout, cap, window, rope = case
    dtype = "f32" if name.startswith("f32") else "bf16"
    lengths = [0, 5, 300, 513] if layout == "contiguous" else [0, 5, 300, 129]
    lengths = [min(x, cap - 4) if layout == "contiguous" else x for x in lengths]
    w = wl.small(name, B=4, Hq=Hq, Hkv=Hkv, d=d, layout=layout, capacity=cap, window=window,
                 rope_base=rope, dtype=dtype, seed=23)
    cache = kvc.Cache.from_workload(w, max_position=4096 if layout == "ring" else 0)
    model = oracle_for(w)
    n = max(lengths)
    k, v = w.prefill_chunk(0, n)
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    check_state(cache, model, w)
    for s in range(3):
        _step(cache, model, w, *w.step_qkv(s))
    assert cache.device_status() == 0


def test_ring_phases_bf16_every_step():
    w = wl.small("ring8", B=2, Hq=4, Hkv=2, d=128, layout="ring", capacity=8, window=8,
                 rope_base=10000.0, seed=5)
    cache = kvc.Cache.from_workload(w, max_position=64)
    model = oracle_for(w)
    for s in range(40):
        _step(cache, model, w, *w.step_qkv(s))
        # slot s holds the newest position congruent to s mod W (ringToList = lastWindow)
        pos = cache.export(kvc.KVC_EXPORT_POSITIONS)[0]
        for slot in range(8):
            assert pos[slot] == max((p for p in range(s + 1) if p % 8 == slot), default=-1)


def test_trim_and_continue_bf16():
    w = wl.small("trim", B=3, Hq=8, Hkv=2, d=128, capacity=512, rope_base=10000.0, seed=31)
    cache = kvc.Cache.from_workload(w)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, 400)
    cache.append_rows(k.cuda(), v.cuda(), counts=[400, 260, 17])
    model.append_rows(host(k), host(v), [400, 260, 17])
    cuts = [123, 260, 0]
    cache.trim(cuts)
    model.trim(cuts)
    check_state(cache, model, w)
    for s in range(4):
        _step(cache, model, w, *w.step_qkv(100 + s))


def test_ring_trim_rules_on_device():
    w = wl.small("ringtrim", B=1, Hq=2, Hkv=1, d=64, layout="ring", capacity=16, window=16,
                 rope_base=10000.0, seed=3)
    cache = kvc.Cache.from_workload(w, max_position=256)
    model = oracle_for(w)
    for s in range(40):
        _step(cache, model, w, *w.step_qkv(s), check=False)
    with pytest.raises(kvc.KvcError) as e:
        cache.trim([20])                          # positions 5..19 were overwritten
    assert e.value.code == kvc.KVC_ERR_EVICTED
    check_state(cache, model, w)                  # a refused trim changes nothing
    with pytest.raises(kvc.KvcError) as e:
        cache.trim([35])                          # needs 20..34, the ring holds 24..39
    assert e.value.code == kvc.KVC_ERR_EVICTED
    cache.trim([39])                              # needs 24..38: all resident
    model.trim([39])
    check_state(cache, model, w)
    with pytest.raises(kvc.KvcError) as e:        # a ring must append before decoding again
        cache.decode(w.step_qkv(0)[0].cuda())
    assert e.value.code == kvc.KVC_ERR_ARG
    for s in range(40, 60):
        _step(cache, model, w, *w.step_qkv(s))


def test_capacity_and_argument_errors():
    w = wl.small("cap", B=2, Hq=2, Hkv=2, d=64, capacity=3, rope_base=0.0)
    cache = kvc.Cache.from_workload(w)
    for s in range(3):
        q, k, v = w.step_qkv(s)
        cache.append(k.cuda(), v.cuda())
    with pytest.raises(kvc.KvcError) as e:
        cache.append(k.cuda(), v.cuda())          # position 3 >= max_seq_len 3
    assert e.value.code == kvc.KVC_ERR_CAPACITY
    assert list(cache.next_positions()) == [3, 3]
    with pytest.raises(kvc.KvcError) as e:
        cache.trim([4, 0])                        # cut beyond next_position
    assert e.value.code == kvc.KVC_ERR_ARG
    empty = kvc.Cache.from_workload(w)
    with pytest.raises(kvc.KvcError):
        empty.decode(q.cuda())                    # nothing cached yet
    with pytest.raises(ValueError):
        cache.decode(q.cuda().float())            # wrong dtype caught by the binding
    assert cache.device_status() == 0


STRICT_CASES = [CASES[0], ("gqa2-d128", 8, 4, 128, "contiguous", 1024, 0, 10000.0), CASES[1], CASES[4], CASES[3],
                CASES[6]]


@pytest.mark.parametrize("case", STRICT_CASES, ids=lambda c: c[0] + "-out-f32")
def test_f32_outputs_strict_tolerance(case):
    # bf16 cache, fp32 outputs: no output rounding, so the plain 2e-3 bound applies; one
    # case for every bf16 decode kernel (g = 1 and 2 at d = 128: the bulk-copy kernel; g = 4
    # and 8: the tensor-copy kernel; ring; the generic kernel at d = 96)
    name, Hq, Hkv, d, layout, cap, window, rope = case
    w = wl.small(name, B=3, Hq=Hq, Hkv=Hkv, d=d, layout=layout, capacity=cap, window=window,
                 rope_base=rope, seed=41)
    cache = kvc.Cache.from_workload(w, max_position=4096 if layout == "ring" else 0, out_dtype="f32")
    model = oracle_for(w)
    lengths = [1, 200, 390]
    k, v = w.prefill_chunk(0, max(lengths))
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    for s in range(2):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        out = cache.decode(q.cuda())
        assert out.dtype == torch.float32
        assert_close(out, model.decode(host(q)), "bf16", "decode f32 out")


@pytest.mark.parametrize("dtype,Hq,d", [("f32", 64, 256), ("bf16", 160, 96)], ids=["f32-g64-d256", "bf16-g160-d96"])
def test_generic_decode_beyond_48kb_shared_memory(dtype, Hq, d):
    # the generic kernel keeps g queries and g x 64 scores per CTA in shared memory: 80 KB
    # (fp32, g = 64, d = 256) and 100 KB (bf16, g = 160, d = 96), above the 48 KB default
    w = wl.small("generic-smem-%s" % dtype, B=2, Hq=Hq, Hkv=1, d=d, capacity=200, rope_base=10000.0,
                 dtype=dtype, seed=19)
    cache = kvc.Cache.from_workload(w)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, 150)
    cache.append_rows(k.cuda(), v.cuda(), counts=[150, 70])
    model.append_rows(host(k), host(v), [150, 70])
    for s in range(2):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        assert_close(cache.decode(q.cuda()), model.decode(host(q)), dtype, "generic smem decode step %d" % s)
    assert cache.device_status() == 0
