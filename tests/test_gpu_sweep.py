"""Seeded random sweeps of the GPU path against the CPU oracle: shapes, layouts, windows,
paging, lengths and split lengths drawn at random (every draw respects the configuration's
documented limits), so that combinations no hand-written case names still meet the same
bar: cache state bit-exact, outputs within the stated tolerance, the INT8 bound sound.

Each sweep's cases are fixed by their seed; a failing case prints its draw.
"""
import numpy as np
import pytest
import torch

from kv_cache_decode_ring_gb300 import kvc
from kv_cache_decode_ring_gb300 import workloads as wl

from _parity import assert_close, check_state, host, oracle_for
from test_gpu_int8 import check_decode_window, check_int8_ring_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_decode_ring_gb300 import build
    build.build()
    torch.cuda.init()


def _pick(rng, xs, p=None):
    return xs[int(rng.choice(len(xs), p=p))]


# ---- bf16 / fp32 decode ---------------------------------------------------------------
def decode_draw(seed):
    rng = np.random.default_rng(7000 + seed)
    dtype = _pick(rng, ["bf16", "f32"], [0.7, 0.3])
    d = _pick(rng, [128, 64, 96, 32], [0.4, 0.3, 0.15, 0.15])
    g = _pick(rng, [1, 2, 4, 8])
    Hkv = _pick(rng, [1, 2, 3])
    layout = _pick(rng, ["contiguous", "ring"])
    paged = bool(rng.random() < 0.35)
    rope = _pick(rng, [0.0, 10000.0])
    B = int(rng.integers(1, 5))
    if layout == "ring":
        W = 16 * int(rng.integers(1, 9)) if paged else int(rng.integers(3, 130))
        cap, window = W, W
        lengths = [int(x) for x in rng.integers(1, 3 * W, B)]
    else:
        cap = 16 * int(rng.integers(4, 40)) if paged else int(rng.integers(40, 640))
        window = 0 if rng.random() < 0.5 else int(rng.integers(1, cap))
        lengths = [int(x) for x in rng.integers(1, cap - 3, B)]
    return dict(dtype=dtype, d=d, Hq=g * Hkv, Hkv=Hkv, layout=layout, paged=paged, rope=rope, B=B, cap=cap,
                window=window, lengths=lengths)


@pytest.mark.parametrize("seed", range(24))
def test_decode_sweep(seed):
    c = decode_draw(seed)
    print(c)
    w = wl.small("sweep-decode-%d" % seed, B=c["B"], Hq=c["Hq"], Hkv=c["Hkv"], d=c["d"], layout=c["layout"],
                 capacity=c["cap"], window=c["window"], rope_base=c["rope"], dtype=c["dtype"], seed=seed)
    ring = c["layout"] == "ring"
    cache = kvc.Cache.from_workload(w, max_position=1024 if ring else 0,
                                    page_pool=c["B"] * (c["cap"] // 16) if c["paged"] else 0)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, max(c["lengths"]))
    cache.append_rows(k.cuda(), v.cuda(), counts=c["lengths"])
    model.append_rows(host(k), host(v), c["lengths"])
    for s in range(3):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        assert_close(cache.decode(q.cuda()), model.decode(host(q)), c["dtype"], "sweep decode %d step %d" % (seed, s))
    check_state(cache, model, w)
    assert cache.device_status() == 0


# ---- INT8 tiers --------------------------------------------------------------------------
def int8_draw(seed):
    rng = np.random.default_rng(8000 + seed)
    quant = _pick(rng, ["int8", "int8-dither"], [0.7, 0.3])
    d = _pick(rng, [128, 64])
    g = _pick(rng, [1, 2, 4, 8])
    Hkv = _pick(rng, [1, 2])
    layout = _pick(rng, ["contiguous", "ring"])
    paged = bool(rng.random() < 0.35)
    B = int(rng.integers(1, 4))
    split = 0 if rng.random() < 0.4 else 64 * int(rng.integers(16, 33))
    if layout == "ring":
        cap = 16 * int(rng.integers(2, 64))
        window = cap
        lengths = [int(x) for x in rng.integers(1, 3 * cap, B)]
    else:
        cap = 16 * int(rng.integers(8, 200))
        window = 0 if rng.random() < 0.5 else int(rng.integers(1, cap))
        lengths = [int(x) for x in rng.integers(1, cap - 3, B)]
    return dict(quant=quant, d=d, Hq=g * Hkv, Hkv=Hkv, layout=layout, paged=paged, B=B, split=split, cap=cap,
                window=window, lengths=lengths)


@pytest.mark.parametrize("seed", range(20))
def test_int8_sweep(seed):
    c = int8_draw(seed)
    print(c)
    extra = {"outliers": (4, 20.0)}
    if c["quant"] == "int8-dither":
        extra.update(dither_key=(0x9E3779B9 ^ seed, 0x7F4A7C15), layer=seed % 5)
    ring = c["layout"] == "ring"
    w = wl.small("sweep-int8-%d" % seed, B=c["B"], Hq=c["Hq"], Hkv=c["Hkv"], d=c["d"], layout=c["layout"],
                 capacity=c["cap"], window=c["window"], rope_base=10000.0, quant=c["quant"], seed=seed, **extra)
    cache = kvc.Cache.from_workload(w, max_position=4096 if ring else 0, out_dtype="f32", int8_split=c["split"],
                                    page_pool=c["B"] * (c["cap"] // 16) if c["paged"] else 0)
    model = oracle_for(w)                    # (with the dither key and layer of Tier B)
    k, v = w.prefill_chunk(0, max(c["lengths"]))
    cache.append_rows(k.cuda(), v.cuda(), counts=c["lengths"])
    model.append_rows(host(k), host(v), c["lengths"])
    for s in range(3):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        check_decode_window(cache, model, q, ring)
    check_int8_ring_state(cache, model)       # (a contiguous cache's blocks are its first S/16)
    assert cache.device_status() == 0


# ---- chunked suffix attention ---------------------------------------------------------------
def chunk_draw(seed):
    rng = np.random.default_rng(9000 + seed)
    g = _pick(rng, [1, 2, 3, 4])
    Hkv = _pick(rng, [1, 2])
    layout = _pick(rng, ["contiguous", "ring"], [0.6, 0.4])
    paged = bool(rng.random() < 0.35)
    B = int(rng.integers(1, 4))
    n = int(rng.integers(1, 260))
    if layout == "ring":
        cap = 16 * int(rng.integers(4, 40))
        window = cap
        lengths = [int(x) for x in rng.integers(0, 2 * cap, B)]
        # a ring trim keeps what the next query needs: any cut while the ring is not full,
        # else the length or one less
        cuts = [int(rng.integers(0, L + 1)) if L < cap else L - int(rng.integers(0, 2)) for L in lengths]
    else:
        cap = (16 * int(rng.integers(8, 60))) if paged else int(rng.integers(100, 1000))
        window = 0 if rng.random() < 0.5 else int(rng.integers(1, min(700, cap)))
        lengths = [int(x) for x in rng.integers(0, cap - n + 1, B)]
        cuts = [int(rng.integers(0, L + 1)) for L in lengths]
    return dict(Hq=g * Hkv, Hkv=Hkv, layout=layout, paged=paged, B=B, n=n, cap=cap, window=window,
                lengths=lengths, cuts=cuts)


@pytest.mark.parametrize("seed", range(16))
def test_chunk_sweep(seed):
    c = chunk_draw(seed)
    print(c)
    ring = c["layout"] == "ring"
    w = wl.small("sweep-chunk-%d" % seed, B=c["B"], Hq=c["Hq"], Hkv=c["Hkv"], d=128, layout=c["layout"],
                 capacity=c["cap"], window=c["window"], rope_base=10000.0, seed=seed)
    pool = c["B"] * (c["cap"] // 16) if c["paged"] else 0
    cache = kvc.Cache.from_workload(w, max_chunk=c["n"], max_position=4096 if ring else 0, out_dtype="f32",
                                    page_pool=pool)
    model = oracle_for(w)
    if max(c["lengths"]) > 0:
        k, v = w.prefill_chunk(0, max(c["lengths"]))
        cache.append_rows(k.cuda(), v.cuda(), counts=c["lengths"])
        model.append_rows(host(k), host(v), c["lengths"])
    cache.trim(c["cuts"])
    model.trim(c["cuts"])
    B, n, Hq, Hkv = c["B"], c["n"], c["Hq"], c["Hkv"]
    q = w.queries((B, n, Hq, 128), "sweep")
    ks = w.keys((B, n, Hkv, 128), "sweep")
    vs = w.values((B, n, Hkv, 128), "sweep")
    out = cache.chunk(q.cuda(), ks.cuda(), vs.cuda())
    assert_close(out, model.chunk(host(q), host(ks), host(vs)), "bf16", "sweep chunk %d" % seed)
    check_state(cache, model, w)
    assert list(cache.next_positions()) == [x + n for x in c["cuts"]]
    assert cache.device_status() == 0
