"""GPU parity of paged caches: K/V in a pool of 16-slot pages mapped by a per-request
block table ([LEAN] §6.1: the logical view must equal the correct interpretation of the
physical pages; [LOOP] §八 Q1: 16-token pages mapped on demand).

Every case runs the same oracle as the unpaged tests.  The logical export, gathered
through the table, must match bit-exact, and the decode outputs must be within
tolerance.  The pool hands out pages in a shuffled order, so the pages of different
requests interleave.
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


def _step(cache, model, w, q, k, v):
    cache.append(k.cuda(), v.cuda())
    model.append(host(k), host(v))
    out = cache.decode(q.cuda())
    assert_close(out, model.decode(host(q)), w.dtype, "paged decode")
    return out


def _pages_ok(cache, model, w):
    """Mapped pages are distinct; a contiguous cache maps exactly the pages its lengths need."""
    tab = cache.export(kvc.KVC_EXPORT_PAGE_TABLE)
    used = tab[tab >= 0]
    assert len(np.unique(used)) == len(used)
    if w.layout == "contiguous":
        for b in range(model.B):
            need = -(-model.length(b) // 16)
            assert (tab[b, :need] >= 0).all() and (tab[b, need:] < 0).all(), b


CASES = [
    # name, Hq, Hkv, d, layout, capacity, window, rope         (kernel that serves it)
    ("mha-d128", 4, 4, 128, "contiguous", 1024, 0, 0.0),                # bf16 fast decode
    ("gqa4-d128-rope", 8, 2, 128, "contiguous", 1024, 0, 10000.0),    # GQA decode
    ("gqa4-d128-window", 8, 2, 128, "contiguous", 1024, 100, 10000.0),  # GQA, window start off a page
    ("gqa8-d64", 8, 1, 64, "contiguous", 704, 0, 0.0),
    ("ring-gqa4-d128", 8, 2, 128, "ring", 128, 128, 10000.0),
    ("ring-mha-d64", 2, 2, 64, "ring", 304, 304, 10000.0),
    ("mha-d128-window", 4, 4, 128, "contiguous", 1024, 77, 10000.0),   # fast decode, window off a page
    ("gqa2-d96-generic", 4, 2, 96, "contiguous", 608, 0, 500.0),      # generic decode
    ("f32-gqa4-d128", 8, 2, 128, "contiguous", 608, 0, 10000.0),      # generic decode, fp32
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_paged_parity(case):
    name, Hq, Hkv, d, layout, cap, window, rope = case
    dtype = "f32" if name.startswith("f32") else "bf16"
    lengths = [0, 5, 300, 513] if layout == "contiguous" else [0, 5, 300, 129]
    lengths = [min(x, cap - 4) if layout == "contiguous" else x for x in lengths]
    w = wl.small(name, B=4, Hq=Hq, Hkv=Hkv, d=d, layout=layout, capacity=cap, window=window,
                 rope_base=rope, dtype=dtype, seed=23)
    cache = kvc.Cache.from_workload(w, max_position=4096 if layout == "ring" else 0, page_pool=4 * cap // 16)
    model = oracle_for(w)
    n = max(lengths)
    k, v = w.prefill_chunk(0, n)
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    check_state(cache, model, w)
    _pages_ok(cache, model, w)
    for s in range(20):                      # crosses page boundaries on single appends
        _step(cache, model, w, *w.step_qkv(s))
    check_state(cache, model, w)
    _pages_ok(cache, model, w)
    assert cache.device_status() == 0


def test_paged_trim_frees_and_reuses_pages():
    w = wl.small("paged-trim", B=3, Hq=8, Hkv=2, d=128, capacity=512, rope_base=10000.0, seed=31)
    pool = 3 * 400 // 16 + 2                # barely enough for the prefill
    cache = kvc.Cache.from_workload(w, page_pool=pool)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, 400)
    cache.append_rows(k.cuda(), v.cuda(), counts=[400, 260, 17])
    model.append_rows(host(k), host(v), [400, 260, 17])
    _pages_ok(cache, model, w)
    cuts = [123, 260, 0]
    cache.trim(cuts)
    model.trim(cuts)
    check_state(cache, model, w)
    _pages_ok(cache, model, w)               # pages past the cuts returned to the pool
    for s in range(30):
        _step(cache, model, w, *w.step_qkv(100 + s))
    check_state(cache, model, w)
    _pages_ok(cache, model, w)


def test_paged_pool_exhaustion_changes_nothing():
    w = wl.small("paged-full", B=2, Hq=4, Hkv=4, d=64, capacity=256, rope_base=0.0, seed=3)
    cache = kvc.Cache.from_workload(w, page_pool=3)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, 32)
    cache.append_rows(k.cuda(), v.cuda(), counts=[32, 16])     # 2 + 1 pages
    model.append_rows(host(k), host(v), [32, 16])
    q, k1, v1 = w.step_qkv(0)
    with pytest.raises(kvc.KvcError) as e:
        cache.append(k1.cuda(), v1.cuda())                     # both requests need a new page
    assert e.value.code == kvc.KVC_ERR_CAPACITY
    assert list(cache.next_positions()) == [32, 16]
    check_state(cache, model, w)
    cache.trim([16, 0])                                        # frees one page of each request
    model.trim([16, 0])
    _step(cache, model, w, q, k1, v1)
    check_state(cache, model, w)


def test_paged_ring_phases_every_step():
    w = wl.small("paged-ring", B=2, Hq=4, Hkv=2, d=128, layout="ring", capacity=32, window=32,
                 rope_base=10000.0, seed=5)
    cache = kvc.Cache.from_workload(w, max_position=128, page_pool=4)
    model = oracle_for(w)
    for s in range(80):                                        # not full, full, replacing
        _step(cache, model, w, *w.step_qkv(s))
        if s % 7 == 0:
            check_state(cache, model, w)
    tab = cache.export(kvc.KVC_EXPORT_PAGE_TABLE)
    assert (tab >= 0).all() and len(np.unique(tab)) == 4       # a full ring holds its two pages


def test_paged_chunk_maps_its_pages():
    # the chunk's suffix rows take pages from the pool like any append (its attention reads
    # them through the block table: parity in test_gpu_chunk.py); a pool too small refuses
    # the call before anything changes
    w = wl.small("paged-chunk", B=1, Hq=8, Hkv=2, d=128, capacity=256, rope_base=10000.0, seed=3)
    cache = kvc.Cache.from_workload(w, max_chunk=32, page_pool=2)
    q = torch.zeros((1, 20, 8, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, 20, 2, 128), dtype=torch.bfloat16, device="cuda")
    cache.chunk(q, kv, kv)
    tab = cache.export(kvc.KVC_EXPORT_PAGE_TABLE)[0]
    assert (tab[:2] >= 0).all() and (tab[2:] == -1).all()         # positions 0..19: two pages
    q2 = torch.zeros((1, 32, 8, 128), dtype=torch.bfloat16, device="cuda")
    kv2 = torch.zeros((1, 32, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        cache.chunk(q2, kv2, kv2)                                   # positions 20..51 need two more pages
    assert e.value.code == kvc.KVC_ERR_CAPACITY
    assert list(cache.next_positions()) == [20]
    assert cache.device_status() == 0
