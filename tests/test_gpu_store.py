"""GPU parity of the prefix store: saved prefills, lookup and copy on reuse.

[PREFIX] "LLM 機制實驗（五）：改了歷史，能否只重算變化的後綴？": the store keeps prefills
keyed by token IDs, scope and signature; a query reuses the longest contiguous common
prefix (ties to the newest entry), copying the kept K, V and positions before the
suffix is computed ("查詢流程與快取所有權"); the nine conditions of "27 例得到的計算量與誤差"
over seeds 7, 11 and 23.  The continued cache must hold, bit for bit, the rows of a full
recompute, and every output must match the oracle.
"""
import numpy as np
import pytest
import torch

from kv_cache_decode_ring_gb300 import kvc
from kv_cache_decode_ring_gb300 import workloads as wl

from _parity import assert_close, check_state, host, oracle_for
from _store_cases import BRANCH, PLAIN, SCOPE, SEEDS, SIGNATURE, VOCAB, read_matrix, rows_of, toy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_decode_ring_gb300 import build
    build.build()
    torch.cuda.init()


def _cache(w, store_slots=2, **kw):
    return kvc.Cache.from_workload(w, max_position=256 if w.layout == "ring" else 0, store_slots=store_slots, **kw)


def _prefill(cache, model, table, ids, b=0):
    """Request b (of a one-request cache) takes the rows of ``ids`` from position 0."""
    q, k, v = rows_of(table, ids)
    cache.append_rows(k.cuda(), v.cuda())
    model.append_rows(host(k), host(v), [len(ids)])


def _continue(cache, model, w, table, ids, start):
    """Append ids[start:] one token at a time; every query's output, checked against the oracle."""
    q, k, v = rows_of(table, ids)
    outs = []
    for i in range(start, len(ids)):
        ki, vi, qi = k[:, :, i].contiguous(), v[:, :, i].contiguous(), q[i][None].contiguous()
        cache.append(ki.cuda(), vi.cuda())
        model.append(host(ki), host(vi))
        out = cache.decode(qi.cuda())
        assert_close(out, model.decode(host(qi)), w.dtype, "token %d" % i)
        outs.append(out.cpu())
    return torch.stack(outs) if outs else None


@pytest.mark.parametrize("seed", SEEDS)
@pytest.mark.parametrize("case", read_matrix(), ids=lambda c: c["name"])
def test_store_matrix(case, seed):
    w = toy(seed, case["ring"])
    table = w.token_table(VOCAB)
    cache, model = _cache(w), oracle_for(w)
    store = kvc.PrefixStore(cache.cfg, 2)
    slots = {}
    for name, ids in (("plain", PLAIN), ("branch", BRANCH)):
        cache.store_load(-1, 0, 0)                          # an empty request
        model.load(0, None, 0)
        _prefill(cache, model, table, ids)
        slots[name] = cache.save_prefix(store, 0, ids, SCOPE, SIGNATURE)
    snaps = {}
    # the oracle's own snapshots of the two prefills
    for name, ids in (("plain", PLAIN), ("branch", BRANCH)):
        m = oracle_for(w)
        m.append_rows(*(host(x) for x in rows_of(table, ids)[1:]), [len(ids)])
        snaps[slots[name]] = m.snapshot(0)
    ids = case["ids"]
    slot, cut = cache.reuse_prefix(store, 0, ids, case["scope"], SIGNATURE)
    assert cut == case["cut"]
    assert slot == (-1 if case["entry"] is None else slots[case["entry"]])
    assert case["proj"] == 6 * (len(ids) - cut)
    model.load(0, snaps.get(slot), cut)
    check_state(cache, model, w)
    got = _continue(cache, model, w, table, ids, cut)
    check_state(cache, model, w)
    # the full recompute on the GPU: same rows, same outputs, bit for bit
    full, fm = _cache(w, store_slots=0), oracle_for(w)
    ref = _continue(full, fm, w, table, ids, 0)
    assert torch.equal(got, ref[cut:])
    for which in (kvc.KVC_EXPORT_POSITIONS, kvc.KVC_EXPORT_NEXT_POSITION):
        assert np.array_equal(cache.export(which), full.export(which))
    live = cache.export(kvc.KVC_EXPORT_POSITIONS)[0] >= 0      # slots past the cut are dead, as after a trim
    for which in (kvc.KVC_EXPORT_K, kvc.KVC_EXPORT_V):
        assert np.array_equal(cache.export(which)[:, :, live].view(np.uint32),
                              full.export(which)[:, :, live].view(np.uint32))
    assert cache.device_status() == 0
    store.close()


def test_store_reuse_then_chunk():
    """Two stored prefills; each request reuses a different one, then a 48-row chunk."""
    w = wl.small("store-gqa", B=2, Hq=8, Hkv=2, d=128, capacity=1024, rope_base=10000.0, seed=29)
    vocab = 512
    table = w.token_table(vocab)
    rng = np.random.default_rng(3)
    pre_a = [int(x) for x in rng.integers(0, vocab, 300)]
    pre_b = pre_a[:120] + [int(x) for x in rng.integers(0, vocab, 180)]
    cache = kvc.Cache.from_workload(w, max_chunk=64, store_slots=2)
    store = kvc.PrefixStore(cache.cfg, 2)
    for ids in (pre_a, pre_b):
        q, k, v = rows_of(table, ids)                       # [1, Hkv, n, d] -> both requests
        cache.store_load(-1, 0, 0)
        cache.store_load(-1, 1, 0)
        cache.append_rows(k.expand(2, -1, -1, -1).contiguous().cuda(), v.expand(2, -1, -1, -1).contiguous().cuda(),
                          counts=[len(ids), 0])
        cache.save_prefix(store, 0, ids, "s", b"w")
    n = 48
    fresh = [int(x) for x in rng.integers(0, vocab, n)]
    queries = [pre_a[:200] + fresh, pre_b[:250] + fresh]     # cut 200 from a, 250 from b
    cuts = []
    for b, ids in enumerate(queries):
        slot, cut = cache.reuse_prefix(store, b, ids, "s", b"w")
        cuts.append(cut)
    assert cuts == [200, 250]
    assert list(cache.next_positions()) == cuts
    # the oracle: each request holds exactly the rows of its reused prefix
    model = oracle_for(w)
    for b, ids in enumerate(queries):
        _, k, v = rows_of(table, ids[:cuts[b]])
        counts = [0, 0]
        counts[b] = cuts[b]
        kk = torch.zeros((2,) + tuple(k.shape[1:]), dtype=k.dtype); kk[b] = k[0]
        vv = torch.zeros_like(kk); vv[b] = v[0]
        model.append_rows(host(kk), host(vv), counts)
    check_state(cache, model, w)
    qs = torch.stack([table[0][ids[cuts[b]:]] for b, ids in enumerate(queries)])        # [2, n, Hq, d]
    ks = torch.stack([table[1][ids[cuts[b]:]] for b, ids in enumerate(queries)])
    vs = torch.stack([table[2][ids[cuts[b]:]] for b, ids in enumerate(queries)])
    out = cache.chunk(qs.cuda(), ks.cuda(), vs.cuda())
    ref = model.chunk(host(qs), host(ks), host(vs))
    assert_close(out, ref, w.dtype, "chunk after reuse")
    check_state(cache, model, w)
    store.close()


def test_store_copy_is_private_and_paged_load():
    """Appending after a load never changes the stored rows; a paged cache loads through its pages."""
    w = wl.small("store-paged", B=3, Hq=4, Hkv=2, d=128, capacity=512, rope_base=10000.0, seed=17)
    cache = kvc.Cache.from_workload(w, store_slots=1, page_pool=3 * 512 // 16)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, 300)
    cache.append_rows(k.cuda(), v.cuda(), counts=[300, 40, 0])
    model.append_rows(host(k), host(v), [300, 40, 0])
    cache.store_save(0, 0, 300)
    snap = model.snapshot(0)
    for cut, b in ((137, 0), (300, 2), (64, 1)):            # request 0 overwrites its own rows first
        cache.store_load(0, b, cut)
        model.load(b, snap, cut)
        check_state(cache, model, w)
        for s in range(5):                                   # continue every request
            q, k1, v1 = w.step_qkv(40 * b + s)
            cache.append(k1.cuda(), v1.cuda())
            model.append(host(k1), host(v1))
            assert_close(cache.decode(q.cuda()), model.decode(host(q)), w.dtype, "paged decode after load")
        check_state(cache, model, w)
    tab = cache.export(kvc.KVC_EXPORT_PAGE_TABLE)
    used = tab[tab >= 0]
    assert len(np.unique(used)) == len(used)
    for b in range(3):
        need = -(-model.length(b) // 16)
        assert (tab[b, :need] >= 0).all() and (tab[b, need:] < 0).all()
    assert cache.device_status() == 0


def test_store_ring_load_keeps_the_resident_rows():
    w = wl.small("store-ring", B=2, Hq=4, Hkv=2, d=64, layout="ring", capacity=64, window=64,
                 rope_base=10000.0, seed=5)
    cache = _cache(w)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, 150)
    cache.append_rows(k.cuda(), v.cuda(), counts=[150, 20])
    model.append_rows(host(k), host(v), [150, 20])
    cache.store_save(1, 0, 150)
    snap = model.snapshot(0)
    with pytest.raises(kvc.KvcError) as e:
        cache.store_load(1, 1, 100)                          # the token at 100 needs position 37: evicted
    assert e.value.code == kvc.KVC_ERR_EVICTED
    with pytest.raises(kvc.KvcError) as e:
        cache.store_load(1, 1, 148)                          # needs 85: the slot holds 86 .. 149
    assert e.value.code == kvc.KVC_ERR_EVICTED
    cache.store_load(1, 1, 149)                              # needs 86 .. 148: resident
    model.load(1, snap, 149)
    check_state(cache, model, w)
    for s in range(70):                                      # across a full turn of the ring
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        assert_close(cache.decode(q.cuda()), model.decode(host(q)), w.dtype, "ring after load")
    check_state(cache, model, w)


def test_store_errors_change_nothing():
    w = wl.small("store-err", B=2, Hq=4, Hkv=2, d=128, capacity=64, rope_base=0.0, seed=2)
    plain = kvc.Cache.from_workload(w)
    with pytest.raises(kvc.KvcError) as e:
        plain.store_save(0, 0, 1)
    assert e.value.code == kvc.KVC_ERR_UNSUPPORTED
    cache = _cache(w, store_slots=2)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, 40)
    cache.append_rows(k.cuda(), v.cuda(), counts=[40, 12])
    model.append_rows(host(k), host(v), [40, 12])
    bad = [lambda: cache.store_save(0, 0, 39),              # n must be the request's length
           lambda: cache.store_save(2, 0, 40),              # no such slot
           lambda: cache.store_load(1, 0, 0),               # slot 1 holds nothing
           lambda: cache.store_load(-1, 0, 5),              # an empty load continues from 0
           lambda: cache.store_load(0, 2, 0)]               # no such request
    for f in bad:
        with pytest.raises(kvc.KvcError) as e:
            f()
        assert e.value.code == kvc.KVC_ERR_ARG
    cache.store_save(0, 1, 12)
    with pytest.raises(kvc.KvcError) as e:
        cache.store_load(0, 0, 13)                           # beyond the saved rows
    assert e.value.code == kvc.KVC_ERR_ARG
    check_state(cache, model, w)
    # a paged cache without pages for the load refuses it and keeps its state
    pw = wl.small("store-err-paged", B=2, Hq=4, Hkv=2, d=128, capacity=64, rope_base=0.0, seed=2)
    pc = kvc.Cache.from_workload(pw, store_slots=1, page_pool=5)
    pm = oracle_for(pw)
    k, v = pw.prefill_chunk(0, 48)
    pc.append_rows(k.cuda(), v.cuda(), counts=[48, 16])    # 3 + 1 pages of 5
    pm.append_rows(host(k), host(v), [48, 16])
    pc.store_save(0, 0, 48)
    with pytest.raises(kvc.KvcError) as e:
        pc.store_load(0, 1, 48)                              # needs 3 pages, has 1 + 1 free
    assert e.value.code == kvc.KVC_ERR_CAPACITY
    check_state(pc, pm, pw)
    pc.store_load(0, 1, 32)                                  # 2 pages: fits
    pm.load(1, pm.snapshot(0), 32)
    check_state(pc, pm, pw)


@pytest.mark.parametrize("paged", [False, True])
def test_store_load_batch(paged):
    """One batched load equals the single loads; a bad entry anywhere changes nothing."""
    w = wl.small("store-batch", B=4, Hq=8, Hkv=2, d=64, capacity=256, rope_base=10000.0, seed=41)
    cache = kvc.Cache.from_workload(w, store_slots=2, page_pool=4 * 256 // 16 if paged else 0)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, 200)
    cache.append_rows(k.cuda(), v.cuda(), counts=[200, 77, 5, 130])
    model.append_rows(host(k), host(v), [200, 77, 5, 130])
    cache.store_save(0, 0, 200)
    cache.store_save(1, 3, 130)
    snaps = {0: model.snapshot(0), 1: model.snapshot(3)}
    with pytest.raises(kvc.KvcError) as e:
        cache.store_load_batch([0, 1], [2, 2], [10, 10])     # one request twice
    assert e.value.code == kvc.KVC_ERR_ARG
    with pytest.raises(kvc.KvcError) as e:
        cache.store_load_batch([0, 1], [1, 2], [10, 131])    # the second is past slot 1's rows
    assert e.value.code == kvc.KVC_ERR_ARG
    check_state(cache, model, w)
    loads = [(1, 0, 129), (-1, 1, 0), (0, 2, 200), (0, 3, 17)]
    cache.store_load_batch(*zip(*loads))
    for slot, b, cut in loads:
        model.load(b, snaps.get(slot), cut)
    check_state(cache, model, w)
    for s in range(3):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        assert_close(cache.decode(q.cuda()), model.decode(host(q)), w.dtype, "decode after batched load")
    check_state(cache, model, w)
    assert cache.device_status() == 0


@pytest.mark.parametrize("dtype,d", [("bf16", 6), ("bf16", 96), ("f32", 256)], ids=["12B-rows", "192B-rows", "1KB-rows"])
def test_store_row_widths(dtype, d):
    """Rows that are not 16-byte multiples (copied by words), and rows of 192 and 1024 bytes
    (copied through shared memory in runs): a save and loads whose cuts end inside, at and
    past a 64-row run."""
    w = wl.small("store-rows-%s-%d" % (dtype, d), B=3, Hq=4, Hkv=2, d=d, capacity=320, rope_base=10000.0,
                 dtype=dtype, seed=43)
    cache = kvc.Cache.from_workload(w, store_slots=1)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, 300)
    cache.append_rows(k.cuda(), v.cuda(), counts=[300, 3, 70])
    model.append_rows(host(k), host(v), [300, 3, 70])
    cache.store_save(0, 0, 300)
    snap = model.snapshot(0)
    cache.store_load_batch([0, 0], [1, 2], [137, 64])
    model.load(1, snap, 137)
    model.load(2, snap, 64)
    check_state(cache, model, w)
    for s in range(3):
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        assert_close(cache.decode(q.cuda()), model.decode(host(q)), w.dtype, "decode after load")
    check_state(cache, model, w)
    assert cache.device_status() == 0
