"""Pins of the oracle's prefix store (CPU only).

[PREFIX] "LLM 機制實驗（五）：改了歷史，能否只重算變化的後綴？": the store keeps at most
two prefills; lookup validates integer IDs, matches scope and signature, takes the
longest contiguous common prefix with ties to the most recent entry, and copies the
kept rows before the suffix is computed ("查詢流程與快取所有權").  The nine conditions
and their cut and projection counts are the table of "27 例得到的計算量與誤差"; the
continued path equals a full recompute and a stale next_position diverges in the nine
partial-reuse cases.
"""
import numpy as np
import pytest

from kv_cache_decode_ring_gb300 import workloads as wl
from oracle import numerics as nm
from oracle.model import DecodeOracle, OracleError
from oracle.store import PrefixStore

from _store_cases import BRANCH, PLAIN, SCOPE, SEEDS, SIGNATURE, VOCAB, read_matrix, rows_of, toy

TOL_F32 = 1e-5


def _model(w):
    return DecodeOracle(1, 1, 1, w.head_dim, w.layout, w.capacity, w.window, w.rope_base, "f32")


def _prefill(m, table, ids):
    q, k, v = rows_of(table, ids)
    m.append_rows(wl.as_numpy(k), wl.as_numpy(v), [len(ids)])


def _continue(m, table, ids, start):
    """Append ids[start:] one token at a time and answer each query: [n - start, d]."""
    q, k, v = rows_of(table, ids)
    q, k, v = wl.as_numpy(q), wl.as_numpy(k), wl.as_numpy(v)
    out = []
    for i in range(start, len(ids)):
        m.append(k[:, :, i], v[:, :, i])
        out.append(m.decode(q[i][None])[0, 0])
    return np.array(out)


def _stale(w, table, ids, cut, old_len):
    """Planted mistake: rows [0, cut) kept, the suffix encoded from the old next_position."""
    q, k, v = (wl.as_numpy(x) for x in rows_of(table, ids))
    K = [nm.rope_rotate(k[0, 0, j], [j], w.rope_base) for j in range(cut)]
    V = [v[0, 0, j] for j in range(cut)]
    out = []
    for i in range(cut, len(ids)):
        p = old_len + (i - cut)
        K.append(nm.rope_rotate(k[0, 0, i], [p], w.rope_base)); V.append(v[0, 0, i])
        qr = nm.rope_rotate(q[i, 0], [p], w.rope_base).astype(np.float64)
        out.append(nm.attend(qr[None], np.stack(K).astype(np.float64), np.stack(V).astype(np.float64),
                             t=len(K) - 1, window=w.window)[0])
    return np.array(out)


def _filled_store(w, table, ring):
    store = PrefixStore(2, ring=ring)
    slots = {}
    for name, ids in (("plain", PLAIN), ("branch", BRANCH)):
        m = _model(w)
        _prefill(m, table, ids)
        slots[name] = store.insert(ids, SCOPE, SIGNATURE, m.snapshot(0))
    return store, slots


@pytest.mark.parametrize("seed", SEEDS)
@pytest.mark.parametrize("case", read_matrix(), ids=lambda c: c["name"])
def test_store_matrix(case, seed):
    w = toy(seed, case["ring"])
    table = w.token_table(VOCAB)
    store, slots = _filled_store(w, table, case["ring"])
    ids = case["ids"]
    slot, cut, snap = store.reuse(ids, case["scope"], SIGNATURE)
    assert cut == case["cut"]
    assert slot == (None if case["entry"] is None else slots[case["entry"]])
    assert case["proj"] == 6 * (len(ids) - cut) and case["full"] == 6 * len(ids)
    m = _model(w)
    m.load(0, snap, cut)
    assert m.length(0) == cut
    got = _continue(m, table, ids, cut)
    full = _model(w)
    ref = _continue(full, table, ids, 0)[cut:]
    assert np.array_equal(got, ref)                     # reuse = full recompute
    assert np.array_equal(m.expected_positions(), full.expected_positions())
    for j in range(len(ids)):
        assert np.array_equal(m.hk[0][j], full.hk[0][j]) and np.array_equal(m.hv[0][j], full.hv[0][j])
    old_len = len(store.entry_ids(slot)) if slot is not None else 0
    if 0 < cut < old_len:                               # the nine partial-reuse cases
        stale = _stale(w, table, ids, cut, old_len)
        assert np.abs(stale - got).max() > 100 * TOL_F32


def test_store_ids_scope_signature():
    s = PrefixStore(2)
    s.insert([1, 2, 3, 4], "a", b"sig", "x")
    assert s.lookup([1, 2, 3, 4, 5], "a", b"sig") == (0, 4)
    assert s.lookup([1, 2, 3, 4, 5], "b", b"sig") == (None, 0)      # scope
    assert s.lookup([1, 2, 3, 4, 5], "a", b"sig2") == (None, 0)     # signature
    with pytest.raises(TypeError):
        s.lookup([1.0, 2, 3, 4, 5], "a", b"sig")                    # 1.0 is not the token 1
    with pytest.raises(TypeError):
        s.lookup([True, 2], "a", b"sig")
    with pytest.raises(ValueError):
        s.lookup([], "a", b"sig")
    assert s.lookup(np.array([1, 2, 3, 9]), "a", b"sig") == (0, 3)   # numpy integers are integers
    assert s.lookup([1, 2, 3, 4], "a", b"sig") == (0, 3)            # identical: recompute the last token


def test_store_capacity_evicts_the_oldest_and_ties_prefer_the_newest():
    s = PrefixStore(2)
    a = s.insert([1, 2, 3], "s", b"", "a")
    b = s.insert([1, 2, 4], "s", b"", "b")
    assert (a, b) == (0, 1)
    assert s.lookup([1, 2, 9], "s", b"") == (1, 2)                   # tie at cut 2: newest
    c = s.insert([1, 2, 5], "s", b"", "c")                           # full: replaces the oldest (a)
    assert c == 0 and s.entry_ids(0) == [1, 2, 5]
    assert s.lookup([1, 2, 3, 7], "s", b"") == (0, 2)                # a is gone; c is newest at cut 2
    assert s.lookup([7], "s", b"") == (None, 0)


def test_store_reuse_copies():
    w = toy(7, False)
    table = w.token_table(VOCAB)
    store, slots = _filled_store(w, table, False)
    _, cut, snap = store.reuse(PLAIN + [9], SCOPE, SIGNATURE)
    snap[0][0][:] = 0.0                                              # scribble on the private copy
    _, _, again = store.reuse(PLAIN + [9], SCOPE, SIGNATURE)
    assert np.abs(again[0][0]).max() > 0


def test_load_refuses_evicted_ring_rows():
    w = toy(11, True)
    table = w.token_table(VOCAB)
    m = _model(w)
    _prefill(m, table, PLAIN)                                         # ring of 4 holds positions 4..7
    snap = m.snapshot(0)
    with pytest.raises(OracleError):
        m.load(0, snap, 2)                                            # needs position 1: evicted
    with pytest.raises(OracleError):
        m.load(0, snap, 6)                                            # the token at 6 sees 3..6: 3 is gone
    m.load(0, snap, 8)
    m.load(0, snap, 7)                                                # the token at 7 sees 4..7: resident
    assert m.length(0) == 7 and list(m.expected_positions()[0]) == [4, 5, 6, -1]
