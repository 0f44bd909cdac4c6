"""Pins of the list model, the physical ring and the prefix rules (CPU only).

[LEAN]   "用Lean4形式化验证滑动窗口KV Cache的正确性" (framerc.cn/news/4505248)
[PREFIX] "LLM 機制實驗（五）：改了歷史，能否只重算變化的後綴？" (huhohoo.com)
"""
import os

import pytest

from oracle.listmodel import (Cell, RingBuffer, last_window, position_invariant, prefix_cut,
                              ring_to_list, ring_trim_allowed, run, step)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def cells(n):
    return [Cell(p, ("k", p), ("v", p)) for p in range(n)]


def test_guard_step_into_empty_cache():
    # [LEAN] §5.4: #guard (step 4 [] kv1) = [kv1]
    kv1 = Cell(0, "k1", "v1")
    assert step(4, [], kv1) == [kv1]


@pytest.mark.parametrize("w", range(1, 9))
def test_run_correct_exhaustive(w):
    # [LEAN] §4.2 run_correct: Valid w tokens (run w tokens), for every prefix length up to 64.
    for n in range(0, 65):
        hs = cells(n)
        c = run(w, hs)
        assert c == last_window(w, hs)
        # §2.4 (1): length never exceeds the window
        assert len(c) == min(w, n) <= w
        # §2.4 (2): the contents are the last W entries of the history
        assert c == hs[max(0, n - w):]
        # §2.4 (3): slot i holds position t - W + 1 + i once full (t = n - 1), else i
        t = n - 1
        for i, cell in enumerate(c):
            assert cell.pos == (t - w + 1 + i if n >= w else i)
        assert position_invariant(c)


@pytest.mark.parametrize("w", range(1, 9))
def test_commuting_equation(w):
    # [LEAN] §2.4 / §4.1: lastWindow w (xs ++ [kv]) = step w (lastWindow w xs) kv
    for n in range(0, 40):
        xs = cells(n)
        kv = Cell(n, ("k", n), ("v", n))
        assert last_window(w, xs + [kv]) == step(w, last_window(w, xs), kv)


def test_position_invariant_detects_gap():
    c = [Cell(3), Cell(4), Cell(6)]
    assert not position_invariant(c)
    assert position_invariant([Cell(5), Cell(6), Cell(7)])


@pytest.mark.parametrize("w", range(1, 9))
def test_physical_ring_simulates_list_model(w):
    # [LEAN] §3.4: ringToList of the head/tail ring equals the list model after every push,
    # through the not-full, exactly-full and first-replacement phases (§1.3, §5.1).
    ring = RingBuffer(w)
    hist = []
    for p in range(0, 3 * w + 5):
        kv = Cell(p, ("k", p), ("v", p))
        slot = ring.push(kv)
        hist.append(kv)
        # the slot the head/count model chose is position mod W (what the GPU writes)
        assert slot == p % w
        assert ring.as_list() == last_window(w, hist)
        if len(hist) < w:
            # not-full phase: the page's all-slots mapping reads empty slots
            naive = ring_to_list(w, ring.buf, ring.head)
            assert any(x is None for x in naive)
        else:
            assert ring_to_list(w, ring.buf, ring.head) == last_window(w, hist)
            # once full, the logical head is (t + 1) mod W
            assert ring.head == (p + 1) % w


def test_ring_phases_w4():
    # The three phases named in [LEAN] §1.3 for W = 4.
    ring = RingBuffer(4)
    for p in range(3):
        ring.push(Cell(p))
    assert [c.pos for c in ring.as_list()] == [0, 1, 2] and ring.count == 3       # not full (t = 2)
    ring.push(Cell(3))
    assert [c.pos for c in ring.as_list()] == [0, 1, 2, 3] and ring.head == 0      # exactly full (t = 3)
    ring.push(Cell(4))
    assert [c.pos for c in ring.as_list()] == [1, 2, 3, 4] and ring.buf[0].pos == 4  # first replacement


def test_signed_base_arithmetic():
    # [LEAN] §4.3/§5.2: the first window position is base = len - min(W, len) = t - W + 1 once
    # full.  Natural-number subtraction evaluates t - W + 1 as (t - W) + 1 with t - W clamped
    # at 0, which is off by one exactly while the ring is not yet past full (len <= W).
    for w in range(1, 9):
        for n in range(1, 20):
            t = n - 1
            base = n - min(w, n)
            assert last_window(w, cells(n))[0].pos == base
            nat_base = max(0, t - w) + 1
            assert (nat_base == base) == (n > w)


@pytest.mark.parametrize("w", range(1, 7))
def test_ring_trim_rule_against_residency(w):
    # The trim rule equals brute-force residency of every position the next query needs.
    for n in range(0, 3 * w + 3):
        ring = RingBuffer(w)
        for p in range(n):
            ring.push(Cell(p))
        resident = {c.pos for c in ring.as_list()}
        for cut in range(0, n + 1):
            need = set(range(max(0, cut - w + 1), cut))
            assert ring_trim_allowed(cut, n, w) == need.issubset(resident), (w, n, cut)


@pytest.mark.parametrize("w", range(1, 6))
def test_ring_truncate_then_continue(w):
    # After an allowed trim (drop the newest entries, keep the head) and one push, the
    # ring again equals lastWindow of the trimmed-and-extended history.
    for n in range(1, 3 * w + 2):
        for cut in range(0, n + 1):
            if not ring_trim_allowed(cut, n, w):
                continue
            ring = RingBuffer(w)
            for p in range(n):
                ring.push(Cell(p, "old"))
            ring.truncate(n - cut, cut % w)
            hist = [Cell(p, "old") for p in range(cut)]
            for p in range(cut, cut + 2 * w + 1):
                kv = Cell(p, "new")
                assert ring.push(kv) == p % w
                hist.append(kv)
                assert ring.as_list() == last_window(w, hist), (w, n, cut, p)


def read_cases():
    rows = []
    with open(os.path.join(GOLDEN, "prefix_reuse_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, old, new, ring, cut, proj, full = [x.strip() for x in line.split("|")]
            rows.append((name, old, [int(x) for x in new.split()], int(ring), int(cut), int(proj), int(full)))
    return rows


@pytest.mark.parametrize("case", read_cases(), ids=lambda c: c[0])
def test_prefix_cut_golden(case):
    name, old, new, ring, cut, proj, full = case
    # projections = layers(2) x Q/K/V(3) x recomputed tokens
    assert proj == 6 * (len(new) - cut) and full == 6 * len(new)
    if old == "store":
        # the two stored branches of the page's store under one scope; the query comes from
        # another scope, so no entry is eligible and everything is recomputed
        from oracle.store import PrefixStore
        store = PrefixStore(2, ring=bool(ring))
        store.insert(list(range(1, 9)), "scope-a", b"sig", None)
        store.insert([1, 2, 3, 4, 5, 20, 21, 22], "scope-a", b"sig", None)
        assert store.lookup(new, "scope-b", b"sig") == (None, cut)
        assert store.lookup(new, "scope-a", b"sig")[1] == 8          # the same query in the stored scope
        return
    assert prefix_cut([int(x) for x in old.split()], new, ring=bool(ring)) == cut


def test_prefix_cut_validation_and_bounds():
    with pytest.raises(ValueError):
        prefix_cut([1, 2], [])
    with pytest.raises(TypeError):
        prefix_cut([1, 2, 3], [1.0, 2, 3])          # 1.0 is not the token 1
    assert prefix_cut([], [5, 6]) == 0
    assert prefix_cut([1, 2, 3], [1, 2, 3]) == 2      # identical query: recompute the last token
    assert prefix_cut([1, 2, 3], [1, 2, 3], ring=True) == 0   # ring: no new suffix -> fall back
    # "change the edit from the fifth to the second token: the cut becomes 1"
    assert prefix_cut(list(range(1, 9)), [1, 20] + list(range(3, 13))) == 1
