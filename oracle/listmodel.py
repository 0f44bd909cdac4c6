"""The KV cache as a list, after [LEAN] §2-§3, plus the prefix-reuse rules of [PREFIX].

TEST INFRASTRUCTURE (see the package docstring).  Pure Python; small cases only.

[LEAN]   "用Lean4形式化验证滑动窗口KV Cache的正确性" (framerc.cn/news/4505248)
[PREFIX] "LLM 機制實驗（五）：改了歷史，能否只重算變化的後綴？" (huhohoo.com)
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Any, List, Optional, Sequence


@dataclass(frozen=True)
class Cell:
    """One cache entry: absolute position plus key and value ([LEAN] §3.2, ``KV Cell``)."""

    pos: int
    key: Any = None
    val: Any = None


def last_window(w: int, hs: Sequence) -> list:
    """The last ``w`` entries of the full history ([LEAN] §2.3, ``lastWindow``).

    Drops ``len(hs) - min(w, len(hs))`` entries from the front; while the history
    is shorter than the window nothing is dropped.
    """
    n = len(hs)
    return list(hs[n - min(w, n):])


def step(w: int, c: Sequence, kv) -> list:
    """Append one entry, then evict the oldest if the list exceeds ``w`` ([LEAN] §3.3, ``step``)."""
    c2 = list(c) + [kv]
    if w < len(c2):
        return c2[1:]
    return c2


def run(w: int, tokens: Sequence) -> list:
    """Fold ``step`` over a token stream from the empty cache ([LEAN] §4.2, ``run``)."""
    c: list = []
    for kv in tokens:
        c = step(w, c, kv)
    return c


def position_invariant(c: Sequence[Cell]) -> bool:
    """Slot i holds position base + i for one base ([LEAN] §3.2, ``PositionInvariant``)."""
    if not c:
        return True
    base = c[0].pos
    return all(cell.pos == base + i for i, cell in enumerate(c))


def ring_to_list(w: int, buf: Sequence, head: int, count: Optional[int] = None) -> list:
    """Read a ring buffer as the logical list ([LEAN] §3.4, ``ringToList``).

    Entry i of the list is ``buf[(head + i) % w]``.  The page maps all ``w`` slots;
    ``count`` limits the read to the live entries, which is what the not-full phase
    needs ([LEAN] §5.1: mapping all w slots before the ring is full reads garbage).
    ``count=None`` reproduces the page's all-slots mapping.
    """
    n = w if count is None else count
    return [buf[(head + i) % w] for i in range(n)]


class RingBuffer:
    """Physical ring: a fixed array with a head index; a push overwrites the oldest ([LEAN] §3.4).

    Formulated with head/count rather than slot arithmetic, so that the GPU's
    ``slot = position mod W`` rule is checked against it rather than copied from it.
    """

    def __init__(self, w: int):
        if w <= 0:
            raise ValueError("window must be positive")
        self.w = w
        self.buf: List[Any] = [None] * w
        self.head = 0
        self.count = 0

    def push(self, kv) -> int:
        """Store ``kv``; returns the slot written."""
        if self.count < self.w:
            slot = (self.head + self.count) % self.w
            self.count += 1
        else:
            slot = self.head
            self.head = (self.head + 1) % self.w
        self.buf[slot] = kv
        return slot

    def as_list(self) -> list:
        return ring_to_list(self.w, self.buf, self.head, self.count)

    def truncate(self, n_drop: int, next_slot: int) -> None:
        """Forget the ``n_drop`` newest entries (a trim); the head stays on the oldest.

        Entries already overwritten are not resident, so at most ``count`` go.  When
        the ring empties, the head moves to ``next_slot`` (where the next push must
        land); otherwise the next push lands at ``head + count``.
        """
        self.count -= min(self.count, n_drop)
        if self.count == 0:
            self.head = next_slot % self.w


def prefix_cut(old_ids: Sequence[int], new_ids: Sequence[int], ring: bool = False) -> int:
    """Rows of a stored prefill that a new query may reuse ([PREFIX]).

    * The cut is the length of the longest *contiguous* common prefix; equal IDs
      after the first difference do not count ("先看一次歷史編輯": old 1..8,
      new 1 2 3 4 20 6 7 8 9 10 11 12 gives cut = 4).
    * At least the last query token is always recomputed: cut <= len(new) - 1
      ("查詢流程與快取所有權").
    * A sliding-window cache is reused only when the whole cached prefix matches
      and the query adds a suffix; a partial hit falls back to cut = 0
      ("為什麼滑窗部分命中必須回退").
    * IDs must be a non-empty sequence of integers; a float such as 1.0 is rejected
      even though it converts to an equal integer ("查詢流程與快取所有權", step 1).
    """
    for ids in (old_ids, new_ids):
        for x in ids:
            if isinstance(x, bool) or not isinstance(x, int):
                raise TypeError("token IDs must be integers")
    if len(new_ids) == 0:
        raise ValueError("empty query")
    lcp = 0
    m = min(len(old_ids), len(new_ids))
    while lcp < m and old_ids[lcp] == new_ids[lcp]:
        lcp += 1
    if ring:
        cut = len(old_ids) if (lcp == len(old_ids) and len(new_ids) > len(old_ids)) else 0
    else:
        cut = lcp
    return min(cut, len(new_ids) - 1)


def ring_trim_allowed(cut: int, next_position: int, w: int) -> bool:
    """Whether a ring of size ``w`` can continue from ``cut`` without evicted rows.

    After the trim the next token sits at position ``cut`` and attends to
    positions ``[cut - w + 1, cut]``, of which ``[max(0, cut - w + 1), cut)`` must
    come from the ring; the ring still holds ``[max(0, next_position - w),
    next_position)``.  Reuse is safe iff that needed range is empty or starts
    inside the resident one: with ``lo = max(0, cut - w + 1)``, ``lo == cut`` or
    ``lo >= max(0, next_position - w)``; and ``cut <= next_position``.
    [PREFIX] "為什麼滑窗部分命中必須回退" states the hazard (rows 0-3 are gone
    from a W=4 ring holding 4-7) and uses the stricter whole-prefix rule, which
    is a special case of this one.
    """
    if cut < 0 or cut > next_position:
        return False
    lo = max(0, cut - w + 1)
    return lo == cut or lo >= max(0, next_position - w)
