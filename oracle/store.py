"""Prefix store: reuse of stored prefill rows by the longest contiguous common prefix.

TEST INFRASTRUCTURE (see the package docstring).

[PREFIX] "LLM 機制實驗（五）：改了歷史，能否只重算變化的後綴？" (huhohoo.com), section
"查詢流程與快取所有權" describes the store and its lookup, in this order:

0. the store keeps at most two prefill results (the page's store; the capacity is a
   parameter here).  The page does not say which entry a third insert replaces; the
   reading taken is the oldest inserted one.
1. the query must be a non-empty sequence of integer token IDs; a float equal to
   an integer (1.0) is not accepted as that integer;
2. only entries with the same application scope and the same computation signature
   (model weights, implementation, window, positional-encoding convention) are
   eligible;
3. among them the entry with the longest contiguous common prefix wins, and on a
   tie the most recently inserted one;
4. the rows to keep (K, V and positions) are copied out of the entry before the
   suffix is computed, so that the query never changes another branch's arrays.

The reusable length of one entry follows :func:`oracle.listmodel.prefix_cut`
(cut <= len(query) - 1; a sliding-window entry only on a whole-prefix match).
"Longest" is compared on that reusable length, which is what the lookup returns.
"""
from __future__ import annotations

import copy
from typing import Any, List, Optional, Sequence, Tuple

from .listmodel import prefix_cut


def _check_ids(ids: Sequence) -> List[int]:
    # step 1: integers only (bool is an int subclass in Python but not a token ID)
    out = []
    for x in ids:
        if isinstance(x, bool) or not hasattr(x, "__index__") or isinstance(x, float):
            raise TypeError("token IDs must be integers, got %r" % (x,))
        out.append(int(x))
    if not out:
        raise ValueError("empty token sequence")
    return out


class _Entry:
    __slots__ = ("ids", "scope", "signature", "payload", "seq")

    def __init__(self, ids, scope, signature, payload, seq):
        self.ids, self.scope, self.signature, self.payload, self.seq = ids, scope, signature, payload, seq


class PrefixStore:
    """A bounded store of prefill results, keyed by token IDs, scope and signature.

    ``payload`` is whatever a prefill produced (cache rows and positions); the store
    deep-copies it on insert and again on reuse, which is step 4's ownership rule.
    ``ring`` selects the sliding-window reuse rule for every entry of this store.
    """

    def __init__(self, capacity: int = 2, ring: bool = False):
        if capacity < 1:
            raise ValueError("capacity must be positive")
        self.capacity = capacity
        self.ring = ring
        self.slots: List[Optional[_Entry]] = [None] * capacity
        self._seq = 0

    def insert(self, ids: Sequence, scope: str, signature: bytes, payload: Any) -> int:
        """Stores a prefill of ``ids``; returns the slot used (a free one, else the oldest)."""
        ids = _check_ids(ids)
        free = [i for i, e in enumerate(self.slots) if e is None]
        slot = free[0] if free else min(range(self.capacity), key=lambda i: self.slots[i].seq)
        self._seq += 1
        self.slots[slot] = _Entry(ids, str(scope), bytes(signature), copy.deepcopy(payload), self._seq)
        return slot

    def lookup(self, ids: Sequence, scope: str, signature: bytes) -> Tuple[Optional[int], int]:
        """(slot, cut) of the best eligible entry, or (None, 0) when nothing is reusable."""
        ids = _check_ids(ids)
        best, best_cut, best_seq = None, 0, -1
        for slot, e in enumerate(self.slots):
            if e is None or e.scope != str(scope) or e.signature != bytes(signature):
                continue
            cut = prefix_cut(e.ids, ids, self.ring)
            if cut > best_cut or (cut == best_cut and cut > 0 and e.seq > best_seq):
                best, best_cut, best_seq = slot, cut, e.seq
        return best, best_cut

    def reuse(self, ids: Sequence, scope: str, signature: bytes) -> Tuple[Optional[int], int, Any]:
        """Lookup, then a private copy of the chosen entry's payload (None on a miss)."""
        slot, cut = self.lookup(ids, scope, signature)
        if slot is None:
            return None, 0, None
        return slot, cut, copy.deepcopy(self.slots[slot].payload)

    def entry_ids(self, slot: int) -> List[int]:
        return list(self.slots[slot].ids)
