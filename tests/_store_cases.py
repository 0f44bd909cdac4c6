"""The prefix-store matrix shared by the oracle and GPU tests.

[PREFIX] "LLM 機制實驗（五）：改了歷史，能否只重算變化的後綴？", sections
"查詢流程與快取所有權" (the store and its lookup) and "27 例得到的計算量與誤差" (nine
conditions, three seeds 7, 11, 23; a single-head model of dimension 16 over a vocabulary
of 32 tokens).  Here one cache layer of that shape stands in for the page's untrained
two-layer decoder: rows are drawn per token ID (equal IDs, equal rows), keys and queries
take RoPE at their positions, fp32.
"""
import os

from kv_cache_decode_ring_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
SEEDS = (7, 11, 23)
VOCAB, D = 32, 16
PLAIN = [1, 2, 3, 4, 5, 6, 7, 8]
BRANCH = [1, 2, 3, 4, 5, 20, 21, 22]
SCOPE = "app"
SIGNATURE = b"toy-1layer-d16-rope10000-f32"
CAPACITY, RING_W = 16, 4


def read_matrix():
    rows = []
    with open(os.path.join(GOLDEN, "prefix_store_matrix.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, store, scope, ids, cut, entry, proj, full = [x.strip() for x in line.split("|")]
            rows.append(dict(name=name, ring=store == "ring", scope=scope, ids=[int(x) for x in ids.split()],
                             cut=int(cut), entry=None if entry == "-" else entry, proj=int(proj), full=int(full)))
    return rows


def toy(seed, ring):
    return wl.small("prefix-store-toy", B=1, Hq=1, Hkv=1, d=D, layout="ring" if ring else "contiguous",
                    capacity=RING_W if ring else CAPACITY, window=RING_W if ring else 0, rope_base=10000.0,
                    dtype="f32", seed=seed)


def rows_of(table, ids):
    """q [n, Hq, d], k and v [1, Hkv, n, d] for the token IDs ``ids`` (CPU tensors)."""
    q, k, v = table
    return q[ids], k[ids].permute(1, 0, 2).unsqueeze(0).contiguous(), v[ids].permute(1, 0, 2).unsqueeze(0).contiguous()
