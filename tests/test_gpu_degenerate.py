"""Degenerate windows on the GPU, against their closed form.

[LEAN] §2.1: the query at position t attends to the W positions ending at t, so a
window of one key keeps only t itself; and at t = 0 every window holds one key.  The
softmax of a single logit is 1, so the output is the newest value row, whatever the
query: out[b, h] = v_t[b, h / g].  Each decode kernel is checked (the MHA kernel, the
GQA kernel, the generic kernel for other head sizes and fp32 caches), on a ring of one
slot and on a contiguous cache with a one-key window, with fp32 outputs at the fp32
tolerance; the oracle's own attention gives the same closed form (pinned on the CPU).
"""
import numpy as np
import pytest
import torch

from kv_cache_decode_ring_gb300 import kvc
from kv_cache_decode_ring_gb300 import workloads as wl
from oracle import numerics as nm

from _parity import assert_close, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_decode_ring_gb300 import build
    build.build()


CASES = [
    # name, Hq, Hkv, d, layout, dtype
    ("mha-d128-ring1", 4, 4, 128, "ring", "bf16"),
    ("gqa4-d128-ring1", 8, 2, 128, "ring", "bf16"),
    ("gqa4-d128-window1", 8, 2, 128, "contiguous", "bf16"),
    ("gqa8-d64-window1", 8, 1, 64, "contiguous", "bf16"),
    ("gqa2-d96-ring1", 4, 2, 96, "ring", "bf16"),
    ("f32-gqa4-d128-ring1", 8, 2, 128, "ring", "f32"),
]


def _values(v, dtype):
    x = host(v)
    return (nm.bf16_to_f32(x) if dtype == "bf16" else x).astype(np.float64)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_window_of_one_returns_the_newest_value(case):
    name, Hq, Hkv, d, layout, dtype = case
    ring = layout == "ring"
    w = wl.small(name, B=3, Hq=Hq, Hkv=Hkv, d=d, layout=layout, capacity=1 if ring else 64, window=1,
                 rope_base=10000.0, dtype=dtype, seed=5)
    cache = kvc.Cache.from_workload(w, max_position=64 if ring else 0, out_dtype="f32")
    g = Hq // Hkv
    for s in range(24):
        q, k, v = w.step_qkv(s)
        cache.append(k.cuda(), v.cuda())
        out = cache.decode(q.cuda())
        want = np.repeat(_values(v, dtype), g, axis=1)          # query head h reads KV head h // g
        assert_close(out, want, "f32", "%s step %d" % (name, s))
    pos = cache.export(kvc.KVC_EXPORT_POSITIONS)
    if ring:
        assert np.array_equal(pos, np.full((3, 1), 23))          # the one slot holds the newest position
    else:
        assert np.array_equal(pos[:, :24], np.broadcast_to(np.arange(24), (3, 24)))
    assert cache.device_status() == 0


@pytest.mark.parametrize("case", CASES[:4], ids=lambda c: c[0])
def test_first_token_attends_to_itself(case):
    # t = 0 with no window limit: one key in the window
    name, Hq, Hkv, d, _, dtype = case
    w = wl.small(name + "-t0", B=3, Hq=Hq, Hkv=Hkv, d=d, capacity=64, rope_base=10000.0, dtype=dtype, seed=6)
    cache = kvc.Cache.from_workload(w, out_dtype="f32")
    q, k, v = w.step_qkv(0)
    cache.append(k.cuda(), v.cuda())
    out = cache.decode(q.cuda())
    assert_close(out, np.repeat(_values(v, dtype), Hq // Hkv, axis=1), "f32", name + " t=0")
    assert cache.device_status() == 0
