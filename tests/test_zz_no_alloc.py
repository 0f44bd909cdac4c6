"""kvc_decode_attn_noalloc: the decode entry point that allocates nothing.

Some callers cannot call cudaMalloc while they decode, for example a serving
engine that reserved all device memory for its KV pool, or a runtime whose own
allocator owns every device buffer.  This variant keeps its split-K scratch in a
fixed array inside the library.  It runs the same kernels on the same inputs as
kvc_decode_attn, so its outputs must be bit-identical to that entry point's, on
two calls in a row (the array keeps the previous call's contents); they are also
held to the oracle within the tolerance of the other parity tests.

This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import os

import numpy as np
import pytest
import torch

from kv_cache_decode_ring_gb300 import kvc
from kv_cache_decode_ring_gb300 import workloads as wl
from oracle import numerics as nm

from _parity import assert_close, host, oracle_for

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20        # KVC_NOALLOC_SCRATCH_BYTES in include/kvc.h


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_decode_ring_gb300 import build
    build.build()


def _filled(w, lengths, **kw):
    """A cache and its oracle model holding the same rows: a prefill of lengths[b] rows,
    then one decode token for every request."""
    cache = kvc.Cache.from_workload(w, **kw)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, max(lengths))
    cache.append_rows(k.cuda(), v.cuda(), counts=lengths)
    model.append_rows(host(k), host(v), lengths)
    q, k1, v1 = w.step_qkv(0)
    cache.append(k1.cuda(), v1.cuda())
    model.append(host(k1), host(v1))
    return cache, q.cuda(), model.decode(host(q))


def _check_twice(cache, q, ref_oracle, dtype):
    ref = cache.decode(q)                                       # the existing entry point
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        kvc.kvc_decode_attn_noalloc(cache.h, q, out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), "noalloc output differs from kvc_decode_attn"
        assert_close(out, ref_oracle, dtype, "noalloc vs the oracle")
    assert cache.device_status() == 0


@pytest.mark.parametrize("layout", ["contiguous", "ring"])
def test_noalloc_matches_decode_attn(layout):
    w = wl.small("noalloc-" + layout, B=5, Hq=16, Hkv=4, d=128, layout=layout,
                 capacity=1024 if layout == "contiguous" else 256,
                 window=0 if layout == "contiguous" else 256, rope_base=10000.0, seed=13)
    cache, q, ref = _filled(w, [1, 37, 200, 555, 1000] if layout == "contiguous" else [1, 37, 200, 555, 300],
                            max_position=4096 if layout == "ring" else 0)
    _check_twice(cache, q, ref, "bf16")


def test_noalloc_matches_decode_attn_paged_gqa():
    # a paged cache is the one layout with an extra split (the window start rounded down to
    # a page) and the combine that knows that origin
    w = wl.small("noalloc-paged", B=4, Hq=16, Hkv=4, d=128, capacity=2048, window=700, rope_base=10000.0,
                 seed=17)
    lengths = [3, 300, 1500, 2000]
    cache, q, ref = _filled(w, lengths, page_pool=4 * (2048 // 16))
    _check_twice(cache, q, ref, "bf16")


def test_noalloc_matches_decode_attn_full_cache_mha():
    # the bench's full-cache MHA shape; the oracle works from the generator's bf16 rows
    w = wl.full_cache_mha()
    ctx = w.extra["context"]
    B, H, d = w.batch, w.n_q_heads, w.head_dim
    cache = kvc.Cache.from_workload(w)
    k, v = w.prefill_chunk(0, ctx, device="cuda")
    cache.append_rows(k, v)
    q, k1, v1 = w.step_qkv(0, device="cuda")
    cache.append(k1, v1)
    hK = np.concatenate([host(k), host(k1)[:, :, None]], axis=2)
    hV = np.concatenate([host(v), host(v1)[:, :, None]], axis=2)
    del k, v
    qf = nm.bf16_to_f32(host(q)).astype(np.float64)
    probs = [(b, h) for b in range(B) for h in range(H)]
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    ref = nm.attend_many([qf[b, h][None] for b, h in probs], [hK[b, h] for b, h in probs],
                         [hV[b, h] for b, h in probs], [ctx] * len(probs), 0, None, nthreads=threads)
    _check_twice(cache, q, np.stack(ref).reshape(B, H, d), "bf16")


def test_noalloc_fp32_generic_kernel():
    w = wl.toy("full")
    cache = kvc.Cache.from_workload(w)
    model = oracle_for(w)
    for s in range(9):
        q, k, v = w.step_qkv(s)
        cache.append(k.cuda(), v.cuda())
        model.append(host(k), host(v))
    _check_twice(cache, q.cuda(), model.decode(host(q)), "f32")


def test_noalloc_rejects_a_problem_larger_than_its_array():
    # 64 query heads per KV head take the generic kernel's 64-key splits: a capacity of
    # 65536 gives 1024 splits, and 16 x 64 x 1024 x (8 + 4 x 128) B = 545 MB of partials
    B, Hq, d, cap = 16, 64, 128, 65536
    need = B * Hq * (cap // 64) * (8 + 4 * d)
    assert need > SCRATCH_BYTES
    w = wl.small("noalloc-big", B=B, Hq=Hq, Hkv=1, d=d, capacity=cap, rope_base=0.0, seed=3)
    cache = kvc.Cache.from_workload(w)
    q, k, v = w.step_qkv(0, device="cuda")
    cache.append(k, v)
    out = torch.zeros_like(q)
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_decode_attn_noalloc(cache.h, q, out)
    assert e.value.code == kvc.KVC_ERR_CAPACITY
    assert not out.any()
