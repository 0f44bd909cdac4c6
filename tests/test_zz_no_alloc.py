"""kvc_decode_attn_noalloc: the decode entry point that allocates nothing.

Some callers cannot call cudaMalloc while they decode, for example a serving
engine that reserved all device memory for its KV pool, or a runtime whose own
allocator owns every device buffer.  This variant keeps its split-K scratch in a
fixed array inside the library.  Its outputs must match kvc_decode_attn's on the
same cache, on two calls in a row (the array keeps the previous call's contents).

This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import pytest
import torch

from kv_cache_decode_ring_gb300 import kvc
from kv_cache_decode_ring_gb300 import workloads as wl

from _parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_decode_ring_gb300 import build
    build.build()


def _filled(w, lengths, **kw):
    cache = kvc.Cache.from_workload(w, **kw)
    k, v = w.prefill_chunk(0, max(lengths), device="cuda")
    cache.append_rows(k, v, counts=lengths)
    q, k1, v1 = w.step_qkv(0, device="cuda")
    cache.append(k1, v1)
    return cache, q


def _check_twice(cache, q, dtype):
    ref = cache.decode(q)                                       # the existing entry point
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        kvc.kvc_decode_attn_noalloc(cache.h, q, out)
        torch.cuda.synchronize()
        assert_close(out, ref.double().cpu().numpy(), dtype, "noalloc vs decode_attn")
    assert cache.device_status() == 0


@pytest.mark.parametrize("layout", ["contiguous", "ring"])
def test_noalloc_matches_decode_attn(layout):
    w = wl.small("noalloc-" + layout, B=5, Hq=16, Hkv=4, d=128, layout=layout,
                 capacity=1024 if layout == "contiguous" else 256,
                 window=0 if layout == "contiguous" else 256, rope_base=10000.0, seed=13)
    cache, q = _filled(w, [1, 37, 200, 555, 1000] if layout == "contiguous" else [1, 37, 200, 555, 300],
                       max_position=4096 if layout == "ring" else 0)
    _check_twice(cache, q, "bf16")


def test_noalloc_matches_decode_attn_full_cache_mha():
    w = wl.full_cache_mha()
    cache, q = _filled(w, [w.extra["context"]] * w.batch)
    _check_twice(cache, q, "bf16")


def test_noalloc_fp32_generic_kernel():
    w = wl.toy("full")
    cache = kvc.Cache.from_workload(w)
    for s in range(9):
        q, k, v = w.step_qkv(s)
        cache.append(k.cuda(), v.cuda())
    _check_twice(cache, q.cuda(), "f32")


def test_noalloc_rejects_a_problem_larger_than_its_array():
    # 16 x 64 query heads x 512 splits x 520 B = 272 MB of partials > 64 MiB
    w = wl.small("noalloc-big", B=16, Hq=64, Hkv=1, d=128, capacity=65536, rope_base=0.0, seed=3)
    cache = kvc.Cache.from_workload(w)
    q, k, v = w.step_qkv(0, device="cuda")
    cache.append(k, v)
    out = torch.zeros_like(q)
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_decode_attn_noalloc(cache.h, q, out)
    assert e.value.code == kvc.KVC_ERR_CAPACITY
    assert not out.any()
