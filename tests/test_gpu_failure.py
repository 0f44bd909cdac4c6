"""Failure detection on the GPU without a fault: a bounded wait that runs out sets the
device error word, the host reads it through kvc_device_status, and the context stays
usable for the next decode step."""
import pytest
import torch

from kv_cache_decode_ring_gb300 import kvc
from kv_cache_decode_ring_gb300 import workloads as wl

from _parity import assert_close, host, oracle_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_decode_ring_gb300 import build
    build.build()
    torch.cuda.init()


def test_bounded_wait_is_reported_and_the_context_survives():
    w = wl.small("failure", B=2, Hq=8, Hkv=2, d=128, capacity=256, rope_base=10000.0, seed=19)
    cache = kvc.Cache.from_workload(w)
    model = oracle_for(w)
    k, v = w.prefill_chunk(0, 100)
    cache.append_rows(k.cuda(), v.cuda())
    model.append_rows(host(k), host(v), [100, 100])
    assert cache.device_status() == 0
    kvc.kvc_check_wait_path(cache.h)             # a wait on a barrier nothing signals
    assert cache.device_status() == 2            # bit 1: a bounded wait gave up
    assert cache.device_status() == 0            # read once, then cleared
    for s in range(3):                           # the same handle and context keep working
        q, k1, v1 = w.step_qkv(s)
        cache.append(k1.cuda(), v1.cuda())
        model.append(host(k1), host(v1))
        assert_close(cache.decode(q.cuda()), model.decode(host(q)), w.dtype, "decode after the failed wait")
    assert cache.device_status() == 0
