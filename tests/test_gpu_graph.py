"""A decode step captured in a CUDA graph and replayed equals the same steps run eagerly,
bit for bit.

[WITCERT] "SGLang 生产级落地与闭环门控修复": the Philox counter of Tier B is self-contained
(request, layer, KV head, token, channel), so the stream is reproduced exactly under CUDA
Graph capture and replay.  The library's kernels read next_position on the device, so one
captured append + decode advances the cache on every replay: each replay writes the next
slot and attends over the new window, for the ring, the contiguous bf16 cache and Tier B.
(The handle's host mirror of next_position counts the captured call once; the test reads
the device state through kvc_export.)
"""
import numpy as np
import pytest
import torch

from kv_cache_decode_ring_gb300 import kvc
from kv_cache_decode_ring_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_decode_ring_gb300 import build
    build.build()
    torch.cuda.init()


CASES = [
    # name, workload kwargs, prefill rows, replays
    ("ring-gqa4", dict(B=2, Hq=8, Hkv=2, d=128, layout="ring", capacity=64, window=64, rope_base=10000.0), 40, 50),
    ("mha-contiguous", dict(B=3, Hq=4, Hkv=4, d=128, capacity=512, rope_base=0.0), 130, 40),
    ("tier-b", dict(B=2, Hq=8, Hkv=2, d=128, capacity=512, rope_base=10000.0, quant="int8-dither",
                    layer=5, dither_key=(0x1234, 0x5678)), 100, 40),
]


def _exports(cache):
    names = [kvc.KVC_EXPORT_POSITIONS, kvc.KVC_EXPORT_NEXT_POSITION]
    if cache.cfg.kv_quant == kvc.KVC_QUANT_NONE:
        names += [kvc.KVC_EXPORT_K, kvc.KVC_EXPORT_V]
    else:
        names += [kvc.KVC_EXPORT_KQ, kvc.KVC_EXPORT_VQ, kvc.KVC_EXPORT_SK, kvc.KVC_EXPORT_SV,
                  kvc.KVC_EXPORT_KTAIL, kvc.KVC_EXPORT_VTAIL]
    return {n: cache.export(n) for n in names}


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_graph_replay_equals_eager(case):
    name, kw, prefill, replays = case
    w = wl.small("graph-" + name, seed=13, **kw)
    mp = 1024 if w.layout == "ring" else 0
    eager = kvc.Cache.from_workload(w, max_position=mp)
    graphed = kvc.Cache.from_workload(w, max_position=mp)
    k, v = w.prefill_chunk(0, prefill, device="cuda")
    for c in (eager, graphed):
        c.append_rows(k, v)
    q0, k0, v0 = w.step_qkv(0, device="cuda")
    sq, sk, sv = q0.clone(), k0.clone(), v0.clone()            # the graph's fixed input buffers
    out_g = torch.empty(q0.shape, dtype=eager.out_dtype, device="cuda")
    # warm the kernels up (attributes, module load) on the eager twin's first step
    eager.append(k0, v0)
    ref0 = eager.decode(q0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        graphed.append(sk, sv)
        graphed.decode(sq, out_g)
    torch.cuda.synchronize()
    for step in range(replays):
        if step == 0:
            q, kk, vv, ref = q0, k0, v0, ref0
        else:
            q, kk, vv = w.step_qkv(step, device="cuda")
            eager.append(kk, vv)
            ref = eager.decode(q)
        sq.copy_(q); sk.copy_(kk); sv.copy_(vv)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g, ref), (name, step)
    a, b = _exports(graphed), _exports(eager)
    for n in a:
        assert np.array_equal(a[n], b[n]), (name, n)
    assert int(a[kvc.KVC_EXPORT_NEXT_POSITION][0]) == prefill + replays
    assert graphed.device_status() == 0 and eager.device_status() == 0
