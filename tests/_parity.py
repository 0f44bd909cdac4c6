"""Shared helpers of the GPU parity tests: drive the CUDA library and the CPU oracle on
the same seeded inputs and compare them (cache state bit-exact, outputs within the
stated tolerance: |gpu - ref| <= atol + rtol |ref| with 1e-5 for fp32 and 2e-3 for bf16)."""
import numpy as np
import torch

from kv_cache_decode_ring_gb300 import kvc
from kv_cache_decode_ring_gb300 import workloads as wl
from oracle import numerics as nm
from oracle.model import DecodeOracle

TOL = {"f32": 1e-5, "bf16": 2e-3}


def oracle_for(w, **kw) -> DecodeOracle:
    if w.quant == "int8-dither":
        kw.setdefault("dither_key", w.extra.get("dither_key", (0, 0)))
        kw.setdefault("layer", w.extra.get("layer", 0))
    return DecodeOracle(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.layout, w.capacity,
                        0 if w.layout == "ring" else w.window, w.rope_base, w.dtype, w.quant, **kw)


def host(t: torch.Tensor) -> np.ndarray:
    return wl.as_numpy(t)


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |x| (8 significant bits: 2^(floor(log2|x|) - 8))."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(ax)).astype(np.int64) - 8)


def assert_close(gpu: torch.Tensor, ref: np.ndarray, dtype: str, what=""):
    """|gpu - ref| <= tol + tol |ref|, tol = 1e-5 (fp32 caches) or 2e-3 (bf16 caches).
    A bf16 *output* is additionally allowed its own rounding, half a bf16 ulp of ref
    (bf16's unit roundoff 2^-8 exceeds 2e-3 once |ref| > ~1)."""
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    tol = TOL[dtype]
    bound = tol + tol * np.abs(ref)
    if gpu.dtype == torch.bfloat16:
        bound = bound + bf16_half_ulp(ref)
    excess = np.abs(g - ref) - bound
    if not np.all(excess <= 0):
        i = np.unravel_index(np.argmax(excess), excess.shape)
        raise AssertionError("%s: %d/%d outside tolerance; worst at %s gpu=%r ref=%r"
                             % (what, int((excess > 0).sum()), excess.size, i, g[i], ref[i]))


def row_bits(row_f32: np.ndarray, dtype: str) -> np.ndarray:
    """Bit patterns of oracle rows (fp32 values) in the cache dtype."""
    if dtype == "bf16":
        return nm.f32_to_bf16(row_f32)
    return np.ascontiguousarray(row_f32, dtype=np.float32).view(np.uint32)


def check_state(cache: kvc.Cache, model: DecodeOracle, w, requests=None):
    """Positions, next_position and every live K/V row, bit-exact."""
    pos = cache.export(kvc.KVC_EXPORT_POSITIONS)
    want = model.expected_positions()
    assert np.array_equal(pos, want), "positions differ"
    npos = cache.export(kvc.KVC_EXPORT_NEXT_POSITION)
    assert np.array_equal(npos, [model.length(b) for b in range(model.B)]), "next_position differs"
    assert np.array_equal(cache.next_positions(), npos)
    K = cache.export(kvc.KVC_EXPORT_K)
    V = cache.export(kvc.KVC_EXPORT_V)
    if w.dtype == "f32":
        K, V = K.view(np.uint32), V.view(np.uint32)
    for b in (range(model.B) if requests is None else requests):
        for which, arr in (("k", K), ("v", V)):
            rows = model.expected_rows(b, which)
            if not rows:
                continue
            slots = np.array(sorted(rows))
            want_bits = row_bits(np.stack([rows[s] for s in slots]), w.dtype)     # [n, Hkv, d]
            got = arr[b][:, slots, :].transpose(1, 0, 2)
            assert np.array_equal(got, want_bits), "%s rows of request %d differ" % (which, b)


def to_dev(*ts):
    return [t.cuda() for t in ts]
