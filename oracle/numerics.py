"""ctypes front end of ``oracle.c`` (number formats, RoPE, fp64 attention, INT8 tier).

TEST INFRASTRUCTURE (see the package docstring).  ``build()`` compiles
``oracle.c`` with gcc; nothing here touches a GPU.

[LEAN]    "用Lean4形式化验证滑动窗口KV Cache的正确性" (framerc.cn/news/4505248)
[LOOP]    "KV Cache 自回归生成推理（增量更新与状态拼接）" (airsota.com/?p=549)
[WITCERT] "WitCert: Sound Runtime Risk Observability and Gating for KV-Cache Quantization"
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
          "-frounding-math", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``oracle/_build/liboracle.so`` (if stale) and return its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            i64, i32, f32, f64, u16 = (ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                       ctypes.c_double, ctypes.c_uint16)
            sig = {
                "orc_version": (i32, []),
                "orc_bf16_to_f32": (f32, [u16]),
                "orc_f32_to_bf16": (u16, [f32]),
                "orc_f32_to_bf16_array": (None, [P, P, i64]),
                "orc_bf16_to_f32_array": (None, [P, P, i64]),
                "orc_f16_value": (f64, [u16]),
                "orc_f32_to_f16_up": (u16, [f32]),
                "orc_rope_cos_sin": (None, [f64, i32, i64, i64, P]),
                "orc_rope_rotate": (None, [P, P, i64, i32, P]),
                "orc_attend_batch": (None, [i32, i32, i32, i32, i64, P, P, P, P, P, P, P, i32]),
                "orc_softmax_weights": (i64, [i32, P, i64, i32, P, i64, i64, i64, P]),
                "orc_quantize_block": (f32, [P, i64, P]),
                "orc_witness_row": (i32, [P, P, f32, i32, i32, P]),
                "orc_residual_row": (None, [P, P, f32, i32, P]),
                "orc_philox4x32_10": (None, [P, P, P]),
                "orc_quantize_block_dither": (f32, [P, P, i64, P]),
                "orc_dither_rows": (None, [P, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, i64, i64, i32,
                                           P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- number formats

def f32_to_bf16(x) -> np.ndarray:
    """Round fp32 values to bf16 bit patterns (nearest, ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16_array(_p(x), _p(y), x.size)
    return y


def bf16_to_f32(b) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    y = np.empty(b.shape, dtype=np.float32)
    lib().orc_bf16_to_f32_array(_p(b), _p(y), b.size)
    return y


def f16_value(h: int) -> float:
    return lib().orc_f16_value(int(h))


def f32_to_f16_up(x: float) -> int:
    """Bit pattern of the smallest fp16 value >= x (x is first taken as fp32)."""
    return int(lib().orc_f32_to_f16_up(float(np.float32(x))))


# ---------------------------------------------------------------- RoPE

def rope_cos_sin(base: float, d: int, p0: int, n: int) -> np.ndarray:
    """{cos, sin} rows for positions p0..p0+n-1: float32 [n, d/2, 2] (see oracle.c for the reading)."""
    cs = np.empty((n, d // 2, 2), dtype=np.float32)
    if n:
        lib().orc_rope_cos_sin(float(base), d, int(p0), int(n), _p(cs))
    return cs


def rope_rotate(x, positions, base: float) -> np.ndarray:
    """Rotate fp32 rows ``x[..., d]`` at the given absolute positions (fp32, one rounding per op)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = x.shape[-1]
    rows = x.reshape(-1, d)
    pos = np.asarray(positions, dtype=np.int64).reshape(-1)
    if pos.size != rows.shape[0]:
        pos = np.broadcast_to(pos.reshape(()) if pos.size == 1 else pos, x.shape[:-1]).reshape(-1)
    # each distinct position's {cos, sin} row once (a position's row does not depend on the
    # others computed with it), then gathered per row
    uniq, inv = np.unique(pos, return_inverse=True)
    if uniq.size and uniq[-1] - uniq[0] < 4 * uniq.size + 64:
        table = rope_cos_sin(base, d, int(uniq[0]), int(uniq[-1] - uniq[0]) + 1)[uniq - uniq[0]]
    else:
        table = np.stack([rope_cos_sin(base, d, int(u), 1)[0] for u in uniq]) if uniq.size else \
            np.empty((0, d // 2, 2), dtype=np.float32)
    cs = np.ascontiguousarray(table[inv.reshape(-1)], dtype=np.float32)
    y = np.empty_like(rows)
    if rows.shape[0]:
        lib().orc_rope_rotate(_p(rows), _p(cs), rows.shape[0], d, _p(y))
    return y.reshape(x.shape)


# ---------------------------------------------------------------- attention

KIND_F32, KIND_BF16, KIND_F64 = 0, 1, 2


def attend(q, hist_k, hist_v, t, window=0, p0=0, kind=None, nthreads=1) -> np.ndarray:
    """Masked attention of one or more query rows over one history ([LEAN] §2.1).

    ``q``: [nq, d] (fp64 or castable); ``hist_k``/``hist_v``: [n, d] as fp32, fp64
    or bf16 bit patterns (uint16); row j holds position ``p0 + j``; ``t`` is the
    query position; ``window`` W > 0 masks positions < t - W + 1.  fp64 result.
    """
    return attend_many([q], [hist_k], [hist_v], [t], window, [p0], kind, nthreads)[0]


def _kind_of(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return KIND_BF16
    if a.dtype == np.float32:
        return KIND_F32
    if a.dtype == np.float64:
        return KIND_F64
    raise TypeError(a.dtype)


def attend_many(qs, ks, vs, ts, window=0, p0s=None, kind=None, nthreads=1) -> list:
    """Independent problems of :func:`attend`, run on ``nthreads`` threads (OpenMP)."""
    nprob = len(qs)
    if nprob == 0:
        return []
    q = np.ascontiguousarray(np.stack([np.atleast_2d(np.asarray(a, dtype=np.float64)) for a in qs]))
    nq, d = q.shape[1], q.shape[2]
    ks = [np.ascontiguousarray(a) for a in ks]
    vs = [np.ascontiguousarray(a) for a in vs]
    kd = _kind_of(ks[0]) if kind is None else kind
    for a in ks + vs:
        assert _kind_of(a) == kd and (a.size == 0 or a.shape[-1] == d)
    n = np.array([a.shape[0] if a.size else 0 for a in ks], dtype=np.int64)
    p0 = np.zeros(nprob, dtype=np.int64) if p0s is None else np.asarray(p0s, dtype=np.int64)
    t = np.asarray(ts, dtype=np.int64)
    kp = (ctypes.c_void_p * nprob)(*[a.ctypes.data for a in ks])
    vp = (ctypes.c_void_p * nprob)(*[a.ctypes.data for a in vs])
    out = np.zeros((nprob, nq, d), dtype=np.float64)
    lib().orc_attend_batch(nprob, nq, d, kd, int(window), _p(q),
                           ctypes.cast(kp, ctypes.c_void_p), ctypes.cast(vp, ctypes.c_void_p),
                           _p(n), _p(p0), _p(t), _p(out), int(nthreads))
    return [out[i] for i in range(nprob)]


def softmax_weights(q, hist_k, t, window=0, p0=0) -> np.ndarray:
    """Softmax weights of one query row over a history, same masks as :func:`attend` (fp64)."""
    q = np.ascontiguousarray(q, dtype=np.float64).reshape(-1)
    k = np.ascontiguousarray(hist_k)
    p = np.zeros(k.shape[0], dtype=np.float64)
    lib().orc_softmax_weights(q.size, _p(q), k.shape[0], _kind_of(k), _p(k), int(p0), int(t),
                              int(window), _p(p))
    return p


# ---------------------------------------------------------------- INT8 tier

def quantize_block(x) -> tuple:
    """(scale, int8 codes) of one block of fp32 values; see ``orc_quantize_block``."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.empty(x.shape, dtype=np.int8)
    s = lib().orc_quantize_block(_p(x), x.size, _p(codes))
    return np.float32(s), codes


def witness_row(x, codes, s, nbands=16) -> np.ndarray:
    """fp16 bit patterns of the per-band residual-norm upper bounds of one key row."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    w = np.empty(nbands, dtype=np.uint16)
    rc = lib().orc_witness_row(_p(x), _p(codes), float(s), x.size, nbands, _p(w))
    if rc != 0:
        raise ArithmeticError("residual not exact in fp32 (rc=%d)" % rc)
    return w


def residual_row(x, codes, s) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    r = np.empty_like(x)
    lib().orc_residual_row(_p(x), _p(codes), float(s), x.size, _p(r))
    return r


def philox4x32_10(ctr, key) -> np.ndarray:
    """Philox4x32-10 of one counter (4 uint32) under one key (2 uint32): 4 uint32 words."""
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint64).astype(np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint64).astype(np.uint32))
    out = np.empty(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


# Subtractive-dither streams ([WITCERT] Tier B: Philox keyed on the five-tuple
# request, layer, KV head, token, channel).  Keys are dithered; values keep the plain
# block quantizer (the tier's certificate concerns the logits, i.e. the keys, and the
# page's counter has no key/value field).  The counter of one call is
#   (position t, channel group, KV head + 65536 * layer, request ID)
# under the cache's 64-bit key; group j covers channels 16 j .. 16 j + 15, and byte i of
# the call (word i/4, least significant byte first) is channel 16 j + i; a channel's
# dither is u = r / 256 - 1/2.
def dither_bytes(key, request, layer, kv_head, position, d) -> np.ndarray:
    """The d key dither bytes of one row as uint8, one Philox call at a time in Python
    (the plain statement of the mapping above)."""
    out = np.empty(d, dtype=np.uint8)
    c2 = (int(kv_head) + 65536 * int(layer)) & 0xFFFFFFFF
    for j in range(d // 16):
        w = philox4x32_10([position, j, c2, request], key)
        out[16 * j:16 * j + 16] = w.view(np.uint8)
    return out


def dither_rows(key, request, layer, kv_head, p0, n, d) -> np.ndarray:
    """dither_bytes of rows p0 .. p0+n-1, [n, d] uint8 (``orc_dither_rows``)."""
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint64).astype(np.uint32))
    out = np.empty((n, d), dtype=np.uint8)
    lib().orc_dither_rows(_p(k), int(request) & 0xFFFFFFFF, int(layer), int(kv_head), int(p0), int(n), int(d),
                          _p(out))
    return out


def dither_values(rbytes) -> np.ndarray:
    """u = r / 256 - 1/2 (exact in fp32)."""
    return (np.asarray(rbytes, dtype=np.float32) / np.float32(256.0) - np.float32(0.5)).astype(np.float32)


def quantize_block_dither(x, u) -> tuple:
    """(scale, int8 codes) of one block with the subtractive dither u; see ``orc_quantize_block_dither``."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = np.ascontiguousarray(u, dtype=np.float32)
    assert u.shape == x.shape
    codes = np.empty(x.shape, dtype=np.int8)
    s = lib().orc_quantize_block_dither(_p(x), _p(u), x.size, _p(codes))
    return np.float32(s), codes


def f16_values(bits) -> np.ndarray:
    """Values of fp16 bit patterns (numpy's binary16 decoding)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)
