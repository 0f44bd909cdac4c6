"""ctypes binding of ``libkvc.so`` (``include/kvc.h``): argument marshalling only.

Every function has the name of the C entry point it calls and raises
:class:`KvcError` on a non-zero status.  Device arguments are torch CUDA tensors
(checked for device, dtype, shape and contiguity here, then passed as raw
pointers); the stream defaults to torch's current stream.  All computation runs
in the library's kernels; if the library has not been built this module raises
on first use -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import numpy as np
import torch

from . import build as _build

KVC_OK, KVC_ERR_ARG, KVC_ERR_CAPACITY, KVC_ERR_EVICTED, KVC_ERR_CUDA, KVC_ERR_UNSUPPORTED, KVC_ERR_DEVICE = range(7)
KVC_F32, KVC_BF16 = 0, 1
KVC_CONTIGUOUS, KVC_RING = 0, 1
KVC_QUANT_NONE, KVC_QUANT_INT8, KVC_QUANT_INT8_DITHER = 0, 1, 2
(KVC_EXPORT_K, KVC_EXPORT_V, KVC_EXPORT_POSITIONS, KVC_EXPORT_NEXT_POSITION, KVC_EXPORT_KQ, KVC_EXPORT_VQ,
 KVC_EXPORT_SK, KVC_EXPORT_SV, KVC_EXPORT_WITNESS, KVC_EXPORT_KTAIL, KVC_EXPORT_VTAIL, KVC_EXPORT_XMAP,
 KVC_EXPORT_PAGE_TABLE) = range(13)

_STATUS_NAMES = {1: "KVC_ERR_ARG", 2: "KVC_ERR_CAPACITY", 3: "KVC_ERR_EVICTED", 4: "KVC_ERR_CUDA",
                 5: "KVC_ERR_UNSUPPORTED", 6: "KVC_ERR_DEVICE"}


class KvcError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s (%s)" % (where, _STATUS_NAMES.get(code, code), kvc_strerror(code)))


class kvc_config(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("layout", ctypes.c_int32), ("kv_quant", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("capacity", ctypes.c_int32), ("window", ctypes.c_int32),
                ("max_position", ctypes.c_int32), ("rope_base", ctypes.c_float), ("max_chunk", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("int8_exact_blocks", ctypes.c_int32), ("page_pool", ctypes.c_int32),
                ("store_slots", ctypes.c_int32), ("layer_index", ctypes.c_int32),
                ("dither_key_lo", ctypes.c_uint32), ("dither_key_hi", ctypes.c_uint32),
                ("int8_split", ctypes.c_int32)]


EXPORTED = ["kvc_state_bytes", "kvc_create", "kvc_destroy", "kvc_append", "kvc_append_rows",
            "kvc_decode_attn", "kvc_trim", "kvc_chunk_attn", "kvc_export_bytes", "kvc_export",
            "kvc_next_positions", "kvc_device_status", "kvc_prefix_cut", "kvc_strerror",
            "kvc_int8_block_risk", "kvc_int8_gate", "kvc_int8_restore",
            "kvc_pstore_create", "kvc_pstore_destroy", "kvc_pstore_insert", "kvc_pstore_lookup",
            "kvc_store_save", "kvc_store_load", "kvc_store_load_batch", "kvc_set_request_id",
            "kvc_check_wait_path"]

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built (no fallback path exists)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError("libkvc.so is not built (%s); run kv_cache_decode_ring_gb300.build.build()" % path)
            L = ctypes.CDLL(path)
            P, i32, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            cfgp = ctypes.POINTER(kvc_config)
            sig = {
                "kvc_state_bytes": [cfgp, ctypes.POINTER(u64)],
                "kvc_create": [cfgp, P, u64, P, ctypes.POINTER(P)],
                "kvc_destroy": [P],
                "kvc_append": [P, P, P, P],
                "kvc_append_rows": [P, P, P, i32, P, P],
                "kvc_decode_attn": [P, P, P, P, P, P, P],
                "kvc_trim": [P, P, P],
                "kvc_chunk_attn": [P, P, P, P, i32, P, P],
                "kvc_export_bytes": [P, i32, ctypes.POINTER(u64)],
                "kvc_export": [P, i32, P, u64, P],
                "kvc_next_positions": [P, P],
                "kvc_device_status": [P, P, ctypes.POINTER(i32)],
                "kvc_prefix_cut": [P, i32, P, i32, i32, ctypes.POINTER(i32)],
                "kvc_decode_attn_noalloc": [P, P, P, P],
                "kvc_int8_block_risk": [P, P, P, P],
                "kvc_int8_gate": [P, i32, i32, i32, ctypes.c_double, i32, P, ctypes.POINTER(i32)],
                "kvc_int8_restore": [P, P, i32, P, P, P],
                "kvc_pstore_create": [cfgp, i32, ctypes.POINTER(P)],
                "kvc_pstore_destroy": [P],
                "kvc_pstore_insert": [P, P, i32, ctypes.c_char_p, P, i32, ctypes.POINTER(i32)],
                "kvc_pstore_lookup": [P, P, i32, ctypes.c_char_p, P, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)],
                "kvc_store_save": [P, i32, i32, i32, P],
                "kvc_store_load": [P, i32, i32, i32, P],
                "kvc_store_load_batch": [P, i32, P, P, P, P],
                "kvc_set_request_id": [P, i32, ctypes.c_uint32, P],
                "kvc_check_wait_path": [P, P],
            }
            for name, args in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            L.kvc_strerror.argtypes = [ctypes.c_int]
            L.kvc_strerror.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _check(rc: int, where: str):
    if rc != KVC_OK:
        raise KvcError(rc, where)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def _dev(t: Optional[torch.Tensor], dtype=None, shape=None, name="tensor") -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return ctypes.c_void_p(t.data_ptr())


def kvc_strerror(code: int) -> str:
    return lib().kvc_strerror(int(code)).decode()


def make_config(dtype="bf16", layout="contiguous", kv_quant=None, batch=1, n_q_heads=1, n_kv_heads=1,
                head_dim=128, capacity=1, window=0, max_position=0, rope_base=0.0, max_chunk=0,
                out_dtype=None, int8_exact_blocks=0, page_pool=0, store_slots=0, layer_index=0,
                dither_key=(0, 0), int8_split=0) -> kvc_config:
    """``out_dtype``: None (the cache dtype), "f32" or "bf16"; ``int8_exact_blocks``: pool
    entries for blocks the gated fallback restores (INT8 caches); ``page_pool``: pages of 16
    slots for paged K/V storage (0 = each request owns ``capacity`` slots); ``store_slots``:
    device slots for saved prefills (prefix store).  ``kv_quant``: None, "int8" (witness
    tier) or "int8-dither" (Tier B, with ``layer_index`` and the 64-bit Philox ``dither_key``
    as (low, high) words); ``int8_split``: positions per quantized split of the INT8 decode
    (a multiple of 64 in [1024, 2048]; 0 = chosen for the device)."""
    od = 0 if out_dtype is None else (KVC_F32 + 1 if out_dtype == "f32" else KVC_BF16 + 1)
    return kvc_config(KVC_BF16 if dtype == "bf16" else KVC_F32,
                      KVC_RING if layout == "ring" else KVC_CONTIGUOUS,
                      {None: KVC_QUANT_NONE, "int8": KVC_QUANT_INT8, "int8-dither": KVC_QUANT_INT8_DITHER}[kv_quant],
                      batch, n_q_heads, n_kv_heads, head_dim, capacity, window, max_position,
                      float(rope_base), max_chunk, od, int(int8_exact_blocks), int(page_pool), int(store_slots),
                      int(layer_index), int(dither_key[0]) & 0xFFFFFFFF, int(dither_key[1]) & 0xFFFFFFFF,
                      int(int8_split))


def kvc_state_bytes(cfg: kvc_config) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().kvc_state_bytes(ctypes.byref(cfg), ctypes.byref(n)), "kvc_state_bytes")
    return n.value


def kvc_create(cfg: kvc_config, state: torch.Tensor, stream=None) -> ctypes.c_void_p:
    h = ctypes.c_void_p(0)
    _check(lib().kvc_create(ctypes.byref(cfg), _dev(state, name="state"), state.numel() * state.element_size(),
                            _stream(stream), ctypes.byref(h)), "kvc_create")
    return h


def kvc_destroy(h) -> None:
    _check(lib().kvc_destroy(h), "kvc_destroy")


def kvc_append(h, k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
    _check(lib().kvc_append(h, _dev(k, name="k"), _dev(v, name="v"), _stream(stream)), "kvc_append")


def kvc_append_rows(h, k: torch.Tensor, v: torch.Tensor, n: int, counts: Optional[Sequence[int]] = None,
                    stream=None) -> None:
    c = None if counts is None else (ctypes.c_int32 * len(counts))(*[int(x) for x in counts])
    _check(lib().kvc_append_rows(h, _dev(k, name="k"), _dev(v, name="v"), int(n),
                                 ctypes.cast(c, ctypes.c_void_p) if c is not None else None, _stream(stream)),
           "kvc_append_rows")


def kvc_decode_attn(h, q, out, cmax=None, tanh=None, ct=None, stream=None) -> None:
    _check(lib().kvc_decode_attn(h, _dev(q, name="q"), _dev(out, name="out"), _dev(cmax, torch.float32, name="cmax"),
                                 _dev(tanh, torch.float32, name="tanh"), _dev(ct, torch.float32, name="ct"),
                                 _stream(stream)), "kvc_decode_attn")


def kvc_int8_block_risk(h, ct, risk, stream=None) -> None:
    _check(lib().kvc_int8_block_risk(h, _dev(ct, torch.float32, name="ct"), _dev(risk, torch.float32, name="risk"),
                                     _stream(stream)), "kvc_int8_block_risk")


def kvc_int8_gate(risk: np.ndarray, tau: float, max_blocks: int) -> np.ndarray:
    """Host selection: [n, 3] int32 (request, KV head, block) triples, highest risk first."""
    r = np.ascontiguousarray(np.asarray(risk, dtype=np.float32))
    if r.ndim != 3:
        raise ValueError("risk must be [B, Hkv, nblk]")
    sel = np.zeros((max(int(max_blocks), 1), 3), dtype=np.int32)
    n = ctypes.c_int32(0)
    _check(lib().kvc_int8_gate(r.ctypes.data_as(ctypes.c_void_p), r.shape[0], r.shape[1], r.shape[2],
                               ctypes.c_double(tau), int(max_blocks), sel.ctypes.data_as(ctypes.c_void_p),
                               ctypes.byref(n)), "kvc_int8_gate")
    return sel[:n.value].copy()


def kvc_int8_restore(h, blocks, k_full, v_full, stream=None) -> None:
    b = np.ascontiguousarray(np.asarray(blocks, dtype=np.int32).reshape(-1, 3))
    _check(lib().kvc_int8_restore(h, b.ctypes.data_as(ctypes.c_void_p) if len(b) else None, len(b),
                                  _dev(k_full, torch.bfloat16, name="k_full"),
                                  _dev(v_full, torch.bfloat16, name="v_full"), _stream(stream)), "kvc_int8_restore")


KVC_NOALLOC_SCRATCH_BYTES = 64 << 20


def kvc_decode_attn_noalloc(h, q, out, stream=None) -> None:
    """Decode attention whose split-K scratch is the library's fixed device array.

    For callers that cannot allocate device memory while they decode; see
    include/kvc.h.  Calls that overlap on the GPU share (and race on) that array."""
    _check(lib().kvc_decode_attn_noalloc(h, _dev(q, name="q"), _dev(out, name="out"), _stream(stream)),
           "kvc_decode_attn_noalloc")


def kvc_trim(h, cuts: Sequence[int], stream=None) -> None:
    c = (ctypes.c_int32 * len(cuts))(*[int(x) for x in cuts])
    _check(lib().kvc_trim(h, ctypes.cast(c, ctypes.c_void_p), _stream(stream)), "kvc_trim")


def kvc_chunk_attn(h, q, k, v, n: int, out, stream=None) -> None:
    _check(lib().kvc_chunk_attn(h, _dev(q, name="q"), _dev(k, name="k"), _dev(v, name="v"), int(n),
                                _dev(out, name="out"), _stream(stream)), "kvc_chunk_attn")


def kvc_export_bytes(h, which: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().kvc_export_bytes(h, int(which), ctypes.byref(n)), "kvc_export_bytes")
    return n.value


def kvc_export(h, which: int, stream=None) -> np.ndarray:
    """Raw bytes of one state array (uint8); callers view them with the documented dtype."""
    n = kvc_export_bytes(h, which)
    buf = np.empty(n, dtype=np.uint8)
    _check(lib().kvc_export(h, int(which), buf.ctypes.data_as(ctypes.c_void_p), n, _stream(stream)), "kvc_export")
    return buf


def kvc_next_positions(h, batch: int) -> np.ndarray:
    out = np.empty(batch, dtype=np.int32)
    _check(lib().kvc_next_positions(h, out.ctypes.data_as(ctypes.c_void_p)), "kvc_next_positions")
    return out


def kvc_device_status(h, stream=None) -> int:
    s = ctypes.c_int32(0)
    _check(lib().kvc_device_status(h, _stream(stream), ctypes.byref(s)), "kvc_device_status")
    return s.value


def kvc_check_wait_path(h, stream=None) -> None:
    _check(lib().kvc_check_wait_path(h, _stream(stream)), "kvc_check_wait_path")


def kvc_prefix_cut(old_ids: Sequence[int], new_ids: Sequence[int], ring: bool = False) -> int:
    for x in list(old_ids) + list(new_ids):
        if isinstance(x, bool) or not isinstance(x, (int, np.integer)):
            raise TypeError("token IDs must be integers")
    o = np.ascontiguousarray(np.asarray(old_ids, dtype=np.int64))
    n = np.ascontiguousarray(np.asarray(new_ids, dtype=np.int64))
    cut = ctypes.c_int32(0)
    _check(lib().kvc_prefix_cut(o.ctypes.data_as(ctypes.c_void_p), len(o), n.ctypes.data_as(ctypes.c_void_p),
                                len(n), 1 if ring else 0, ctypes.byref(cut)), "kvc_prefix_cut")
    return cut.value


def _token_ids(ids) -> np.ndarray:
    """Token IDs as int64, refusing anything that is not an integer (1.0 is not the token 1)."""
    if isinstance(ids, torch.Tensor):
        if ids.dtype.is_floating_point or ids.dtype == torch.bool or ids.dtype.is_complex:
            raise TypeError("token IDs must be integers, got %s" % ids.dtype)
        return np.ascontiguousarray(ids.detach().cpu().numpy().astype(np.int64).reshape(-1))
    if isinstance(ids, np.ndarray):
        if ids.dtype.kind not in "iu":
            raise TypeError("token IDs must be integers, got %s" % ids.dtype)
        return np.ascontiguousarray(ids.astype(np.int64).reshape(-1))
    for x in ids:
        if isinstance(x, bool) or not isinstance(x, (int, np.integer)):
            raise TypeError("token IDs must be integers, got %r" % (x,))
    return np.ascontiguousarray(np.asarray(list(ids), dtype=np.int64).reshape(-1))


def _sig(signature) -> bytes:
    return signature.encode() if isinstance(signature, str) else bytes(signature)


def kvc_pstore_create(cfg: kvc_config, capacity: int) -> ctypes.c_void_p:
    ps = ctypes.c_void_p(0)
    _check(lib().kvc_pstore_create(ctypes.byref(cfg), int(capacity), ctypes.byref(ps)), "kvc_pstore_create")
    return ps


def kvc_pstore_destroy(ps) -> None:
    _check(lib().kvc_pstore_destroy(ps), "kvc_pstore_destroy")


def kvc_pstore_insert(ps, ids, scope: str, signature=b"") -> int:
    a, sg = _token_ids(ids), _sig(signature)
    slot = ctypes.c_int32(-1)
    _check(lib().kvc_pstore_insert(ps, a.ctypes.data_as(ctypes.c_void_p) if len(a) else None, len(a),
                                   scope.encode(), sg or None, len(sg), ctypes.byref(slot)), "kvc_pstore_insert")
    return slot.value


def kvc_pstore_lookup(ps, ids, scope: str, signature=b"") -> tuple:
    a, sg = _token_ids(ids), _sig(signature)
    slot, cut = ctypes.c_int32(-1), ctypes.c_int32(0)
    _check(lib().kvc_pstore_lookup(ps, a.ctypes.data_as(ctypes.c_void_p) if len(a) else None, len(a),
                                   scope.encode(), sg or None, len(sg), ctypes.byref(slot), ctypes.byref(cut)),
           "kvc_pstore_lookup")
    return slot.value, cut.value


def kvc_store_save(h, slot: int, b: int, n: int, stream=None) -> None:
    _check(lib().kvc_store_save(h, int(slot), int(b), int(n), _stream(stream)), "kvc_store_save")


def kvc_store_load(h, slot: int, b: int, cut: int, stream=None) -> None:
    _check(lib().kvc_store_load(h, int(slot), int(b), int(cut), _stream(stream)), "kvc_store_load")


def kvc_set_request_id(h, b: int, request_id: int, stream=None) -> None:
    _check(lib().kvc_set_request_id(h, int(b), int(request_id) & 0xFFFFFFFF, _stream(stream)), "kvc_set_request_id")


def kvc_store_load_batch(h, slots, bs, cuts, stream=None) -> None:
    arr = [np.ascontiguousarray(np.asarray(x, dtype=np.int32).reshape(-1)) for x in (slots, bs, cuts)]
    n = len(arr[0])
    if any(len(x) != n for x in arr):
        raise ValueError("slots, requests and cuts must have one entry per load")
    ptr = [x.ctypes.data_as(ctypes.c_void_p) if n else None for x in arr]
    _check(lib().kvc_store_load_batch(h, n, ptr[0], ptr[1], ptr[2], _stream(stream)), "kvc_store_load_batch")


class PrefixStore:
    """Host policy of the prefix store (see include/kvc.h): which stored prefill a query
    reuses, and how many rows.  The rows live in a Cache's store slots."""

    def __init__(self, cfg: kvc_config, capacity: int = 2):
        self.capacity = capacity
        self.ps = kvc_pstore_create(cfg, capacity)

    def insert(self, ids, scope: str, signature=b"") -> int:
        return kvc_pstore_insert(self.ps, ids, scope, signature)

    def lookup(self, ids, scope: str, signature=b"") -> tuple:
        """(slot, cut); slot -1 when nothing is reusable."""
        return kvc_pstore_lookup(self.ps, ids, scope, signature)

    def close(self):
        if self.ps is not None and self.ps.value:
            kvc_pstore_destroy(self.ps)
        self.ps = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Cache:
    """A KV cache of one layer on the current CUDA device: the state buffer (a torch
    uint8 tensor) plus its library handle.  Thin wrapper over the functions above."""

    _EXPORT_DTYPES = {KVC_EXPORT_POSITIONS: np.int32, KVC_EXPORT_NEXT_POSITION: np.int32, KVC_EXPORT_KQ: np.int8,
                      KVC_EXPORT_VQ: np.int8, KVC_EXPORT_SK: np.float32, KVC_EXPORT_SV: np.float32,
                      KVC_EXPORT_WITNESS: np.uint16, KVC_EXPORT_KTAIL: np.uint16, KVC_EXPORT_VTAIL: np.uint16,
                      KVC_EXPORT_XMAP: np.int32, KVC_EXPORT_PAGE_TABLE: np.int32}

    def __init__(self, cfg: kvc_config, device="cuda", stream=None):
        self.cfg = cfg
        self.torch_dtype = torch.bfloat16 if cfg.dtype == KVC_BF16 else torch.float32
        if cfg.out_dtype == 0:
            self.out_dtype = self.torch_dtype
        else:
            self.out_dtype = torch.float32 if cfg.out_dtype == KVC_F32 + 1 else torch.bfloat16
        nbytes = kvc_state_bytes(cfg)
        self.state = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.h = kvc_create(cfg, self.state, stream)

    @classmethod
    def from_workload(cls, w, max_chunk=0, max_position=0, device="cuda", out_dtype=None, int8_exact_blocks=0,
                      page_pool=0, store_slots=0, int8_split=0):
        cfg = make_config(w.dtype, w.layout, w.quant, w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.capacity,
                          0 if w.layout == "ring" else w.window, max_position, w.rope_base, max_chunk, out_dtype,
                          int8_exact_blocks, page_pool, store_slots, w.extra.get("layer", 0),
                          w.extra.get("dither_key", (0, 0)), int8_split)
        return cls(cfg, device)

    def close(self):
        if self.h is not None and self.h.value:
            kvc_destroy(self.h)
        self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # shapes
    @property
    def B(self): return self.cfg.batch
    @property
    def Hq(self): return self.cfg.n_q_heads
    @property
    def Hkv(self): return self.cfg.n_kv_heads
    @property
    def d(self): return self.cfg.head_dim
    @property
    def S(self): return self.cfg.capacity

    def append(self, k, v, stream=None):
        _dev(k, self.torch_dtype, (self.B, self.Hkv, self.d), "k")
        _dev(v, self.torch_dtype, (self.B, self.Hkv, self.d), "v")
        kvc_append(self.h, k, v, stream)

    def append_rows(self, k, v, counts=None, stream=None):
        n = k.shape[2]
        _dev(k, self.torch_dtype, (self.B, self.Hkv, n, self.d), "k")
        _dev(v, self.torch_dtype, (self.B, self.Hkv, n, self.d), "v")
        kvc_append_rows(self.h, k, v, n, counts, stream)

    def decode(self, q, out=None, cmax=None, tanh=None, ct=None, stream=None):
        _dev(q, self.torch_dtype, (self.B, self.Hq, self.d), "q")
        if out is None:
            out = torch.empty(q.shape, dtype=self.out_dtype, device=q.device)
        _dev(out, self.out_dtype, (self.B, self.Hq, self.d), "out")
        kvc_decode_attn(self.h, q, out, cmax, tanh, ct, stream)
        return out

    def trim(self, cuts, stream=None):
        if len(cuts) != self.B:
            raise ValueError("need one cut per request")
        kvc_trim(self.h, cuts, stream)

    def chunk(self, q, k, v, out=None, stream=None):
        n = q.shape[1]
        _dev(q, self.torch_dtype, (self.B, n, self.Hq, self.d), "q")
        _dev(k, self.torch_dtype, (self.B, n, self.Hkv, self.d), "k")
        _dev(v, self.torch_dtype, (self.B, n, self.Hkv, self.d), "v")
        if out is None:
            out = torch.empty(q.shape, dtype=self.out_dtype, device=q.device)
        _dev(out, self.out_dtype, (self.B, n, self.Hq, self.d), "out")
        kvc_chunk_attn(self.h, q, k, v, n, out, stream)
        return out

    def export(self, which, stream=None) -> np.ndarray:
        raw = kvc_export(self.h, which, stream)
        if which in (KVC_EXPORT_K, KVC_EXPORT_V):
            dt = np.uint16 if self.cfg.dtype == KVC_BF16 else np.float32
            return raw.view(dt).reshape(self.B, self.Hkv, self.S, self.d)
        arr = raw.view(self._EXPORT_DTYPES[which])
        shapes = {KVC_EXPORT_POSITIONS: (self.B, self.S), KVC_EXPORT_NEXT_POSITION: (self.B,),
                  KVC_EXPORT_KQ: (self.B, self.Hkv, self.S, self.d),
                  KVC_EXPORT_VQ: (self.B, self.Hkv, self.S, self.d),
                  KVC_EXPORT_SK: (self.B, self.Hkv, self.S // 16), KVC_EXPORT_SV: (self.B, self.Hkv, self.S // 16),
                  KVC_EXPORT_WITNESS: (self.B, self.Hkv, self.S, 16), KVC_EXPORT_KTAIL: (self.B, self.Hkv, 16, self.d),
                  KVC_EXPORT_VTAIL: (self.B, self.Hkv, 16, self.d),
                  KVC_EXPORT_XMAP: (self.B, self.Hkv, self.S // 16),
                  KVC_EXPORT_PAGE_TABLE: (self.B, self.S // 16)}
        return arr.reshape(shapes[which])

    def next_positions(self) -> np.ndarray:
        return kvc_next_positions(self.h, self.B)

    # gated fallback of the INT8 tier
    def block_risk(self, ct, risk=None, stream=None):
        """Per complete block, the largest c_t over its tokens and the KV head's query heads."""
        _dev(ct, torch.float32, (self.B, self.Hq, self.S), "ct")
        if risk is None:
            risk = torch.empty((self.B, self.Hkv, self.S // 16), dtype=torch.float32, device=ct.device)
        _dev(risk, torch.float32, (self.B, self.Hkv, self.S // 16), "risk")
        kvc_int8_block_risk(self.h, ct, risk, stream)
        return risk

    def restore(self, blocks, k_full, v_full, stream=None):
        _dev(k_full, torch.bfloat16, (self.B, self.Hkv, self.S, self.d), "k_full")
        _dev(v_full, torch.bfloat16, (self.B, self.Hkv, self.S, self.d), "v_full")
        kvc_int8_restore(self.h, blocks, k_full, v_full, stream)

    def device_status(self, stream=None) -> int:
        return kvc_device_status(self.h, stream)

    def set_request_id(self, b, request_id, stream=None):
        kvc_set_request_id(self.h, b, request_id, stream)

    # prefix store
    def store_save(self, slot, b, n, stream=None):
        kvc_store_save(self.h, slot, b, n, stream)

    def store_load(self, slot, b, cut, stream=None):
        kvc_store_load(self.h, slot, b, cut, stream)

    def store_load_batch(self, slots, bs, cuts, stream=None):
        kvc_store_load_batch(self.h, slots, bs, cuts, stream)

    def save_prefix(self, store: PrefixStore, b, ids, scope: str, signature=b"", stream=None) -> int:
        """Records request b's prefill of ``ids`` in ``store`` and copies its rows to the slot."""
        slot = store.insert(ids, scope, signature)
        kvc_store_save(self.h, slot, b, len(_token_ids(ids)), stream)
        return slot

    def reuse_prefix(self, store: PrefixStore, b, ids, scope: str, signature=b"", stream=None) -> tuple:
        """Request b continues from the longest reusable stored prefix of ``ids``: (slot, cut)."""
        slot, cut = store.lookup(ids, scope, signature)
        kvc_store_load(self.h, slot, b, cut, stream)
        return slot, cut
