"""Seeded synthetic inputs shaped like the decode workloads (no method arithmetic here).

Both the CUDA path and the CPU oracle take their inputs from this module; it
draws random numbers and nothing else.  Every tensor comes from its own
``torch.Generator`` seeded from (workload seed, tensor name), so the values do
not depend on the order in which tensors are drawn.  Draws on a CUDA device and
on the CPU give different (equally valid) streams for the same seed; a
comparison always draws on one device and copies to the other.

Distributions: standard normal drawn in fp32, optionally scaled in fp32, then
rounded to the cache dtype by ``Tensor.to`` (round to nearest even).
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass, field
from typing import List, Optional

import torch


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1000003 + zlib.crc32(name.encode())) & 0x7FFFFFFFFFFFFFFF)
    return g


def normal(shape, seed: int, name: str, device="cpu", dtype=torch.float32, scale: float = 1.0):
    """N(0,1) values of ``shape`` from the stream (seed, name), times ``scale`` in fp32."""
    x = torch.randn(tuple(shape), generator=_gen(seed, name, device), device=device,
                    dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(dtype)


def uniform_int(n: int, lo: int, hi: int, seed: int, name: str) -> List[int]:
    """n integers uniform in [lo, hi] (inclusive), drawn on the CPU."""
    g = _gen(seed, name, "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def outlier_channels(n_heads: int, d: int, count: int, seed: int, name: str) -> torch.Tensor:
    """``count`` distinct channels per head, [n_heads, count] (int64, CPU)."""
    g = _gen(seed, name, "cpu")
    return torch.stack([torch.randperm(d, generator=g)[:count].sort().values for _ in range(n_heads)])


@dataclass
class Workload:
    """Shape and seeds of one decode workload; the fields mirror ``kvc_config``."""

    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    layout: str            # "contiguous" or "ring"
    capacity: int          # max_seq_len (contiguous) or ring size W
    window: int            # attention window (0 = full); a ring uses its size
    rope_base: float       # 0 = no rotary embedding
    dtype: str             # "f32" or "bf16"
    quant: Optional[str]   # None or "int8"
    seed: int
    key_scale: float = 1.0
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    # ------------------------------------------------------------------ draws
    def keys(self, shape, name, device="cpu"):
        return normal(shape, self.seed, "k/" + name, device, self.torch_dtype, self.key_scale)

    def values(self, shape, name, device="cpu"):
        return normal(shape, self.seed, "v/" + name, device, self.torch_dtype)

    def queries(self, shape, name, device="cpu"):
        return normal(shape, self.seed, "q/" + name, device, self.torch_dtype)

    def step_qkv(self, step: int, device="cpu"):
        """q [B, Hq, d], k and v [B, Hkv, d] of decode step ``step`` (pre-RoPE)."""
        B, Hq, Hkv, d = self.batch, self.n_q_heads, self.n_kv_heads, self.head_dim
        k = self.keys((B, Hkv, d), "step%d" % step, device)
        if self.extra.get("outliers"):
            k = self.apply_outliers(k)
        return (self.queries((B, Hq, d), "step%d" % step, device), k,
                self.values((B, Hkv, d), "step%d" % step, device))

    def token_table(self, vocab: int, device="cpu"):
        """Rows keyed by token ID: q [vocab, Hq, d], k and v [vocab, Hkv, d] (pre-RoPE).

        A prefill of token IDs ``ids`` takes rows ``k[ids]``, ``v[ids]``; equal IDs give
        equal rows, which is what prefix reuse by token ID relies on.
        """
        Hq, Hkv, d = self.n_q_heads, self.n_kv_heads, self.head_dim
        return (self.queries((vocab, Hq, d), "tokens", device), self.keys((vocab, Hkv, d), "tokens", device),
                self.values((vocab, Hkv, d), "tokens", device))

    def prefill_chunk(self, chunk: int, rows: int, device="cpu"):
        """k, v [B, Hkv, rows, d] for positions chunk*rows .. chunk*rows+rows-1."""
        B, Hkv, d = self.batch, self.n_kv_heads, self.head_dim
        k = self.keys((B, Hkv, rows, d), "prefill%d" % chunk, device)
        if self.extra.get("outliers"):
            k = self.apply_outliers(k)
        return k, self.values((B, Hkv, rows, d), "prefill%d" % chunk, device)

    def apply_outliers(self, k: torch.Tensor) -> torch.Tensor:
        """Scale the seeded outlier channels of every KV head (before RoPE), in fp32."""
        count, factor = self.extra["outliers"]
        ch = outlier_channels(self.n_kv_heads, self.head_dim, count, self.seed, "outliers")
        kf = k.float()
        for h in range(self.n_kv_heads):
            idx = ch[h].to(k.device)
            kf[:, h, ..., idx] = kf[:, h, ..., idx] * factor
        return kf.to(k.dtype)


# ---------------------------------------------------------------------- the workloads

def toy(variant: str = "full") -> Workload:
    """Toy decode, fp32: B=1, H=2, d=4, seed 7; 64 steps.

    variant "full": contiguous max_seq_len 64; "ring": ring W=4; "trim": contiguous
    history of 8 tokens trimmed at cut=4 and continued with 8 new tokens.
    """
    if variant == "ring":
        return Workload("toy-ring", 1, 2, 2, 4, "ring", 4, 4, 0.0, "f32", None, 7)
    if variant == "trim":
        return Workload("toy-trim", 1, 2, 2, 4, "contiguous", 64, 0, 0.0, "f32", None, 7,
                        extra={"history": 8, "cut": 4, "suffix": 8})
    return Workload("toy-full", 1, 2, 2, 4, "contiguous", 64, 0, 0.0, "f32", None, 7)


def full_cache_mha() -> Workload:
    """Full-cache MHA decode, bf16: B=32, Hq=Hkv=32, d=128, context 4096 + 128 steps, cache 8192.

    Keys are N(0,1) times 1/sqrt(2) (fp32) rounded to bf16; seed 11.
    """
    return Workload("full-cache-mha-bf16", 32, 32, 32, 128, "contiguous", 8192, 0, 0.0, "bf16",
                    None, 11, key_scale=2.0 ** -0.5, extra={"context": 4096, "steps": 128})


def sliding_window_gqa() -> Workload:
    """Sliding-window GQA decode, bf16: B=64, Hq=32, Hkv=8, d=128, ring W=4096, RoPE 10000.

    Per-request current position L_b - 1 with L_b uniform in [1, 32768] (seed 23).
    """
    w = Workload("sliding-window-gqa-bf16", 64, 32, 8, 128, "ring", 4096, 4096, 10000.0, "bf16",
                 None, 23, extra={"max_len": 32768})
    w.extra["lengths"] = uniform_int(w.batch, 1, 32768, w.seed, "lengths")
    return w


def prefix_reuse(windowed: bool = False) -> Workload:
    """Prefix-reuse suffix recompute, bf16: 16 requests, Hq=32, Hkv=8, d=128, prefix 8192, suffix 512.

    Cuts uniform in [0, 8191] (seed 7); RoPE 10000; full attention or W=4096.
    """
    w = Workload("prefix-reuse-%s-bf16" % ("w4096" if windowed else "full"), 16, 32, 8, 128,
                 "contiguous", 8192 + 512, 4096 if windowed else 0, 10000.0, "bf16", None, 7,
                 extra={"prefix": 8192, "suffix": 512})
    w.extra["cuts"] = uniform_int(w.batch, 0, 8191, w.seed, "cuts")
    return w


def int8_witness() -> Workload:
    """INT8 KV with witnesses: B=8, Hq=32, Hkv=8, d=128, context 131072, RoPE 10000, seed 7.

    Keys N(0,1) with 4 seeded outlier channels per head scaled x20 before RoPE.
    """
    return Workload("int8-witness-bf16", 8, 32, 8, 128, "contiguous", 131072 + 16, 0, 10000.0,
                    "bf16", "int8", 7, extra={"context": 131072, "steps": 16, "outliers": (4, 20.0)})


def int8_witness_ring() -> Workload:
    """The INT8 + witness workload on a sliding-window ring of W = 32768 slots: the same
    tokens (context 131072, 4 outlier channels per head x 20, RoPE 10000, seed 7), of which
    the ring keeps the newest 2048 complete blocks and the exact tail."""
    w = int8_witness()
    w.name, w.layout, w.capacity, w.window = "int8-witness-ring-bf16", "ring", 32768, 32768
    return w


def int8_dither() -> Workload:
    """Tier B at the INT8 workload's shape: the same tokens, subtractive-dither INT8 codes
    without witnesses; Philox key (0x243F6A88, 0x85A308D3), layer 0."""
    w = int8_witness()
    w.name, w.quant = "int8-dither-bf16", "int8-dither"
    w.extra.update(dither_key=(0x243F6A88, 0x85A308D3), layer=0)
    return w


def small(name="small", B=2, Hq=4, Hkv=2, d=128, layout="contiguous", capacity=300, window=0,
          rope_base=10000.0, dtype="bf16", quant=None, seed=11, **extra) -> Workload:
    """A parity-sized workload of any shape (several tiles and a ragged tail)."""
    return Workload(name, B, Hq, Hkv, d, layout, capacity, window, rope_base, dtype, quant, seed,
                    extra=dict(extra))


def as_numpy(t: torch.Tensor):
    """Host copy for the oracle: fp32 values as float32, bf16 as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
