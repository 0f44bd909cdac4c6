#!/usr/bin/env python
"""Decode-step benchmark: one JSON line on stdout (rank 0).

A step is one pass of the hot path for the whole batch: ``kvc_append`` (k_t, v_t
at position t, RoPE if configured) followed by ``kvc_decode_attn`` (split-K
decode attention of the new query over its cached window).  The default workload
is full-cache MHA decode in bf16: 32 requests, 32 query = 32 KV heads, head_dim
128, contiguous cache of 8192, context 4096 plus one token per step; after 128
steps every request is trimmed back to 4096 (one ``kvc_trim``), so contexts cycle
through 4097..4224 keys.  Inputs are synthetic (seeded N(0,1), keys x 1/sqrt 2).

value    = decode-attention KV bytes per second over the timed steps (whole job),
           KV bytes = sum over requests and KV heads of keys x d x 2 (K and V) x 2 B.
e2e      = the same metric through the C ABI with host buffers: every step copies
           q, k, v from pinned host memory and the output back, inside the timing.
roofline = the decode-attention call (split-K kernel + combine) timed with CUDA
           events on its stream; algorithmic bytes = KV bytes + q + out per call.

lines    = (default run only) the same measurement, value and roofline with its own
           clocks, for the INT8 + witness decode, the sliding-window GQA decode, the
           chunked suffix attention (full and W = 4096) and the INT8 Tier B decode.

--gpus N without torchrun starts N ranks under torch.distributed.run, one replica of
the workload per GPU (weak scaling, no collective on the data path).
--impl reference times the CPU oracle instead (fp64 attention by definition, on
the host cores) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
CSRC = os.path.join(ROOT, "kv_cache_decode_ring_gb300", "csrc")

# DRAM traffic (ncu dram__bytes_read.sum + dram__bytes_write.sum) of the dominant kernel
# per byte of the bench's traffic basis (the decode call's algorithmic bytes; for the chunk
# kernel the K/V bytes of the step), from the small-case captures summarised in profiles/;
# valid only while the kernel source is the one captured (sha256 prefix), otherwise the
# JSON line reports null.
TRAFFIC_PER_BYTE = {
    "full-cache-mha": ("decode_fast.cu", "ea05ecaf8cc06944", (268707328 + 4217088) / 268632064),
    "sliding-window-gqa": ("decode_gqa.cu", "68a52c99893be10e", (268102912 + 3000064) / 268148736),
    "int8-witness": ("int8.cu", "8753292bf0d3a988", (302857984 + 2983168) / 302551040),
    "bf16-at-int8-shape": ("decode_gqa.cu", "68a52c99893be10e", (536976640 + 3210240) / 536907776),
    # (the chunk's reads also include the query, 16.8 MB in this 4-request capture, which the
    # K/V basis leaves out)
    "prefix-reuse": ("chunk.cu", "de37e058599ee090", (83959552 + 3649792) / 60850176),
    "prefix-reuse-w4096": ("chunk.cu", "de37e058599ee090", (77292288 + 3273984) / 60850176),
    "int8-dither": ("int8.cu", "8753292bf0d3a988", (269328128 + 3047936) / 268996608),
    # (2 requests: 16 x (2048 blocks of codes, witnesses and scales + 3 tail rows) = 151.28 MB)
    "int8-witness-ring": ("int8.cu", "8753292bf0d3a988", (151496448 + 3245312) / 151281664),
    "full-cache-mha-paged": ("decode_fast.cu", "ea05ecaf8cc06944", (268708608 + 4353280) / 268632064),
    "sliding-window-gqa-paged": ("decode_gqa.cu", "68a52c99893be10e", (268100608 + 2968064) / 268148736),
    "prefix-reuse-store": ("chunk.cu", "de37e058599ee090", (83959552 + 3649792) / 60850176),   # the same chunk launch
    # the store's batched row copy (8 requests' cuts, 297.9 MB read + written): writes still in L2
    # at the end of the launch are not counted, so the ratio is below 1
    "store-load": ("store.cu", "817adec9d1411abf", (149277440 + 95578624) / 297918464),
}


def traffic_per_launch(workload, basis_bytes):
    import hashlib
    entry = TRAFFIC_PER_BYTE.get(workload)
    if not entry:
        return None
    src, sha, ratio = entry
    with open(os.path.join(CSRC, src), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest()[:16] != sha:
            return None
    return int(ratio * basis_bytes)
FALLBACK_HBM_GBS = 6800.0
METRIC = "decode-attention KV bytes/s (GB/s, % of HBM peak) and decode steps/s at 1 GB300"


def hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 TFLOP/s sustained over a seconds-long loop (the timed region is one)."""
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1700.0, "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9 and parts[0].isdigit() and int(parts[0]) == self.gpu_index:
                self.rows.append(parts)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in self.rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x for x in vis.split(",") if x.strip()]
    if ids and all(x.strip().isdigit() for x in ids) and local_rank < len(ids):
        return int(ids[local_rank])
    return local_rank


# ----------------------------------------------------------------------------- workloads

def kv_bytes_per_step(nkeys_per_request, Hkv, d, elem=2):
    return sum(nkeys_per_request) * Hkv * d * 2 * elem


class DecodeBench:
    """Common driver: a cache, a cycle of per-step inputs on the device, and the step
    ``kvc_append`` + ``kvc_decode_attn``.  Subclasses fill the cache and count bytes."""

    CYCLE = 64
    PAGED = False                       # K/V in 16-slot pages behind a block table
    kernel = "kvc_decode_attn (split-K decode + combine)"
    metric = METRIC
    unit = "GB/s"
    bound = "hbm"

    def _inputs(self, device):
        import torch
        w = self.w
        steps = [w.step_qkv(s, device=device) for s in range(self.CYCLE)]
        self.q = [s[0] for s in steps]
        self.k = [s[1] for s in steps]
        self.v = [s[2] for s in steps]
        self.out = torch.empty_like(self.q[0])
        self.done = 0
        torch.cuda.synchronize()

    def io_bytes(self):
        w = self.w
        return (2 * w.batch * w.n_q_heads * w.head_dim) * 2      # q read + out write (bf16)

    def traffic_basis(self, attn_bytes):
        return attn_bytes                                        # DRAM traffic scales with these

    def launches_per_step(self):
        return 3                                                 # append, split-K decode, combine

    def before_step(self):
        return 0                                                 # extra launches (e.g. a trim)

    def decode(self, q):
        self.cache.decode(q, self.out)

    def step(self, ev=None):
        j = self.done % self.CYCLE
        extra = self.before_step()
        self.cache.append(self.k[j], self.v[j])
        if ev is not None:
            ev[0].record()
        self.decode(self.q[j])
        if ev is not None:
            ev[1].record()
        self.done += 1
        return extra

    # ---- end to end through the public API, with host buffers -----------------
    # Every step uploads its inputs from pinned host memory and downloads its output;
    # two device slots for each and a copy stream let one step's copies overlap its
    # neighbours' kernels.  Subclasses say which host inputs step n uses and how a step
    # computes from device inputs into a given output.
    def e2e_setup(self):
        import torch
        self.hq = [t.cpu().pin_memory() for t in self.q]
        self.hk = [t.cpu().pin_memory() for t in self.k]
        self.hv = [t.cpu().pin_memory() for t in self.v]
        return self.e2e_init([self.hq[0], self.hk[0], self.hv[0]], self.out)

    def e2e_host_inputs(self, n):
        j = n % self.CYCLE
        return self.hq[j], self.hk[j], self.hv[j]

    def e2e_compute(self, dev, out):
        q, k, v = dev
        self.before_step()
        self.cache.append(k, v)
        keep = self.out
        self.out = out
        self.decode(q)
        self.out = keep

    def e2e_init(self, host_example, out_example):
        import torch
        self.e2e_dev = [[torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in host_example] for _ in range(2)]
        self.e2e_dout = [torch.empty_like(out_example) for _ in range(2)]
        self.e2e_hout = [torch.empty(out_example.shape, dtype=out_example.dtype).pin_memory() for _ in range(2)]
        # uploads and downloads on streams of their own, so the two copy directions overlap
        self.up_stream = torch.cuda.Stream()
        self.down_stream = torch.cuda.Stream()
        self.ev_in = [torch.cuda.Event() for _ in range(2)]      # slot's inputs uploaded
        self.ev_used = [torch.cuda.Event() for _ in range(2)]    # slot's inputs consumed, output written
        self.ev_read = [torch.cuda.Event() for _ in range(2)]    # slot's output downloaded
        self.e2e_next = None                                     # step whose inputs are in flight
        return sum(t.numel() * t.element_size() for t in host_example), \
            self.e2e_hout[0].numel() * self.e2e_hout[0].element_size()

    def _upload(self, n):
        """Upload stream: the inputs of step n into slot n % 2 once that slot is free."""
        import torch
        s = n % 2
        with torch.cuda.stream(self.up_stream):
            self.up_stream.wait_event(self.ev_used[s])
            for dst, src in zip(self.e2e_dev[s], self.e2e_host_inputs(n)):
                dst.copy_(src, non_blocking=True)
            self.ev_in[s].record(self.up_stream)

    def e2e_step(self):
        """One step: its inputs uploaded, its kernels, its output downloaded.  The next
        step's upload is issued now, so it overlaps this step's kernels, and this step's
        download overlaps the next step's kernels."""
        import torch
        n = self.done
        s = n % 2
        if self.e2e_next != n:
            self._upload(n)
        self._upload(n + 1)
        self.e2e_next = n + 1
        cur = torch.cuda.current_stream()
        cur.wait_event(self.ev_in[s])
        cur.wait_event(self.ev_read[s])                          # the slot's previous output downloaded
        self.e2e_compute(self.e2e_dev[s], self.e2e_dout[s])
        self.ev_used[s].record(cur)
        with torch.cuda.stream(self.down_stream):
            self.down_stream.wait_event(self.ev_used[s])
            self.e2e_hout[s].copy_(self.e2e_dout[s], non_blocking=True)
            self.ev_read[s].record(self.down_stream)
        self.done += 1

    def e2e_flush(self):
        """The current stream waits for the last download; a pending upload is dropped
        (the next step uploads its own inputs again)."""
        import torch
        for st in (self.up_stream, self.down_stream):
            done = torch.cuda.Event()
            done.record(st)
            torch.cuda.current_stream().wait_event(done)
        self.e2e_next = None


def full_cache_config(w, ctx, cycle):
    """The full-cache MHA line's config (both arms print it)."""
    return {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
            "head_dim": w.head_dim, "layout": "contiguous", "max_seq_len": w.capacity,
            "context": "%d + step (cycles %d..%d keys)" % (ctx, ctx + 1, ctx + cycle),
            "l2": "inputs larger than L2: %.2f GB of K/V read per step vs 129 MB L2"
                  % (kv_bytes_per_step([ctx + 1] * w.batch, w.n_kv_heads, w.head_dim) / 1e9)}


class FullCacheBench(DecodeBench):
    """Full-cache MHA decode, bf16: B=32, H=32, d=128, contiguous 8192, context 4096 + steps;
    every 128 steps the requests are trimmed back to 4096."""

    CYCLE = 128

    def __init__(self, device, batch=None, total_steps=0):
        from kv_cache_decode_ring_gb300 import kvc
        from kv_cache_decode_ring_gb300 import workloads as wl
        self.w = w = wl.full_cache_mha()
        if batch:
            w.batch = batch                   # smaller case for profiler captures
        self.ctx = w.extra["context"]
        # a paged cache gets exactly the pages the cycle needs: ceil((ctx + CYCLE) / 16) a request
        pool = w.batch * -(-(self.ctx + self.CYCLE) // 16) if self.PAGED else 0
        self.cache = kvc.Cache.from_workload(w, device=device, page_pool=pool)
        k, v = w.prefill_chunk(0, self.ctx, device=device)
        self.cache.append_rows(k, v)
        del k, v
        self.cuts = [self.ctx] * w.batch
        self._inputs(device)

    def before_step(self):
        if self.done % self.CYCLE == 0 and self.done > 0:
            self.cache.trim(self.cuts)
            return 1
        return 0

    def units(self):
        """KV bytes read by the decode of the step about to run (the cycle position is done mod 128)."""
        n = self.ctx + (self.done % self.CYCLE) + 1
        return kv_bytes_per_step([n] * self.w.batch, self.w.n_kv_heads, self.w.head_dim)

    def reset(self):
        import torch
        self.cache.trim(self.cuts)
        self.done = 0
        torch.cuda.synchronize()

    def cpu_problem(self):
        return self.ctx + 1, 1

    def config(self):
        return full_cache_config(self.w, self.ctx, self.CYCLE)


class SlidingWindowBench(DecodeBench):
    """Sliding-window GQA decode, bf16: B=64, Hq=32, Hkv=8, d=128, ring W=4096, RoPE 10000,
    request b starts at position L_b - 1 (L_b uniform in [1, 32768]) and advances one token a step."""

    def __init__(self, device, batch=None, total_steps=0):
        from kv_cache_decode_ring_gb300 import kvc
        from kv_cache_decode_ring_gb300 import workloads as wl
        self.w = w = wl.sliding_window_gqa()
        if batch:
            w.batch = batch                   # smaller case for profiler captures: the first requests
            w.extra["lengths"] = w.extra["lengths"][:batch]
        self.W = w.capacity
        self.L = list(w.extra["lengths"])
        maxp = w.extra["max_len"] + total_steps + 64
        pool = w.batch * (self.W // 16) if self.PAGED else 0   # every ring fills its window
        self.cache = kvc.Cache.from_workload(w, max_position=maxp, device=device, page_pool=pool)
        chunk = 4096
        for c in range((max(self.L) + chunk - 1) // chunk):
            counts = [int(min(max(L - 1 - c * chunk, 0), chunk)) for L in self.L]
            if any(counts):
                k, v = w.prefill_chunk(c, chunk, device=device)
                self.cache.append_rows(k, v, counts=counts)
                del k, v
        self._inputs(device)

    def units(self):
        n = [min(L + self.done, self.W) for L in self.L]
        return kv_bytes_per_step(n, self.w.n_kv_heads, self.w.head_dim)

    def reset(self):
        import torch
        torch.cuda.synchronize()              # a ring keeps advancing; nothing to undo

    def cpu_problem(self):
        return self.W, self.w.n_q_heads // self.w.n_kv_heads

    def config(self):
        w = self.w
        return {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
                "head_dim": w.head_dim, "layout": "ring", "window": self.W, "rope_base": w.rope_base,
                "context": "L_b - 1 + step, L_b uniform in [1, 32768] (seed 23)",
                "l2": "inputs larger than L2: %.2f GB of K/V read per step vs 129 MB L2" % (self.units() / 1e9)}


class Int8Bench(DecodeBench):
    """INT8 KV with witnesses: B=8, Hq=32, Hkv=8, d=128, context 131072 prefilled through the
    block quantizer; each step appends one token and runs the fused decode + bound."""

    kernel = "kvc_decode_attn INT8 (fused decode + witness bound + combine)"

    def __init__(self, device, batch=None, total_steps=0):
        import torch
        from kv_cache_decode_ring_gb300 import kvc
        self.w = w = self.make_workload()
        if batch:
            w.batch = batch                   # smaller case for profiler captures
        self.ctx = w.extra["context"]
        w.capacity = self.ctx + 16 * ((total_steps + 16 + 15) // 16)
        self.cache = kvc.Cache.from_workload(w, device=device, int8_exact_blocks=self.pool_blocks())
        chunk = 8192
        for c in range(self.ctx // chunk):
            k, v = w.prefill_chunk(c, chunk, device=device)
            self.cache.append_rows(k, v)
            del k, v
        B, Hq = w.batch, w.n_q_heads
        self.cmax = torch.empty((B, Hq), device=device)
        self.tanh = torch.empty((B, Hq), device=device)
        self._inputs(device)

    def make_workload(self):
        from kv_cache_decode_ring_gb300 import workloads as wl
        return wl.int8_witness()

    def pool_blocks(self):
        return 0

    def decode(self, q):
        self.cache.decode(q, self.out, self.cmax, self.tanh)

    def units(self):
        """Bytes the fused decode reads: codes, witnesses and scales of complete blocks, exact tail rows
        (and the bf16 rows of blocks restored by the gated fallback)."""
        w = self.w
        n = self.ctx + self.done + 1
        nfull = n // 16 * 16
        per_head = nfull * (2 * w.head_dim + 32) + (nfull // 16) * 8 + (n - nfull) * 4 * w.head_dim
        return w.batch * w.n_kv_heads * per_head + getattr(self, "restored", 0) * 16 * 4 * w.head_dim

    def reset(self):
        import torch
        torch.cuda.synchronize()

    def cpu_problem(self):
        return 4096, self.w.n_q_heads // self.w.n_kv_heads

    def config(self):
        w = self.w
        return {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
                "head_dim": w.head_dim, "layout": "contiguous int8 + witnesses", "context": "131072 + step",
                "l2": "inputs larger than L2: %.2f GB read per step vs 129 MB L2" % (self.units() / 1e9)}


class Int8RingBench(Int8Bench):
    """INT8 + witness on a ring of 32768 slots at the INT8 workload's shape: the 131072-token
    prefill streams through the ring (blocks overwritten within the call are never stored),
    then each step appends one token and runs the fused decode over the window."""

    kernel = "kvc_decode_attn INT8 on a ring (fused decode + witness bound + combine)"

    def __init__(self, device, batch=None, total_steps=0):
        import torch
        from kv_cache_decode_ring_gb300 import kvc
        from kv_cache_decode_ring_gb300 import workloads as wl
        self.w = w = wl.int8_witness_ring()
        if batch:
            w.batch = batch                   # smaller case for profiler captures
        self.ctx = w.extra["context"]
        self.W = w.capacity
        self.cache = kvc.Cache.from_workload(w, device=device, max_position=self.ctx + total_steps + 64)
        chunk = 8192
        for c in range(self.ctx // chunk):
            k, v = w.prefill_chunk(c, chunk, device=device)
            self.cache.append_rows(k, v)
            del k, v
        B, Hq = w.batch, w.n_q_heads
        self.cmax = torch.empty((B, Hq), device=device)
        self.tanh = torch.empty((B, Hq), device=device)
        self._inputs(device)

    def units(self):
        """Bytes the fused decode reads: the ring's complete blocks (codes, witnesses, scales) and
        the exact tail rows."""
        w = self.w
        n = self.ctx + self.done + 1
        nblk = min(n // 16, self.W // 16)
        per_head = nblk * 16 * (2 * w.head_dim + 32) + nblk * 8 + (n - n // 16 * 16) * 4 * w.head_dim
        return w.batch * w.n_kv_heads * per_head

    def config(self):
        c = super().config()
        c["workload"] = self.w.name
        c["layout"] = "ring of %d slots, int8 + witnesses" % self.W
        c["context"] = "131072 + step positions, window %d" % self.W
        return c


class Int8CtBench(Int8Bench):
    """The INT8 workload with the decode also writing every cached token's c_t (fp32
    [B][Hq][capacity]), the input of the gated fallback's block risk: the same reads plus
    B x Hq x n_keys x 4 bytes written per step."""

    kernel = "kvc_decode_attn INT8 with per-token c_t (fused decode + witness bound + c_t write + combine)"

    def __init__(self, device, batch=None, total_steps=0):
        import torch
        super().__init__(device, batch, total_steps)
        self.ct = torch.zeros((self.w.batch, self.w.n_q_heads, self.cache.S), device=device)

    def decode(self, q):
        self.cache.decode(q, self.out, self.cmax, self.tanh, self.ct)

    def units(self):
        w = self.w
        return super().units() + w.batch * w.n_q_heads * (self.ctx + self.done + 1) * 4

    def config(self):
        c = super().config()
        c["workload"] = "int8-witness-ct"
        c["ct"] = "fp32 c_t of every cached token written per step (%.3f GB)" % (
            self.w.batch * self.w.n_q_heads * (self.ctx + 1) * 4 / 1e9)
        return c


class Int8DitherBench(Int8Bench):
    """Tier B at the INT8 workload's shape: subtractive-dither INT8 codes and scales, no
    witnesses (Philox key 0x85A308D3243F6A88, layer 0, request IDs 0..7); each step appends
    one token and runs the decode, which regenerates every dither it reads."""

    kernel = "kvc_decode_attn INT8 Tier B (Philox dither regenerated in the decode + combine)"

    def make_workload(self):
        from kv_cache_decode_ring_gb300 import workloads as wl
        return wl.int8_dither()

    def decode(self, q):
        self.cache.decode(q, self.out)

    def units(self):
        """Bytes the decode reads: codes and scales of complete blocks, exact tail rows."""
        w = self.w
        n = self.ctx + self.done + 1
        nfull = n // 16 * 16
        per_head = nfull * 2 * w.head_dim + (nfull // 16) * 8 + (n - nfull) * 4 * w.head_dim
        return w.batch * w.n_kv_heads * per_head

    def config(self):
        c = super().config()
        c["layout"] = "contiguous int8 Tier B (subtractive dither, no witnesses)"
        return c


class Int8GatedBench(Int8Bench):
    """The INT8 workload after one gated fallback: a decode with per-token c_t, block risk,
    gate at tau = 0.2 with a budget of 1 % of the complete blocks (highest risk first),
    restore from a bf16 backing store; then the same decode steps as the INT8 bench, with
    the restored blocks served exactly.  The gate's own cost (risk, selection, restore) is
    reported in the config."""

    TAU = 0.2
    BUDGET_FRAC = 0.01

    def pool_blocks(self):
        w = self.w
        return max(1, int(self.BUDGET_FRAC * w.batch * w.n_kv_heads * (w.extra["context"] // 16)))

    def __init__(self, device, batch=None, total_steps=0):
        import copy
        import time
        import numpy as np
        import torch
        from kv_cache_decode_ring_gb300 import kvc
        super().__init__(device, batch, total_steps)
        w = self.w
        # backing store: the same tokens in a bf16 cache, exported to device tensors
        wb = copy.copy(w)
        wb.quant = None
        full = kvc.Cache.from_workload(wb, device=device)
        for c in range(self.ctx // 8192):
            k, v = w.prefill_chunk(c, 8192, device=device)
            full.append_rows(k, v)
            del k, v
        kf = torch.from_numpy(full.export(kvc.KVC_EXPORT_K).view(np.int16)).view(torch.bfloat16).to(device)
        vf = torch.from_numpy(full.export(kvc.KVC_EXPORT_V).view(np.int16)).view(torch.bfloat16).to(device)
        full.close()
        del full
        torch.cuda.empty_cache()
        # one decode with c_t, then the gate
        B, Hq = w.batch, w.n_q_heads
        ct = torch.zeros((B, Hq, self.cache.S), device=device)
        self.cache.decode(self.q[0], self.out, self.cmax, self.tanh, ct)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        risk = self.cache.block_risk(ct).cpu().numpy()
        t1 = time.perf_counter()
        sel = kvc.kvc_int8_gate(risk, self.TAU, self.pool_blocks())
        t2 = time.perf_counter()
        self.cache.restore(sel, kf, vf)
        torch.cuda.synchronize()
        t3 = time.perf_counter()
        self.restored = len(sel)
        self.risky = int((np.tanh(risk.astype(np.float64)) > self.TAU).sum())
        self.gate_ms = {"risk_and_readback": round((t1 - t0) * 1e3, 3), "select": round((t2 - t1) * 1e3, 3),
                        "restore": round((t3 - t2) * 1e3, 3)}
        del ct, kf, vf
        torch.cuda.empty_cache()

    def config(self):
        c = super().config()
        c["workload"] = "int8-witness-gated"
        c["gate"] = {"tau": self.TAU, "budget_blocks": self.pool_blocks(), "risky_blocks": self.risky,
                     "restored_blocks": self.restored, "ms": self.gate_ms}
        return c


class FullCachePagedBench(FullCacheBench):
    """The full-cache MHA workload on a paged cache (pages handed out in a shuffled order)."""
    PAGED = True

    def config(self):
        c = super().config()
        c["workload"] += "-paged"
        c["layout"] = "contiguous, paged (16-slot pages, block table)"
        return c


class SlidingWindowPagedBench(SlidingWindowBench):
    """The sliding-window GQA workload on a paged ring."""
    PAGED = True

    def config(self):
        c = super().config()
        c["workload"] += "-paged"
        c["layout"] = "ring, paged (16-slot pages, block table)"
        return c


class Bf16AtInt8ShapeBench(DecodeBench):
    """The bf16 decode at the INT8 workload's shape (B=8, Hq=32, Hkv=8, d=128, context 131072,
    same keys with outlier channels and RoPE), for comparison with the INT8 tier: the same
    tokens cost 512 B per KV head in bf16 against 288.5 B quantized."""

    def __init__(self, device, batch=None, total_steps=0):
        from kv_cache_decode_ring_gb300 import kvc
        from kv_cache_decode_ring_gb300 import workloads as wl
        self.w = w = wl.int8_witness()
        w.quant = None
        w.name = "bf16-at-int8-shape"
        if batch:
            w.batch = batch                   # smaller case for profiler captures
        self.ctx = w.extra["context"]
        w.capacity = self.ctx + total_steps + 16
        self.cache = kvc.Cache.from_workload(w, device=device)
        chunk = 8192
        for c in range(self.ctx // chunk):
            k, v = w.prefill_chunk(c, chunk, device=device)
            self.cache.append_rows(k, v)
            del k, v
        self._inputs(device)

    def units(self):
        w = self.w
        return kv_bytes_per_step([self.ctx + self.done + 1] * w.batch, w.n_kv_heads, w.head_dim)

    def reset(self):
        import torch
        torch.cuda.synchronize()

    def cpu_problem(self):
        return 4096, self.w.n_q_heads // self.w.n_kv_heads

    def config(self):
        w = self.w
        return {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
                "head_dim": w.head_dim, "layout": "contiguous bf16", "context": "131072 + step",
                "l2": "inputs larger than L2: %.2f GB read per step vs 129 MB L2" % (self.units() / 1e9)}


class ChunkBench(DecodeBench):
    """Prefix-reuse suffix recompute, bf16: 16 requests, Hq=32, Hkv=8, d=128, prefix 8192 rows
    (RoPE 10000), cuts uniform in [0, 8191] (seed 7).  A step trims every request to its cut and
    runs kvc_chunk_attn on a 512-token suffix (append, rotate, causal tcgen05 attention)."""

    kernel = "kvc_chunk_attn (suffix append + tcgen05 causal attention with the query rotation fused)"
    metric = "chunked suffix attention FLOP/s (TFLOP/s, % of bf16 tensor peak) at 1 GB300"
    unit = "TFLOP/s"
    bound = "tensor"

    def __init__(self, device, batch=None, total_steps=0, windowed=False):
        import torch
        from kv_cache_decode_ring_gb300 import kvc
        from kv_cache_decode_ring_gb300 import workloads as wl
        self.w = w = wl.prefix_reuse(windowed)
        if batch:
            w.batch = batch                   # smaller case for profiler captures: the first requests
            w.extra["cuts"] = w.extra["cuts"][:batch]
        self.n = w.extra["suffix"]
        self.cache = self.make_cache(w, device)
        pre = w.extra["prefix"]
        for c in range(pre // 2048):
            k, v = w.keys((w.batch, w.n_kv_heads, 2048, w.head_dim), "prefix%d" % c, device), \
                w.values((w.batch, w.n_kv_heads, 2048, w.head_dim), "prefix%d" % c, device)
            self.cache.append_rows(k, v)
            del k, v
        self.cuts = list(w.extra["cuts"])
        B, n, Hq, Hkv, d = w.batch, self.n, w.n_q_heads, w.n_kv_heads, w.head_dim
        self.q = w.queries((B, n, Hq, d), "suffix", device)
        self.k = w.keys((B, n, Hkv, d), "suffix", device)
        self.v = w.values((B, n, Hkv, d), "suffix", device)
        self.out = torch.empty_like(self.q)
        self.done = 0
        W = w.window
        keys = 0
        for c in self.cuts:
            for i in range(n):
                p = c + i
                keys += p + 1 - (max(0, p - W + 1) if W else 0)
        self.flops = 4.0 * keys * Hq * d
        torch.cuda.synchronize()

    def make_cache(self, w, device):
        from kv_cache_decode_ring_gb300 import kvc
        return kvc.Cache.from_workload(w, max_chunk=self.n, device=device)

    def launches_per_step(self):
        return 4                                   # trim, append rows, advance, attention

    def traffic_basis(self, flops):
        w = self.w                                 # the K/V rows a step's attention reads
        return sum(c + self.n for c in self.cuts) * w.n_kv_heads * w.head_dim * 4

    def step(self, ev=None):
        self.cache.trim(self.cuts)
        if ev is not None:
            ev[0].record()
        self.cache.chunk(self.q, self.k, self.v, self.out)
        if ev is not None:
            ev[1].record()
        self.done += 1
        return 0

    def units(self):
        return self.flops

    def io_bytes(self):
        return 0

    def e2e_setup(self):
        self.hq, self.hk, self.hv = (t.cpu().pin_memory() for t in (self.q, self.k, self.v))
        return self.e2e_init([self.hq, self.hk, self.hv], self.out)

    def e2e_host_inputs(self, n):
        return self.hq, self.hk, self.hv

    def e2e_compute(self, dev, out):
        self.cache.trim(self.cuts)
        self.cache.chunk(dev[0], dev[1], dev[2], out)

    def reset(self):
        import torch
        torch.cuda.synchronize()

    def cpu_problem(self):
        return 4096, self.w.n_q_heads // self.w.n_kv_heads

    def config(self):
        w = self.w
        return {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
                "head_dim": w.head_dim, "prefix": w.extra["prefix"], "suffix": self.n, "window": w.window,
                "cuts": "uniform in [0, 8191], seed 7", "gflop_per_step": round(self.flops / 1e9, 2),
                "l2": "K/V of a step %.2f GB (> 129 MB L2)"
                      % (sum(c + self.n for c in self.cuts) * w.n_kv_heads * w.head_dim * 4 / 1e9)}


class ChunkWindowBench(ChunkBench):
    def __init__(self, device, batch=None, total_steps=0):
        super().__init__(device, batch, total_steps, windowed=True)


class ChunkStoreBench(ChunkBench):
    """The prefix-reuse workload through the prefix store: every request's 8192-row prefill is
    saved in a store slot under its token IDs; a step looks up each request's query (the first
    cut IDs of its prefill, then 512 new IDs) on the host, copies the kept rows back into the
    request (kvc_store_load), and runs kvc_chunk_attn on the suffix."""

    def __init__(self, device, batch=None, total_steps=0):
        import numpy as np
        import torch
        from kv_cache_decode_ring_gb300 import kvc
        super().__init__(device, batch, total_steps)
        w, B = self.w, self.w.batch
        self.store = kvc.PrefixStore(self.cache.cfg, B)
        rng = np.random.default_rng(w.seed)
        pre = w.extra["prefix"]
        self.queries = []
        for r in range(B):
            ids = rng.integers(0, 1 << 31, pre, dtype=np.int64)      # token IDs labelling the prefill rows
            slot = self.cache.save_prefix(self.store, r, ids, "bench", b"prefix-reuse")
            assert slot == r
            new = rng.integers(1 << 32, 1 << 33, self.n, dtype=np.int64)   # never equal to a stored ID
            self.queries.append(np.concatenate([ids[:self.cuts[r]], new]))
        self.load_bytes = 4 * sum(self.cuts) * w.n_kv_heads * w.head_dim * 2    # K and V, read and written
        self.load_ev = []
        torch.cuda.synchronize()

    def make_cache(self, w, device):
        from kv_cache_decode_ring_gb300 import kvc
        return kvc.Cache.from_workload(w, max_chunk=self.n, device=device, store_slots=w.batch)

    def launches_per_step(self):
        return 4                                   # batched load, append rows, advance, attention

    def reuse(self, ev=False):
        import torch
        if ev:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
        slots, cuts = [], []
        for r in range(self.w.batch):                 # host lookups, then one batched load
            slot, cut = self.store.lookup(self.queries[r], "bench", b"prefix-reuse")
            slots.append(slot)
            cuts.append(cut)
        self.cache.store_load_batch(slots, list(range(self.w.batch)), cuts)
        if ev:
            b.record()
            self.load_ev.append((a, b))

    def step(self, ev=None):
        self.reuse(ev is not None)
        if ev is not None:
            ev[0].record()
        self.cache.chunk(self.q, self.k, self.v, self.out)
        if ev is not None:
            ev[1].record()
        self.done += 1
        return 0

    def e2e_compute(self, dev, out):
        self.reuse()
        self.cache.chunk(dev[0], dev[1], dev[2], out)

    def extra_report(self, peak_hbm):
        ms = [a.elapsed_time(b) for a, b in self.load_ev]
        avg = sum(ms) / len(ms)
        gbs = self.load_bytes / (avg / 1e3) / 1e9
        return {"store_load": {"kernel": "host lookups + kvc_store_load_batch (row copy of every request)",
                               "bytes_per_step": self.load_bytes, "avg_ms": round(avg, 5),
                               "achieved": round(gbs, 2), "unit": "GB/s", "peak": peak_hbm,
                               "frac": round(gbs / peak_hbm, 4),
                               "traffic": traffic_per_launch("store-load", self.load_bytes)}}

    def config(self):
        c = super().config()
        c["workload"] = self.w.name + "-store"
        c["store"] = "%d slots, one per request; lookup over %d entries of %d IDs" % (
            self.w.batch, self.w.batch, self.w.extra["prefix"])
        return c


BENCHES = {"full-cache-mha": FullCacheBench, "sliding-window-gqa": SlidingWindowBench, "int8-witness": Int8Bench,
           "bf16-at-int8-shape": Bf16AtInt8ShapeBench, "int8-witness-gated": Int8GatedBench,
           "int8-dither": Int8DitherBench, "int8-witness-ct": Int8CtBench, "int8-witness-ring": Int8RingBench,
           "full-cache-mha-paged": FullCachePagedBench, "sliding-window-gqa-paged": SlidingWindowPagedBench,
           "prefix-reuse": ChunkBench, "prefix-reuse-w4096": ChunkWindowBench, "prefix-reuse-store": ChunkStoreBench}


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(w, seconds: float, threads: int, heads_per_call=None, problem=None):
    """Time the oracle's fp64 attention (C, OpenMP) on (request, KV head) problems of the
    workload (``problem`` = (keys, query heads per KV head)); returns (GB/s of KV bytes,
    seconds, problems, description)."""
    import numpy as np
    from kv_cache_decode_ring_gb300 import workloads as wl
    from oracle import numerics as nm
    ctx, g = problem if problem else (w.extra.get("context", 4096) + 1, w.n_q_heads // w.n_kv_heads)
    d = w.head_dim
    nprob = heads_per_call or max(threads, 8)
    k = wl.as_numpy(w.keys((nprob, ctx, d), "cpu-sample"))
    v = wl.as_numpy(w.values((nprob, ctx, d), "cpu-sample"))
    q = wl.as_numpy(w.queries((nprob, g, d), "cpu-sample"))
    qf = nm.bf16_to_f32(q).astype(np.float64)
    ks = [k[i] for i in range(nprob)]
    vs = [v[i] for i in range(nprob)]
    done, t0 = 0, time.perf_counter()
    while True:
        nm.attend_many([qf[i] for i in range(nprob)], ks, vs, [ctx - 1] * nprob, 0, None, nthreads=threads)
        done += nprob
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    by = done * ctx * d * 2 * 2
    desc = ("%d (request, KV head) problems of %d query heads at %d keys, d=%d, bf16 inputs, fp64 math"
            % (done, g, ctx, d))
    return by / el / 1e9, el, done, desc


# ----------------------------------------------------------------------------- main

def replica_aggregate(ms_local, units_local, dist=None, device="cpu"):
    """Whole-job timing of replicas: (the slowest rank's milliseconds, the units all ranks
    processed).  Every rank runs its own copy of the workload (weak scaling, no data-path
    collective); only these two numbers cross ranks.  `dist` is torch.distributed with an
    initialised process group (NCCL: device "cuda"; gloo: "cpu"), or None for one process."""
    import torch
    t = torch.tensor([float(ms_local)], device=device, dtype=torch.float64)
    u = torch.tensor([float(units_local)], device=device, dtype=torch.float64)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# Lines that the default run times after the headline one, each in the same way (warm-up,
# K timed steps with CUDA events around the dominant call, clocks sampled meanwhile).
EXTRA_LINES = ("int8-witness", "sliding-window-gqa", "prefix-reuse", "prefix-reuse-w4096", "int8-dither",
               "prefix-reuse-store", "int8-witness-ring")


def call_samples(K):
    """The timed steps whose dominant call is bracketed by CUDA events: every 8th (every 4th
    below 64 steps) from the second on.  The first step follows the synchronize that opens
    the timed region, so its launches start from an idle GPU."""
    stride = 8 if K >= 64 else 4
    return list(range(1, K, stride)) or [0]


def time_steps(bench, K, warmup, local_rank, dist):
    """W untimed steps, then K timed steps bracketed by a barrier and a synchronize on both
    sides.  The dominant call of the steps call_samples(K) names is bracketed by its own
    pair of CUDA events on the stream it is launched on: an event between two kernels keeps
    the second from starting as a dependent launch during the first's tail, so events on
    every step would add their own gaps (7-8 us a step) to the step time they measure.
    Returns the slowest rank's milliseconds, the units all ranks processed, the sampled
    steps' units and call milliseconds, launches and clocks."""
    import torch

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(warmup):
        bench.step()
    bench.reset()
    sampled = call_samples(K)
    ev = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for i in sampled}
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_index(local_rank))
    sampler.start()
    time.sleep(0.3)
    barrier()
    wall0 = time.perf_counter()
    t0e.record()
    units, launches, step_units = 0, 0, []
    for i in range(K):
        u = bench.units()
        launches += bench.launches_per_step() + bench.step(ev.get(i))
        units += u
        if i in ev:
            step_units.append(u)
    t1e.record()
    barrier()
    wall = time.perf_counter() - wall0
    sampler.stop()
    ms_total, all_units = replica_aggregate(t0e.elapsed_time(t1e), units, dist, "cuda")
    return {"ms": ms_total, "units": all_units, "step_units": step_units,
            "call_ms": [ev[i][0].elapsed_time(ev[i][1]) for i in sampled], "launches": launches,
            "clocks": sampler.summary(),
            "wall": wall}


def line_summary(bench, workload, t, K):
    """Throughput of the timed steps and the roofline of the dominant call."""
    peak, peak_kind = hbm_peak() if bench.bound == "hbm" else tensor_peak()
    scale = 1e9 if bench.unit == "GB/s" else 1e12
    value = t["units"] / (t["ms"] / 1e3) / scale
    n = len(t["call_ms"])                                   # the sampled calls
    call_units = sum(u + bench.io_bytes() for u in t["step_units"]) / n
    call_ms = sum(t["call_ms"]) / n
    achieved = call_units / (call_ms / 1e3) / scale
    return {
        "value": round(value, 2), "unit": bench.unit, "ms_per_step": round(t["ms"] / K, 5), "steps": K,
        "steps_per_s": round(K / (t["ms"] / 1e3), 2), "frac_of_%s_peak" % peak_kind: round(value / peak, 4),
        "roofline": {"bound": bench.bound, "achieved": round(achieved, 2), "peak": peak, "unit": bench.unit,
                     "frac": round(achieved / peak, 4),
                     "traffic": traffic_per_launch(workload, bench.traffic_basis(call_units)),
                     "kernel": bench.kernel, "peak_kind": peak_kind,
                     "%s_per_launch" % ("bytes" if bench.unit == "GB/s" else "flops"): int(call_units),
                     "avg_launch_ms": round(call_ms, 5), "launches_timed": n},
        "gpu_launches": t["launches"], "clocks": t["clocks"], "config": bench.config(),
    }


def free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_replicas(n: int, argv) -> int:
    """Start n ranks of this script under torch.distributed.run (one per GPU, rendezvous
    on 127.0.0.1); rank 0 prints the line."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(n),
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def dry_run(args, world, rank):
    """The replica launcher without a GPU: every rank joins a gloo group, runs K trivial
    CPU steps and reports one unit per step; rank 0 prints the aggregate line.  Tests use
    it to check that --gpus N really starts N ranks."""
    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    x = torch.ones(1024)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        x = x * 1.0
    ms = (time.perf_counter() - t0) * 1e3
    ms, units = replica_aggregate(max(ms, 1e-6), args.steps, dist, "cpu")
    ranks = replica_aggregate(0.0, 1.0, dist, "cpu")[1]
    if rank == 0:
        print(json.dumps({"metric": "dry run of the replica launcher (no GPU work)", "value": units / (ms / 1e3),
                          "unit": "steps/s", "n_gpus": world, "ranks_run": int(ranks), "steps": args.steps,
                          "warmup": args.warmup, "dry_run": True}), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=None,
                    help="replicas, one per GPU (default: WORLD_SIZE under torchrun, else 1); without "
                         "torchrun, N > 1 starts N ranks itself")
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="kvc", choices=["kvc", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-lines", action="store_true",
                    help="time only the chosen workload (the default run also times %s)" % ", ".join(EXTRA_LINES))
    ap.add_argument("--dry-run", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--batch", type=int, default=0, help="override the batch (profiling a smaller case)")
    ap.add_argument("--workload", default="full-cache-mha", choices=sorted(BENCHES),
                    help="full-cache-mha (the headline line) or any other workload")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)

    env_world = os.environ.get("WORLD_SIZE")
    if env_world is None and args.gpus is not None and args.gpus > 1:
        return launch_replicas(args.gpus, argv)
    world = int(env_world) if env_world is not None else 1
    if args.gpus is not None and args.gpus != world:
        print("bench.py: --gpus %d disagrees with WORLD_SIZE=%d" % (args.gpus, world), file=sys.stderr)
        return 2
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)

    if args.dry_run:
        return dry_run(args, world, rank)
    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args, world, threads)

    import torch
    if local_rank >= torch.cuda.device_count():
        print("bench.py: rank %d has no GPU (%d visible)" % (local_rank, torch.cuda.device_count()), file=sys.stderr)
        return 2
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    from __graft_entry__ import build
    build()
    e2e_steps = 0 if args.no_e2e else min(args.steps, 400) + 3
    bench = BENCHES[args.workload]("cuda", args.batch, args.warmup + args.steps + e2e_steps)
    K = args.steps
    t = time_steps(bench, K, args.warmup, local_rank, dist)
    head = line_summary(bench, args.workload, t, K)

    # end-to-end through the ABI with host buffers
    e2e = None
    if not args.no_e2e:
        bench.reset()
        hb, db = bench.e2e_setup()
        Ke = min(K, 400)
        for i in range(3):
            bench.e2e_step()
        bench.e2e_flush()
        bench.reset()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        eu = 0
        for i in range(Ke):
            eu += bench.units()
            bench.e2e_step()
        bench.e2e_flush()
        b.record()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        ems, eut = replica_aggregate(a.elapsed_time(b), eu, dist, "cuda")
        scale = 1e9 if bench.unit == "GB/s" else 1e12
        e2e = {"value": round(eut / (ems / 1e3) / scale, 2), "unit": bench.unit,
               "h2d_bytes_per_step": hb, "d2h_bytes_per_step": db, "steps": Ke}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        gbps, el, nprob, desc = oracle_sample(bench.w, args.cpu_seconds, threads, problem=bench.cpu_problem())
        cpu = {"value": round(gbps, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": desc + ", %.1f s" % el}
    extra = bench.extra_report(hbm_peak()[0]) if hasattr(bench, "extra_report") else {}
    bench = None
    torch.cuda.empty_cache()

    # the other lines the decode step's targets name, timed the same way
    lines = {}
    if args.workload == "full-cache-mha" and not args.no_lines and not args.batch:
        for name in EXTRA_LINES:
            lb = BENCHES[name]("cuda", 0, args.warmup + K)
            lines[name] = line_summary(lb, name, time_steps(lb, K, args.warmup, local_rank, dist), K)
            if hasattr(lb, "extra_report"):
                lines[name].update(lb.extra_report(hbm_peak()[0]))
            lb = None
            torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": BENCHES[args.workload].metric,
            "value": head["value"], "unit": head["unit"], "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "steps_per_s": head["steps_per_s"],
        }
        line.update({k: v for k, v in head.items() if k.startswith("frac_of_")})
        line.update({"config": head["config"], "roofline": head["roofline"], "cpu_baseline": cpu, "e2e": e2e,
                     "gpu_launches": head["gpu_launches"],
                     "clocks": head["clocks"], "wall_s": round(t["wall"], 3)})
        line.update(extra)
        if lines:
            line["lines"] = lines
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_reference(args, world, threads):
    if args.workload != "full-cache-mha":
        # the reference arm times the oracle on the default line only
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm (the CPU oracle) times the "
                          "full-cache-mha line only, not %s" % args.workload}), flush=True)
        return 0
    from kv_cache_decode_ring_gb300 import workloads as wl
    from oracle import numerics as nm
    nm.build()
    w = wl.full_cache_mha()
    # size each step so the whole run stays within about a minute; at most one full
    # decode step (B x Hkv problems) per step, drawn from a pool of 64 distinct problems
    budget = 60.0 / (args.steps + args.warmup)
    _, el, n, _ = oracle_sample(w, 0.0, threads, heads_per_call=threads)
    per_prob = el / max(n, 1)
    per_step = max(1, min(w.batch * w.n_kv_heads, int(budget / per_prob)))
    import numpy as np
    ctx = w.extra["context"] + 1
    d, g = w.head_dim, w.n_q_heads // w.n_kv_heads
    pool = min(64, per_step)
    k = wl.as_numpy(w.keys((pool, ctx, d), "ref-sample"))
    v = wl.as_numpy(w.values((pool, ctx, d), "ref-sample"))
    q = nm.bf16_to_f32(wl.as_numpy(w.queries((pool, g, d), "ref-sample"))).astype(np.float64)
    ks = [k[i % pool] for i in range(per_step)]
    vs = [v[i % pool] for i in range(per_step)]
    qs = [q[i % pool] for i in range(per_step)]
    for _ in range(args.warmup):
        nm.attend_many(qs, ks, vs, [ctx - 1] * per_step, 0, None, nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        nm.attend_many(qs, ks, vs, [ctx - 1] * per_step, 0, None, nthreads=threads)
    el = time.perf_counter() - t0
    by = args.steps * per_step * ctx * d * 2 * 2
    value = by / el / 1e9
    full_step = kv_bytes_per_step([ctx] * w.batch, w.n_kv_heads, d)
    sample = ("each step: %d of the %d (request, KV head) problems of one decode step at %d keys (fp64 oracle)"
              % (per_step, w.batch * w.n_kv_heads, ctx))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "steps_per_s": round(value * 1e9 / full_step, 6),
            "config": full_cache_config(w, w.extra["context"], FullCacheBench.CYCLE),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
