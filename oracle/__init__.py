"""Plain CPU oracle for one KV-cache decode step.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The GPU library
(``kv_cache_decode_ring_gb300``) never imports it and shares no code with it.

Sources, cited by page title and section:

* [LEAN]    "用Lean4形式化验证滑动窗口KV Cache的正确性" (framerc.cn/news/4505248)
* [PREFIX]  "LLM 機制實驗（五）：改了歷史，能否只重算變化的後綴？"
            (huhohoo.com/zh-TW/docs/llm/longest-prefix-reuse)
* [LOOP]    "KV Cache 自回归生成推理（增量更新与状态拼接）" (airsota.com/?p=549)
* [WITCERT] "WitCert: Sound Runtime Risk Observability and Gating for KV-Cache
            Quantization" (agifrontier.github.io tutorial)

Layout of the package:

* ``listmodel``  -- the cache as a list (lastWindow, step, run, ringToList), the
                    physical ring, the prefix cut and the trim rules.
* ``numerics``   -- ctypes front end of ``oracle.c``: bf16/fp16 rounding, RoPE,
                    fp64 masked attention, INT8 quantizer and witnesses, Philox4x32-10
                    and the Tier B dither streams.
* ``model``      -- a whole decode-step oracle built from the two: per request the
                    full history of cells, decode by masked attention over it, the
                    expected physical cache state, trim, chunk, the INT8 tier, its
                    gated fallback (block risk, gate selection, restore) and Tier B.
* ``store``      -- the prefix store: bounded entries, scope and signature
                    eligibility, the longest reusable prefix, the newest on ties.

Every function here that has no independent pin says so in its docstring
("parity unpinned"); all others are pinned by ``tests/test_oracle_*.py``.
"""
from .listmodel import (  # noqa: F401
    Cell,
    last_window,
    step,
    run,
    position_invariant,
    ring_to_list,
    RingBuffer,
    prefix_cut,
    ring_trim_allowed,
)
from . import numerics  # noqa: F401
from .numerics import build  # noqa: F401
