"""The C-ABI library loads, exports every entry point include/kvc.h declares, and its
host-only logic is right (CPU only: no kernel is launched here)."""
import os
import re
import subprocess

import pytest

from kv_cache_decode_ring_gb300 import build as kbuild
from kv_cache_decode_ring_gb300 import kvc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kvc.lib()


def declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(kvc_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared()
    for want in ["kvc_create", "kvc_append", "kvc_trim", "kvc_decode_attn", "kvc_chunk_attn"]:
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", kvc.library_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (kvc_\w+)", out))
    missing = [n for n in declared() if n not in exported]
    assert not missing, missing
    for n in declared():
        assert hasattr(lib, n)


def test_state_bytes_validation(lib):
    ok = kvc.make_config("bf16", "contiguous", None, 32, 32, 32, 128, 8192)
    n = kvc.kvc_state_bytes(ok)
    assert n >= 2 * 32 * 32 * 8192 * 128 * 2 + 32 * 8192 * 4
    bad = [
        kvc.make_config("bf16", "contiguous", None, 2, 3, 2, 128, 64),          # Hq % Hkv
        kvc.make_config("bf16", "contiguous", None, 1, 1, 1, 7, 64),            # odd head_dim
        kvc.make_config("bf16", "ring", None, 1, 1, 1, 128, 64, window=32),     # ring window != W
        kvc.make_config("bf16", "ring", None, 1, 1, 1, 128, 64, rope_base=1e4),  # ring RoPE needs max_position
        kvc.make_config("f32", "contiguous", "int8", 1, 1, 1, 128, 64),         # INT8 needs bf16
        kvc.make_config("bf16", "contiguous", "int8", 1, 1, 1, 128, 60),        # INT8 capacity % 16
        kvc.make_config("bf16", "ring", "int8", 1, 1, 1, 128, 72),              # INT8 ring W % 16
        kvc.make_config("bf16", "ring", "int8", 1, 4, 1, 128, 64, int8_exact_blocks=4),   # gate on a ring
        kvc.make_config("bf16", "contiguous", None, 0, 1, 1, 128, 64),          # empty batch
        kvc.make_config("bf16", "contiguous", "int8", 1, 4, 1, 128, 64, window=32,
                        int8_exact_blocks=4),                                    # gate with a window
        kvc.make_config("bf16", "contiguous", None, 1, 1, 1, 128, 64, int8_exact_blocks=4),  # pool needs INT8
        kvc.make_config("bf16", "contiguous", "int8", 1, 4, 1, 128, 64, int8_exact_blocks=-1),
        kvc.make_config("bf16", "contiguous", "int8", 1, 4, 1, 128, 64, page_pool=8,
                        int8_exact_blocks=4),                                    # gate pool of a paged cache
        kvc.make_config("bf16", "contiguous", None, 1, 4, 1, 128, 72, page_pool=8),     # capacity % 16
        kvc.make_config("bf16", "ring", None, 1, 4, 1, 128, 40, page_pool=8, max_position=64),  # W % 16
        kvc.make_config("bf16", "contiguous", None, 1, 4, 1, 128, 64, page_pool=-1),
        kvc.make_config("bf16", "contiguous", None, 1, 4, 1, 128, 64, store_slots=-1),
        kvc.make_config("bf16", "contiguous", "int8", 1, 4, 1, 128, 64, store_slots=2),   # store of INT8
        kvc.make_config("bf16", "contiguous", "int8-dither", 1, 4, 1, 128, 64, int8_exact_blocks=4),  # no gate
        kvc.make_config("bf16", "contiguous", "int8-dither", 1, 4, 1, 128, 64, layer_index=65536),   # 16-bit layer
        kvc.make_config("bf16", "contiguous", "int8-dither", 1, 4, 1, 128, 64, layer_index=-1),
        kvc.make_config("bf16", "ring", "int8-dither", 1, 4, 1, 128, 56),
        kvc.make_config("f32", "contiguous", "int8-dither", 1, 4, 1, 128, 64),
        kvc.make_config("bf16", "contiguous", None, 1, 4, 1, 128, 64, int8_split=1024),   # split needs INT8
        kvc.make_config("bf16", "contiguous", "int8", 1, 4, 1, 128, 64, int8_split=1000),  # not a multiple of 64
        kvc.make_config("bf16", "contiguous", "int8", 1, 4, 1, 128, 64, int8_split=960),   # below 1024
        kvc.make_config("bf16", "contiguous", "int8", 1, 4, 1, 128, 64, int8_split=2112),  # above 2048
        kvc.make_config("f32", "contiguous", None, 1, 256, 1, 256, 64),         # generic decode: 320 KB of smem
    ]
    # the INT8 tiers on a ring (W % 16 == 0) or with a window
    for c in [kvc.make_config("bf16", "ring", "int8", 1, 4, 1, 128, 64),
              kvc.make_config("bf16", "ring", "int8-dither", 1, 4, 1, 128, 64),
              kvc.make_config("bf16", "contiguous", "int8", 1, 4, 1, 128, 64, window=8),
              kvc.make_config("bf16", "contiguous", "int8", 1, 4, 1, 128, 64, page_pool=8),
              kvc.make_config("bf16", "ring", "int8-dither", 1, 4, 1, 128, 64, page_pool=8),
              kvc.make_config("bf16", "contiguous", "int8", 1, 4, 1, 128, 64, int8_split=1088),
              kvc.make_config("bf16", "ring", "int8-dither", 1, 4, 1, 128, 64, int8_split=2048),
              kvc.make_config("f32", "contiguous", None, 1, 181, 1, 256, 64)]:           # 227 KB: the limit
        assert kvc.kvc_state_bytes(c) > 0
    for c in bad:
        with pytest.raises(kvc.KvcError) as e:
            kvc.kvc_state_bytes(c)
        assert e.value.code == kvc.KVC_ERR_ARG


def test_paged_state_is_the_pool_not_the_capacity(lib):
    # a paged cache sizes K/V by its pool, whatever the per-request capacity
    big = kvc.kvc_state_bytes(kvc.make_config("bf16", "contiguous", None, 64, 32, 8, 128, 32768))
    paged = kvc.kvc_state_bytes(kvc.make_config("bf16", "contiguous", None, 64, 32, 8, 128, 32768, page_pool=1024))
    assert paged < big / 20


def test_prefix_cut_matches_golden(lib):
    import test_oracle_listmodel as golden
    for name, old, new, ring, cut, _, _ in golden.read_cases():
        if old == "store":
            continue
        assert kvc.kvc_prefix_cut([int(x) for x in old.split()], new, bool(ring)) == cut, name
    with pytest.raises(kvc.KvcError):
        kvc.kvc_prefix_cut([1, 2], [])
    with pytest.raises(TypeError):
        kvc.kvc_prefix_cut([1, 2], [1.0, 2])


def test_prefix_cut_matches_oracle_exhaustively(lib):
    import itertools
    from oracle.listmodel import prefix_cut
    alphabet = [1, 2]
    for n_old in range(0, 5):
        for n_new in range(1, 5):
            for old in itertools.product(alphabet, repeat=n_old):
                for new in itertools.product(alphabet, repeat=n_new):
                    for ring in (False, True):
                        assert kvc.kvc_prefix_cut(list(old), list(new), ring) == prefix_cut(list(old), list(new), ring)


def test_strerror(lib):
    for code in range(7):
        assert kvc.kvc_strerror(code)


@pytest.mark.parametrize("seed", range(8))
def test_int8_gate_matches_oracle_selection(lib, seed):
    # the host gate of the C ABI against the oracle's selection on the same fp32 risks,
    # including ties, values at atanh(tau) and budgets
    import math
    import numpy as np
    from oracle.model import gate_select
    rng = np.random.default_rng(seed)
    B, H, nb = int(rng.integers(1, 4)), int(rng.integers(1, 4)), int(rng.integers(0, 40))
    pool = np.array([0.0, 0.05, 0.2, math.atanh(0.2), 0.25, 0.7, 0.7, 3.0], dtype=np.float32)
    risk = rng.choice(pool, (B, H, nb)).astype(np.float32)
    for tau in (0.0, 0.2, 0.5):
        for budget in (0, 1, 5, B * H * nb + 1):
            got = kvc.kvc_int8_gate(risk, tau, budget)
            want = gate_select({(b, h): risk[b, h] for b in range(B) for h in range(H)}, tau, budget)
            assert [tuple(x) for x in got] == want, (tau, budget)


def _pstore(ring, capacity=2):
    cfg = kvc.make_config("f32", "ring" if ring else "contiguous", None, 1, 1, 1, 16, 4 if ring else 16,
                          max_position=64, rope_base=10000.0, store_slots=capacity)
    return kvc.PrefixStore(cfg, capacity)


def test_pstore_matrix_through_the_abi(lib):
    from _store_cases import BRANCH, PLAIN, SCOPE, SIGNATURE, read_matrix
    for case in read_matrix():
        ps = _pstore(case["ring"])
        slots = {"plain": ps.insert(PLAIN, SCOPE, SIGNATURE), "branch": ps.insert(BRANCH, SCOPE, SIGNATURE)}
        slot, cut = ps.lookup(case["ids"], case["scope"], SIGNATURE)
        assert cut == case["cut"], case["name"]
        assert slot == (-1 if case["entry"] is None else slots[case["entry"]]), case["name"]
        ps.close()


def test_pstore_validation_and_state_bytes(lib):
    ps = _pstore(False)
    with pytest.raises(TypeError):
        ps.lookup([1.0, 2], "s")                          # 1.0 is not the token 1
    with pytest.raises(TypeError):
        ps.insert(__import__("numpy").array([1.5, 2.0]), "s")
    with pytest.raises(kvc.KvcError) as e:
        ps.lookup([], "s")
    assert e.value.code == kvc.KVC_ERR_ARG
    assert ps.lookup([1, 2], "s") == (-1, 0)             # empty store
    with pytest.raises(kvc.KvcError):
        kvc.PrefixStore(kvc.make_config("bf16", "contiguous", None, 1, 1, 1, 128, 64), 0)
    base = kvc.kvc_state_bytes(kvc.make_config("bf16", "contiguous", None, 2, 8, 2, 128, 512))
    two = kvc.kvc_state_bytes(kvc.make_config("bf16", "contiguous", None, 2, 8, 2, 128, 512, store_slots=2))
    assert two - base >= 2 * (2 * 2 * 512 * 128 * 2 + 512 * 4)


@pytest.mark.parametrize("seed", range(6))
def test_pstore_matches_oracle_store(lib, seed):
    """Random insert/lookup sequences: the C policy and the oracle's agree on every slot and cut."""
    import random
    from oracle.store import PrefixStore as OracleStore
    rng = random.Random(seed)
    for ring in (False, True):
        cap = rng.choice([1, 2, 3])
        ps, ref = _pstore(ring, cap), OracleStore(cap, ring=ring)
        for _ in range(200):
            ids = [rng.choice([1, 2, 3]) for _ in range(rng.randint(1, 6))]
            scope, sig = rng.choice(["a", "b"]), rng.choice([b"", b"w1", b"w2"])
            if rng.random() < 0.3:
                assert ps.insert(ids, scope, sig) == ref.insert(ids, scope, sig, None)
            else:
                s_ref, c_ref = ref.lookup(ids, scope, sig)
                assert ps.lookup(ids, scope, sig) == (-1 if s_ref is None else s_ref, c_ref), (ids, scope, sig)
        ps.close()


def test_dither_state_has_no_witnesses(lib):
    w8 = kvc.kvc_state_bytes(kvc.make_config("bf16", "contiguous", "int8", 2, 8, 2, 128, 4096))
    wd = kvc.kvc_state_bytes(kvc.make_config("bf16", "contiguous", "int8-dither", 2, 8, 2, 128, 4096,
                                             layer_index=7, dither_key=(1, 2)))
    assert w8 - wd >= 2 * 2 * 4096 * 16 * 2 - 4096                  # 32 B per token and head fewer


def test_config_struct_matches_the_header():
    # the ctypes mirror of kvc_config lists the header's fields in the header's order,
    # with 32-bit members throughout (a mismatch would shift every later field)
    import ctypes
    src = open(os.path.join(ROOT, "include", "kvc.h")).read()
    start = src.index("typedef struct {", src.index("configuration")) + len("typedef struct {")
    body = src[start:src.index("} kvc_config;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = []
    for decl in body.split(";"):
        m = re.match(r"\s*(int32_t|uint32_t|float)\s+(.+)", decl.strip(), flags=re.S)
        if m:
            fields += [(m.group(1), n.strip()) for n in m.group(2).split(",")]
    mirror = kvc.kvc_config._fields_
    assert [n for _, n in fields] == [n for n, _ in mirror]
    ctype = {"int32_t": ctypes.c_int32, "uint32_t": ctypes.c_uint32, "float": ctypes.c_float}
    assert [ctype[t] for t, _ in fields] == [t for _, t in mirror]
