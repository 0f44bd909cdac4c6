"""Host-side logic of bench.py, on the CPU.

- `traffic`: a stored DRAM-to-algorithmic ratio is reported only while the kernel source
  still hashes to the value it was captured from; any edit turns it into null.
- The algorithmic bytes of a bf16 decode step: K and V read once per KV head.
- Both arms of the bench print the same config for the full-cache MHA line.
"""
import hashlib
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from kv_cache_decode_ring_gb300 import workloads as wl  # noqa: E402


def test_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    src = os.path.join(bench.CSRC, "decode_fast.cu")
    dst = tmp_path / "decode_fast.cu"
    shutil.copy(src, dst)
    sha = hashlib.sha256(dst.read_bytes()).hexdigest()[:16]
    monkeypatch.setattr(bench, "CSRC", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC_PER_BYTE", {"w": ("decode_fast.cu", sha, 1.25)})
    assert bench.traffic_per_launch("w", 1000) == 1250
    assert bench.traffic_per_launch("other", 1000) is None          # no capture for that workload
    with open(dst, "ab") as f:
        f.write(b"\n")                                               # the kernel changed since the capture
    assert bench.traffic_per_launch("w", 1000) is None


def test_every_traffic_entry_names_a_kernel_source():
    for name, (src, sha, ratio) in bench.TRAFFIC_PER_BYTE.items():
        assert os.path.exists(os.path.join(bench.CSRC, src)), name
        assert len(sha) == 16 and int(sha, 16) >= 0, name
        assert 0.5 < ratio < 2.0, name                               # DRAM bytes near the algorithmic bytes


def test_kv_bytes_per_step():
    # K and V of every key, once per KV head: 2 tensors x 2 bytes x d
    assert bench.kv_bytes_per_step([4097] * 32, 32, 128) == 32 * 32 * 4097 * 128 * 4
    assert bench.kv_bytes_per_step([1, 10], 8, 64) == (1 + 10) * 8 * 64 * 4


def test_both_arms_share_the_full_cache_config():
    w = wl.full_cache_mha()
    c = bench.full_cache_config(w, w.extra["context"], bench.FullCacheBench.CYCLE)
    assert c["workload"] == "full-cache-mha-bf16" and c["batch"] == 32 and c["head_dim"] == 128
    assert c["max_seq_len"] == 8192 and c["context"] == "4096 + step (cycles 4097..4224 keys)"


def test_reference_arm_names_the_lines_it_does_not_time():
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "int8-witness", "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and "full-cache-mha" in line["unavailable"]
