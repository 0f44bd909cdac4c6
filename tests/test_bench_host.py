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


def _run_bench(args, env=None, timeout=300):
    import json
    import subprocess
    e = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        e.pop(k, None)
    e.update(env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                       timeout=timeout, env=e)
    lines = [l for l in r.stdout.strip().splitlines() if l.startswith("{")]
    return r.returncode, (json.loads(lines[-1]) if lines else None), r.stderr


def test_gpus_flag_starts_that_many_ranks():
    # without torchrun, --gpus 2 starts two ranks itself (gloo in the dry run, no GPU work);
    # the line counts the ranks that really ran
    rc, line, err = _run_bench(["--gpus", "2", "--dry-run", "--steps", "3", "--warmup", "3"])
    assert rc == 0, err
    assert line["n_gpus"] == 2 and line["ranks_run"] == 2 and line["dry_run"]
    rc, line, err = _run_bench(["--dry-run", "--steps", "3"])
    assert rc == 0 and line["n_gpus"] == 1 and line["ranks_run"] == 1


def test_gpus_flag_must_agree_with_the_launcher():
    rc, line, err = _run_bench(["--gpus", "3", "--dry-run", "--steps", "1"],
                               env={"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"})
    assert rc == 2 and line is None and "disagrees" in err


def test_default_run_times_every_targeted_line():
    # the INT8 decode, the sliding-window GQA decode and the chunk kernel each get a line
    for name in ("int8-witness", "sliding-window-gqa", "prefix-reuse", "prefix-reuse-w4096", "int8-dither",
                 "prefix-reuse-store", "int8-witness-ring"):
        assert name in bench.EXTRA_LINES and name in bench.BENCHES


def test_call_samples_skip_the_first_step_and_thin_out():
    # the dominant call is timed on a sample of the steps (events between kernels cost the
    # dependent launches their overlap); never the first step after the synchronize
    assert bench.call_samples(1) == [0]
    assert bench.call_samples(20) == [1, 5, 9, 13, 17]
    s = bench.call_samples(1500)
    assert s[0] == 1 and all(b - a == 8 for a, b in zip(s, s[1:])) and s[-1] < 1500
