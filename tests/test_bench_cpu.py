"""Host-side checks of bench.py's contract (no GPU needed).

- The reference arm (the oracle on the host's cores) prints one JSON line with
  the GPU arm's metric, unit and workload, its CPU baseline and an end-to-end
  figure with no host-device traffic; a rank other than 0 does no work.
- The GPU arm fails loudly without a GPU: no line, non-zero exit (there is no
  CPU fallback to measure by mistake).
- The DRAM traffic table parses, and a figure is reported only for the kernel
  sources it was captured on.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _run(args, env=None, timeout=240):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=timeout)


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.strip().startswith("{")]


def test_reference_arm_line():
    r = _run(["--impl", "reference", "--steps", "2", "--warmup", "3"], env={"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == bench.WORKLOAD
    assert d["steps"] == 2 and d["warmup"] >= 3 and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]


def test_reference_arm_other_rank_does_nothing():
    r = _run(["--impl", "reference", "--steps", "1", "--warmup", "3"], env={"RANK": "1", "WORLD_SIZE": "2"},
             timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert _json_lines(r.stdout) == []


@pytest.mark.skipif(os.path.exists("/dev/nvidia0") or os.path.exists("/dev/nvidiactl"),
                    reason="a GPU is present")
def test_gpu_arm_fails_without_gpu():
    r = _run(["--steps", "1", "--warmup", "3"], timeout=120)
    assert r.returncode != 0
    assert _json_lines(r.stdout) == []


def test_dram_traffic_table():
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    rows = []
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            op, workload, nbytes, sha = line.split()
            assert op in bench._KERNEL_FILES and workload in ("video", "image")
            assert int(nbytes) > 0 and len(sha) == 16 and int(sha, 16) >= 0
            rows.append((op, workload, int(nbytes), sha))
    assert rows
    for op, workload, nbytes, sha in rows:
        cur = bench.kernel_sha(op)
        assert len(cur) == 16
        # reported only while the sources hash to the captured value
        assert bench.dram_traffic(op, workload) == (nbytes if cur == sha else None)


def test_step_bytes_are_the_algorithmic_bytes():
    """Every input read once and every output written once, bf16."""
    T = 32760 * 5120 * 2
    assert bench.V_LN_BYTES == 4 * T                  # x, scale, shift, out
    assert bench.V_TANH_BYTES == 4 * T + 5120 * 2     # x, g, r, out + weight
    assert bench.V_STEP_BYTES == 8 * T + 10240 == 2_683_709_440
    assert abs(bench.ROW_BYTES * 32760 - bench.V_STEP_BYTES) < 1e-3
    t = 2 * 4352 * 3072 * 2
    assert bench.I_LN_BYTES == 2 * t + 2 * 2 * 3072 * 2
    assert bench.I_RGA_BYTES == 3 * t + 2 * 3072 * 2
