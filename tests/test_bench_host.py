"""Host-side checks of bench.py (no GPU): the committed ncu summary of the
headline kernel matches the current kernel sources (so the roofline
reports the measured DRAM traffic rather than null); the algorithmic byte
counts; the reference arm's JSON line, alone and under torchrun with two
ranks; the warm-up floor; and the CPU-baseline block of the GPU arm."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_profiled_traffic_matches_current_headline_sources():
    t = bench.profiled_traffic()
    assert t is not None, ("headline kernel sources changed since the committed DRAM counters were taken: "
                           f"re-take them (digest now {bench.kernel_source_digest()})")
    # reads alone are 2 B per element (536.9 MB); writes fall short of the
    # algorithmic 277 MB only by what is still dirty in L2 at launch end
    assert 2 * 65536 * 4096 <= t <= bench.algorithmic_bytes(65536, 4096, "mxfp8")


def test_algorithmic_bytes():
    # 2H read + H codes + H/32 scales + 4 inv_rms per row at H = 4096
    assert bench.algorithmic_bytes(1, 4096, "mxfp8") == 12420
    assert bench.algorithmic_bytes(1, 4096, "mxfp4") == 10372
    assert bench.baseline_bytes(1, 4096) == 28804


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the CPU oracle on the host cores) prints
    one JSON line with the benchmark contract's keys."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["ms_per_step"] > 0 and d["config"]["workload"] == "llama3_8b_65536x4096"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["cpu"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_warmup_below_three_is_refused():
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "2"], capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_reference_arm_under_torchrun_prints_once():
    """Launched the way a multi-GPU run is (torchrun, two ranks), the
    reference arm runs on rank 0 alone and prints one JSON line; the other
    rank exits 0 without work."""
    import json
    import socket
    import subprocess
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0])["impl"] == "reference"


def test_cpu_baseline_fields():
    """The GPU arm's cpu_baseline block (the oracle on the host cores, on a
    bounded sample) carries the keys the benchmark line needs."""
    from mx_scale_reusing_gb300 import synth
    xb = synth.make_activations(synth.WORKLOADS["llama3_8b_65536x4096"], rows=512)
    cb = bench.cpu_baseline(xb, 2, 64)
    assert cb["kind"] == "oracle" and cb["unit"] == "tokens/s" and cb["cores"] >= 1 and cb["cpu"]
    assert cb["value"] > 0 and cb["single_thread_tokens_per_s"] > 0
    assert abs(cb["GB/s"] - cb["value"] * 12420 / 1e9) <= 1e-3 + 1e-3 * cb["GB/s"]
    assert "rows" in cb["sample"]
