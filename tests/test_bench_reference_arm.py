"""The reference arm of bench.py: the CPU oracle timed on a bounded sample of
the bench's workload, printed as one JSON line with the bench's metric, unit
and workload (no GPU needed)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "32e-top4-h2880"
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == d["value"] and cpu["cores"] >= 1
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_route_kernel_count_follows_the_library_rule():
    """bench.py counts one routing kernel for the batches the library routes in
    a single CTA (the boundaries the GPU routing tests exercise), two otherwise."""
    sys.path.insert(0, ROOT)
    import bench
    one = [(64, 32, 4), (128, 32, 8), (128, 8, 8), (64, 64, 8), (32, 128, 8), (1, 32, 1)]
    two = [(4096, 32, 4), (129, 32, 4), (65, 64, 2), (33, 128, 4), (1, 256, 8), (64, 256, 8), (200, 16, 8)]
    assert all(bench.route_kernels(*a) == 1 for a in one)
    assert all(bench.route_kernels(*a) == 2 for a in two)
