"""bench.py on the GPU: the JSON line carries every key of the benchmark
contract (the value, the roofline of the dominant kernel with its measured
peak, the oracle baseline, the end-to-end figure with its host-link bytes, the
launch count and the clocks), with plausible values."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_step_line_has_the_contract_keys(gpu):
    d = _run("--steps", "50", "--warmup", "3", "--cpu-seconds", "1")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 50 and d["warmup"] >= 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["config"]["workload"] == "llama7b_b64"
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert 0.3 < r["frac"] < 1.3                       # a copy-rate denominator: about 1 at most
    assert r["traffic"] is None or r["traffic"] > 0
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["value"] < d["value"] * 1.05              # the host link can only cost
    assert d["gpu_launches"] == 2 * d["steps"]
    # the decode's own duration comes from a long decode-only loop, and a
    # kernel cannot take longer than the step it sits in
    assert r["launches_timed"] >= 200
    assert d["decode_ms"] <= d["ms_per_step"]
    clk = d["clocks"]
    assert clk is not None and clk["samples"] >= 5 and clk["sm_mhz"] > 0
    # the other workloads, timed in the same run
    side = d["workloads"]["results"]
    for w in ("tiny", "cb_mix", "shared_prefix", "long_ctx", "cb_mix_1k", "cb_mix_4k"):
        assert side[w]["decode_ms"] > 0 and side[w]["launches"] >= 200, w
        if w != "tiny":                                   # HBM-bound: a copy-rate fraction
            assert 0.3 < side[w]["unique_frac"] < 1.3, (w, side[w])
    for w in ("shared_prefix", "shared_prefix_4k"):
        c = side[w + "_shared_call"]
        assert c["speedup_vs_plain"] > 1.0 and 0.3 < c["unique_frac"] < 1.3, (w, c)


def test_shared_prefix_line(gpu):
    d = _run("--op", "shared_prefix", "--steps", "20", "--warmup", "3")
    assert d["value"] > 0 and d["speedup_vs_plain"] > 1.0
    r = d["roofline"]
    assert r["bound"] == "hbm" and 0.2 < r["frac"] < 1.3
    assert r["traffic"] is None or r["traffic"] > 0
