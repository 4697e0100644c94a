"""bench.py's reference arm (the fp64 oracle on the host cores) prints one JSON line with the
fields the benchmark contract asks for (CPU only, tiny workload)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_prints_the_contract_line():
    d = _run("--impl", "reference", "--workload", "tiny_nvfp4", "--steps", "2", "--warmup", "0")
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["steps"] == 2 and d["warmup"] >= 3  # at least three warm-up steps, whatever was asked
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["unit"] == "tokens/s" and d["dtype"] == "f64" and d["data"] == "synthetic"
    assert d["config"]["workload"] == "tiny_nvfp4"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_tensor_peak_follows_the_clock_regime():
    """Burst peak when the median SM clock sat at its maximum with no power cap, sustained peak
    under the power cap or a lower clock, and the larger (burst) peak when nothing was sampled."""
    b = _bench_module()
    assert b.tensor_peak({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}, 1890.0, 1710.0)[0] == 1890.0
    assert b.tensor_peak({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}, 1890.0,
                         1710.0)[0] == 1710.0
    assert b.tensor_peak({"sm_mhz": 1700.0, "sm_max_mhz": 2070.0, "reasons": []}, 1890.0, 1710.0)[0] == 1710.0
    assert b.tensor_peak({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}, 1890.0, 1710.0)[0] == 1890.0


def test_kernel_table_fractions_and_shares():
    b = _bench_module()
    alg = {"gemm_fc1_swiglu_aq": ("tensor", 1e12), "fakequant_w": ("hbm", 1e9)}
    prof = {"gemm_fc1_swiglu_aq": (2.0, 2), "fakequant_w": (1.0, 4), "route_permute": (0.5, 2), "combine": (0.0, 0)}
    k = b.kernel_table(prof, 2, alg, 2000.0, 2000.0, 1000.0, 5000.0)
    g = k["gemm_fc1_swiglu_aq"]
    assert abs(g["achieved_tflops"] - 1000.0) < 1e-9 and abs(g["frac"] - 0.5) < 1e-12
    assert abs(g["frac_of_sustained"] - 1.0) < 1e-12 and abs(g["frac_of_burst"] - 0.5) < 1e-12
    f = k["fakequant_w"]
    assert abs(f["achieved_gbs"] - 4000.0) < 1e-9 and abs(f["frac"] - 0.8) < 1e-12
    assert abs(f["frac_of_nominal_8tbs"] - 0.5) < 1e-12
    assert "combine" not in k and k["route_permute"]["share"] is None
    assert abs(g["share"] - 2.0 / 3.0) < 1e-12 and abs(f["share"] - 1.0 / 3.0) < 1e-12


def test_algorithmic_bytes_and_flops_per_launch():
    """2 R N K FLOPs per GEMM launch over the routed rows; the weight fake-quant moves 2 B read +
    the fp32 scale share + 2 B written per weight (averaged over its two launches); with deployed
    nvfp4 scales it also writes each deployed scale, and the tensor-scale pass reads each scale."""
    b = _bench_module()
    cfg = dict(T=16384, topk=8, d=2048, F=768, E=128, fmt=0)
    alg = b.algorithmic_per_launch(cfg)
    R = 16384 * 8
    assert alg["gemm_fc1_swiglu_aq"] == ("tensor", 2.0 * R * 1536 * 2048)
    assert alg["gemm_fc2"] == ("tensor", 2.0 * R * 2048 * 768)
    n = 128 * 1536 * 2048 + 128 * 2048 * 768
    assert alg["fakequant_w"] == ("hbm", (2 + 0.25 + 2) * n / 2)
    assert "deploy_scales" not in alg
    dep = b.algorithmic_per_launch(dict(cfg, fmt=6))
    assert dep["fakequant_w"] == ("hbm", (2 + 0.5 + 2) * n / 2)
    assert dep["deploy_scales"] == ("hbm", 4.0 * n / 16)


def test_memory_phase_with_the_side_stream():
    """The fake-quant entry's memory-phase rate: its own bytes over its launches plus the bytes of
    the side-stream kernels (routing maps, token rows read once and written to each routed row),
    over the phase (the longer of the fake-quant launches and the side-stream launches); absent
    when nothing ran beside it."""
    b = _bench_module()
    cfg = dict(T=16384, topk=8, d=2048, F=768, E=128, fmt=0)
    R = 16384 * 8
    assert b.side_stream_bytes(cfg) == 4.0 * R + 12.0 * R + 2.0 * 16384 * 2048 + 2.0 * R * 2048
    alg = {"fakequant_w": ("hbm", 1e9)}
    prof = {"fakequant_w": (1.0, 4), "route_permute": (0.5, 2)}
    k = b.kernel_table(prof, 2, alg, 2000.0, 2000.0, 1000.0, 5000.0, side_bytes=1e9)
    ph = k["fakequant_w"]["with_side_stream"]
    assert ph["bytes_per_step"] == 3e9 and abs(ph["achieved_gbs"] - 6000.0) < 1e-9 and abs(ph["frac"] - 1.2) < 1e-12
    # a side stream longer than the fake-quant sets the phase: 0.5 + 0.25 ms
    prof = {"fakequant_w": (1.0, 4), "route_permute": (1.0, 2), "gather_rows": (0.5, 2)}
    ph = b.kernel_table(prof, 2, alg, 2000.0, 2000.0, 1000.0, 5000.0, side_bytes=1e9)["fakequant_w"]["with_side_stream"]
    assert abs(ph["phase_ms"] - 0.75) < 1e-12 and abs(ph["achieved_gbs"] - 4000.0) < 1e-9
    k = b.kernel_table({"fakequant_w": (1.0, 4)}, 2, alg, 2000.0, 2000.0, 1000.0, 5000.0, side_bytes=1e9)
    assert "with_side_stream" not in k["fakequant_w"]
