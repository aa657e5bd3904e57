"""Host-side logic of bench.py, on the CPU: the JSON line of the reference
arm (the CPU oracle timed on the host cores) at one rank and under torchrun
with two ranks, the roofline arithmetic against closed-form counts of the
layer's work, the clock record parsed from nvidia-smi samples, and the
output error report."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
REF_ARGS = ["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1", "--ref-tokens", "16"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", *REF_ARGS], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    j = lines[0]
    assert j["impl"] == "reference" and j["unit"] == "tokens/s" and j["higher_is_better"] is True
    assert j["n_gpus"] == 1 and j["steps"] == 2
    assert j["warmup"] == 3                                   # raised to the minimum of three
    assert j["value"] > 0 and j["vs_baseline"] is None and j["scaling"] == "weak"
    assert j["ms_per_step"] == pytest.approx(16 / j["value"] * 1e3, rel=1e-9)
    assert j["config"]["workload"].startswith("tiny: T=256 d=256 E=8 top_k=2 F=512")
    assert "0.00315 GB" in j["config"]["l2"]                  # 8 experts x 3 x 512 x 256 e4m3 bytes
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == j["value"] and cb["cores"] >= 1 and cb["sample"]
    assert j["e2e"] == {"value": j["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_two_ranks_rank0_alone():
    """Launched as the multi-GPU bench is, only rank 0 runs the oracle and
    prints; the other rank exits 0 without work."""
    env = dict(os.environ, MASTER_ADDR="127.0.0.1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--gpus", "2", *REF_ARGS]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def test_roofline_arithmetic_closed_forms():
    """The algorithmic work behind each fraction, for the large layer with
    every leg timed at 1 ms: 6 A d F flops for the two GEMMs (A = T k routed
    rows, GEMM1 2F wide, GEMM2 d wide), and the bytes each HBM step must move."""
    import bench
    from block_scaled_fp8_router_gb300 import synthetic as S
    cfg = S.CONFIGS["large"]
    T, d, E, k, F = 8192, 7168, 256, 8, 2048
    A = T * k
    avg = {key: 1.0 for key in ("ffn", "quant", "dispatch", "combine", "route")}
    peaks = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0, "source": "measured"}
    ffn, extra = bench.rooflines(cfg, avg, peaks)
    assert ffn["achieved"] == pytest.approx((2 * A * d * 2 * F + 2 * A * F * d) / 1e-3 / 1e12)
    assert ffn["achieved"] == pytest.approx(5772.436, rel=1e-6)
    assert ffn["peak"] == 4000.0 and ffn["frac"] == pytest.approx(ffn["achieved"] / 4000.0)
    # 1x128 quantiser: bf16 in, e4m3 codes and one fp32 scale per 128 channels out
    assert extra["quant_1x128"]["GB/s"] == pytest.approx((T * d * 2 + T * d + T * d // 128 * 4) / 1e-3 / 1e9)
    # dispatch: the ids, both maps, and the quantised rows read once per token, written once per slot
    row = d + d // 128 * 4
    assert extra["dispatch"]["GB/s"] == pytest.approx((A * 4 + 2 * A * 4 + T * row + A * row) / 1e-3 / 1e9)
    # combine: A bf16 expert rows, the map and the gates in, y out
    assert extra["combine"]["GB/s"] == pytest.approx((A * d * 2 + A * 4 + A * 4 + T * d * 2) / 1e-3 / 1e9)
    assert extra["combine"]["frac_hbm"] == pytest.approx(extra["combine"]["GB/s"] / 8000.0)
    # router: logits over all experts, one fma (two flops) per token, channel and expert
    assert extra["route_topk"]["fp32 TFLOP/s"] == pytest.approx(2 * T * d * E / 1e-3 / 1e12)
    # the gathered form moves no rows in dispatch
    _, g = bench.rooflines(cfg, avg, peaks, gathered=True)
    assert g["dispatch"]["GB/s"] == pytest.approx((A * 4 + 2 * A * 4) / 1e-3 / 1e9)


def test_padded_fraction_and_weight_bytes():
    import bench
    from block_scaled_fp8_router_gb300 import synthetic as S
    assert bench.padded_fraction([0, 1, 128, 129]) == pytest.approx((0 + 128 + 128 + 256) / 258)
    assert bench.padded_fraction([]) == 0.0
    assert bench.fp8_weight_bytes(S.CONFIGS["large"]) == 256 * (2 * 2048 * 7168 + 7168 * 2048)


def test_clock_summary_from_samples():
    """The clock record beside the number: median SM clock under load, the
    maximum, and every throttle reason seen active in any sample (the query's
    fields in order: index, SM clock, its maximum, power, the active-reasons
    mask, four reason flags, GPU utilisation)."""
    import bench
    c = bench.Clocks(0)
    c.f.write("0, 2070, 2070, 190.5, 0x0, Not Active, Not Active, Not Active, Not Active, 0\n"
              "0, 2070, 2070, 210.0, 0x0, Not Active, Not Active, Not Active, Not Active, 3\n"
              "0, 1950, 2070, 1380.0, 0x4, Not Active, Not Active, Not Active, Active, 100\n"
              "0, 1965, 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active, 98\n"
              "0, 1980, 2070, 1210.0, 0x0, Not Active, Not Active, Not Active, Not Active, 100\n"
              "garbage line\n")
    s = c.summary()
    assert s["sm_mhz"] == 1965.0 and s["sm_max_mhz"] == 2070.0   # the idle samples are left out
    assert s["samples"] == 5 and s["samples_under_load"] == 3
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1380.0
    c = bench.Clocks(0)                                           # no utilisation reading: all samples
    c.f.write("0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active\n"
              "0, 2055, 2070, 1380.0, 0x4, Not Active, Not Active, Not Active, Active\n"
              "0, 2070, 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active, [N/A]\n")
    s = c.summary()
    assert s["sm_mhz"] == 2070.0 and s["samples"] == 3 and s["samples_under_load"] == 0
    c = bench.Clocks(0)
    c.f.write("0, 1500, 2070, [N/A], 0x0, Active, Not Active, Active, Not Active\n")
    s = c.summary()
    assert s["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"] and s["power_w_max"] is None
    assert bench.Clocks(0).summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}


def test_error_report_closed_form():
    """Row error is max |y - ref| over the row's largest |ref|; element error
    divides by max(|ref|, 1e-2 rowmax)."""
    import numpy as np
    import torch
    import bench
    bits = lambda a: torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref = [[4.0, -2.0, 0.0, 1.0], [1.0, 1.0, 1.0, 1.0]]
    y = [[4.0, -2.0, 0.03125, 1.0], [1.0, 1.0, 1.0, 1.0]]
    r = bench.error_report(bits(y), bits(ref))
    assert r["tokens"] == 2 and r["bar_row_rel_err"] == 2e-2
    assert r["row_rel_err_max"] == pytest.approx(0.03125 / 4.0)
    assert r["elem_rel_err_max"] == pytest.approx(0.03125 / 0.04)
    assert r["elem_rel_err_mean"] == pytest.approx(0.03125 / 0.04 / 8)
