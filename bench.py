"""Throughput of the MoE layer with router replay and block-scaled FP8 on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload large] [--impl reference]

A step is one forward of the whole hot path over one batch of synthetic
tokens, with inputs resident in HBM: router top-k (or payload replay) ->
1x128 FP8 quantisation of x -> dispatch -> grouped FP8 SwiGLU FFN ->
combine.  Default workload "large": T=8192 tokens, d=7168, 256 experts,
top-8, F=2048, sigmoid top-k gating (the large-MoE shape of the metric).
The FP8 weights (11.3 GB) are quantised once before timing (they change once
per weight update, not per step) and are streamed from HBM every step, so
each step's working set is far larger than the 129 MB L2.

Reported (one JSON line, rank 0):
  value      tokens/s over all ranks (device-resident inputs, CUDA events)
  e2e        tokens/s through the public layer API with pinned host x in and
             y out (host<->device copies inside the timed region)
  roofline   grouped FFN call (its two tcgen05 GEMM kernels): algorithmic
             FLOPs 6*A*d*F per call / its event-timed duration, against the
             FP8 dense peak (2 x measured bf16 peak)
  extra      the other steps' event times and their own rooflines
  cpu_baseline  the CPU oracle on a bounded token sample, on the host cores
Multi-GPU: each rank runs its own batch (token sharding, no exchange);
value = tokens of all ranks / max time over ranks.

--impl reference times the CPU oracle (the only reference this method has)
on the same workload, a bounded token sample per step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
L2_FLUSH_BYTES = 512 * 1024 * 1024      # written between timed steps (not timed) so no step starts warm
FP32_ALU_TFLOPS_DERIVED = 152 * 128 * 2 * 2.07e9 / 1e12   # 152 SMs x 128 FMA lanes x 2 FLOP x 2.07 GHz
# DRAM bytes (read + write) per routed row of the grouped FFN at d=7168, F=2048,
# ~256 rows per expert: ncu capture of grouped_gemm_kernel<1> and <2> on the
# large_e64 profiling shape (A = 16384 rows): 2.0422e9 + 0.0353e9 + 0.9750e9 +
# 0.2185e9 bytes.  Valid for the kernel that capture measured.
FFN_DRAM_BYTES_PER_ROW = (2.0422e9 + 0.0353e9 + 0.9750e9 + 0.2185e9) / 16384
KERNELS_PER_STEP = {"route": 1, "replay": 1, "quant": 1, "dispatch": 4, "ffn": 2, "combine": 1}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def fp8_peak_tflops(dev, n: int = 8192, reps: int = 10):
    """Dense FP8 (e4m3 x e4m3 -> bf16) GEMM throughput of cuBLASLt through
    torch._scaled_mm at n^3, best of `reps` with CUDA events: the measured
    FP8 peak beside the nominal 2 x bf16 one.  None if unsupported."""
    import torch
    try:
        g = torch.Generator(device=dev).manual_seed(7)
        a = torch.randn((n, n), generator=g, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), generator=g, device=dev).to(torch.float8_e4m3fn)
        one = torch.ones((), dtype=torch.float32, device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1)
            best = t if best is None else min(best, t)
        del a, b
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except Exception:                                   # a measurement beside the line, not a step of it
        return None


def cpu_model() -> str:
    """The host CPU's name (x86 model name, or Arm implementer/part)."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    for line in info.splitlines():
        if line.lower().startswith("model name"):
            return line.split(":", 1)[1].strip()
    impl = part = None
    for line in info.splitlines():
        if line.startswith("CPU implementer"):
            impl = line.split(":", 1)[1].strip()
        elif line.startswith("CPU part"):
            part = line.split(":", 1)[1].strip()
    names = {("0x41", "0xd4f"): "Arm Neoverse V2 (NVIDIA Grace)", ("0x41", "0xd40"): "Arm Neoverse V1",
             ("0x41", "0xd0c"): "Arm Neoverse N1"}
    if impl and part:
        return names.get((impl, part), f"Arm implementer {impl} part {part}")
    return "unknown"


def fp8_weight_bytes(cfg) -> int:
    """One layer's e4m3 expert weights (W13 [2F, d] and W2 [d, F] per expert),
    without their 128x128 scales."""
    return cfg.E * 3 * cfg.F * cfg.d


def padded_fraction(counts, bm: int = 128) -> float:
    """Rows the grouped GEMM computes (each expert's rows rounded up to whole
    bm-row tiles) over the rows routed."""
    c = [int(v) for v in counts]
    A = max(sum(c), 1)
    return sum(bm * ((v + bm - 1) // bm) for v in c) / A


class Clocks:
    """nvidia-smi sampling (every 100 ms) during the timed region.  The SM
    clock reported is the median of the samples taken under load (GPU
    utilisation at least 50%; all samples if none was); a throttle reason
    counts if any sample shows it."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")
    PERIOD_MS = 100

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()

    def summary(self):
        self.f.flush()
        rows = []
        try:
            for line in open(self.f.name):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        finally:
            os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        util = lambda r: float(r[9]) if len(r) > 9 and r[9].replace(".", "").isdigit() else -1.0
        loaded = [r for r in rows if util(r) >= 50.0]
        sm = [float(r[1]) for r in (loaded or rows)]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "power_w_max": max((float(r[3]) for r in rows if r[3].replace(".", "").isdigit()), default=None),
                "samples": len(rows), "samples_under_load": len(loaded), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ workload

def build_weights(cfg, dev, seed, layer=0, ue8m0=False):
    """One layer's router weights and 128x128-quantised expert weights (bf16
    drawn 16 experts at a time, quantised, freed)."""
    import torch
    from block_scaled_fp8_router_gb300 import synthetic as S
    from block_scaled_fp8_router_gb300.layer import MoEWeightsFP8, quantize_weights

    E, d, F = cfg.E, cfg.d, cfg.F
    sdt = torch.uint8 if ue8m0 else torch.float32     # power-of-two exponents or fp32 scales
    w = MoEWeightsFP8(S.make_router_w(cfg, dev, seed, layer),
                      torch.empty((E, 2 * F, d), dtype=torch.uint8, device=dev),
                      torch.empty((E, 2 * F // 128, d // 128), dtype=sdt, device=dev),
                      torch.empty((E, d, F), dtype=torch.uint8, device=dev),
                      torch.empty((E, d // 128, F // 128), dtype=sdt, device=dev))
    chunk = 16
    for e0 in range(0, E, chunk):
        n = min(chunk, E - e0)
        w13 = torch.stack([S.make_w13_expert(cfg, e, dev, seed, layer) for e in range(e0, e0 + n)])
        w2 = torch.stack([S.make_w2_expert(cfg, e, dev, seed, layer) for e in range(e0, e0 + n)])
        quantize_weights(w13, w2, out=w, e0=e0)
        del w13, w2
    return w


def build_workload(cfg, dev, seed, gathered=False, ue8m0=False):
    from block_scaled_fp8_router_gb300 import synthetic as S
    from block_scaled_fp8_router_gb300.layer import MoELayerFP8

    w = build_weights(cfg, dev, seed, 0, ue8m0)
    layer = MoELayerFP8(w, cfg.T, cfg.k, cfg.score_fn, cfg.renorm, cfg.route_scale, gathered=gathered)
    x = S.make_x(cfg, dev, seed)
    replay = S.make_replay_payload(cfg.with_(layers=1), dev, seed)[0] if cfg.mode == "replay" else None
    return layer, x, replay


def run_gpu(args, rank, world, workload=None, with_e2e=True, steps=None, ue8m0=False):
    import torch
    from block_scaled_fp8_router_gb300 import moe_r3 as Lb
    from block_scaled_fp8_router_gb300 import synthetic as S

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    cfg = S.CONFIGS[workload or args.workload]
    if cfg.layers > 1:
        cfg = cfg.with_(layers=1)   # one layer of a stacked workload per step
    steps = steps or args.steps
    gathered = args.form == "gathered" and not ue8m0
    layer, x, replay = build_workload(cfg, dev, rank_seed(args.seed, rank), gathered, ue8m0)
    T, k, d, F, E = cfg.T, cfg.k, cfg.d, cfg.F, cfg.E
    A = T * k
    stream = torch.cuda.current_stream()

    ev = lambda: torch.cuda.Event(enable_timing=True)
    marks = {n: [] for n in ("route", "quant", "dispatch", "ffn", "combine")}

    def step(record):
        if record:
            e = [ev() for _ in range(6)]
            e[0].record()
        layer.route(x, replay)
        if record: e[1].record()
        if ue8m0:
            Lb.fp8_block_quant_ue8m0(x, 1, q=layer.xq[:T], scale_exp=layer.xs[:T])
        else:
            Lb.fp8_block_quant(x, 1, q=layer.xq[:T], scales=layer.xs[:T])
        if record: e[2].record()
        if ue8m0:
            Lb.moe_dispatch(layer.ids[:T], E, rows=layer.xq[:T], expert_counts=layer.counts,
                            expert_offsets=layer.offsets, sorted_to_slot=layer.s2s[:A], slot_to_sorted=layer.sl2[:A],
                            rows_sorted=layer.xq_sorted[:A], workspace=layer.dsp_ws, dev_status=layer.dev_status)
        elif gathered:
            Lb.moe_dispatch(layer.ids[:T], E, expert_counts=layer.counts, expert_offsets=layer.offsets,
                            sorted_to_slot=layer.s2s[:A], slot_to_sorted=layer.sl2[:A], workspace=layer.dsp_ws,
                            dev_status=layer.dev_status)
        else:
            Lb.moe_dispatch(layer.ids[:T], E, rows=layer.xq[:T], row_scales=layer.xs[:T],
                            expert_counts=layer.counts, expert_offsets=layer.offsets,
                            sorted_to_slot=layer.s2s[:A], slot_to_sorted=layer.sl2[:A],
                            rows_sorted=layer.xq_sorted[:A], scales_sorted=layer.xs_sorted[:A],
                            workspace=layer.dsp_ws, dev_status=layer.dev_status)
        if record: e[3].record()
        if ue8m0:
            Lb.moe_grouped_ffn_mx(layer.xq_sorted[:A], layer.xs[:T], layer.s2s[:A], k, layer.offsets, layer.w.w13_q,
                                  layer.w.w13_s, layer.w.w2_q, layer.w.w2_s, out_sorted=layer.out_sorted[:A],
                                  workspace=layer.ffn_ws, dev_status=layer.dev_status)
        elif gathered:
            Lb.moe_grouped_ffn_fp8_gathered(layer.xq[:T], layer.xs[:T], k, layer.s2s[:A], layer.offsets,
                                            layer.w.w13_q, layer.w.w13_s, layer.w.w2_q, layer.w.w2_s,
                                            out_slots=layer.out_sorted[:A], workspace=layer.ffn_ws,
                                            dev_status=layer.dev_status)
        else:
            Lb.moe_grouped_ffn_fp8(layer.xq_sorted[:A], layer.xs_sorted[:A], layer.offsets, layer.w.w13_q,
                                   layer.w.w13_s, layer.w.w2_q, layer.w.w2_s, out_sorted=layer.out_sorted[:A],
                                   workspace=layer.ffn_ws, dev_status=layer.dev_status)
        if record: e[4].record()
        if gathered:
            Lb.moe_combine_slots(layer.out_sorted[:A], layer.sl2[:A], layer.gates[:T], y=layer.y[:T])
        else:
            Lb.moe_combine(layer.out_sorted[:A], layer.sl2[:A], layer.gates[:T], y=layer.y[:T])
        if record:
            e[5].record()
            return e
        return None

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        flush.zero_()
        step(False)
    barrier()
    # ---- device-resident timed region: K steps, each bracketed by its own
    # events, with an L2 flush (a 512 MB write) before each step outside them ----
    with Clocks(dev.index) as clk:
        t0, t1 = ev(), ev()
        t0.record()
        per = []
        for _ in range(steps):
            flush.zero_()
            per.append(step(True))
        t1.record()
        barrier()
    clocks = clk.summary()
    total_ms = sum(e[0].elapsed_time(e[5]) for e in per)
    bracket_ms = t0.elapsed_time(t1)
    for e in per:
        for i, n in enumerate(("route", "quant", "dispatch", "ffn", "combine")):
            marks[n].append(e[i].elapsed_time(e[i + 1]))
    status = Lb.check_status(layer.dev_status)
    padded = padded_fraction(layer.counts.cpu())

    if not with_e2e:
        avg = {n: sum(v) / len(v) for n, v in marks.items()}
        total_ms = reduce_max([total_ms], world)[0]
        return dict(cfg=cfg, total_ms=total_ms, avg=avg, clocks=clocks, status=status, steps=steps, padded=padded)

    # ---- end to end through the public layer API: pinned host x in, y out,
    # copies overlapped with compute by HostStreamer (two copy streams) ----
    from block_scaled_fp8_router_gb300.layer import HostStreamer
    xh = torch.empty((T, d), dtype=torch.bfloat16, pin_memory=True)
    xh.copy_(x.cpu())
    yhs = [torch.empty((T, d), dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    rh = None
    if replay is not None:
        rh = torch.empty(replay.shape, dtype=torch.int32, pin_memory=True)
        rh.copy_(replay.cpu())
    streamer = HostStreamer(layer, T)

    def e2e_run(n):
        # the same pinned input batch every step (one batch of synthetic tokens)
        reps = None
        if rh is not None:
            rd = torch.empty_like(replay)
            rd.copy_(rh, non_blocking=True)
            reps = [rd] * n
        streamer.run([xh] * n, [yhs[i & 1] for i in range(n)], reps)

    e2e_run(max(1, args.warmup))
    streamer.synchronize()
    barrier()
    a, b = ev(), ev()
    a.record()
    streamer.h2d.wait_event(a)
    streamer.d2h.wait_event(a)
    e2e_run(steps)
    torch.cuda.current_stream().wait_stream(streamer.d2h)
    b.record()
    streamer.synchronize()
    barrier()
    e2e_ms = a.elapsed_time(b)
    h2d = T * d * 2 + (rh.numel() * 4 if rh is not None else 0)

    total_ms, e2e_ms = reduce_max([total_ms, e2e_ms], world)
    avg = {n: sum(v) / len(v) for n, v in marks.items()}
    return dict(cfg=cfg, total_ms=total_ms, e2e_ms=e2e_ms, avg=avg, clocks=clocks, status=status, h2d=h2d,
                d2h=T * d * 2, x=x, layer=layer, padded=padded, bracket_ms=bracket_ms)


def reduce_max(vals, world):
    """Max over ranks of per-rank timings (the slowest rank sets the job's
    time); a no-op for one rank.  Uses the process group's own device (CUDA
    for NCCL, host for gloo)."""
    import torch
    if world <= 1:
        return list(vals)
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor(list(vals), dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.cpu().tolist()


def job_throughput(tokens_per_rank, steps, world, total_ms):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time
    (token sharding, weak scaling: each rank runs its own batch)."""
    return tokens_per_rank * steps * world / (total_ms * 1e-3)


def rank_seed(seed, rank):
    """Each rank draws its own batch (and its own replica weights)."""
    return seed + rank


def rooflines(cfg, avg, peaks, gathered=False, ue8m0=False):
    T, k, d, F, E = cfg.T, cfg.k, cfg.d, cfg.F, cfg.E
    A = T * k
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    flops_ffn = 6.0 * A * d * F
    ffn = {"bound": "tensor", "kernel": ("moe_grouped_ffn_fp8_gathered" if gathered else "moe_grouped_ffn_fp8")
                                         + " (GEMM1+SwiGLU+requant, GEMM2)",
           "achieved": flops_ffn / (avg["ffn"] * 1e-3) / 1e12, "peak": fp8_peak, "unit": "TFLOP/s",
           "peak_note": "FP8 dense = 2 x measured bf16 burst (nominal FP8:BF16 ratio)" if peaks["source"] == "measured"
           else "FP8 dense = 2 x fallback bf16",
           "traffic": FFN_DRAM_BYTES_PER_ROW * A if cfg.d == 7168 and cfg.F == 2048 else None,
           "traffic_note": "dram read+write bytes of both GEMM kernels from one ncu capture of the profiling shape "
                           "(large_e64: same per-expert shape, 1/4 of the experts), scaled by routed rows"}
    ffn["frac"] = ffn["achieved"] / ffn["peak"]
    if peaks.get("fp8_tflops_measured"):
        ffn["peak_fp8_measured"] = peaks["fp8_tflops_measured"]
        ffn["frac_of_fp8_measured"] = ffn["achieved"] / peaks["fp8_tflops_measured"]
        ffn["fp8_measured_note"] = "cuBLASLt e4m3 GEMM 8192^3 via torch._scaled_mm, best of 10, this run"
    hbm = peaks["hbm_gbs"]
    row = d + (1 if ue8m0 else 4) * d / 128     # one FP8 row with its 1x128 scales (fp32 or exponent bytes)
    bytes_quant = T * d * 2 + T * row
    if ue8m0:
        row = d                                 # dispatch moves the codes only (the exponents stay token-major)
    bytes_disp = A * 4 + 2 * A * 4 + (0 if gathered else T * row + A * row)  # ids, two maps (+ row copy)
    bytes_comb = A * d * 2 + A * 4 + T * k * 4 + T * d * 2  # A bf16 rows + map + gates in, y out
    route_flops = 2.0 * T * d * E if cfg.mode == "route" else 2.0 * T * d * k
    extra = {
        "quant_1x128": {"ms": avg["quant"], "GB/s": bytes_quant / (avg["quant"] * 1e-3) / 1e9},
        "dispatch": {"ms": avg["dispatch"], "GB/s": bytes_disp / (avg["dispatch"] * 1e-3) / 1e9},
        "combine": {"ms": avg["combine"], "GB/s": bytes_comb / (avg["combine"] * 1e-3) / 1e9},
        ("route_topk" if cfg.mode == "route" else "route_replay"):
            {"ms": avg["route"], "fp32 TFLOP/s": route_flops / (avg["route"] * 1e-3) / 1e12,
             "frac_of_fp32_alu_derived": route_flops / (avg["route"] * 1e-3) / 1e12 / FP32_ALU_TFLOPS_DERIVED,
             "fp32_alu_peak_derived": FP32_ALU_TFLOPS_DERIVED,
             "peak_note": "derived, not measured: 152 SMs x 128 FMA lanes x 2 FLOP x 2.07 GHz"},
        "ffn": {"ms": avg["ffn"]},
    }
    for key in ("quant_1x128", "dispatch", "combine"):
        extra[key]["frac_hbm"] = extra[key]["GB/s"] / hbm
    return ffn, extra


def run_multilayer(dev, seed, steps, warmup, peaks):
    """The stacked replay workload as written: 8 layers of the large shape
    (d=7168, 256 experts, top-8, F=2048), T=16384 tokens, one routed-experts
    payload [8, 8, 16384] (30% of slots to 8 hot experts, 8 experts that
    receive nothing).  All 8 layers' FP8 weights stay resident (8 x 11.3 GB);
    one sweep runs every layer in turn: replay of its payload slab (gates
    from its router) -> 1x128 quantisation -> dispatch -> grouped FFN ->
    combine.  A 512 MB L2 flush precedes each timed sweep."""
    import torch
    from block_scaled_fp8_router_gb300 import moe_r3 as Lb
    from block_scaled_fp8_router_gb300 import synthetic as S
    from block_scaled_fp8_router_gb300.layer import MoELayerFP8
    cfg = S.CONFIGS["multilayer_replay"]
    Ln, T, k, d, F, E = cfg.layers, cfg.T, cfg.k, cfg.d, cfg.F, cfg.E
    A = T * k
    payload = S.make_replay_payload(cfg, dev, seed)                 # [L, k, T]
    weights = [build_weights(cfg, dev, seed, l) for l in range(Ln)]
    xs = [S.make_x(cfg, dev, seed, l) for l in range(Ln)]
    layer = MoELayerFP8(weights[0], T, k, cfg.score_fn, cfg.renorm, cfg.route_scale)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    padded = []

    def sweep(ffn_ev=None):
        for l in range(Ln):
            layer.w = weights[l]
            layer.route(xs[l], payload[l])
            xq, xsc = Lb.fp8_block_quant(xs[l], 1, q=layer.xq[:T], scales=layer.xs[:T])
            Lb.moe_dispatch(layer.ids[:T], E, rows=xq, row_scales=xsc, expert_counts=layer.counts,
                            expert_offsets=layer.offsets, sorted_to_slot=layer.s2s[:A], slot_to_sorted=layer.sl2[:A],
                            rows_sorted=layer.xq_sorted[:A], scales_sorted=layer.xs_sorted[:A], workspace=layer.dsp_ws,
                            dev_status=layer.dev_status)
            if ffn_ev: ffn_ev[l][0].record()
            Lb.moe_grouped_ffn_fp8(layer.xq_sorted[:A], layer.xs_sorted[:A], layer.offsets, layer.w.w13_q,
                                   layer.w.w13_s, layer.w.w2_q, layer.w.w2_s, out_sorted=layer.out_sorted[:A],
                                   workspace=layer.ffn_ws, dev_status=layer.dev_status)
            if ffn_ev: ffn_ev[l][1].record()
            Lb.moe_combine(layer.out_sorted[:A], layer.sl2[:A], layer.gates[:T], y=layer.y[:T])
            if ffn_ev is not None and len(padded) < Ln:
                padded.append(layer.counts.clone())

    for _ in range(warmup):
        flush.zero_()
        sweep()
    torch.cuda.synchronize()
    per, ffn = [], []
    for _ in range(steps):
        flush.zero_()
        a, b = ev(), ev()
        fe = [[ev(), ev()] for _ in range(Ln)]
        a.record()
        sweep(fe)
        b.record()
        per.append((a, b))
        ffn.append(fe)
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in per) / steps
    ffn_ms = sum(sum(e[0].elapsed_time(e[1]) for e in fe) for fe in ffn) / steps
    flops = 6.0 * A * d * F * Ln
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    out = {"workload": f"multilayer_replay: {Ln} layers x T={T} d={d} E={E} top_k={k} F={F}, payload "
                       f"[{Ln}, {k}, {T}] (8 hot / 8 empty experts per layer), all layers' FP8 weights resident "
                       f"({Ln * (3 * E * d * F) / 1e9:.1f} GB)",
           "tokens_x_layers/s": T * Ln / (ms * 1e-3), "ms_per_sweep": ms, "ms_per_layer": ms / Ln,
           "ffn_ms_per_layer": ffn_ms / Ln, "ffn_TFLOP/s": flops / (ffn_ms * 1e-3) / 1e12,
           "ffn_frac": flops / (ffn_ms * 1e-3) / 1e12 / fp8_peak, "peak": fp8_peak,
           "gemm_padded_rows_per_layer": [padded_fraction(c.cpu()) for c in padded],
           "steps": steps, "status": Lb.check_status(layer.dev_status)}
    if peaks.get("fp8_tflops_measured"):
        out["ffn_frac_of_fp8_measured"] = flops / (ffn_ms * 1e-3) / 1e12 / peaks["fp8_tflops_measured"]
    del weights, xs, layer, payload
    torch.cuda.empty_cache()
    return out


def run_dispatch_combine(dev, seed, steps, warmup, peaks):
    """Dispatch + combine alone on the long-context shape (T=131072, d=7168
    bf16 rows, 256 experts, top-8, replayed uniform ids, Dirichlet gates,
    identity experts): replay copy -> dispatch (maps + bf16 row gather) ->
    combine.  Inputs (1.9 GB of x, 15 GB of dispatched rows) dwarf L2."""
    import torch
    from block_scaled_fp8_router_gb300 import moe_r3 as Lb
    from block_scaled_fp8_router_gb300 import synthetic as S
    cfg = S.CONFIGS["long_dispatch"]
    T, k, d, E = cfg.T, cfg.k, cfg.d, cfg.E
    A = T * k
    payload = S.make_replay_payload(cfg, dev, seed)[0]
    gates = S.make_dirichlet_gates(cfg, dev, seed)
    x = S.make_x(cfg, dev, seed)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    rows = torch.empty((A, d), dtype=torch.bfloat16, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    s2s = torch.empty(A, dtype=torch.int32, device=dev)
    sl2 = torch.empty(A, dtype=torch.int32, device=dev)
    ws = torch.empty(Lb.moe_dispatch_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    y = torch.empty_like(x)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def step(e=None):
        if e: e[0].record()
        Lb.moe_route_replay(payload, E, topk_ids=ids, dev_status=st)
        Lb.moe_dispatch(ids, E, rows=x, expert_counts=counts, expert_offsets=offs, sorted_to_slot=s2s,
                        slot_to_sorted=sl2, rows_sorted=rows, workspace=ws, dev_status=st)
        if e: e[1].record()
        Lb.moe_combine(rows, sl2, gates, y=y)
        if e: e[2].record()

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    evs = [[ev(), ev(), ev()] for _ in range(steps)]
    for e in evs:
        step(e)
    torch.cuda.synchronize()
    t_disp = sum(e[0].elapsed_time(e[1]) for e in evs) / steps
    t_comb = sum(e[1].elapsed_time(e[2]) for e in evs) / steps
    exact = bool(torch.equal(y.view(torch.int16), x.view(torch.int16)))
    b_disp = 2 * A * 4 + A * 4 + 2 * A * 4 + T * d * 2 + A * d * 2   # replay in/out, ids, maps, rows
    b_comb = A * d * 2 + A * 4 + T * k * 4 + T * d * 2
    gbs = (b_disp + b_comb) / ((t_disp + t_comb) * 1e-3) / 1e9
    out = {"workload": f"long_dispatch: T={T} d={d} bf16 rows E={E} top_k={k}, identity experts",
           "ms": t_disp + t_comb, "dispatch_ms": t_disp, "combine_ms": t_comb, "GB/s": gbs,
           "frac": gbs / peaks["hbm_gbs"], "peak_GB/s": peaks["hbm_gbs"],
           "bytes": b_disp + b_comb, "bytes_rows_only": 2 * T * d * (2 + 2 * k),
           "combine_of_dispatch_exact": exact, "status": Lb.check_status(st)}
    del rows, x, y
    torch.cuda.empty_cache()
    return out


def run_backward(cfg, dev, seed, steps, warmup, peaks):
    """Backward of the expert path with the routing fixed (as the trainer
    replays it): forward(train=True) once, then per step combine backward ->
    dgrad GEMM (W2^T) -> SwiGLU backward -> dgrad GEMM (W13^T) -> dispatch
    backward, timed by CUDA events between the calls."""
    import torch
    from block_scaled_fp8_router_gb300 import moe_r3 as Lb
    layer, x, replay = build_workload(cfg, dev, seed)
    layer.forward(x, replay_kT=replay, train=True)
    layer.backward(torch.zeros_like(x))               # allocates the gradient buffers and the W^T copies
    torch.cuda.synchronize()
    T, k, d, F, E = cfg.T, cfg.k, cfg.d, cfg.F, cfg.E
    A = T * k
    dy = torch.empty_like(x).normal_(0.0, 1.0, generator=torch.Generator(device=dev).manual_seed(seed + 1))
    b = layer._bw
    w2t_q, w2t_s, w13t_q, w13t_s = layer.w.transposed()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    names = ("combine_bwd", "dgrad_gemm2", "swiglu_bwd", "dgrad_gemm1", "dispatch_bwd")

    def step(e=None):
        if e: e[0].record()
        Lb.moe_combine_backward(dy, layer.gates[:T], layer.out_sorted[:A], layer.sl2[:A], d_out_q=b["d_out_q"][:A],
                                d_out_s=b["d_out_s"][:A], d_gates=b["d_gates"][:T], dev_status=layer.dev_status)
        if e: e[1].record()
        Lb.moe_grouped_gemm_fp8(b["d_out_q"][:A], b["d_out_s"][:A], layer.offsets, w2t_q, w2t_s, out=b["d_act"][:A],
                                dev_status=layer.dev_status)
        if e: e[2].record()
        Lb.moe_swiglu_backward(b["d_act"][:A], layer.h[:A], dh_q=b["dh_q"][:A], dh_s=b["dh_s"][:A])
        if e: e[3].record()
        Lb.moe_grouped_gemm_fp8(b["dh_q"][:A], b["dh_s"][:A], layer.offsets, w13t_q, w13t_s,
                                out=b["dx_sorted"][:A], dev_status=layer.dev_status)
        if e: e[4].record()
        Lb.moe_dispatch_backward(b["dx_sorted"][:A], layer.sl2[:A], T, k, dx=b["dx"][:T])
        if e: e[5].record()

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0, t1 = ev(), ev()
    evs = [[ev() for _ in range(6)] for _ in range(steps)]
    t0.record()
    for e in evs:
        step(e)
    t1.record()
    torch.cuda.synchronize()
    total = t0.elapsed_time(t1) / steps
    split = {n: sum(e[i].elapsed_time(e[i + 1]) for e in evs) / steps for i, n in enumerate(names)}
    gemm_ms = split["dgrad_gemm2"] + split["dgrad_gemm1"]
    # weight gradients (four 128 x 1 operand quantisations, two grouped GEMMs)
    for _ in range(warmup):
        layer._weight_grads(dy, T)
    torch.cuda.synchronize()
    a, bb = ev(), ev()
    a.record()
    for _ in range(steps):
        layer._weight_grads(dy, T)
    bb.record()
    torch.cuda.synchronize()
    wg_ms = a.elapsed_time(bb) / steps
    # the same calls split by events (pad offsets + d_out quantisation, act
    # quantisation, dW2 GEMM, dh quantisation, x quantisation, dW13 GEMM)
    wg_names = ("quant_d_out", "quant_act", "gemm_dW2", "quant_dh", "quant_x", "gemm_dW13")
    wevs = [[ev() for _ in range(7)] for _ in range(steps)]
    for e in wevs:
        layer._weight_grads(dy, T, events=e)
    torch.cuda.synchronize()
    wg_split = {n: sum(e[i].elapsed_time(e[i + 1]) for e in wevs) / steps for i, n in enumerate(wg_names)}
    # the router's backward (ids fixed): d_logits alone, + dx, + dW_r, each
    # timed over `steps` calls; the splits are the differences
    dgates = b["d_gates"][:T]
    rb_dl = torch.empty((T, k), dtype=torch.float32, device=dev)
    rb_dx = torch.empty((T, d), dtype=torch.float32, device=dev)
    rb_dw = torch.empty((E, d), dtype=torch.float32, device=dev)

    def rb_call(with_dx, with_dw):
        Lb.moe_router_backward(x, layer.w.w_router, layer.ids[:T], dgates, layer.score_fn, layer.renorm,
                               layer.route_scale, d_logits=rb_dl, dx=rb_dx if with_dx else None,
                               dw_router=rb_dw if with_dw else None, sorted_to_slot=layer.s2s[:A],
                               expert_offsets=layer.offsets, dev_status=layer.dev_status)

    rb_ms = {}
    for key, flags in (("dl", (False, False)), ("dl_dx", (True, False)), ("all", (True, True))):
        for _ in range(warmup):
            rb_call(*flags)
        torch.cuda.synchronize()
        a, bb = ev(), ev()
        a.record()
        for _ in range(steps):
            rb_call(*flags)
        bb.record()
        torch.cuda.synchronize()
        rb_ms[key] = a.elapsed_time(bb) / steps
    flops = 6.0 * A * d * F
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    hbm = peaks["hbm_gbs"]
    row = d + 4 * d / 128
    b_comb = T * d * 2 + A * d * 2 + A * row + A * 4 + T * k * 8
    b_swi = A * F * 2 + A * 2 * F * 4 + A * 2 * F * (1 + 4 / 128)
    b_disp = A * d * 2 + A * 4 + T * d * 2
    out = {"workload": f"{cfg.name}: T={T} d={d} E={E} top_k={k} F={F}, expert-path backward (dgrad) with the "
                       "routing fixed", "tokens/s": T / (total * 1e-3), "ms_per_step": total,
           "steps": {n: {"ms": v} for n, v in split.items()},
           "dgrad_gemms": {"ms": gemm_ms, "TFLOP/s": flops / (gemm_ms * 1e-3) / 1e12,
                           "frac": flops / (gemm_ms * 1e-3) / 1e12 / fp8_peak, "peak": fp8_peak},
           "weight_grads": {"ms": wg_ms, "TFLOP/s (dW2 + dW13 GEMMs, algorithmic)": flops / (wg_ms * 1e-3) / 1e12,
                            "note": "includes the four 128x1 operand quantisations and the fp32 dW writes "
                                    f"({4 * 3 * E * d * F / 1e9:.1f} GB)",
                            "steps": {n: {"ms": v} for n, v in wg_split.items()}},
           "status": Lb.check_status(layer.dev_status)}
    dx_ms, dw_ms = rb_ms["dl_dx"] - rb_ms["dl"], rb_ms["all"] - rb_ms["dl_dx"]
    out["router_bwd"] = {
        "ms": rb_ms["all"],
        "note": "gradients of the router for the fixed ids: d_logits (the chosen logits re-formed, gate "
                "derivative), dx [T, d] and dW_r [E, d] in fp32; not part of ms_per_step",
        "d_logits": {"ms": rb_ms["dl"], "router row bytes through L1": T * k * d * 2,
                     "fp32 TFLOP/s": 2 * T * k * d / (rb_ms["dl"] * 1e-3) / 1e12},
        "dx": {"ms": dx_ms, "bytes": T * d * 4 + T * k * 8, "GB/s": (T * d * 4 + T * k * 8) / (dx_ms * 1e-3) / 1e9,
               "frac_hbm": (T * d * 4 + T * k * 8) / (dx_ms * 1e-3) / 1e9 / hbm},
        "dW_r": {"ms": dw_ms, "x row bytes per routed row (L2)": A * d * 2, "bytes (HBM: x once, dW_r written)":
                 T * d * 2 + E * d * 4}}
    for n, nb in (("combine_bwd", b_comb), ("swiglu_bwd", b_swi), ("dispatch_bwd", b_disp)):
        out["steps"][n]["GB/s"] = nb / (split[n] * 1e-3) / 1e9
        out["steps"][n]["frac_hbm"] = out["steps"][n]["GB/s"] / hbm
    # the weight-gradient GEMMs are bound by their fp32 stores: output bytes
    # per launch over the launch time, against the measured copy bandwidth
    # the 128 x 1 operand quantisations: source rows read once per routed row
    # (dy and x gathered per slot), codes and scales over the padded rows P
    cnt = (layer.offsets[1:E + 1] - layer.offsets[:E]).cpu().to(torch.int64)
    P = int((((cnt + 127) // 128) * 128).sum())
    codes = lambda C: C * P * (1 + 4 / 128)
    b_q = {"quant_d_out": A * d * 2 + A * 8 + codes(d), "quant_act": A * 2 * F * 4 + codes(F),
           "quant_dh": A * F * 2 + A * 2 * F * 4 + codes(2 * F), "quant_x": A * d * 2 + A * 4 + codes(d)}
    for n, nb in b_q.items():
        st = out["weight_grads"]["steps"][n]
        st["bytes"] = nb
        st["GB/s"] = nb / (st["ms"] * 1e-3) / 1e9
        st["frac_hbm"] = st["GB/s"] / hbm
    out["weight_grads"]["padded_rows"] = P
    for n, nb in (("gemm_dW2", 4.0 * E * d * F), ("gemm_dW13", 4.0 * E * 2 * F * d)):
        st = out["weight_grads"]["steps"][n]
        st["store GB/s"] = nb / (st["ms"] * 1e-3) / 1e9
        st["frac_hbm"] = st["store GB/s"] / hbm
    del layer, x, b
    torch.cuda.empty_cache()
    return out


def run_nvfp4_layer(cfg, dev, seed, steps, warmup, peaks):
    """The layer with NVFP4 activations and expert weights (E2M1 codes, E4M3
    scales per 16 elements, fp32 tensor scales; the FP4 variant) on the large
    workload: route -> NVFP4 x -> dispatch -> moe_grouped_ffn_nvfp4 (two
    kind::mxf4nvf4 block-scaled GEMMs with act requantised between them) ->
    combine.  Weights quantised once before timing; an L2 flush before each
    step."""
    import torch
    from block_scaled_fp8_router_gb300 import moe_r3 as Lb
    from block_scaled_fp8_router_gb300 import synthetic as S
    from block_scaled_fp8_router_gb300.layer import (MoELayerNVFP4, MoEWeightsNVFP4, finish_nvfp4_weights,
                                                     quantize_weights_nvfp4)
    T, k, d, F, E = cfg.T, cfg.k, cfg.d, cfg.F, cfg.E
    A = T * k
    e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
    W = MoEWeightsNVFP4(S.make_router_w(cfg, dev, seed), e((E, 2 * F, d // 2), torch.uint8),
                        e((E, 2 * F, d // 16), torch.uint8), e((E,), torch.float32), None,
                        e((E, d, F // 2), torch.uint8), e((E, d, F // 16), torch.uint8), e((E,), torch.float32), None)
    for e0 in range(0, E, 16):
        n = min(16, E - e0)
        w13 = torch.stack([S.make_w13_expert(cfg, i, dev, seed) for i in range(e0, e0 + n)])
        w2 = torch.stack([S.make_w2_expert(cfg, i, dev, seed) for i in range(e0, e0 + n)])
        quantize_weights_nvfp4(W.w_router, w13, w2, out=W, e0=e0)
        del w13, w2
    finish_nvfp4_weights(W)
    layer = MoELayerNVFP4(W, T, k, cfg.score_fn, cfg.renorm, cfg.route_scale)
    x = S.make_x(cfg, dev, seed)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def ffn():
        Lb.moe_grouped_ffn_nvfp4(layer.xq_sorted[:A], layer.xs_sorted[:A], layer.x_ts, layer.offsets, W.w13_q,
                                 W.w13_sf, W.w13_enc, W.w2_q, W.w2_sf, W.w2_enc, out_sorted=layer.out_sorted[:A],
                                 workspace=layer.ffn_ws, dev_status=layer.dev_status)

    for _ in range(warmup):
        flush.zero_()
        layer.forward(x)
    torch.cuda.synchronize()
    per = []
    for _ in range(steps):
        flush.zero_()
        a, b = ev(), ev()
        a.record()
        layer.forward(x)
        b.record()
        per.append((a, b))
    fper = []
    for _ in range(steps):
        flush.zero_()
        a, b = ev(), ev()
        a.record()
        ffn()
        b.record()
        fper.append((a, b))
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in per) / steps
    ffn_ms = sum(a.elapsed_time(b) for a, b in fper) / steps
    flops = 6.0 * A * d * F
    fp4_peak = 6.0 * peaks["bf16_tflops"]
    out = {"workload": f"{cfg.name}: T={T} d={d} E={E} top_k={k} F={F}, NVFP4 activations and weights "
                       f"({E * 3 * d * F / 2 / 1e9:.2f} GB of E2M1 weight codes)",
           "tokens/s": T / (ms * 1e-3), "ms_per_step": ms, "ffn_ms": ffn_ms,
           "ffn_TFLOP/s": flops / (ffn_ms * 1e-3) / 1e12,
           "ffn_frac_of_fp4_peak": flops / (ffn_ms * 1e-3) / 1e12 / fp4_peak, "fp4_peak": fp4_peak,
           "peak_note": "FP4 dense = 6 x measured bf16 burst (the nominal FP4:BF16 ratio, 13.5 / 2.25 PFLOP/s)",
           "status": Lb.check_status(layer.dev_status)}
    del layer, W, x
    torch.cuda.empty_cache()
    return out


def run_nvfp4_quant(cfg, dev, seed, steps, warmup, peaks):
    """The NVFP4 quantiser (fp8_quant_nvfp4: tensor amax pass, then E4M3 block
    scales and packed E2M1 codes) on the layer's activations [T, d] bf16."""
    import torch
    from block_scaled_fp8_router_gb300 import moe_r3 as Lb
    from block_scaled_fp8_router_gb300 import synthetic as S
    x = S.make_x(cfg, dev, seed)
    T, d = x.shape
    q = torch.empty((T, d // 2), dtype=torch.uint8, device=dev)
    s = torch.empty((T, d // 16), dtype=torch.uint8, device=dev)
    ts = torch.empty((2,), dtype=torch.float32, device=dev)
    for _ in range(warmup):
        Lb.fp8_quant_nvfp4(x, q=q, scales=s, tensor_scale=ts)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        Lb.fp8_quant_nvfp4(x, q=q, scales=s, tensor_scale=ts)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    nbytes = T * d * (2 + 2 + 0.5 + 1 / 16)      # x read by both passes, codes and scales written
    return {"workload": f"x [{T}, {d}] bf16 -> NVFP4 (16-element E4M3-scaled blocks, fp32 tensor scale)",
            "ms": ms, "GB/s": nbytes / (ms * 1e-3) / 1e9, "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "launches": 2, "note": "x (117 MB) fits L2, so the second pass may read it from L2"}


def run_payload(dev, seed, steps, warmup, peaks):
    """The routed-experts payload at one byte per id: a [64, 8, 131072] int32
    payload (64 layers x top-8 x 128K tokens, 268 MB, replayed-id
    distribution) packed to uint8 and unpacked again on the device, one
    layer slab replayed from bytes and from int32 (ids only), and the
    payload's host->device copy from pinned memory at both widths."""
    import torch
    from block_scaled_fp8_router_gb300 import moe_r3 as Lb
    from block_scaled_fp8_router_gb300 import synthetic as S
    cfg = S.CONFIGS["long_dispatch"].with_(layers=64)
    L_, k, T, E = cfg.layers, cfg.k, cfg.T, cfg.E
    n = L_ * k * T
    payload = S.make_replay_payload(cfg, dev, seed)            # [L, k, T] int32
    packed = torch.empty_like(payload, dtype=torch.uint8)
    back = torch.empty_like(payload)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    h32 = torch.empty(payload.shape, dtype=torch.int32, pin_memory=True)
    h8 = torch.empty(payload.shape, dtype=torch.uint8, pin_memory=True)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = ev(), ev()
        a.record()
        for _ in range(steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    t_pack = timed(lambda: Lb.moe_payload_pack_u8(payload, E, out=packed, dev_status=st))
    t_unpack = timed(lambda: Lb.moe_payload_unpack_u8(packed, out=back))
    exact = bool(torch.equal(back, payload))
    t_r32 = timed(lambda: Lb.moe_route_replay(payload[7], E, topk_ids=ids, dev_status=st))
    t_r8 = timed(lambda: Lb.moe_route_replay(packed[7], E, topk_ids=ids, dev_status=st))
    t_h32 = timed(lambda: payload.copy_(h32, non_blocking=True))
    t_h8 = timed(lambda: packed.copy_(h8, non_blocking=True))
    gbs = lambda b, t: b / (t * 1e-3) / 1e9
    out = {"workload": f"routed-experts payload [{L_}, {k}, {T}] (E={E}), replayed-id distribution",
           "ids": n, "bytes_int32": 4 * n, "bytes_u8": n,
           "pack_ms": t_pack, "pack_GB/s": gbs(5 * n, t_pack), "pack_frac_hbm": gbs(5 * n, t_pack) / peaks["hbm_gbs"],
           "unpack_ms": t_unpack, "unpack_GB/s": gbs(5 * n, t_unpack),
           "unpack_frac_hbm": gbs(5 * n, t_unpack) / peaks["hbm_gbs"], "round_trip_exact": exact,
           "replay_layer_ids_only_ms": {"int32": t_r32, "u8": t_r8},
           "h2d_ms": {"int32": t_h32, "u8": t_h8}, "h2d_GB/s": {"int32": gbs(4 * n, t_h32), "u8": gbs(n, t_h8)},
           "status": Lb.check_status(st)}
    del payload, packed, back, h32, h8
    torch.cuda.empty_cache()
    return out


def run_hbm_kernels(dev, seed, steps, warmup, peaks):
    """The HBM-bound kernels alone on a profiling shape larger than L2 and a
    few GB in total: T=16384 tokens, d=7168, E=256, top-8, replayed uniform
    ids.  1x128 quantiser (235 MB of x), dispatch with FP8 rows + scales
    (940 MB of rows), combine of bf16 expert rows (1.9 GB), one-byte payload
    pack/unpack of a [64, 8, 131072] payload (268 MB)."""
    import torch
    from block_scaled_fp8_router_gb300 import moe_r3 as Lb
    from block_scaled_fp8_router_gb300 import synthetic as S
    cfg = S.CONFIGS["long_dispatch"].with_(T=16384)
    T, k, d, E = cfg.T, cfg.k, cfg.d, cfg.E
    A = T * k
    x = S.make_x(cfg, dev, seed)
    ids = S.make_replay_payload(cfg, dev, seed)[0].t().contiguous()
    gates = S.make_dirichlet_gates(cfg, dev, seed)
    q = torch.empty((T, d), dtype=torch.uint8, device=dev)
    sc = torch.empty((T, d // 128), dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    s2s = torch.empty(A, dtype=torch.int32, device=dev)
    sl2 = torch.empty(A, dtype=torch.int32, device=dev)
    rows = torch.empty((A, d), dtype=torch.uint8, device=dev)
    rsc = torch.empty((A, d // 128), dtype=torch.float32, device=dev)
    ws = torch.empty(Lb.moe_dispatch_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
    out = torch.empty((A, d), dtype=torch.bfloat16, device=dev).normal_(0.0, 0.1, generator=torch.Generator(device=dev).manual_seed(seed))
    y = torch.empty_like(x)
    pl = S.make_replay_payload(S.CONFIGS["long_dispatch"].with_(layers=64), dev, seed)
    packed = torch.empty_like(pl, dtype=torch.uint8)
    back = torch.empty_like(pl)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = ev(), ev()
        a.record()
        for _ in range(steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    gbs = lambda nbytes, ms: nbytes / (ms * 1e-3) / 1e9
    row = d + 4 * d / 128
    res = {}
    t = timed(lambda: Lb.fp8_block_quant(x, 1, q=q, scales=sc))
    res["quant_1x128"] = {"ms": t, "bytes": T * d * 2 + T * row, "GB/s": gbs(T * d * 2 + T * row, t)}
    t = timed(lambda: Lb.moe_dispatch(ids, E, rows=q, row_scales=sc, expert_counts=counts, expert_offsets=offs,
                                      sorted_to_slot=s2s, slot_to_sorted=sl2, rows_sorted=rows, scales_sorted=rsc,
                                      workspace=ws, dev_status=st))
    nb = A * 4 + 2 * A * 4 + T * row + A * row
    res["dispatch_fp8_rows"] = {"ms": t, "bytes": nb, "GB/s": gbs(nb, t)}
    t = timed(lambda: Lb.moe_combine(out, sl2, gates, y=y))
    nb = A * d * 2 + A * 4 + A * 4 + T * d * 2
    res["combine"] = {"ms": t, "bytes": nb, "GB/s": gbs(nb, t)}
    n = pl.numel()
    t = timed(lambda: Lb.moe_payload_pack_u8(pl, E, out=packed, dev_status=st))
    res["payload_pack_u8"] = {"ms": t, "bytes": 5 * n, "GB/s": gbs(5 * n, t)}
    t = timed(lambda: Lb.moe_payload_unpack_u8(packed, out=back))
    res["payload_unpack_u8"] = {"ms": t, "bytes": 5 * n, "GB/s": gbs(5 * n, t)}
    del x, q, sc, rows, rsc, out, y, pl, packed, back, ws
    torch.cuda.empty_cache()
    # the backward's HBM-bound steps on the large layer's shape (T=8192,
    # 256 rows per expert, so the 128 x 1 legs have no padding): combine
    # backward, SwiGLU backward and the four 128 x 1 operand quantisations
    Tb, F = 8192, 2048
    Ab = Tb * k
    g = torch.Generator(device=dev).manual_seed(seed + 7)
    dy = torch.randn((Tb, d), generator=g, device=dev).to(torch.bfloat16)
    outb = torch.randn((Ab, d), generator=g, device=dev).to(torch.bfloat16)
    gb = torch.rand((Tb, k), generator=g, device=dev)
    slb = torch.randperm(Ab, generator=g, device=dev).to(torch.int32)             # slot -> sorted row
    s2b = torch.empty_like(slb)
    s2b[slb.long()] = torch.arange(Ab, device=dev, dtype=torch.int32)
    offb = torch.arange(E + 1, device=dev, dtype=torch.int32) * (Ab // E)
    padb = Lb.moe_wgrad_pad_offsets(offb)
    ld = (Ab // 128 + E) * 128
    h = torch.randn((Ab, 2 * F), generator=g, device=dev)
    d_act = torch.randn((Ab, F), generator=g, device=dev).to(torch.bfloat16)
    qb = torch.empty((max(d, 2 * F), ld), dtype=torch.uint8, device=dev)
    sbf = torch.empty((ld // 128) * max(d, 2 * F), dtype=torch.float32, device=dev)
    sb = lambda C: sbf[:(ld // 128) * C].view(ld // 128, C)
    dq = torch.empty((Ab, d), dtype=torch.uint8, device=dev)
    ds = torch.empty((Ab, d // 128), dtype=torch.float32, device=dev)
    dg = torch.empty((Tb, k), dtype=torch.float32, device=dev)
    hq = torch.empty((Ab, 2 * F), dtype=torch.uint8, device=dev)
    hs = torch.empty((Ab, 2 * F // 128), dtype=torch.float32, device=dev)
    codes = lambda C: C * Ab * (1 + 4 / 128)
    bw = {
        "combine_backward": (lambda: Lb.moe_combine_backward(dy, gb, outb, slb, d_out_q=dq, d_out_s=ds, d_gates=dg,
                                                             dev_status=st),
                             Tb * d * 2 + Ab * d * 2 + Ab * row + Ab * 8),
        "swiglu_backward": (lambda: Lb.moe_swiglu_backward(d_act, h, dh_q=hq, dh_s=hs),
                            Ab * F * 2 + Ab * 2 * F * 4 + codes(2 * F)),
        "wgrad_quant_d_out": (lambda: Lb.moe_wgrad_quant(0, offb, padb, d, ld, True, dy=dy, gates=gb.view(-1),
                                                         sorted_to_slot=s2b, k=k, q=qb[:d], scales=sb(d)),
                              Ab * d * 2 + Ab * 8 + codes(d)),
        "wgrad_quant_act": (lambda: Lb.moe_wgrad_quant(1, offb, padb, F, ld, True, h=h, F=F, q=qb[:F],
                                                       scales=sb(F)),
                            Ab * 2 * F * 4 + codes(F)),
        "wgrad_quant_dh": (lambda: Lb.moe_wgrad_quant(2, offb, padb, 2 * F, ld, True, h=h, d_act=d_act, F=F,
                                                      q=qb[:2 * F], scales=sb(2 * F)),
                           Ab * F * 2 + Ab * 2 * F * 4 + codes(2 * F)),
        "wgrad_quant_x": (lambda: Lb.moe_wgrad_quant(3, offb, padb, d, ld, True, x=dy, sorted_to_slot=s2b, k=k,
                                                     q=qb[:d], scales=sb(d)),
                          Ab * d * 2 + Ab * 4 + codes(d)),
    }
    for name, (fn, nb) in bw.items():
        t = timed(fn)
        res[name] = {"ms": t, "bytes": nb, "GB/s": gbs(nb, t)}
    for v in res.values():
        v["frac_hbm"] = v["GB/s"] / peaks["hbm_gbs"]
    return {"workload": f"HBM kernels: T={T} d={d} E={E} top_k={k} (replayed uniform ids); payload [64, 8, 131072]; "
                        f"backward steps at T={Tb} F={F} (256 rows per expert)",
            "peak_GB/s": peaks["hbm_gbs"], "kernels": res, "status": Lb.check_status(st)}


def run_router_kernels(dev, seed, steps, warmup):
    """The router kernels alone (no expert weights on the device): route_topk
    on the large layer's shape (T=8192, d=7168, E=256, top-8, sigmoid) and
    route_replay of one layer of the replay workload (T=16384, skewed
    replayed ids, gates from the router logits)."""
    import torch
    from block_scaled_fp8_router_gb300 import moe_r3 as Lb
    from block_scaled_fp8_router_gb300 import synthetic as S
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = ev(), ev()
        a.record()
        for _ in range(steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    res = {}
    c = S.CONFIGS["large"]
    x = S.make_x(c, dev, seed)
    wr = S.make_router_w(c, dev, seed)
    ids = torch.empty((c.T, c.k), dtype=torch.int32, device=dev)
    g = torch.empty((c.T, c.k), dtype=torch.float32, device=dev)
    t = timed(lambda: Lb.moe_route_topk(x, wr, c.k, c.score_fn, c.renorm, c.route_scale, topk_ids=ids, topk_gates=g))
    res["route_topk"] = {"workload": f"T={c.T} d={c.d} E={c.E} top_k={c.k}", "ms": t,
                         "fp32 TFLOP/s": 2.0 * c.T * c.d * c.E / (t * 1e-3) / 1e12}
    # the router's backward for these ids: d_logits, dx, dW_r (the dispatch
    # maps for dW_r; a seeded upstream gradient)
    s2s = torch.empty(c.T * c.k, dtype=torch.int32, device=dev)
    offs = torch.empty(c.E + 1, dtype=torch.int32, device=dev)
    Lb.moe_dispatch(ids, c.E, expert_offsets=offs, sorted_to_slot=s2s)
    dgates = torch.empty((c.T, c.k), dtype=torch.float32, device=dev).normal_(
        0.0, 1.0, generator=torch.Generator(device=dev).manual_seed(seed + 2))
    dl = torch.empty_like(dgates)
    dxr = torch.empty((c.T, c.d), dtype=torch.float32, device=dev)
    dwr = torch.empty((c.E, c.d), dtype=torch.float32, device=dev)
    t = timed(lambda: Lb.moe_router_backward(x, wr, ids, dgates, c.score_fn, c.renorm, c.route_scale, d_logits=dl,
                                             dx=dxr, dw_router=dwr, sorted_to_slot=s2s, expert_offsets=offs))
    res["router_backward"] = {"workload": f"T={c.T} d={c.d} E={c.E} top_k={c.k}", "ms": t,
                              "dx bytes written": c.T * c.d * 4, "router row bytes through L1": c.T * c.k * c.d * 2}
    del x
    r = S.CONFIGS["multilayer_replay"]
    x = S.make_x(r, dev, seed)
    payload = S.make_replay_payload(r.with_(layers=1), dev, seed)[0]
    ids = torch.empty((r.T, r.k), dtype=torch.int32, device=dev)
    g = torch.empty((r.T, r.k), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    t = timed(lambda: Lb.moe_route_replay(payload, r.E, x, wr, r.score_fn, r.renorm, r.route_scale, topk_ids=ids,
                                          topk_gates=g, dev_status=st))
    res["route_replay"] = {"workload": f"T={r.T} d={r.d} E={r.E} top_k={r.k}", "ms": t,
                           "fp32 TFLOP/s": 2.0 * r.T * r.d * r.k / (t * 1e-3) / 1e12,
                           "W_r row bytes read from L2 per launch": r.T * r.k * r.d * 2}
    return {"kernels": res, "status": Lb.check_status(st)}


# ------------------------------------------------------------------ CPU oracle

class OracleSample:
    """A bounded sample of the workload for the CPU oracle: the first n tokens
    and the experts they route to.  Inputs come from the seeded generators
    (on `gen_dev`, CUDA when present since it is faster, then copied to the
    host); the sample's expert weights are quantised by the oracle here, once
    (per-weight-update work, untimed, as on the GPU)."""

    def __init__(self, cfg, n_tokens, seed, gen_dev):
        import numpy as np
        import torch
        from block_scaled_fp8_router_gb300 import synthetic as S
        from oracle import oracle as O
        O.build()
        self.cfg, self.n = cfg, n_tokens
        bits = lambda t: t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
        self.xb = bits(S.make_x(cfg, gen_dev, seed)[:n_tokens])
        self.wrb = bits(S.make_router_w(cfg, gen_dev, seed))
        self.replay = None
        if cfg.mode == "replay":
            self.replay = np.ascontiguousarray(
                S.make_replay_payload(cfg.with_(layers=1), gen_dev, seed)[0][:, :n_tokens].cpu().numpy())
        ids = self._ids(O.router_logits(self.xb, self.wrb))
        used = np.unique(ids)
        w = [[], [], [], []]
        for e in used:
            q, s = O.quant_128x128(bits(S.make_w13_expert(cfg, int(e), gen_dev, seed))); w[0].append(q); w[1].append(s)
            q, s = O.quant_128x128(bits(S.make_w2_expert(cfg, int(e), gen_dev, seed))); w[2].append(q); w[3].append(s)
        self.w = [np.stack(a) for a in w]
        self.remap = np.full(cfg.E, -1, np.int32)
        self.remap[used] = np.arange(len(used), dtype=np.int32)

    def _ids(self, logits):
        from oracle import oracle as O
        return O.topk(logits, self.cfg.k) if self.replay is None else O.replay(self.replay, self.cfg.E)[0]

    def run(self, n: int | None = None, with_y: bool = False):
        """One timed pass of the whole layer over the first n tokens of the
        sample (all of it by default); returns seconds (and y's bf16 bits)."""
        import numpy as np
        from oracle import oracle as O
        cfg = self.cfg
        n = self.n if n is None else n
        xb = np.ascontiguousarray(self.xb[:n])
        replay = None if self.replay is None else np.ascontiguousarray(self.replay[:, :n])
        t0 = time.perf_counter()
        l = O.router_logits(xb, self.wrb)
        ids = O.topk(l, cfg.k) if replay is None else O.replay(replay, cfg.E)[0]
        g = O.gates(l, ids, cfg.score_fn, cfg.renorm, cfg.route_scale)
        xq, xs = O.quant_1x128(xb)
        counts, offsets, s2s, sl2, _ = O.dispatch(ids, cfg.E)
        A = n * cfg.k
        row_e = self.remap[np.repeat(np.arange(cfg.E, dtype=np.int32), counts)]
        _, _, _, out = O.expert_ffn(O.gather_rows(xq, s2s, A, cfg.k), O.gather_rows(xs, s2s, A, cfg.k),
                                    row_e, *self.w)
        y = O.combine(out, sl2, g)
        secs = time.perf_counter() - t0
        return (secs, y) if with_y else secs

    def describe(self, secs):
        cfg = self.cfg
        return (f"{self.n} tokens of the {cfg.name} workload through the whole layer (router logits over all "
                f"{cfg.E} experts or replay, top-k, gates, 1x128 quant, dispatch, SwiGLU FFN of the "
                f"{self.n * cfg.k} expert rows, combine); expert weight quantisation untimed; {secs:.2f} s")


def error_report(y_gpu_bits, y_ref_bits):
    """The output comparison of the layer contract on a token sample: per row
    max |y - ref| / max(max |ref|, 1e-6) (the bar, 2e-2), and element-wise
    |y - ref| / max(|ref|, 1e-2 * rowmax)."""
    import numpy as np
    import torch
    to64 = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double().numpy()
    y, ref = to64(y_gpu_bits), to64(y_ref_bits)
    rowmax = np.abs(ref).max(axis=1, keepdims=True)
    row = np.abs(y - ref).max(axis=1) / np.maximum(rowmax[:, 0], 1e-6)
    elem = np.abs(y - ref) / np.maximum(np.abs(ref), 1e-2 * rowmax)
    return {"tokens": int(y.shape[0]), "row_rel_err_max": float(row.max()), "elem_rel_err_max": float(elem.max()),
            "elem_rel_err_mean": float(elem.mean()), "bar_row_rel_err": 2e-2}


def cpu_baseline(cfg, seed, n_tokens, gen_dev, y_gpu_bits=None):
    """The CPU oracle on the host cores: all cores over n_tokens, one thread
    over n_tokens / 16, and (given the GPU layer's y for the same tokens) the
    output error of the GPU against it."""
    import os as _os
    from oracle import oracle as O
    smp = OracleSample(cfg, n_tokens, seed, gen_dev)
    secs, y = smp.run(with_y=True)
    cores = O.num_threads()
    out = {"value": n_tokens / secs, "unit": "tokens/s", "cores": cores, "kind": "oracle",
           "sample": smp.describe(secs), "cpu_model": cpu_model(), "host_cpus": _os.cpu_count()}
    n1 = max(8, n_tokens // 16)
    O.set_num_threads(1)
    try:
        s1 = smp.run(n1)
    finally:
        O.set_num_threads(cores)
    out["single_thread"] = {"value": n1 / s1, "unit": "tokens/s", "cores": 1,
                            "sample": f"the first {n1} tokens of the same sample, one thread; {s1:.2f} s"}
    if y_gpu_bits is not None:
        out["gpu_vs_oracle"] = error_report(y_gpu_bits[:n_tokens], y)
    out["configs"] = cpu_config_legs(seed, gen_dev)
    return out


def cpu_config_legs(seed, gen_dev):
    """The oracle on the other workloads (all host cores, bounded samples):
    the tiny and replay layers through the whole layer, and the long-context
    dispatch + combine of bf16 rows with identity experts."""
    import numpy as np
    import torch
    from block_scaled_fp8_router_gb300 import synthetic as S
    from oracle import oracle as O
    legs = {}
    for name, n in (("tiny", 256), ("replay", 512)):
        c = S.CONFIGS[name]
        secs = OracleSample(c, n, seed, gen_dev).run()
        legs[name] = {"value": n / secs, "unit": "tokens/s", "sample": f"{n} of {c.T} tokens, whole layer, "
                                                                       f"{secs:.2f} s"}
    c = S.CONFIGS["long_dispatch"]
    n = 8192
    bits = lambda t: t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    xb = bits(S.make_x(c, gen_dev, seed, T=n))
    ids = np.ascontiguousarray(S.make_replay_payload(c.with_(layers=1), gen_dev, seed)[0][:, :n].t().cpu().numpy())
    g = np.ascontiguousarray(S.make_dirichlet_gates(c, gen_dev, seed)[:n].cpu().numpy())
    t0 = time.perf_counter()
    _, _, s2s, sl2, _ = O.dispatch(ids, c.E)
    rows = O.gather_rows(xb, s2s, n * c.k, c.k)
    O.combine(rows, sl2, g)
    secs = time.perf_counter() - t0
    nbytes = 2 * n * c.d * (2 + 2 * c.k)
    legs["long_dispatch"] = {"value": n / secs, "unit": "tokens/s", "GB/s": nbytes / secs / 1e9,
                             "sample": f"{n} of {c.T} tokens, dispatch + row gather + combine of bf16 rows "
                                       f"(identity experts), {secs:.2f} s"}
    return legs


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="large")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=1024, help="token sample of the CPU baseline")
    ap.add_argument("--ref-tokens", type=int, default=32, help="token sample per step of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dispatch-combine", action="store_true")
    ap.add_argument("--no-replay", action="store_true", help="skip the replay-workload line")
    ap.add_argument("--no-mx", action="store_true",
                    help="skip the power-of-two-scale (block-scaled MMA) line and the NVFP4 quantiser timing")
    ap.add_argument("--no-backward", action="store_true", help="skip the expert-path backward line")
    ap.add_argument("--no-multilayer", action="store_true",
                    help="skip the 8-layer replay sweep (all layers' FP8 weights resident)")
    ap.add_argument("--router-kernels", action="store_true",
                    help="time only the router kernels (route_topk, route_replay) and print their line")
    ap.add_argument("--hbm-kernels", action="store_true",
                    help="time only the HBM-bound kernels on a profiling shape (T=16384) and print their line")
    ap.add_argument("--scales", default="fp32", choices=["fp32", "ue8m0"],
                    help="block scales of the timed layer: fp32 (the recipe) or power-of-two (block-scaled MMA)")
    ap.add_argument("--form", default="sorted", choices=["sorted", "gathered"],
                    help="sorted: dispatch copies rows into expert order; gathered: the FFN gathers its rows "
                         "(tile::gather4) and stores outputs in slot order")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    from block_scaled_fp8_router_gb300 import synthetic as S
    cfg = S.CONFIGS[args.workload]
    config = {"workload": f"{cfg.name}: T={cfg.T} d={cfg.d} E={cfg.E} top_k={cfg.k} F={cfg.F} "
                          f"{'sigmoid' if cfg.score_fn else 'softmax'} {cfg.mode}",
              "tokens_per_gpu": cfg.T, "parallelism": f"token-sharded x{world}" if world > 1 else "single GPU",
              "l2": "flushed: a 512 MB device write before every timed step, outside the step's events "
                    f"(the FP8 expert weights, {fp8_weight_bytes(cfg) / 1e9:.3g} GB, are streamed from HBM "
                    "every step as well)",
              "form": args.form, "scales": args.scales}
    metric = "MoE-layer tokens/s (7168d/256e/top-8 FP8)" if cfg.name == "large" else f"MoE-layer tokens/s ({cfg.name})"

    if args.router_kernels:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        print(json.dumps(run_router_kernels(torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))), args.seed,
                                            args.steps, args.warmup)))
        return

    if args.hbm_kernels:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        print(json.dumps(run_hbm_kernels(torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))), args.seed,
                                         args.steps, args.warmup, _peaks())))
        return

    if args.impl == "reference":
        if rank != 0:
            return
        import torch
        from oracle import oracle as O
        gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
        smp = OracleSample(cfg, args.ref_tokens, args.seed, gen_dev)
        times = [smp.run() for _ in range(args.warmup + args.steps)][args.warmup:]
        total = sum(times)
        value = args.ref_tokens * args.steps / total
        print(json.dumps({"impl": "reference", "metric": metric, "value": value, "unit": "tokens/s",
                          "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
                          "vs_baseline": None, "dtype": "f64 block sums, f32 fma chains (CPU oracle)",
                          "data": "synthetic", "config": config,
                          "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": O.num_threads(),
                                           "kind": "oracle", "sample": smp.describe(total / args.steps),
                                           "cpu_model": cpu_model()},
                          "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    import __graft_entry__
    __graft_entry__.build()
    peaks = _peaks()
    peaks["fp8_tflops_measured"] = fp8_peak_tflops(torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))))
    main_mx = args.scales == "ue8m0"
    r = run_gpu(args, rank, world, ue8m0=main_mx)
    cfg = r["cfg"]
    y_first = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        y_first = r["layer"].y[:args.cpu_tokens].contiguous().cpu().view(torch.int16).numpy().view("uint16")
    value = job_throughput(cfg.T, args.steps, world, r["total_ms"])
    e2e = job_throughput(cfg.T, args.steps, world, r["e2e_ms"])
    gathered = args.form == "gathered" and not main_mx
    ffn, extra = rooflines(cfg, r["avg"], peaks, gathered, main_mx)
    if main_mx:
        ffn["kernel"] = "moe_grouped_ffn_mx (block-scaled MMA, GEMM1+SwiGLU+requant, GEMM2)"
        ffn["traffic"] = None
    launches = sum(KERNELS_PER_STEP[n] for n in ("quant", "dispatch", "ffn", "combine")) + 1 - int(gathered)
    out = {"metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": r["total_ms"] / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e4m3 -> fp32 (GEMMs); fp32 router; bf16 io",
           "data": "synthetic (seeded N(0,1) tokens, N(0,0.006) weights, N(0,0.02) router)", "config": config,
           "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": r["h2d"],
                   "d2h_bytes_per_step": r["d2h"]},
           "roofline": ffn, "extra": extra, "gpu_launches": launches * args.steps, "clocks": r["clocks"],
           "dev_status": r["status"], "peaks_source": peaks["source"],
           "gemm_padded_rows": {"tile_rows": 128, "fraction": r["padded"],
                                "note": "rows the grouped GEMMs compute (each expert rounded up to 128-row "
                                        "tiles) over the routed rows"},
           "timing": {"ms_sum_of_steps": r["total_ms"], "ms_bracket_with_flushes": r["bracket_ms"]}}
    if cfg.name == "large" and not args.no_replay:
        import torch
        del r
        torch.cuda.empty_cache()
        rr = run_gpu(args, rank, world, workload="multilayer_replay", with_e2e=False, steps=max(3, args.steps // 2))
        rcfg = rr["cfg"]
        rffn, rextra = rooflines(rcfg, rr["avg"], peaks, gathered)
        out["replay_layer"] = {
            "workload": f"multilayer_replay (one layer): T={rcfg.T} d={rcfg.d} E={rcfg.E} top_k={rcfg.k} "
                        f"F={rcfg.F}, replayed payload with 8 hot and 8 empty experts, sigmoid gates",
            "tokens/s": job_throughput(rcfg.T, rr["steps"], world, rr["total_ms"]),
            "ms_per_step": rr["total_ms"] / rr["steps"], "ffn_TFLOP/s": rffn["achieved"],
            "ffn_frac": rffn["frac"], "ffn_frac_of_fp8_measured": rffn.get("frac_of_fp8_measured"),
            "gemm_padded_rows": rr["padded"], "steps": rextra, "dev_status": rr["status"]}
        del rr
        torch.cuda.empty_cache()
    if cfg.name == "large" and not args.no_multilayer and not main_mx:
        import torch
        torch.cuda.empty_cache()
        out["multilayer_sweep"] = run_multilayer(torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))),
                                                 rank_seed(args.seed, rank), max(3, args.steps // 4), 3, peaks)
    if cfg.name in ("large", "large_e16") and not args.no_backward and not main_mx:
        import torch
        torch.cuda.empty_cache()
        out["backward_layer"] = run_backward(cfg, torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))),
                                             rank_seed(args.seed, rank), max(3, args.steps // 2), 3, peaks)
    if cfg.name == "large" and not args.no_mx and not main_mx:
        import torch
        torch.cuda.empty_cache()
        rm = run_gpu(args, rank, world, workload=cfg.name, with_e2e=False, steps=max(3, args.steps // 2), ue8m0=True)
        mffn, mextra = rooflines(cfg, rm["avg"], peaks, ue8m0=True)
        mffn["kernel"] = "moe_grouped_ffn_mx (block-scaled MMA, GEMM1+SwiGLU+requant, GEMM2)"
        mffn["traffic"] = None
        out["mx_layer"] = {
            "workload": config["workload"] + ", power-of-two (UE8M0) block scales on the block-scaled MMA",
            "tokens/s": job_throughput(cfg.T, rm["steps"], world, rm["total_ms"]),
            "ms_per_step": rm["total_ms"] / rm["steps"], "ffn": mffn, "steps": mextra, "dev_status": rm["status"]}
        del rm
        torch.cuda.empty_cache()
    if cfg.name == "large" and not args.no_dispatch_combine:
        import torch
        torch.cuda.empty_cache()
        out["dispatch_combine"] = run_dispatch_combine(torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))),
                                                       args.seed + rank, max(3, args.steps // 2), 3, peaks)
    if cfg.name == "large" and not args.no_dispatch_combine:
        out["payload"] = run_payload(torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))),
                                     args.seed + rank, max(3, args.steps // 2), 3, peaks)
    if cfg.name in ("large", "large_e64") and not args.no_mx:
        import torch
        torch.cuda.empty_cache()
        out["nvfp4_layer"] = run_nvfp4_layer(cfg, torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))),
                                             rank_seed(args.seed, rank), max(3, args.steps // 2), 3, peaks)
        try:
            out["nvfp4_quant"] = run_nvfp4_quant(cfg, torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))),
                                                 args.seed + rank, max(3, args.steps // 2), 3, peaks)
        except Exception as exc:   # an extra measurement: report, do not lose the line
            out["nvfp4_quant"] = {"error": f"{type(exc).__name__}: {exc}"[:300]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg, args.seed, args.cpu_tokens, "cuda", y_first)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
