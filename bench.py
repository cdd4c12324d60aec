"""Benchmark of the latent-MoE layer tail on GB300.

One step = one klt_forward (routing, permutation, routed FP8/NVFP4 experts, combine,
RMSNorm, up-projection + BF16 shared expert) over one batch of synthetic tokens.  Prints
one JSON line.  By default every workload is measured in the same run (tiny M=4, decode
M=16, decode M=128, prefill M=4096, prefill M=8192 NVFP4, plus decode M=16 from the hidden
state alone, prefill M=4096 with MXFP8 routed weights and prefill M=8192 with NVFP4 weights
and activations); the line's top-level figures
are the decode batch of 16 tokens (E=64, top-8, routed intermediate 1024 with FP8 128x128
block scales, shared intermediate 2048, H=7168, L=3584) and `workloads` holds every
workload's record (roofline, end to end, clocks, the oracle on the host cores).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload all|NAME]

Multi-GPU (under torchrun): the tail has no exchange step, so every rank runs an
independent replica on its own tokens (weak scaling); time = max over ranks.
`--impl reference` times the CPU float64 oracle (the only other implementation) on the
headline workload (the whole decode batch per step).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-tail tokens/sec & µs/layer at M=16..8192; % of HBM or tensor roofline"
HBM_NOMINAL_GBS = 8000.0


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def max_over_ranks(value: float, ws: int, device: str = "cuda") -> float:
    """The largest of every rank's value: a replicated job runs as long as its slowest
    replica."""
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ws: int, m: int, steps: int, ms_total: float) -> float:
    """Tokens per second of the whole job: every replica processes m tokens a step."""
    return ws * m * steps / (ms_total / 1e3)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the dominant
# kernel (block-scaled layers: both GEMM launches), from one ncu launch-list capture of
# `bench.py --workload W --steps 2 --warmup 3 --no-cpu-baseline` (the steady-state forward),
# valid only while the kernel sources hash to the recorded digest.
NCU_TRAFFIC = {
    ("decode_m16_e64_k8_fp8", "gemm_fused"): (715542784, "630ce809b733f263"),
    ("tiny_m4_e16_k4", "gemm_fused"): (191047680, "630ce809b733f263"),
    ("decode_m128_e64_k8_fp8_biased", "gemm_fused"): (839586816, "630ce809b733f263"),
    ("prefill_m4096_e64_k8_fp8_zipf", "gemm_fused"): (1678991104, "630ce809b733f263"),
    ("prefill_m8192_e128_k8_nvfp4", "gemm_fused"): (6972542464, "630ce809b733f263"),
    ("prefill_m4096_e64_k8_mxfp8_zipf", "gemm_routed+gemm_dense"): (1722151424,
                                                                     "630ce809b733f263"),
    ("prefill_m8192_e128_k8_nvfp4_w4a4", "gemm_routed+gemm_dense"): (3541166848,
                                                                      "630ce809b733f263"),
    ("decode_m16_e64_k8_fp8+hidden", "gemm_fused"): (781824000, "630ce809b733f263"),
}
KERNEL_SOURCES = ("klt_gemm.cu", "klt_wide.cu", "klt_device.cuh", "klt_internal.h", "klt_api.cu",
                  "klt_route.cu")


def kernel_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "latent_moe_layer_route_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    rec = NCU_TRAFFIC.get((workload, kernel))
    if rec is None or rec[1] != kernel_digest():
        return None
    return rec[0]


def algorithmic_bytes(cfg, cnt: np.ndarray, M: int):
    """Bytes each launch must move at least once (weights of touched experts, token
    inputs, stage outputs), per the tail's data flow."""
    H, L, I, Is, k, E = cfg.H, cfg.L, cfg.I, cfg.Is, cfg.topk, cfg.E
    touched = int((cnt > 0).sum())
    Mk = M * k
    # routed weight bytes per element: codes plus scales
    wb = {"fp8": 1.0, "mxfp8": 1.0 + 1.0 / 32, "nvfp4": 0.5 + 1.0 / 16,
          "nvfp4_w4a4": 0.5 + 1.0 / 16}[cfg.routed_fmt]
    # quantised routed activation bytes per element (latent input, SwiGLU output)
    qb = {"mxfp8": 1.0 + 1.0 / 32, "nvfp4_w4a4": 0.5 + 1.0 / 16}.get(cfg.routed_fmt, 1.0)
    w13 = touched * 2 * I * L * wb
    w2 = touched * L * I * wb
    g1 = 2 * Is * H * 2 + M * H * 2 + w13 + Mk * L * qb + Mk * I * qb + M * Is * 2
    g2 = w2 + Mk * I * qb + M * L * 4
    norm = M * L * 4 + M * L * 2
    g3 = H * L * 2 + H * Is * 2 + M * L * 2 + M * Is * 2 + M * H * 2
    route = M * E * 4 + M * L * 2 + M * L * qb + M * L * 4
    perm = Mk * L * qb * 2
    total = g1 + g2 + norm + g3 + route + perm
    return {"gemm_l1": g1, "gemm_l2": g2, "norm": norm, "gemm_out": g3, "route": route,
            "perm": perm, "total": total, "touched_experts": touched}


def launch_names(cfg, nt: int, phased: bool, hidden: bool):
    """Names of a forward's launches, in order, from the tail's launch count `nt`: the
    routing launches (one fused launch for a small batch; else routing, the expert
    histogram above one permutation block, scatter, gather), then the GEMM launches."""
    bs = cfg.routed_fmt in ("mxfp8", "nvfp4_w4a4")  # routed and dense GEMM launches
    gemms = (["gemm_l1", "gemm_l2", "norm", "gemm_out"] if phased else
             ["gemm_routed", "gemm_dense"] if bs else ["gemm_fused"])
    routing = {1: ["route_perm"], 3: ["route", "perm_scatter", "perm_gather"],
               4: ["route", "perm_hist", "perm_scatter", "perm_gather"]}[nt - len(gemms)]
    return (["proj"] if hidden else []) + routing + gemms


def flops(cfg, M: int):
    H, L, I, Is, k = cfg.H, cfg.L, cfg.I, cfg.Is, cfg.topk
    routed = 2.0 * M * k * (2 * I * L + L * I)
    dense = 2.0 * M * (2 * Is * H + H * Is + H * L)
    return routed, dense


HEADLINE = "decode_m16_e64_k8_fp8"


def dtype_of(cfg) -> str:
    if cfg.routed_fmt == "fp8":
        return "fp8e4m3+bf16 (fp32 accumulate)"
    if cfg.routed_fmt == "mxfp8":
        return "mxfp8 (e4m3, power-of-two scales per 32, block-scaled MMA) + bf16 (fp32 accumulate)"
    if cfg.routed_fmt == "nvfp4_w4a4":
        return ("nvfp4 weights and activations (e2m1, e4m3 scales per 16, block-scaled FP4 "
                "MMA) + bf16 (fp32 accumulate)")
    return "nvfp4 weights (bf16-exact MMA) + fp8e4m3 activations + bf16 (fp32 accumulate)"


def run_reference(cfg, args, ws, rank):
    """The CPU float64 oracle as it stands, on a bounded token sample per step (the whole
    batch for decode workloads)."""
    if rank != 0:
        return
    from latent_moe_layer_route_gb300 import inputs
    from oracle import model as oracle_model
    act, w = inputs.make_inputs(cfg)
    sample = min(cfg.M, 16)  # a decode batch whole; prefill batches: 16 tokens per step
    tok = np.arange(sample)
    for _ in range(args.warmup):
        oracle_model.tail(act, w, cfg, tokens=tok)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_model.tail(act, w, cfg, tokens=tok)
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    value = sample * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "M": cfg.M, "sample_tokens": sample,
                   "same_config": sample == cfg.M},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {sample} of {cfg.M} tokens per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(cfg, act, w):
    """The oracle as it stands on the first (at most 16) tokens of the workload, repeated
    for about 10 s; the routing and permutation still cover the whole batch."""
    from oracle import model as oracle_model
    cores = len(os.sched_getaffinity(0))
    sample = min(cfg.M, 16)
    tok = np.arange(sample)
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle_model.tail(act, w, cfg, tokens=tok)
        n += 1
        if time.perf_counter() - t0 > 10.0 or n >= 5:
            break
    dt = time.perf_counter() - t0
    return {"value": sample * n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} step(s) of the first {sample} of {cfg.M} tokens, {dt:.1f} s"}


def measure(cfg, args, ws, rank, local, flush, with_cpu: bool, hidden: bool = False):
    """Every figure of one workload: device-timed steps, graph replay, per-launch times,
    end to end with host buffers, roofline of the dominant launch, oracle on the host.
    `hidden`: the step runs from the hidden state alone (klt_forward_hidden: the latent
    input and router logits are computed by the library first)."""
    import torch
    from latent_moe_layer_route_gb300 import binding as B
    from latent_moe_layer_route_gb300 import inputs

    M = cfg.M
    act_cpu, w_cpu = inputs.make_inputs(cfg)
    if hidden:
        w_cpu.update(inputs.make_projection_weights(cfg))
    w = {k: v.cuda() for k, v in w_cpu.items()}
    act = {k: v.cuda() for k, v in act_cpu.items()}
    flags = (B.KLT_FLAG_PHASED if args.phased else 0) | \
        (B.KLT_FLAG_DETERMINISTIC if args.deterministic else 0)
    tail = B.LatentMoETail(cfg, w, flags=flags)
    del w
    out = torch.empty((M, cfg.H), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    cnt = torch.zeros(cfg.E, dtype=torch.int32, device="cuda")
    ro = B.KltRouting(None, None, cnt.data_ptr(), None, None, None, None)
    if hidden:
        tail.forward_hidden(act["x"], out=out, routing=ro)
    else:
        tail.forward(act["x"], act["z"], act["logits"], out=out, routing=ro)
    torch.cuda.synchronize()
    assert tail.status() == B.KLT_OK
    nl = tail.launch_count(M) + (1 if hidden else 0)

    base_dbg = None
    if args.tile_n:
        base_dbg = B.KltDebug()
        base_dbg.force_bn = args.tile_n

    def step():
        if hidden:
            tail.forward_hidden(act["x"], out=out, debug=base_dbg)
        else:
            tail.forward(act["x"], act["z"], act["logits"], out=out, debug=base_dbg)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()

    # ---- timed region: device time of each step, L2 flushed between steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]

    def load_for(seconds):  # the same steps, untimed, so clock samples see the timed load
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            for _ in range(10):
                flush.zero_()
                step()
            torch.cuda.synchronize()

    with Clocks(local) as clk:
        load_for(0.5)
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        load_for(0.5)
    if ws > 1:
        dist.barrier()
    ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)), ws)
    ms_step = ms / args.steps
    value = job_throughput(ws, M, args.steps, ms)
    assert tail.status() == B.KLT_OK

    # ---- the same step captured once in a CUDA graph (kernels chained by programmatic
    # dependent launch edges) and replayed, L2 flushed before each replay
    try:
        graph_obj = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        with torch.cuda.graph(graph_obj):
            step()
        torch.cuda.synchronize()
        gs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ge = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            gs[i].record(stream)
            graph_obj.replay()
            ge[i].record(stream)
        torch.cuda.synchronize()
        assert tail.status() == B.KLT_OK
        gms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(gs, ge)), ws)
        graph = {"value": job_throughput(ws, M, args.steps, gms), "unit": "tokens/s",
                 "ms_per_step": gms / args.steps,
                 "how": "one klt_forward captured in a CUDA graph, replayed per step"}
        del graph_obj
    except Exception as exc:  # report, do not fail the line
        graph = {"unavailable": f"{type(exc).__name__}: {str(exc)[:160]}"}

    # ---- per-launch breakdown (events between launches; separate loop)
    nev = nl + 1
    assert nl <= 8
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    for row in evs:  # torch creates the CUDA event on first record
        for ev in row:
            ev.record(stream)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        dbg = B.KltDebug()
        dbg.force_bn = args.tile_n
        evs[i][0].record(stream)
        for j in range(nl):
            dbg.events[j] = evs[i][j + 1].cuda_event
        if hidden:
            tail.forward_hidden(act["x"], out=out, debug=dbg)
        else:
            tail.forward(act["x"], act["z"], act["logits"], out=out, debug=dbg)
    torch.cuda.synchronize()
    per = np.zeros(nl)
    for i in range(args.steps):
        for j in range(nl):
            per[j] += evs[i][j].elapsed_time(evs[i][j + 1])
    per /= args.steps
    names = launch_names(cfg, nl - (1 if hidden else 0), args.phased, hidden)
    per_launch_us = {n: round(float(v) * 1e3, 2) for n, v in zip(names, per)}

    # ---- end to end through the public API with host buffers
    xh = act_cpu["x"].pin_memory()
    zh = act_cpu["z"].pin_memory()
    lh = act_cpu["logits"].pin_memory()
    oh = torch.empty((M, cfg.H), dtype=torch.bfloat16).pin_memory()
    xd, zd, ld = torch.empty_like(act["x"]), torch.empty_like(act["z"]), torch.empty_like(
        act["logits"])
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        e0[i].record(stream)
        xd.copy_(xh, non_blocking=True)
        if hidden:
            tail.forward_hidden(xd, out=out, debug=base_dbg)
        else:
            zd.copy_(zh, non_blocking=True)
            ld.copy_(lh, non_blocking=True)
            tail.forward(xd, zd, ld, out=out, debug=base_dbg)
        oh.copy_(out, non_blocking=True)
        e1[i].record(stream)
    torch.cuda.synchronize()
    ems = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(e0, e1)), ws)
    e2e = job_throughput(ws, M, args.steps, ems)
    h2d = xh.numel() * 2 + (0 if hidden else zh.numel() * 2 + lh.numel() * 4)
    d2h = oh.numel() * 2

    # ---- roofline of the dominant launch
    cnt_h = cnt.cpu().numpy()
    ab = algorithmic_bytes(cfg, cnt_h, M)
    hbm, bf16_tf, peak_src = _peaks()
    if "gemm_routed" in per_launch_us:  # block-scaled layers: both GEMM launches together
        dom = "gemm_routed+gemm_dense"
        per_launch_us[dom] = round(per_launch_us["gemm_routed"] + per_launch_us["gemm_dense"], 2)
        dom_bytes = ab["gemm_l1"] + ab["gemm_l2"] + ab["norm"] + ab["gemm_out"]
    elif "gemm_fused" in per_launch_us:
        dom = "gemm_fused"
        dom_bytes = ab["gemm_l1"] + ab["gemm_l2"] + ab["norm"] + ab["gemm_out"]
    else:
        dom = max(("gemm_l1", "gemm_l2", "gemm_out"), key=lambda n: per_launch_us[n])
        dom_bytes = ab[dom]
    routed_f, dense_f = flops(cfg, M)
    if hidden:  # the projection: its weights, x again, z and logits written
        ab["total"] += (cfg.L + cfg.E) * cfg.H * 2 + M * cfg.H * 2 + M * (cfg.L * 2 + cfg.E * 4)
        dense_f += 2.0 * M * cfg.H * (cfg.L + cfg.E)
    # fp8 routed contractions run at twice the bf16 rate and fp4 x fp4 ones at six times
    # (the nominal dense ratios 4.5 : 2.25 and 13.5 : 2.25 PFLOP/s applied to the measured
    # bf16 peak); the fused launch's mixed peak follows from the flop mix
    rr = 6.0 if cfg.routed_fmt == "nvfp4_w4a4" else 2.0
    t_tensor = routed_f / (rr * bf16_tf * 1e12) + dense_f / (bf16_tf * 1e12)
    dom_s = per_launch_us[dom] * 1e-6
    traffic = recorded_traffic(cfg.name + ("+hidden" if hidden else ""), dom)
    if t_tensor > dom_bytes / (hbm * 1e9):
        mixed_peak = (routed_f + dense_f) / t_tensor / 1e12
        achieved = (routed_f + dense_f) / dom_s / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1),
                "peak": round(mixed_peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / mixed_peak, 4),
                "peak_source": f"{peak_src} bf16 burst, routed share at {rr:g}x",
                "traffic": traffic, "algorithmic_flops": routed_f + dense_f,
                "algorithmic_bytes": int(dom_bytes)}
    else:
        achieved = dom_bytes / dom_s / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "peak_source": f"{peak_src} copy bandwidth", "traffic": traffic,
                "algorithmic_bytes": int(dom_bytes)}
    roof_time_us = max(ab["total"] / (HBM_NOMINAL_GBS * 1e9), t_tensor) * 1e6

    rec = {
        "value": value, "unit": "tokens/s", "ms_per_step": ms_step,
        "us_per_layer": ms_step * 1e3, "dtype": dtype_of(cfg),
        "config": {"workload": cfg.name + ("+hidden" if hidden else ""), "M": M, "H": cfg.H,
                   "L": cfg.L, "E": cfg.E,
                   "inputs": "hidden state x only (latent input and router logits computed "
                             "by the library)" if hidden else "x, z, logits",
                   "topk": cfg.topk, "I": cfg.I, "Is": cfg.Is, "routed_fmt": cfg.routed_fmt,
                   "router": cfg.router, "gemm_engine": tail.gemm_tile(M, args.tile_n),
                   "l2": "flushed (512 MB write) before every timed step",
                   "schedule": "phased" if args.phased else "fused",
                   "combine": "fixed order" if args.deterministic else "arrival order",
                   "parallelism": f"replicas x{ws}"},
        "roofline": roof,
        "step_roofline": {"algorithmic_bytes": int(ab["total"]),
                          "touched_experts": ab["touched_experts"],
                          "roofline_us_at_8TBps": round(roof_time_us, 2),
                          "frac_of_roofline": round(roof_time_us / (ms_step * 1e3), 4),
                          "achieved_GBps": round(ab["total"] / (ms_step * 1e-3) / 1e9, 1)},
        "per_launch_us": per_launch_us,
        "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": nl * args.steps,
        "graph": graph,
        "clocks": {**clk.summary(),
                   "window": "nvidia-smi every 200 ms, timed steps bracketed by 0.5 s of the "
                             "same steps on each side"},
    }
    tail.close()
    del act, out, xd, zd, ld
    torch.cuda.empty_cache()
    if with_cpu:
        rec["cpu_baseline"] = cpu_baseline(cfg, act_cpu, w_cpu)
    return rec


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all",
                    help="one workload name, or 'all' (default): every workload measured in "
                         "this run, decode M=16 as the headline of the printed line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--phased", action="store_true",
                    help="one launch per GEMM stage instead of the fused persistent launch")
    ap.add_argument("--deterministic", action="store_true",
                    help="fixed-order combine of the routed experts (KLT_FLAG_DETERMINISTIC)")
    ap.add_argument("--tile-n", type=int, default=0,
                    help="GEMM engine / token-tile width: 16..128 feature-major, 256 "
                         "token-major (0 = library choice)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from latent_moe_layer_route_gb300 import configs
    # a workload name with "+hidden" runs that workload from the hidden state alone
    if args.workload == "all":  # the five workloads, the step before the tail, the MX and
        # FP4 x FP4 variants
        names = [c.name for c in configs.ALL] + [HEADLINE + "+hidden",
                                                 configs.PREFILL_M4096_MX.name,
                                                 configs.PREFILL_M8192_W4A4.name]
    else:  # one name, or several separated by commas (the first is the headline)
        names = args.workload.split(",")
    cfgs = [(configs.BY_NAME[n.split("+")[0]], n.endswith("+hidden")) for n in names]
    head = configs.BY_NAME[HEADLINE] if args.workload == "all" else cfgs[0][0]
    ws, rank, local = _dist()

    if args.impl == "reference":
        run_reference(head, args, ws, rank)
        return

    import torch
    import torch.distributed as dist
    from latent_moe_layer_route_gb300 import binding as B
    from latent_moe_layer_route_gb300 import build

    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl")
    build.build()
    B.load_library()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    with_cpu = rank == 0 and ws == 1 and not args.no_cpu_baseline
    recs = {}
    for cfg, hid in cfgs:
        recs[cfg.name + ("+hidden" if hid else "")] = measure(cfg, args, ws, rank, local,
                                                              flush, with_cpu and not hid, hid)
    h = recs[head.name] if head.name in recs else next(iter(recs.values()))
    line = {
        "metric": METRIC, "value": h["value"], "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": h["ms_per_step"],
        "us_per_layer": h["us_per_layer"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": h["dtype"],
        "data": "synthetic (seeded numpy draws, random-init weights)",
    }
    line.update({k: v for k, v in h.items() if k not in line})
    if len(recs) > 1:
        line["workloads"] = {
            n: {k: v for k, v in r.items() if k not in ("graph",)} for n, r in recs.items()}
        line["gpu_launches_all_workloads"] = sum(r["gpu_launches"] for r in recs.values())
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
