#!/usr/bin/env python
"""Benchmark: the Qwen2-7B-shaped decode linear set at M=1, W4A8.

One step = one pass of the whole hot path over one decode token: for the
eight linears (q, k, v, o, gate, up, down, lm_head) the fused kernel
quantizes the fp16 activation to INT8, streams the packed INT4 weights,
accumulates in int32 and rescales to fp32.  Projections that read the same
activation in the model share one grouped launch (q/k/v; gate/up), so a step
is five launches.  Weights (389.8 MB per set) are resident in HBM; two copies
alternate between steps, so nothing is reused from the 129 MB L2.  The step is
replayed as a CUDA graph of programmatically dependent launches.

Reported (one JSON line, rank 0):
  value     effective weight GB/s (packed INT4 + fp32 scales per set / time)
  e2e       the same with the activations copied in from pinned host memory
            and the outputs read back, every step, inside the timed region
  roofline  the dominant kernel (lm_head, 273 MB) against measured HBM peak
  cpu_baseline  the CPU oracle timed on the host on a sample of the set

`--impl reference` times the CPU oracle alone (the reference arm).
Under torchrun with N > 1 every rank runs an independent replica (weak
scaling); the path has no data exchange.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/decode-step linear set & effective weight GB/s (% of GB300 HBM peak), M=1 W4A8"
# (name, K in-features, N out-features)
LINEARS = [("q", 3584, 3584), ("k", 3584, 512), ("v", 3584, 512), ("o", 3584, 3584),
           ("gate", 3584, 18944), ("up", 3584, 18944), ("down", 18944, 3584),
           ("lm_head", 3584, 152064)]
# Launches of one decode step: projections that read the same activation share
# one grouped launch (q/k/v; gate/up), as they do in the model.
LAUNCHES = [("qkv", ("q", "k", "v")), ("o", ("o",)), ("gate_up", ("gate", "up")),
            ("down", ("down",)), ("lm_head", ("lm_head",))]
WEIGHT_SEED0 = 1000
ACT_SEED_OFFSET = 500
OUTLIER_FRAC = 0.001
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = ("Qwen2-7B-shaped decode linear set, M=1, W4A8: q 3584->3584, k 3584->512, "
            "v 3584->512, o 3584->3584, gate 3584->18944, up 3584->18944, down 18944->3584, "
            "lm_head 3584->152064; weights N(0,0.02), x N(0,1) fp16 with 0.1% outliers x20")
CPU_SAMPLE_STRIDE = 8


def activation_seed(name: str) -> int:
    """Seed of the activation read by linear `name` (shared inside a launch)."""
    names = [l[0] for l in LINEARS]
    first = next(members[0] for _, members in LAUNCHES if name in members)
    return WEIGHT_SEED0 + names.index(first) + ACT_SEED_OFFSET


def weight_bytes(K: int, N: int) -> int:
    """Algorithmic bytes of one W4A8 linear: packed INT4 weights + fp32 scales."""
    return N * K // 2 + 4 * N


SET_BYTES = sum(weight_bytes(K, N) for _, K, N in LINEARS)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-busy-s", type=float, default=0.6,
                    help="keep the GPU busy at least this long before timing (clock samples)")
    ap.add_argument("--only", choices=[l[0] for l in LAUNCHES], default=None,
                    help="profiling aid: time one launch kind alone, eagerly, without PDL "
                         "(not the headline metric)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------

def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, uuid: str):
        self.uuid = uuid
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + CLOCK_FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9 or (self.uuid and self.uuid not in f[0]):
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        os.unlink(self.file.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


def gpu_uuid() -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return ""


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_weight_quantized_w4a8_gb300", "csrc")
    for name in ("gemv.cu", "plan.h", "ptx.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic():
    """dram bytes per lm_head launch from the committed ncu summary, or None
    when the kernel sources changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("source_sha256") != kernel_source_hash():
        return None
    return t.get("dram_bytes_per_launch")


def cpu_sample_inputs(dev):
    """Every CPU_SAMPLE_STRIDE-th output row of each linear, quantized by the
    oracle on the host (weights drawn by the generator's GPU twin: same bits)."""
    import oracle
    import synth
    orc = oracle.load()
    out = []
    for idx, (name, K, N) in enumerate(LINEARS):
        seed = WEIGHT_SEED0 + idx
        W = synth.normal_gpu(seed, (N, K), 0.02, device=dev)
        W_rows = W[::CPU_SAMPLE_STRIDE].cpu().numpy()
        del W
        Wq, sw = orc.w4_quantize(W_rows)
        X = synth.activation(activation_seed(name), 1, K, outlier_frac=OUTLIER_FRAC)
        out.append((X, Wq, sw, N))
    return orc, out


def time_oracle_sample(orc, inputs, min_s=2.0, max_reps=50):
    """Seconds the oracle takes for one full set, extrapolated from the row sample."""
    reps, t_total = 0, 0.0
    while reps < max_reps and (t_total < min_s or reps < 2):
        t0 = time.perf_counter()
        for (X, Wq, sw, _) in inputs:
            orc.w4a8_linear(X, Wq, sw)
        t_total += time.perf_counter() - t0
        reps += 1
    rows_sampled = sum(Wq.shape[0] for (_, Wq, _, _) in inputs)
    rows_total = sum(N for (_, _, _, N) in inputs)
    return t_total / reps * rows_total / rows_sampled, reps


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle alone
# ---------------------------------------------------------------------------

def run_reference(args, world, rank):
    import torch
    if rank != 0:
        return
    dev = torch.device("cuda") if torch.cuda.is_available() else None
    import oracle
    import synth
    orc = oracle.load()
    if dev is not None:
        orc, inputs = cpu_sample_inputs(dev)
        sample = "every %dth output row of each linear (%.1f%% of the set's weights)" % (
            CPU_SAMPLE_STRIDE, 100.0 / CPU_SAMPLE_STRIDE)
    else:
        raise SystemExit(json.dumps({"impl": "reference", "unavailable": "no CUDA device for input generation"}))
    for _ in range(args.warmup):
        for (X, Wq, sw, _) in inputs:
            orc.w4a8_linear(X, Wq, sw)
    rows_sampled = sum(Wq.shape[0] for (_, Wq, _, _) in inputs)
    rows_total = sum(N for (_, _, _, N) in inputs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for (X, Wq, sw, _) in inputs:
            orc.w4a8_linear(X, Wq, sw)
    dt = (time.perf_counter() - t0) / args.steps * rows_total / rows_sampled
    value = SET_BYTES / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4xint8->int32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1, "set_weight_bytes": SET_BYTES},
        "cpu_baseline": {"kind": "oracle", "value": round(value, 4), "unit": "GB/s", "cores": 1,
                         "sample": sample + "; per step, scaled to the full set"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, world, rank):
    import torch
    import synth
    import bit_weight_quantized_w4a8_gb300 as w4

    w4.build()
    w4.w4a8_set_tuning(reset=True)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream(dev)
    PDL = w4.LAUNCH_PDL

    # --- inputs: one activation per launch, outputs in one buffer -----------
    names = [l[0] for l in LINEARS]
    lin = {name: (i, K, N) for i, (name, K, N) in enumerate(LINEARS)}
    act_K = [lin[members[0]][1] for _, members in LAUNCHES]
    k_off = np.cumsum([0] + act_K)
    n_off = np.cumsum([0] + [N for _, _, N in LINEARS])
    X_host = np.concatenate([
        synth.activation(activation_seed(members[0]), 1, lin[members[0]][1],
                         outlier_frac=OUTLIER_FRAC)[0] for _, members in LAUNCHES])
    X_all = torch.from_numpy(X_host).to(dev)
    Y_all = torch.zeros(int(n_off[-1]), dtype=torch.float32, device=dev)
    Xs = [X_all[k_off[j]:k_off[j + 1]].view(1, -1) for j in range(len(LAUNCHES))]
    Ys = [Y_all[n_off[i]:n_off[i + 1]].view(1, -1) for i in range(len(LINEARS))]

    # --- weights: generated on the GPU, quantized by the library -----------
    copies = []
    for c in range(2):
        Wqs, sws = [], []
        for i, (_, K, N) in enumerate(LINEARS):
            W = synth.normal_gpu(WEIGHT_SEED0 + i, (N, K), 0.02, device=dev)
            Wq, sw = w4.w4_quantize_weights(W)
            del W
            Wqs.append(Wq)
            sws.append(sw)
        copies.append((Wqs, sws))
    ws_bytes = max(w4.w4a8_workspace_bytes(1, act_K[j], sum(lin[n][2] for n in members))
                   for j, (_, members) in enumerate(LAUNCHES))
    ws = torch.zeros(max(ws_bytes, 4096), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def launch(c, j, flags):
        Wqs, sws = copies[c]
        idx = [lin[n][0] for n in LAUNCHES[j][1]]
        if len(idx) == 1:
            w4.w4a8_linear(Xs[j], Wqs[idx[0]], sws[idx[0]], Y=Ys[idx[0]], ws=ws, flags=flags)
        else:
            w4.w4a8_linear_grouped(Xs[j], [Wqs[i] for i in idx], [sws[i] for i in idx],
                                   Ys=[Ys[i] for i in idx], ws=ws, flags=flags)

    def launch_set(c):
        for j in range(len(LAUNCHES)):
            launch(c, j, PDL)

    # eager warm-up (sets kernel attributes), then graphs per weight copy
    with torch.cuda.stream(stream):
        launch_set(0)
        launch_set(1)
    torch.cuda.synchronize()
    graphs, e2e_graphs = [], []
    X_pin = torch.from_numpy(X_host).pin_memory()
    Y_pin = torch.empty(int(n_off[-1]), dtype=torch.float32).pin_memory()
    for c in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            launch_set(c)
        graphs.append(g)
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=stream):
            X_all.copy_(X_pin, non_blocking=True)
            launch_set(c)
            Y_pin.copy_(Y_all, non_blocking=True)
        e2e_graphs.append(g2)
    torch.cuda.synchronize()

    clocks = ClockSampler(gpu_uuid())
    clocks.start()
    # warm-up: at least W steps, and long enough for clock samples under load
    with torch.cuda.stream(stream):
        t_end = time.time() + args.min_busy_s
        k = 0
        while k < args.warmup or time.time() < t_end:
            graphs[k % 2].replay()
            k += 1
            if k % 200 == 0:
                stream.synchronize()
    stream.synchronize()

    # --- headline: K steps of the set --------------------------------------
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for k in range(args.steps):
            graphs[k % 2].replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_step = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)

    # --- dominant kernel: lm_head, CUDA events around each launch ------------
    jl = [l[0] for l in LAUNCHES].index("lm_head")
    _, K_lm, N_lm = LINEARS[lin["lm_head"][0]]
    n_lm = max(20, min(args.steps, 400))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_lm)]
    with torch.cuda.stream(stream):
        for k in range(n_lm):
            evs[k][0].record(stream)
            launch(k % 2, jl, 0)
            evs[k][1].record(stream)
    torch.cuda.synchronize()
    lm_ms = float(np.mean([a.elapsed_time(b) for a, b in evs[2:]]))

    # --- e2e: pinned host in, results out, every step ---------------------
    with torch.cuda.stream(stream):
        for k in range(max(3, args.warmup)):
            e2e_graphs[k % 2].replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k in range(args.steps):
            e2e_graphs[k % 2].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    Y_check = Y_pin.numpy()
    assert np.isfinite(Y_check).all()

    # --- per-launch times: a graph of 20 launches of one kind (no PDL) -------
    per_launch = {}
    for j, (lname, members) in enumerate(LAUNCHES):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(20):
                launch(k % 2, j, 0)
        with torch.cuda.stream(stream):
            g.replay()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(5):
                g.replay()
            a1.record(stream)
        torch.cuda.synchronize()
        us = a0.elapsed_time(a1) / 100 * 1e3
        nbytes = sum(weight_bytes(lin[n][1], lin[n][2]) for n in members)
        per_launch[lname] = {"us": round(us, 2), "GBps": round(nbytes / us / 1e3, 1)}
        del g
    errors = w4.w4a8_device_error()
    if errors:
        raise SystemExit("device error word %#x" % errors)

    peak, peak_kind = measured_peak()
    value = SET_BYTES * world / (ms_step * 1e-3) / 1e9
    lm_bytes = weight_bytes(K_lm, N_lm)
    achieved = lm_bytes / (lm_ms * 1e-3) / 1e9
    traffic = profiled_traffic()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4xint8->int32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1, "set_weight_bytes": SET_BYTES,
                   "l2": "two weight copies alternate (780 MB > 129 MB L2)",
                   "launch": "CUDA graph of 5 fused launches (q/k/v and gate/up grouped) with programmatic dependent launch",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "us_per_set": round(ms_step * 1e3, 2),
        "pct_hbm_peak": {"of_measured": round(SET_BYTES / (ms_step * 1e-3) / 1e9 / peak, 4),
                         "measured_gbs": peak, "of_nominal_8tbs":
                         round(SET_BYTES / (ms_step * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4)},
        "roofline": {"bound": "hbm", "kernel": "gemv_kernel<W4A8, M=1, fused> on lm_head 3584->152064",
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": lm_bytes, "avg_launch_us": round(lm_ms * 1e3, 2)},
        "e2e": {"value": round(SET_BYTES * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "us_per_set": round(e2e_ms * 1e3, 2),
                "h2d_bytes_per_step": int(X_pin.numel() * X_pin.element_size()),
                "d2h_bytes_per_step": int(Y_pin.numel() * Y_pin.element_size()),
                "how": "CUDA graph: pinned H2D of the 5 activations, 5 fused launches, D2H of the 8 outputs"},
        "clocks": clk,
        "gpu_launches": len(LAUNCHES) * args.steps,
        "per_launch_no_pdl": per_launch,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        orc, inputs = cpu_sample_inputs(dev)
        t_set, reps = time_oracle_sample(orc, inputs)
        line["cpu_baseline"] = {
            "value": round(SET_BYTES / t_set / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "us_per_set": round(t_set * 1e6, 1),
            "sample": "every %dth output row of each linear, %d repetitions, scaled to the full set"
                      % (CPU_SAMPLE_STRIDE, reps)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_only(args, lname):
    """Profiling aid: `warmup` then `steps` eager launches of one launch kind on
    two alternating weight copies, CUDA events around the timed launches."""
    import torch
    import synth
    import bit_weight_quantized_w4a8_gb300 as w4
    w4.build()
    w4.w4a8_set_tuning(reset=True)
    dev = torch.device("cuda", torch.cuda.current_device())
    members = dict(LAUNCHES)[lname]
    names = [l[0] for l in LINEARS]
    idx = [names.index(n) for n in members]
    K = LINEARS[idx[0]][1]
    X = torch.from_numpy(synth.activation(activation_seed(members[0]), 1, K,
                                          outlier_frac=OUTLIER_FRAC)).to(dev)
    copies = []
    for c in range(2):
        ws_, ss_ = [], []
        for i in idx:
            W = synth.normal_gpu(WEIGHT_SEED0 + i, (LINEARS[i][2], K), 0.02, device=dev)
            Wq, sw = w4.w4_quantize_weights(W)
            del W
            ws_.append(Wq)
            ss_.append(sw)
        copies.append((ws_, ss_))
    Ys = [torch.empty((1, LINEARS[i][2]), dtype=torch.float32, device=dev) for i in idx]
    wsb = torch.zeros(max(w4.w4a8_workspace_bytes(1, K, sum(LINEARS[i][2] for i in idx)), 4096),
                      dtype=torch.uint8, device=dev)

    def one(k):
        Wqs, sws = copies[k % 2]
        if len(idx) == 1:
            w4.w4a8_linear(X, Wqs[0], sws[0], Y=Ys[0], ws=wsb)
        else:
            w4.w4a8_linear_grouped(X, Wqs, sws, Ys=Ys, ws=wsb)

    for k in range(args.warmup):
        one(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for k in range(args.steps):
        one(k)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / args.steps * 1e3
    nbytes = sum(weight_bytes(K, LINEARS[i][2]) for i in idx)
    print(json.dumps({"only": lname, "members": list(members), "steps": args.steps,
                      "us_per_launch": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
                      "note": "eager launches, host launch gaps included; profiling aid"}),
          flush=True)


def main():
    args = parse()
    world, rank, _ = dist_setup(args)
    if args.only is not None:
        if rank == 0:
            run_only(args, args.only)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
