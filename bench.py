#!/usr/bin/env python
"""Benchmark: the Qwen2-7B-shaped decode linear set at M=1, W4A8.

One step = one pass of the whole hot path over one decode token: for the
eight linears (q, k, v, o, gate, up, down, lm_head) the fused kernel
quantizes the fp16 activation to INT8, streams the packed INT4 weights,
accumulates in int32 and rescales to fp32.  Projections that read the same
activation in the model share one grouped launch (q/k/v; gate/up), so a step
is five launches.  Weights (389.8 MB per set) are resident in HBM; two copies
alternate between steps, so nothing is reused from the 129 MB L2.  Steps are
replayed as CUDA graphs of two steps each (copy 0, then copy 1) whose launches
are programmatically dependent.

Reported (one JSON line, rank 0):
  value     effective weight GB/s (packed INT4 + fp32 scales per set / time)
  e2e       the same with the activations copied in from pinned host memory
            and the outputs read back, every step, inside the timed region
  roofline  the dominant kernel (lm_head, 273 MB) against measured HBM peak
  cpu_baseline  the CPU oracle timed on the host on a sample of the set
  decode_step_28_layers  a full 28-layer decode step of the same shapes
            (linear layers only) plus lm_head: ms per token
  skinny_batch  gate and down at M = 1 ... 64 activation rows
  w8a16_set the ChatGLM2-6B-shaped W8A16 GEMVs at M=1
  group_scale_set  the M=1 set with group-wise INT4 scales (group 128)
  index_softmax  the IntAttention page's integer softmax on 32 x 1024 x 4096
            int32 attention logits

`--impl reference` times the CPU oracle alone (the reference arm).
Under torchrun with N > 1 every rank runs an independent replica (weak
scaling); the path has no data exchange.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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
# L2 prefetch hint of a decode step (w4a8_linear_prefetch): the launch
# before lm_head (down, latency-bound at one row, so HBM has room) brings the
# first 16 MiB of lm_head's weights into L2.  Measured: the set 78.5 -> 73.9
# us; hints before the other launches gained nothing and cost the 28-layer
# step 1%.
PREFETCH_NEXT = {"down": 16 << 20}
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
IO_BYTES = sum(2 * K + 4 * N for _, K, N in LINEARS)  # M = 1: activation in, output out


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sample-stride", type=int, default=0,
                    help="the oracle's sample: every n-th output row of each linear (default: "
                         "%d for our arm's cpu_baseline, 1 = the whole set for --impl reference)"
                         % CPU_SAMPLE_STRIDE)
    ap.add_argument("--no-prefetch", action="store_true",
                    help="launch the decode steps without the L2 prefetch hints (PREFETCH_NEXT)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the 28-layer step, the skinny-batch sweep and the W8A16 set")
    ap.add_argument("--min-busy-s", type=float, default=0.6,
                    help="keep the GPU busy at least this long before timing (clock samples)")
    ap.add_argument("--only", choices=[l[0] for l in LAUNCHES] + ["w8_" + l[0] for l in W8A16_SET]
                    + ["isx"],
                    default=None,
                    help="profiling aid: time one launch kind alone, eagerly, without PDL "
                         "(not the headline metric)")
    ap.add_argument("--m", type=int, default=1,
                    help="with --only: activation rows of the W4A8 launch (3..64 take the tensor cores)")
    ap.add_argument("--group", type=int, default=0,
                    help="with --only: group-wise INT4 scales of this group size")
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
    for name in ("gemv_kernel.cuh", "gemv.cu", "plan.h", "ptx.cuh", "actq.cuh"):
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


def cpu_sample_inputs(dev, stride=CPU_SAMPLE_STRIDE):
    """Every stride-th output row of each linear, quantized by the oracle on
    the host.  Weights are drawn on the host by the C twin of the generator
    (the same bits as the numpy definition and the GPU twin), so no GPU is
    involved; the oracle quantizes row chunks on host threads (set-up, not
    timed)."""
    import concurrent.futures as cf
    import oracle
    import synth
    orc = oracle.load()
    out = []
    threads = os.cpu_count() or 4
    for idx, (name, K, N) in enumerate(LINEARS):
        seed = WEIGHT_SEED0 + idx
        W_rows = np.ascontiguousarray(synth.normal_host(seed, (N, K), 0.02)[::stride])
        n = W_rows.shape[0]
        Wq = np.empty((n, K // 2), np.uint8)
        sw = np.empty(n, np.float32)
        step = -(-n // (4 * threads))

        def quant(r0):
            Wq[r0:r0 + step], sw[r0:r0 + step] = orc.w4_quantize(W_rows[r0:r0 + step])

        with cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(quant, range(0, n, step)))
        del W_rows
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


def time_oracle_sample_threads(orc, inputs, threads, min_s=2.0, max_reps=50):
    """The same sample with each linear's rows split over `threads` host
    threads, each calling the unchanged oracle on its slice (rows are
    independent, so the results are the same; the C oracle runs without the
    interpreter lock)."""
    import concurrent.futures as cf
    import numpy as np
    jobs = []
    for (X, Wq, sw, _) in inputs:
        for rows in np.array_split(np.arange(Wq.shape[0]), threads):
            if rows.size:
                jobs.append((X, np.ascontiguousarray(Wq[rows]), np.ascontiguousarray(sw[rows])))
    reps, t_total = 0, 0.0
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        while reps < max_reps and (t_total < min_s or reps < 2):
            t0 = time.perf_counter()
            for f in [ex.submit(orc.w4a8_linear, *j) for j in jobs]:
                f.result()
            t_total += time.perf_counter() - t0
            reps += 1
    rows_sampled = sum(Wq.shape[0] for (_, Wq, _, _) in inputs)
    rows_total = sum(N for (_, _, _, N) in inputs)
    return t_total / reps * rows_total / rows_sampled, reps


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle alone
# ---------------------------------------------------------------------------

def run_reference(args, world, rank):
    if rank != 0:
        return
    stride = args.sample_stride or 1
    orc, inputs = cpu_sample_inputs(None, stride)
    sample = ("the whole set (every output row of each linear)" if stride == 1 else
              "every %dth output row of each linear (%.2f%% of the set's weights)" % (stride, 100.0 / stride))
    for _ in range(args.warmup):
        for (X, Wq, sw, _) in inputs:
            orc.w4a8_linear(X, Wq, sw)
    rows_sampled = sum(Wq.shape[0] for (_, Wq, _, _) in inputs)
    rows_total = sum(N for (_, _, _, N) in inputs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for (X, Wq, sw, _) in inputs:
            orc.w4a8_linear(X, Wq, sw)
    measured = (time.perf_counter() - t0) / args.steps
    dt = measured * rows_total / rows_sampled
    value = SET_BYTES / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4xint8->int32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1, "set_weight_bytes": SET_BYTES},
        "cpu_baseline": {"kind": "oracle", "value": round(value, 4), "unit": "GB/s", "cores": 1,
                         "sample": sample + ("; timed per step" if stride == 1 else
                                             "; per step, scaled to the full set"),
                         "measured_s_per_step": round(measured, 4)},
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
        pf, pb = None, 0
        if not args.no_prefetch and LAUNCHES[j][0] in PREFETCH_NEXT and j + 1 < len(LAUNCHES):
            pf, pb = Wqs[lin[LAUNCHES[j + 1][1][0]][0]], PREFETCH_NEXT[LAUNCHES[j][0]]
        if len(idx) == 1:
            w4.w4a8_linear(Xs[j], Wqs[idx[0]], sws[idx[0]], Y=Ys[idx[0]], ws=ws, flags=flags,
                           prefetch=pf, prefetch_bytes=pb)
        else:
            w4.w4a8_linear_grouped(Xs[j], [Wqs[i] for i in idx], [sws[i] for i in idx],
                                   Ys=[Ys[i] for i in idx], ws=ws, flags=flags, prefetch=pf,
                                   prefetch_bytes=pb)

    def launch_set(c):
        for j in range(len(LAUNCHES)):
            launch(c, j, PDL)

    X_pin = torch.from_numpy(X_host).pin_memory()
    Y_pin = torch.empty(int(n_off[-1]), dtype=torch.float32).pin_memory()

    def e2e_set(c):
        X_all.copy_(X_pin, non_blocking=True)
        launch_set(c)
        Y_pin.copy_(Y_all, non_blocking=True)

    # eager warm-up (sets kernel attributes), then graphs: a pair of steps
    # (weight copy 0, then copy 1) and a single step for an odd remainder
    with torch.cuda.stream(stream):
        launch_set(0)
        launch_set(1)
    torch.cuda.synchronize()

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    pair = capture(lambda: (launch_set(0), launch_set(1)))
    single = capture(lambda: launch_set(0))
    e2e_pair = capture(lambda: (e2e_set(0), e2e_set(1)))
    e2e_single = capture(lambda: e2e_set(0))
    torch.cuda.synchronize()

    def run_steps(n, two, one):
        for _ in range(n // 2):
            two.replay()
        if n % 2:
            one.replay()

    clocks = ClockSampler(gpu_uuid())
    clocks.start()
    # warm-up: at least W steps, and long enough for clock samples under load
    with torch.cuda.stream(stream):
        t_end = time.time() + args.min_busy_s
        k = 0
        while k < args.warmup or time.time() < t_end:
            pair.replay()
            k += 2
            if k % 400 == 0:
                stream.synchronize()
    stream.synchronize()

    # --- headline: K steps of the set --------------------------------------
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        run_steps(args.steps, pair, single)
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_step = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)

    # --- dominant kernel: lm_head.  Its steady-state launch duration: CUDA
    # events on the stream around replays of a graph of 20 back-to-back
    # launches (PDL, the two weight copies alternating: 546 MB > L2), as it
    # runs inside the set; and one launch on its own (ramp-up and tail
    # included), for reference
    jl = [l[0] for l in LAUNCHES].index("lm_head")
    _, K_lm, N_lm = LINEARS[lin["lm_head"][0]]
    lm_chain_us = _graph_us(torch, stream, lambda: [launch(k % 2, jl, PDL) for k in range(20)], 20,
                            reps=10)
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
        run_steps(max(4, args.warmup), e2e_pair, e2e_single)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_steps(args.steps, e2e_pair, e2e_single)
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
    peak, peak_kind = measured_peak()
    extra = {}
    if not args.no_extra:
        extra["skinny_batch"] = measure_skinny(torch, w4, synth, dev, stream, copies, lin)
        extra["mlp_m1"] = measure_mlp(torch, w4, synth, dev, stream, lin)
        extra["w8a16_set"] = measure_w8a16(torch, w4, synth, dev, stream)
        extra["group_scale_set"] = measure_group_set(torch, w4, synth, dev, stream, lin)
        extra["index_softmax"] = measure_index_softmax(torch, w4, synth, dev, stream, peak)
        del copies
        torch.cuda.empty_cache()
        extra["decode_step_28_layers"] = measure_decode_step(torch, w4, synth, dev, stream, ws, peak,
                                                             no_prefetch=args.no_prefetch)
    errors = w4.w4a8_device_error()
    if errors:
        raise SystemExit("device error word %#x" % errors)

    value = SET_BYTES * world / (ms_step * 1e-3) / 1e9
    lm_bytes = weight_bytes(K_lm, N_lm)
    achieved = lm_bytes / (lm_chain_us * 1e-6) / 1e9
    traffic = profiled_traffic()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4xint8->int32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1, "set_weight_bytes": SET_BYTES,
                   "l2": "two weight copies alternate (780 MB > 129 MB L2)",
                   "launch": "CUDA graphs of two steps (weight copy 0, then 1; a one-step graph for an odd count), 5 fused launches a step (q/k/v and gate/up grouped), programmatic dependent launch",
                   "l2_prefetch": "none" if args.no_prefetch else
                   "down (the launch before lm_head) brings the first 16 MiB of lm_head's weights into L2 (w4a8_linear_prefetch)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "us_per_set": round(ms_step * 1e3, 2),
        # the same time over weights + fp16 activation in + fp32 output bytes of every linear
        "GBps_with_io": round((SET_BYTES + IO_BYTES) / (ms_step * 1e-3) / 1e9, 2),
        "pct_hbm_peak": {"of_measured": round(SET_BYTES / (ms_step * 1e-3) / 1e9 / peak, 4),
                         "measured_gbs": peak, "of_nominal_8tbs":
                         round(SET_BYTES / (ms_step * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4)},
        "roofline": {"bound": "hbm", "kernel": "gemv_kernel<W4A8, M=1, fused> on lm_head 3584->152064",
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": lm_bytes, "avg_launch_us": round(lm_chain_us, 2),
                     "how": "graph of 20 back-to-back lm_head launches (PDL, two weight copies), "
                            "CUDA events around 10 replays on the launching stream",
                     "isolated_launch_us": round(lm_ms * 1e3, 2),
                     "isolated_frac": round(lm_bytes / (lm_ms * 1e-3) / 1e9 / peak, 4)},
        "e2e": {"value": round(SET_BYTES * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "us_per_set": round(e2e_ms * 1e3, 2),
                "h2d_bytes_per_step": int(X_pin.numel() * X_pin.element_size()),
                "d2h_bytes_per_step": int(Y_pin.numel() * Y_pin.element_size()),
                "how": "CUDA graphs of two steps: per step pinned H2D of the 5 activations, 5 fused launches, D2H of the 8 outputs"},
        "clocks": clk,
        "gpu_launches": len(LAUNCHES) * args.steps,
        "per_launch_no_pdl": per_launch,
    }
    line.update(extra)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        stride = args.sample_stride or CPU_SAMPLE_STRIDE
        orc, inputs = cpu_sample_inputs(dev, stride)
        t_set, reps = time_oracle_sample(orc, inputs)
        line["cpu_baseline"] = {
            "value": round(SET_BYTES / t_set / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "us_per_set": round(t_set * 1e6, 1),
            "sample": "every %dth output row of each linear, %d repetitions, scaled to the full set"
                      % (stride, reps)}
        threads = os.cpu_count() or 1
        t_all, reps_all = time_oracle_sample_threads(orc, inputs, threads)
        line["cpu_baseline"]["all_cores"] = {
            "value": round(SET_BYTES / t_all / 1e9, 4), "unit": "GB/s", "cores": threads,
            "us_per_set": round(t_all * 1e6, 1),
            "sample": "the same rows split over %d host threads, %d repetitions" % (threads, reps_all)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def _graph_us(torch, stream, fn, per_replay, reps=5):
    """Captures fn() as one CUDA graph, replays it once untimed and `reps`
    times timed; returns microseconds per unit (per_replay units a replay)."""
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    with torch.cuda.stream(stream):
        g.replay()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(reps):
            g.replay()
        a1.record(stream)
    torch.cuda.synchronize()
    return a0.elapsed_time(a1) / (reps * per_replay) * 1e3


DECODE_LAYERS = 28


def measure_decode_step(torch, w4, synth, dev, stream, ws, peak, no_prefetch=False):
    """A full 28-layer Qwen2-7B-shaped decode step, linear layers only: per
    layer q/k/v (grouped), o, gate/up (grouped), down, then lm_head once;
    per-layer weights (seed 1000 * (layer + 1) + index), 3.54 GB resident;
    activations pre-generated per launch (the linears do not chain without
    attention and norms); one CUDA graph of 113 dependent launches."""
    names = [l[0] for l in LINEARS]
    layers = []
    for layer in range(DECODE_LAYERS):
        Wq, sw = {}, {}
        for i, (n, K, N) in enumerate(LINEARS[:-1]):
            W = synth.normal_gpu(1000 * (layer + 1) + i, (N, K), 0.02, device=dev)
            Wq[n], sw[n] = w4.w4_quantize_weights(W)
            del W
        Xs = {}
        for lname, members in LAUNCHES[:-1]:
            K = LINEARS[names.index(members[0])][1]
            Xs[lname] = torch.from_numpy(synth.activation(
                1000 * (layer + 1) + names.index(members[0]) + ACT_SEED_OFFSET, 1, K,
                outlier_frac=OUTLIER_FRAC)).to(dev)
        layers.append((Wq, sw, Xs))
    i_lm = names.index("lm_head")
    _, K_lm, N_lm = LINEARS[i_lm]
    W = synth.normal_gpu(WEIGHT_SEED0 + i_lm, (N_lm, K_lm), 0.02, device=dev)
    Wq_lm, sw_lm = w4.w4_quantize_weights(W)
    del W
    X_lm = torch.from_numpy(synth.activation(activation_seed("lm_head"), 1, K_lm,
                                             outlier_frac=OUTLIER_FRAC)).to(dev)
    Ys = {n: torch.empty((1, N), dtype=torch.float32, device=dev) for n, _, N in LINEARS}
    torch.cuda.synchronize()

    def step():
        for li, (Wq, sw, Xs) in enumerate(layers):
            for j, (lname, members) in enumerate(LAUNCHES[:-1]):
                pf, pb = None, 0
                if not no_prefetch and lname in PREFETCH_NEXT and j + 1 == len(LAUNCHES) - 1 \
                        and li + 1 == len(layers):
                    pf, pb = Wq_lm, PREFETCH_NEXT[lname]  # the last down: lm_head follows
                if len(members) == 1:
                    w4.w4a8_linear(Xs[lname], Wq[members[0]], sw[members[0]], Y=Ys[members[0]],
                                   ws=ws, flags=w4.LAUNCH_PDL, prefetch=pf, prefetch_bytes=pb)
                else:
                    w4.w4a8_linear_grouped(Xs[lname], [Wq[n] for n in members],
                                           [sw[n] for n in members], Ys=[Ys[n] for n in members],
                                           ws=ws, flags=w4.LAUNCH_PDL, prefetch=pf, prefetch_bytes=pb)
        w4.w4a8_linear(X_lm, Wq_lm, sw_lm, Y=Ys["lm_head"], ws=ws, flags=w4.LAUNCH_PDL)

    us = _graph_us(torch, stream, step, 1, reps=10)
    nbytes = DECODE_LAYERS * sum(weight_bytes(K, N) for _, K, N in LINEARS[:-1]) + \
        weight_bytes(K_lm, N_lm)
    del layers
    return {"workload": "28 layers x (q/k/v, o, gate/up, down) + lm_head, M=1, W4A8",
            "launches": DECODE_LAYERS * (len(LAUNCHES) - 1) + 1, "weight_bytes": nbytes,
            "ms_per_token": round(us / 1e3, 4), "tok_per_s": round(1e6 / us, 1),
            "GBps": round(nbytes / us / 1e3, 1), "of_measured_peak": round(nbytes / us / 1e3 / peak, 4)}


SKINNY_M = (1, 2, 4, 8, 16, 32, 64)


def measure_skinny(torch, w4, synth, dev, stream, copies, lin):
    """gate 3584->18944 and down 18944->3584 at M = 1 ... 64 rows, and
    lm_head 3584->152064 at 2 ... 16: a graph of ten calls on the two
    alternating weight copies, each row with the kernel that served it
    (0 dp4a GEMV, 1 tcgen05 tensor cores, 2 row-per-thread dp4a, 3 warp-level
    e4m3 MMA)."""
    out = {}
    for name in ("gate", "down", "lm_head"):
        i, K, N = lin[name]
        res = {}
        for M in (SKINNY_M if name != "lm_head" else (2, 4, 8, 16)):
            X = torch.from_numpy(synth.activation(WEIGHT_SEED0 + i + ACT_SEED_OFFSET, M, K,
                                                  outlier_frac=OUTLIER_FRAC)).to(dev)
            Y = torch.empty((M, N), dtype=torch.float32, device=dev)
            ws = torch.zeros(max(w4.w4a8_workspace_bytes(M, K, N), 4096), dtype=torch.uint8,
                             device=dev)

            def calls():
                for k in range(10):
                    Wqs, sws = copies[k % 2]
                    w4.w4a8_linear(X, Wqs[i], sws[i], Y=Y, ws=ws, flags=w4.LAUNCH_PDL)

            us = _graph_us(torch, stream, calls, 10)
            res[str(M)] = {"us": round(us, 2), "GBps": round(weight_bytes(K, N) / us / 1e3, 1),
                           "kernel": w4.w4a8_plan_info(M, K, N)["kernel"]}
        out[name] = res
    return out


def measure_mlp(torch, w4, synth, dev, stream, lin):
    """The Qwen2-7B-shaped MLP at one row, gate/up 3584 -> 18944 and down
    18944 -> 3584 (102 MB of weights): fused, the gate/up launch writing
    h = fp16(silu(g) * u) from its epilogue (row-interleaved gate/up weights)
    and down reading h; unfused, the grouped gate/up launch, the gated
    product as a launch of its own, then down.  PDL, two weight copies
    alternating, graphs of ten MLPs."""
    ig, K, N = lin["gate"]
    iu = lin["up"][0]
    idn = lin["down"][0]
    mats = []
    for c in range(2):
        q = {}
        for i in (ig, iu, idn):
            n_, k_ = LINEARS[i][2], LINEARS[i][1]
            W = synth.normal_gpu(WEIGHT_SEED0 + i + 100 * c, (n_, k_), 0.02, device=dev)
            q[i] = w4.w4_quantize_weights(W)
            del W
        q["gu"] = w4.w4_interleave_rows(q[ig][0], q[ig][1], q[iu][0], q[iu][1])
        mats.append(q)
    X = torch.from_numpy(synth.activation(activation_seed("gate"), 1, K, outlier_frac=OUTLIER_FRAC)).to(dev)
    H = torch.empty((1, N), dtype=torch.float16, device=dev)
    Ygu = torch.empty((1, 2 * N), dtype=torch.float32, device=dev)
    Yg = torch.empty((1, N), dtype=torch.float32, device=dev)
    Yu = torch.empty((1, N), dtype=torch.float32, device=dev)
    Yd = torch.empty((1, K), dtype=torch.float32, device=dev)
    ws = torch.zeros(max(w4.w4a8_gate_up_silu_workspace_bytes(1, K, N), w4.w4a8_workspace_bytes(1, K, 2 * N),
                         w4.w4a8_workspace_bytes(1, N, K), 4096), dtype=torch.uint8, device=dev)
    PDL = w4.LAUNCH_PDL

    def fused():
        for k in range(10):
            q = mats[k % 2]
            w4.w4a8_gate_up_silu(X, q["gu"][0], q["gu"][1], H=H, Y_gu=Ygu, ws=ws, flags=PDL)
            w4.w4a8_linear(H, q[idn][0], q[idn][1], Y=Yd, ws=ws, flags=PDL)

    def unfused():
        for k in range(10):
            q = mats[k % 2]
            w4.w4a8_linear_grouped(X, [q[ig][0], q[iu][0]], [q[ig][1], q[iu][1]], Ys=[Yg, Yu], ws=ws, flags=PDL)
            w4.w4a8_silu_mul(Yg, Yu, H=H, flags=PDL)
            w4.w4a8_linear(H, q[idn][0], q[idn][1], Y=Yd, ws=ws, flags=PDL)

    nbytes = 2 * weight_bytes(K, N) + weight_bytes(N, K)
    res = {"workload": "Qwen2-7B MLP, M=1: gate/up 3584->18944, silu(g)*u, down 18944->3584", "weight_bytes": nbytes}
    for name, fn in (("fused", fused), ("unfused", unfused)):
        us = _graph_us(torch, stream, fn, 10, reps=10)
        res[name] = {"us": round(us, 2), "GBps": round(nbytes / us / 1e3, 1), "launches": 2 if name == "fused" else 3}
    del mats
    return res


GROUP_SIZE = 128


def measure_group_set(torch, w4, synth, dev, stream, lin, gs=GROUP_SIZE):
    """The headline set with group-wise INT4 scales (one fp32 scale per 128
    codes): same shapes, seeds, activations and launch structure (five
    launches, q/k/v and gate/up grouped, PDL, two weight copies alternating
    in graphs of two steps).  Bytes per linear: N * (K/2 + 4 * stride)."""
    names = [l[0] for l in LINEARS]
    copies = []
    for c in range(2):
        Wqs, sgs = [], []
        for i, (_, K, N) in enumerate(LINEARS):
            W = synth.normal_gpu(WEIGHT_SEED0 + i, (N, K), 0.02, device=dev)
            Wq, sg = w4.w4g_quantize_weights(W, gs)
            del W
            Wqs.append(Wq)
            sgs.append(sg)
        copies.append((Wqs, sgs))
    Xs, Ys = [], [torch.empty((1, N), dtype=torch.float32, device=dev) for _, _, N in LINEARS]
    for _, members in LAUNCHES:
        K = lin[members[0]][1]
        Xs.append(torch.from_numpy(synth.activation(activation_seed(members[0]), 1, K,
                                                    outlier_frac=OUTLIER_FRAC)).to(dev))
    ws_bytes = max(w4.w4a8g_workspace_bytes(1, lin[m[0]][1], sum(lin[n][2] for n in m), gs)
                   for _, m in LAUNCHES)
    ws = torch.zeros(max(ws_bytes, 4096), dtype=torch.uint8, device=dev)

    def launch(c, j, flags):
        Wqs, sgs = copies[c]
        idx = [names.index(n) for n in LAUNCHES[j][1]]
        if len(idx) == 1:
            w4.w4a8g_linear(Xs[j], Wqs[idx[0]], sgs[idx[0]], gs, Y=Ys[idx[0]], ws=ws, flags=flags)
        else:
            w4.w4a8g_linear_grouped(Xs[j], [Wqs[i] for i in idx], [sgs[i] for i in idx], gs,
                                    Ys=[Ys[i] for i in idx], ws=ws, flags=flags)

    def pair():
        for c in range(2):
            for j in range(len(LAUNCHES)):
                launch(c, j, w4.LAUNCH_PDL)

    us = _graph_us(torch, stream, pair, 2, reps=20)
    nbytes = sum(N * (K // 2 + 4 * w4.w4g_scale_stride(K, gs)) for _, K, N in LINEARS)
    jl = [l[0] for l in LAUNCHES].index("lm_head")
    us_lm = _graph_us(torch, stream, lambda: [launch(k % 2, jl, w4.LAUNCH_PDL) for k in range(20)], 20)
    _, K_lm, N_lm = LINEARS[names.index("lm_head")]
    lm_bytes = N_lm * (K_lm // 2 + 4 * w4.w4g_scale_stride(K_lm, gs))
    # batches on gate and down (2..8 rows take the row-per-thread kernel,
    # 9..64 the tensor cores)
    skinny = {}
    for name in ("gate", "down"):
        i = names.index(name)
        _, K, N = LINEARS[i]
        res = {}
        for M in (1, 2, 4, 8, 16, 64):
            X = torch.from_numpy(synth.activation(WEIGHT_SEED0 + i + ACT_SEED_OFFSET, M, K,
                                                  outlier_frac=OUTLIER_FRAC)).to(dev)
            Y = torch.empty((M, N), dtype=torch.float32, device=dev)
            wsm = torch.zeros(max(w4.w4a8g_workspace_bytes(M, K, N, gs), 4096), dtype=torch.uint8,
                              device=dev)
            us_m = _graph_us(torch, stream, lambda: [w4.w4a8g_linear(X, copies[k % 2][0][i], copies[k % 2][1][i],
                                                                     gs, Y=Y, ws=wsm, flags=w4.LAUNCH_PDL)
                                                     for k in range(10)], 10)
            nb = N * (K // 2 + 4 * w4.w4g_scale_stride(K, gs))
            res[str(M)] = {"us": round(us_m, 2), "GBps": round(nb / us_m / 1e3, 1)}
        skinny[name] = res
    del copies
    return {"workload": "the M=1 set above with group-wise INT4 scales, group %d" % gs,
            "weight_bytes": nbytes, "us_per_set": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
            "lm_head_in_chain": {"us": round(us_lm, 2), "GBps": round(lm_bytes / us_lm / 1e3, 1),
                                 "how": "graph of 20 back-to-back launches, PDL, two weight copies"},
            "skinny_batch": skinny}


ISX_HEADS, ISX_QUERIES, ISX_KEYS = 32, 1024, 4096


def measure_index_softmax(torch, w4, synth, dev, stream, peak):
    """IndexSoftmax on int32 attention logits of 32 heads x 1024 query rows x
    4096 keys (d = 128, per-tensor INT8 scales 4/127, dequantized logits with
    standard deviation 4): two logit buffers alternate (2 x 512 MB > L2), a
    graph of 10 launches; bytes per launch = 4 per logit in + 1 per
    probability out."""
    rows, cols = ISX_HEADS * ISX_QUERIES, ISX_KEYS
    s = float(np.float32(4 / 127))
    scale = 4.0 * math.sqrt(128) / (s * s)
    bufs = []
    for c in range(2):
        A = torch.empty((rows, cols), dtype=torch.int32, device=dev)
        for r0 in range(0, rows, 2048):
            z = synth.normal_gpu(4242 + c, (2048, cols), 1.0, offset=r0 * cols, device=dev)
            A[r0:r0 + 2048] = torch.round(z.double() * scale).int()
            del z
        bufs.append(A)
    P = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    c_int = w4.index_softmax_c_int(w4.ISX_DEFAULT_C, 128, s, s)
    lut = w4.index_softmax_lut()
    us = _graph_us(torch, stream, lambda: [w4.index_softmax_u8(bufs[k % 2], c_int, lut=lut, P=P)
                                           for k in range(10)], 10)
    nbytes = rows * cols * 5
    del bufs
    return {"workload": "IndexSoftmax (b=5, c=6.6) of int32 logits, %d heads x %d query rows x %d keys"
                        % (ISX_HEADS, ISX_QUERIES, ISX_KEYS),
            "bytes_per_launch": nbytes, "us": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
            "of_measured_peak": round(nbytes / us / 1e3 / peak, 4),
            "Gelem_per_s": round(rows * cols / us / 1e3, 1)}


W8A16_SET = [("h_to_4h", 4096, 27392), ("qkv", 4096, 4608), ("4h_to_h", 13696, 4096)]


def measure_w8a16(torch, w4, synth, dev, stream):
    """ChatGLM2-6B-shaped W8A16 GEMVs at M=1 (per-channel INT8 weights, fp16
    scale, fp16 activation): two weight copies alternate, one graph."""
    copies = []
    for c in range(2):
        cp = []
        for j, (_, K, N) in enumerate(W8A16_SET):
            W = synth.normal_gpu(2000 + j, (N, K), 0.02, device=dev)
            cp.append(w4.w8_quantize_weights(W))
            del W
        copies.append(cp)
    Xs = [torch.from_numpy(synth.activation(2500 + j, 1, K)).to(dev)
          for j, (_, K, _) in enumerate(W8A16_SET)]
    Ys = [torch.empty((1, N), dtype=torch.float32, device=dev) for _, _, N in W8A16_SET]
    ws = torch.zeros(max(max(w4.w8a16_workspace_bytes(1, K, N) for _, K, N in W8A16_SET), 4096),
                     dtype=torch.uint8, device=dev)

    def sets():
        for c in range(2):
            for j in range(len(W8A16_SET)):
                Wq8, sw16 = copies[c][j]
                w4.w8a16_gemv(Xs[j], Wq8, sw16, Y=Ys[j], ws=ws, flags=w4.LAUNCH_PDL)

    us = _graph_us(torch, stream, sets, 2, reps=10)
    nbytes = sum(N * K + 2 * N for _, K, N in W8A16_SET)
    del copies
    return {"workload": "W8A16 GEMVs 4096->27392, 4096->4608, 13696->4096, M=1",
            "weight_bytes": nbytes, "us_per_set": round(us, 2), "GBps": round(nbytes / us / 1e3, 1)}


def run_only(args, lname):
    """Profiling aid: `warmup` then `steps` eager launches of one launch kind on
    two alternating weight copies, CUDA events around the timed launches."""
    import torch
    import synth
    import bit_weight_quantized_w4a8_gb300 as w4
    w4.build()
    w4.w4a8_set_tuning(reset=True)
    dev = torch.device("cuda", torch.cuda.current_device())
    if lname.startswith("w8_"):
        return run_only_w8(args, lname[3:], torch, synth, w4, dev)
    if lname == "isx":
        return run_only_isx(args, torch, synth, w4, dev)
    members = dict(LAUNCHES)[lname]
    names = [l[0] for l in LINEARS]
    idx = [names.index(n) for n in members]
    K = LINEARS[idx[0]][1]
    M = args.m
    X = torch.from_numpy(synth.activation(activation_seed(members[0]), M, K,
                                          outlier_frac=OUTLIER_FRAC)).to(dev)
    gs = args.group
    copies = []
    for c in range(2):
        ws_, ss_ = [], []
        for i in idx:
            W = synth.normal_gpu(WEIGHT_SEED0 + i, (LINEARS[i][2], K), 0.02, device=dev)
            Wq, sw = w4.w4g_quantize_weights(W, gs) if gs else w4.w4_quantize_weights(W)
            del W
            ws_.append(Wq)
            ss_.append(sw)
        copies.append((ws_, ss_))
    Ys = [torch.empty((M, LINEARS[i][2]), dtype=torch.float32, device=dev) for i in idx]
    N_all = sum(LINEARS[i][2] for i in idx)
    nws = w4.w4a8g_workspace_bytes(M, K, N_all, gs) if gs else w4.w4a8_workspace_bytes(M, K, N_all)
    wsb = torch.zeros(max(nws, 4096), dtype=torch.uint8, device=dev)

    def one(k):
        Wqs, sws = copies[k % 2]
        if gs and len(idx) == 1:
            w4.w4a8g_linear(X, Wqs[0], sws[0], gs, Y=Ys[0], ws=wsb)
        elif gs:
            w4.w4a8g_linear_grouped(X, Wqs, sws, gs, Ys=Ys, ws=wsb)
        elif len(idx) == 1:
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
    if gs:
        nbytes = sum(LINEARS[i][2] * (K // 2 + 4 * w4.w4g_scale_stride(K, gs)) for i in idx)
    else:
        nbytes = sum(weight_bytes(K, LINEARS[i][2]) for i in idx)
    print(json.dumps({"only": lname, "members": list(members), "M": M, "group": gs, "steps": args.steps,
                      "us_per_launch": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
                      "note": "eager launches, host launch gaps included; profiling aid"}),
          flush=True)


def run_only_isx(args, torch, synth, w4, dev):
    """Profiling aid: eager IndexSoftmax launches on the benchmark's logits."""
    rows, cols = ISX_HEADS * ISX_QUERIES, ISX_KEYS
    s = float(np.float32(4 / 127))
    A = torch.empty((rows, cols), dtype=torch.int32, device=dev)
    for r0 in range(0, rows, 2048):
        z = synth.normal_gpu(4242, (2048, cols), 1.0, offset=r0 * cols, device=dev)
        A[r0:r0 + 2048] = torch.round(z.double() * (4.0 * math.sqrt(128) / (s * s))).int()
        del z
    P = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    c_int = w4.index_softmax_c_int(w4.ISX_DEFAULT_C, 128, s, s)
    lut = w4.index_softmax_lut()
    for _ in range(args.warmup):
        w4.index_softmax_u8(A, c_int, lut=lut, P=P)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        w4.index_softmax_u8(A, c_int, lut=lut, P=P)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / args.steps * 1e3
    print(json.dumps({"only": "isx", "steps": args.steps, "us_per_launch": round(us, 2),
                      "GBps": round(rows * cols * 5 / us / 1e3, 1),
                      "note": "eager launches on one logit buffer; profiling aid"}), flush=True)


def run_only_w8(args, name, torch, synth, w4, dev):
    """Profiling aid for one W8A16 GEMV of the ChatGLM2-6B-shaped set."""
    j = [l[0] for l in W8A16_SET].index(name)
    _, K, N = W8A16_SET[j]
    copies = []
    for c in range(2):
        W = synth.normal_gpu(2000 + j, (N, K), 0.02, device=dev)
        copies.append(w4.w8_quantize_weights(W))
        del W
    X = torch.from_numpy(synth.activation(2500 + j, 1, K)).to(dev)
    Y = torch.empty((1, N), dtype=torch.float32, device=dev)
    wsb = torch.zeros(max(w4.w8a16_workspace_bytes(1, K, N), 4096), dtype=torch.uint8, device=dev)

    def one(k):
        Wq8, sw16 = copies[k % 2]
        w4.w8a16_gemv(X, Wq8, sw16, Y=Y, ws=wsb)

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
    print(json.dumps({"only": "w8_" + name, "steps": args.steps, "us_per_launch": round(us, 2),
                      "GBps": round((N * K + 2 * N) / us / 1e3, 1),
                      "note": "eager launches, host launch gaps included; profiling aid"}), flush=True)


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
