"""Benchmark of the MoE layer forward on B300: one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference] [--no-cpu-baseline]

A step is one moe_layer_forward (router, dispatch, grouped expert FFN,
combine, statistics) over one batch of the workload, inputs resident in HBM.
Steps rotate over several input + weight sets whose total exceeds the L2
cache, so no step reads the previous step's data from L2.

Under torchrun (N > 1) every rank runs its own independent batch (the layer
is token-parallel; nothing is exchanged on the data path), the K steps are
bracketed by a barrier and a device synchronisation, the time is the maximum
over ranks and ``value`` is the total tokens of all ranks per second.

``--impl reference`` times the CPU oracle instead (rank 0 only), each step a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mixture_experts_layer_99_b300 import workloads as W  # noqa: E402

METRIC = ("MoE-layer fwd tokens/s at 1 B300; expert-GEMM TFLOP/s % of BF16 peak; "
          "router/dispatch GB/s")
UNIT = "tokens/s"
L2_BYTES = 126 * 1024 * 1024
# B300 dense bf16 tensor-core rate (no sparsity), NVIDIA's nominal figure
NOMINAL_BF16_TFLOPS = 2250.0


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def max_over_ranks(v: float, pg, device) -> float:
    """The maximum of a per-rank value over all ranks (the value itself
    without a process group). Used for step times only."""
    if pg is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def rank_seed(w, rank: int, i: int) -> int:
    """Seed of input set i on a rank: every rank draws its own batch."""
    return w.seed + 1000 * rank + i


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0,
                source="fallback")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "timestamp")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.t_start = self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, "t_" + which, time.time())

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                stamp, frac = parts[9].rsplit(".", 1)
                t = time.mktime(time.strptime(stamp, "%Y/%m/%d %H:%M:%S")) + float("0." + frac)
                rows.append(dict(t=t, sm=float(parts[1]), smax=float(parts[2]), w=float(parts[3]),
                                 mask=parts[4], hw=parts[5], hwt=parts[6], swt=parts[7],
                                 pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["no samples"])
        # samples (~20 ms apart) taken while the timed steps ran
        inside = [r for r in rows if self.t_start is not None and self.t_end is not None
                  and self.t_start <= r["t"] <= self.t_end]
        window = "timed region"
        if len(inside) < 3:
            inside, window = rows, "whole sampling period (timed region too short)"
        reasons = set()
        for r in inside:
            if r["hw"] == "Active":
                reasons.add("hw_slowdown")
            if r["hwt"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return dict(sm_mhz=statistics.median(r["sm"] for r in inside),
                    sm_max_mhz=max(r["smax"] for r in rows), reasons=sorted(reasons),
                    power_w=statistics.median(r["w"] for r in inside),
                    active_masks=sorted({r["mask"] for r in inside}),
                    samples=len(inside), window=window)


# ---------------------------------------------------------------- work model
def algorithmic(w, kept: int, n_active: int):
    """Algorithmic FLOPs and bytes of one layer call (what the method must
    compute or move), per part."""
    s = w.elem_bytes
    T, d, E, k, H = w.T, w.d, w.E, w.k, w.H
    nm = w.nmat
    router_b = T * d * s + E * d * s + (T * E * 4 if w.noise else 0) + T * k * 8 + E * 4
    router_f = 2 * T * d * E
    disp_b = T * k * 4 * 2 + 2 * kept * d * s + 8 * E
    gemm_f = kept * 2 * nm * d * H
    gemm_b = n_active * nm * d * H * s + 2 * kept * d * s
    comb_b = kept * d * s + T * k * 8 + T * d * s
    return dict(router_bytes=router_b, router_flops=router_f, dispatch_bytes=disp_b,
                gemm_flops=gemm_f, gemm_bytes=gemm_b, combine_bytes=comb_b,
                tc_router=w.dtype == "bf16" and E <= 64)


def footprint_bytes(inp):
    return sum(v.numel() * v.element_size() for v in inp.values() if v is not None)


def rotating_sets(fp: int) -> int:
    """Input + weight sets the GPU arm rotates over: their total exceeds three
    times the L2 cache, so no step finds the previous step's data in L2."""
    return max(2, math.ceil(3 * L2_BYTES / fp))


def bench_config(w, capacity: int, kept: int, n_active: int, nsets: int, fp: int,
                 world: int) -> dict:
    """The ``config`` object of both arms' JSON lines (the same keys and
    values, so that the two lines describe one workload)."""
    return dict(workload=w.name, T=w.T, d=w.d, E=w.E, k=w.k, H=w.H, act=w.act,
                capacity=capacity, kept_rows=kept, active_experts=n_active,
                parallelism=f"replicas x{world}",
                launch="one CUDA graph per input set, one layer call each",
                l2=f"{nsets} rotating input+weight sets of {fp / 2**20:.0f} MiB "
                   f"(> L2 between reuses)")


def time_backward(w, cfg, inp, ws, stream, dev, kept, reps):
    """ms per moe_layer_backward call (loss = sum <dy, y> + 0.01 L_balance),
    and the GEMM work it executes (tensor cores for bf16, FMA for fp32): the recomputed
    pre-activations (unless cfg keeps them from the forward), dh = dY W2,
    dxd = dact [W1; W3] and the weight gradients, kept * 2 * d * H *
    (3 (nm - 1) + 2) flops, (nm - 1) fewer with kept pre-activations."""
    from mixture_experts_layer_99_b300 import moe
    keep = bool(cfg.flags & moe.MOE_FLAG_KEEP_PREACT)
    out = moe.alloc_outputs(cfg, dev)
    moe.layer_forward(cfg, inp, ws=ws, out=out)
    dy = torch.randn(w.T, w.d, generator=torch.Generator().manual_seed(5)).to(
        w.torch_dtype).to(dev)
    bws = moe.workspace_backward(cfg, dev)
    grads = moe.alloc_grads(cfg, inp, dev)
    for _ in range(2):
        moe.layer_backward(cfg, inp, out, dy, 0.01, ws=ws, bws=bws, grads=grads)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        moe.layer_backward(cfg, inp, out, dy, 0.01, ws=ws, bws=bws, grads=grads)
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / reps
    # the forward of the same configuration, eager calls (with kept
    # pre-activations its GEMM1 also stores them)
    a.record(stream)
    for _ in range(reps):
        moe.layer_forward(cfg, inp, ws=ws, out=out)
    b.record(stream)
    torch.cuda.synchronize(dev)
    fwd_ms = a.elapsed_time(b) / reps
    flops = kept * 2 * w.d * w.H * ((2 if keep else 3) * (w.nmat - 1) + 2)
    return dict(ms_per_call=ms, calls=reps, gemm_tflops_executed=flops / (ms / 1e3) / 1e12,
                forward_ms_per_call=fwd_ms,
                tokens_per_s=w.T / (ms / 1e3), loss="sum <dy, y> + 0.01 L_balance",
                note=("eager calls on one input set; the forward kept the pre-activations "
                      "(MOE_FLAG_KEEP_PREACT)" if keep else
                      "eager calls on one input set; GEMM work includes the recomputed "
                      "pre-activations"))


def traffic_record(kernel_src_sha, workload):
    """The committed ncu DRAM traffic of the grouped GEMM, if it was taken on
    this workload from the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    if rec.get("source_sha256") != kernel_src_sha or rec.get("workload") != workload:
        return None
    return rec


def source_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mixture_experts_layer_99_b300", "csrc")
    with open(os.path.join(csrc, "ffn_tc.cu"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()


# ---------------------------------------------------------------- CPU oracle
def time_oracle(w, target_s=12.0, seed=0):
    """Times the oracle (fp64 numpy, all host cores its BLAS uses) on the
    first n tokens of the workload's batch taken as a batch of their own."""
    from oracle import moe_oracle as ORC
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:  # pragma: no cover
        cores = os.cpu_count()
    inp = W.make_inputs(w)

    def run(n):
        sub = dict(inp)
        sub["x"] = inp["x"][:n]
        if inp.get("noise") is not None:
            sub["noise"] = inp["noise"][:n]
        t0 = time.perf_counter()
        ORC.moe_forward(sub, k=w.k, c=w.c, act=w.act, tau=w.tau)
        return time.perf_counter() - t0

    n = min(w.T, 64)
    t = run(n)
    while t < target_s / 2 and n < w.T:
        n = min(w.T, max(n * 2, int(n * target_s / max(t, 1e-3) / 2)))
        t = run(n)
    return dict(value=n / t, unit=UNIT, cores=cores, kind="oracle",
                sample=sample_label(w, n, t), seconds=t, tokens=n)


def sample_label(w, n: int, t: float) -> str:
    head = "" if n == w.T else f"extrapolated ({n} of {w.T} tokens): "
    return (f"{head}first {n} of {w.T} tokens of the seed-{w.seed} {w.name} batch as a "
            f"batch of their own (capacity recomputed): full fp64 numpy forward "
            f"(router, top-k, dispatch, experts, combine, statistics) in {t:.2f} s")


def oracle_routing_summary(w, inp):
    """Kept rows and active experts of the whole batch, from the oracle's own
    routing (the reference arm's copy of the GPU arm's config keys)."""
    from oracle import moe_oracle as ORC
    T = inp["x"].shape[0]
    C = ORC.capacity(w.c, w.k, T, w.E)
    lg = ORC.router_logits(inp["x"], inp["Wg"], inp.get("bias"), inp.get("noise"), w.tau)
    r = ORC.route_from_logits(lg, w.k, C)
    return C, int(r["offset"][-1]), int((np.diff(r["offset"]) > 0).sum())


def run_reference(args, w):
    rank, _, world = dist_env()
    if rank != 0:
        return
    # each step is a sample of about three seconds of oracle work (so that a
    # run of 20 + 5 steps ends in a couple of minutes): at a few dozen tokens
    # the oracle's fixed cost (each expert's weights converted to fp64) would
    # dominate its per-token rate
    per_step = time_oracle(w, target_s=6.0)
    n = per_step["tokens"]
    from oracle import moe_oracle as ORC
    inp = W.make_inputs(w)
    sub = dict(inp)
    sub["x"] = inp["x"][:n]
    if inp.get("noise") is not None:
        sub["noise"] = inp["noise"][:n]
    for _ in range(args.warmup):
        ORC.moe_forward(sub, k=w.k, c=w.c, act=w.act, tau=w.tau)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ORC.moe_forward(sub, k=w.k, c=w.c, act=w.act, tau=w.tau)
    dt = (time.perf_counter() - t0) / args.steps
    value = n / dt
    C, kept, n_active = oracle_routing_summary(w, inp)
    fp = footprint_bytes(inp)
    cfg = bench_config(w, C, kept, n_active, rotating_sets(fp), fp, world)
    line = dict(metric=METRIC, value=value, unit=UNIT, n_gpus=args.gpus, steps=args.steps,
                warmup=args.warmup, ms_per_step=dt * 1e3, higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
                impl="reference",
                config=cfg,
                cpu_baseline=dict(value=value, unit=UNIT, cores=per_step["cores"],
                                  kind="oracle", sample=sample_label(w, n, dt)),
                e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- stage times
STAGES = ["router", "dispatch", "gemm1", "gemm2", "combine_stats"]


def _stage_avg(evs):
    n = len(evs)
    st = {name: sum(r[j].elapsed_time(r[j + 1]) for r in evs) / n
          for j, name in enumerate(STAGES)}
    st["layer"] = sum(r[0].elapsed_time(r[5]) for r in evs) / n
    return st


def stage_times(moe, cfg, sets, nsets, ws, out, stream, dev, want):
    """Per-stage device times of the layer call, averaged over about ``want``
    calls. The calls run as replays of one CUDA graph of M consecutive
    moe_layer_forward_profiled calls (rotating over the input sets), each with
    its own six events, which become event nodes of the graph; so the
    stages are timed on the same graph-launched path as the timed steps (an
    event node between two kernels does stop the next kernel's prologue from
    overlapping its predecessor's tail). Falls back to eager calls if the
    capture fails."""
    M = 8
    reps = max(2, math.ceil(want / M))

    def new_events(n):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n)]
        for row in evs:
            for e in row:
                e.record(stream)  # create the events
        return evs

    try:
        evs = new_events(M)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(M):
                moe.layer_forward_profiled(cfg, sets[i % nsets], evs[i], ws=ws, out=out)
        g.replay()  # warm-up replay
        torch.cuda.synchronize(dev)
        acc = []
        for _ in range(reps):
            g.replay()
            torch.cuda.synchronize(dev)
            acc.append(_stage_avg(evs))
        st = {k: sum(a[k] for a in acc) / len(acc) for k in acc[0]}
        return st, (f"CUDA-graph replays: {reps} x {M} consecutive moe_layer_forward_profiled "
                    f"calls with event nodes at the stage boundaries")
    except Exception as exc:  # pragma: no cover - capture not available
        torch.cuda.synchronize(dev)
        evs = new_events(want)
        torch.cuda.synchronize(dev)
        for i in range(want):
            moe.layer_forward_profiled(cfg, sets[i % nsets], evs[i], ws=ws, out=out)
        torch.cuda.synchronize(dev)
        return _stage_avg(evs), f"eager moe_layer_forward_profiled calls ({exc.__class__.__name__})"


def router_context(moe, cfg, sets, nsets, ws, out, stream, dev, reps=4):
    """The router step on its own, to read its stage time inside the layer:
    CUDA-graph replays of M moe_router_topk calls over the rotating input sets
    (the router kernel and the small kernel that sums its probability
    partials), each between two event nodes, (a) alone, (b) right after a
    memset of the layer's output y (T x d), which leaves y's lines dirty in
    L2 as the previous layer call's combine does, so that the router's loads
    also carry their write-back, and (c) two event nodes with nothing
    between them (the floor of one event-pair measurement). Medians in ms."""
    M = 8

    def med(kind):
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
               for _ in range(M)]
        for row in evs:
            for e in row:
                e.record(stream)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(M):
                s = sets[i % nsets]
                if kind == "after_write":
                    out["y"].zero_()
                evs[i][0].record(stream)
                if kind != "floor":
                    moe.router_topk(cfg, s["x"], s["Wg"], s.get("bias"), s.get("noise"),
                                    ws=ws, logits=True)
                evs[i][1].record(stream)
        g.replay()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(reps):
            g.replay()
            torch.cuda.synchronize(dev)
            ts += [r[0].elapsed_time(r[1]) for r in evs]
        ts.sort()
        return ts[len(ts) // 2]

    try:
        return {k: med(k) for k in ("alone", "after_write", "floor")}
    except Exception:  # pragma: no cover - capture not available
        torch.cuda.synchronize(dev)
        return None


# ---------------------------------------------------------------- GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    # the shared-expert variant (moe_layer_forward_shared) is covered by the
    # parity tests; the bench times the routed layer
    ap.add_argument("--workload", default="mixtral",
                    choices=sorted(n for n, v in W.WORKLOADS.items() if v.shared_H == 0))
    ap.add_argument("--impl", default="b300", choices=["b300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return

    from mixture_experts_layer_99_b300 import moe

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    # all work on one non-default stream (CUDA graphs cannot be captured on
    # the legacy default stream)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    peaks = load_peaks()

    # ---- inputs: rotating sets, different seed per rank and per set
    base = W.make_inputs(w, seed=rank_seed(w, rank, 0))
    fp = footprint_bytes(base)
    nsets = rotating_sets(fp)
    sets = [W.to_device(base, dev)]
    for i in range(1, nsets):
        sets.append(W.to_device(W.make_inputs(w, seed=rank_seed(w, rank, i)), dev))
    cfg = moe.config_from_workload(w)
    ws = moe.workspace(cfg, dev, host_io=True)
    out = moe.alloc_outputs(cfg, dev, full=True)

    # ---- routing statistics of set 0 (for the algorithmic work model)
    moe.layer_forward(cfg, sets[0], ws=ws, out=out)
    torch.cuda.synchronize(dev)
    offs = out["expert_offset"].cpu().numpy()
    kept = int(offs[-1])
    n_active = int((np.diff(offs) > 0).sum())
    work = algorithmic(w, kept, n_active)

    def step_eager(i):
        moe.layer_forward(cfg, sets[i % nsets], ws=ws, out=out)

    for i in range(args.warmup):
        step_eager(i)
    torch.cuda.synchronize(dev)
    # one CUDA graph per input set, each holding one layer call; a step
    # replays the next set's graph (the same kernels and arguments as the
    # eager call, without the host launch overhead)
    graphs = []
    for i in range(nsets):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step_eager(i)
        graphs.append(g)
    torch.cuda.synchronize(dev)

    def step(i):
        graphs[i % nsets].replay()

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    # then keep stepping, untimed, until the GPU has run the layer for about
    # 1.5 s: the timed region starts in the clock and power state of a long
    # run (dense layers reach the power limit within milliseconds, and its
    # throttle reason is reported only once the limit has held for a while).
    # The clock sampler starts first, so that the GPU does not idle between
    # these steps and the timed ones.
    clocks = ClockSampler(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
    t_warm = time.time() + 1.5
    i = args.warmup
    while time.time() < t_warm:
        step(i)
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clocks:
        clocks.mark("start")
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.mark("end")
    if pg:
        pg.barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
    # the same K steps as direct (eager) calls, for comparison, right after
    # the timed ones (the same clock and power state)
    ev0.record(stream)
    for i in range(args.steps):
        step_eager(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    eager_ms = ev0.elapsed_time(ev1) / args.steps
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(ms, pg, dev)
    value = w.T * world / (ms / 1e3)
    status = moe.device_status(ws)

    # ---- live stage times: the same steps through moe_layer_forward_profiled,
    # which records CUDA events on this stream at the stage boundaries
    st, stage_how = stage_times(moe, cfg, sets, nsets, ws, out, stream, dev,
                                max(10, min(args.steps, 200)))
    rctx = (router_context(moe, cfg, sets, nsets, ws, out, stream, dev)
            if work["tc_router"] else None)

    # ---- end to end through the host-buffer C call (pinned host x and y):
    # every step copies its tokens in, runs the layer and copies y (and
    # L_balance) out, through moe_layer_forward_host_pipelined as a serving
    # loop would run it: copies in, layers and copies out on three streams,
    # two workspaces (each with its three events) taken in turn, so one
    # step's copies overlap the neighbouring steps' layers while the layers
    # run one after another
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    e2e_ws = [ws, moe.workspace(cfg, dev, host_io=True)]
    e2e_ev = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]
    xh = [s["x"].cpu().pin_memory() for s in sets[:2]]
    yh = [torch.empty_like(xh[0]).pin_memory() for _ in range(2)]
    Lh = [torch.empty(1, dtype=torch.float32).pin_memory() for _ in range(2)]
    e2e_steps = max(10, min(args.steps, 500))

    def e2e_step(i):
        j = i % 2
        moe.layer_forward_host_pipelined(cfg, xh[i % 2], sets[i % nsets], yh[j], ws=e2e_ws[j],
                                         events=e2e_ev[j], copy_in=s_in, compute=stream,
                                         copy_out=s_out, L_host=Lh[j])

    # the same steady state as the timed device steps: about 1 s of untimed
    # steps first, clocks sampled during the timed ones
    e2e_clocks = ClockSampler(local_rank) if rank == 0 else None
    if e2e_clocks:
        e2e_clocks.start()
    t_warm = time.time() + 1.0
    i = 0
    while time.time() < t_warm or i < 4:
        e2e_step(i)
        i += 1
        if i % 8 == 0:
            s_out.synchronize()
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if e2e_clocks:
        e2e_clocks.mark("start")
    a.record(stream)
    s_in.wait_event(a)
    s_out.wait_event(a)
    for i in range(e2e_steps):
        e2e_step(i)
    done = torch.cuda.Event()
    done.record(s_out)
    stream.wait_event(done)
    b.record(stream)
    torch.cuda.synchronize(dev)
    if e2e_clocks:
        e2e_clocks.mark("end")
    e2e_clk = e2e_clocks.stop() if e2e_clocks else None
    e2e_ms = max_over_ranks(a.elapsed_time(b) / e2e_steps, pg, dev)
    bytes_x = cfg.T * cfg.d * sets[0]["x"].element_size()

    # ---- roofline of the dominant kernel (the grouped GEMM, two launches per
    # call): tensor-bound, or HBM-bound where streaming the experts' weights
    # takes longer than their flops (a decode-sized batch)
    gemm_ms = st["gemm1"] + st["gemm2"]
    achieved = work["gemm_flops"] / (gemm_ms / 1e3) / 1e12
    peak = peaks["bf16_tflops"]
    gemm_gbs = work["gemm_bytes"] / (gemm_ms / 1e3) / 1e9
    rec = traffic_record(source_sha(), w.name)
    g1_flops = work["gemm_flops"] * (w.nmat - 1) / w.nmat
    g2_flops = work["gemm_flops"] / w.nmat
    common = dict(kernel="grouped_gemm_tc_kernel (GEMM1 + GEMM2 launches per layer call)",
                  traffic=None if rec is None else rec["bytes_per_launch"],
                  algorithmic_flops_per_launch=work["gemm_flops"] / 2,
                  algorithmic_bytes_per_launch=work["gemm_bytes"] / 2,
                  launch_ms=gemm_ms / 2,
                  gemm1=dict(ms=st["gemm1"], tflops=g1_flops / (st["gemm1"] / 1e3) / 1e12),
                  gemm2=dict(ms=st["gemm2"], tflops=g2_flops / (st["gemm2"] / 1e3) / 1e12))
    if gemm_gbs / peaks["hbm_gbs"] > achieved / peak:
        roof = dict(bound="hbm", achieved=gemm_gbs, peak=peaks["hbm_gbs"], unit="GB/s",
                    frac=gemm_gbs / peaks["hbm_gbs"],
                    peak_source=f"{peaks['source']} HBM copy bandwidth (MEASURED_PEAKS.json)",
                    **common)
    else:
        roof = dict(bound="tensor", achieved=achieved, peak=peak, unit="TFLOP/s",
                    frac=achieved / peak,
                    peak_source=f"{peaks['source']} burst bf16 (MEASURED_PEAKS.json)",
                    frac_of_sustained=(achieved / peaks["bf16_tflops_sustained"]
                                       if peaks.get("bf16_tflops_sustained") else None),
                    frac_of_nominal_dense=achieved / NOMINAL_BF16_TFLOPS, **common)

    # ---- backward pass of the same layer call (moe_layer_backward), timed
    # alone with CUDA events after one forward call that left its state in ws
    bwd = None
    if w.shared_H == 0:
        bwd = time_backward(w, cfg, sets[0], ws, stream, dev, kept, max(3, args.steps // 20))
    if w.dtype == "bf16" and w.shared_H == 0:
        # a training forward that keeps the pre-activations, and its backward
        cfg_k = moe.config_from_workload(w, keep_preact=True)
        ws_k = moe.workspace(cfg_k, dev)
        bwd["keep_preact"] = time_backward(w, cfg_k, sets[0], ws_k, stream, dev, kept,
                                           max(3, args.steps // 20))
        del ws_k

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = time_oracle(w)
        cpu = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}

    if rank == 0:
        hbm = peaks["hbm_gbs"]
        comb_ms = st["combine_stats"] if w.k > 1 or not work["tc_router"] else None
        line = dict(
            metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps,
            warmup=args.warmup, ms_per_step=ms, eager_ms_per_step=eager_ms,
            higher_is_better=True, scaling="weak",
            vs_baseline=None, dtype="bf16" if w.dtype == "bf16" else "f32",
            data="synthetic (seeded N(0,1) tokens, N(0,1/fan_in) weights)",
            config=bench_config(w, cfg.capacity, kept, n_active, nsets, fp, world),
            roofline=roof,
            cpu_baseline=cpu,
            e2e=dict(value=w.T * world / (e2e_ms / 1e3), unit=UNIT, h2d_bytes_per_step=bytes_x,
                     d2h_bytes_per_step=bytes_x + 4, ms_per_step=e2e_ms,
                     call="moe_layer_forward_host_pipelined: copies in, layers and copies out on three streams, two workspaces in turn",
                     clocks=e2e_clk),
            gpu_launches=moe.lib().moe_layer_forward_launch_count(moe.ctypes.byref(cfg))
            * args.steps,
            clocks=clk,
            stages_ms=st,
            stages_roofline=dict(
                router_gbs=work["router_bytes"] / (st["router"] / 1e3) / 1e9,
                router_hbm_frac=work["router_bytes"] / (st["router"] / 1e3) / 1e9 / hbm,
                dispatch_gbs=work["dispatch_bytes"] / (st["dispatch"] / 1e3) / 1e9,
                dispatch_hbm_frac=work["dispatch_bytes"] / (st["dispatch"] / 1e3) / 1e9 / hbm,
                combine_gbs=(None if comb_ms is None
                             else work["combine_bytes"] / (comb_ms / 1e3) / 1e9),
                combine_hbm_frac=(None if comb_ms is None
                                  else work["combine_bytes"] / (comb_ms / 1e3) / 1e9 / hbm),
                gemm_tflops=achieved, gemm_frac_burst=achieved / peak,
                gemm_frac_nominal_dense=achieved / NOMINAL_BF16_TFLOPS,
                gemm_weight_gbs=work["gemm_bytes"] / (gemm_ms / 1e3) / 1e9,
                gemm_weight_hbm_frac=work["gemm_bytes"] / (gemm_ms / 1e3) / 1e9 / hbm,
                router_context_ms=rctx,
                router_alone_gbs=(None if not rctx
                                  else work["router_bytes"] / (rctx["alone"] / 1e3) / 1e9),
                router_alone_hbm_frac=(None if not rctx else
                                       work["router_bytes"] / (rctx["alone"] / 1e3) / 1e9 / hbm),
                hbm_peak_gbs=hbm,
                bytes=dict(router=work["router_bytes"], dispatch=work["dispatch_bytes"],
                           combine=work["combine_bytes"], gemm=work["gemm_bytes"]),
                note=(f"stage times from {stage_how}; router_context_ms: moe_router_topk "
                      f"alone, after a memset of y (the previous call's output lines dirty in "
                      f"L2, as after a combine), and an empty event pair, each between event "
                      f"nodes of a CUDA graph; dispatch = per-tile dispatch + gather "
                      f"launches; " + ("for k = 1 the combine runs inside GEMM2 (no combine "
                                       "stage)" if comb_ms is None else
                                       "combine = the combine launch"))),
            device_status=status[0],
            backward=bwd,
        )
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
