"""Benchmark of the quantized MoE expert path on GB300.

One step = the whole path over one batch of routed tokens: routing sort,
activation quantisation, grouped gate/up GEMM + SwiGLU (+ intermediate
quantisation), grouped down GEMM, weighted combine.  Default workload: the
MXFP4 x FP8 prefill layer at T=4096 (hidden 4096, 512 experts, top-10,
inter 1024).  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun each rank runs its own replica on its own tokens (weak
scaling; the layer needs no exchange between ranks).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_mixture_experts_moe_gb300 import inputs as gen  # noqa: E402

METRIC = "grouped-MoE prefill TFLOP/s & tokens/s at T=4096; % of tensor/HBM roofline"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 10**6  # GB300 L2

# DRAM bytes (read + write) of one stage-1 GEMM launch from an ncu capture,
# divided by that launch's algorithmic bytes.  Keyed by workload where the
# capture ran on the workload itself, else by scheme (a capture on a smaller
# workload with the same tokens per expert, whose traffic scales with the
# units processed).  An entry is removed when its kernel changes.
TRAFFIC_RATIO_GEMM1 = {
    # MXFP4, 512 tokens over 64 experts (~80 per expert, as at T=4096 over 512), 112-row tiles
    "mxfp4": (309262592 + 6259456) / 287375360,
    # MXFP4 TP4 shard (I 256) with stage 1 gathering x: 1024 tokens over 128 experts (~80 per expert,
    # as at T=4096 over 512), 112-row tiles
    "mxfp4_tp4_T4096": (147034368 + 3652352) / 146931712,
    # MXFP4 decode, 16-row tiles, on the workloads themselves
    "decode_T1": (45416448 + 161024) / 44568704,
    "decode_T4": (127116032 + 2582016) / 124797440,
    # W4A16 on the workload itself (T=2048)
    "w4a16": (298661120 + 18805248) / 234881024,
    # W8A8 and W4A8, 1024 tokens over 8 experts (~1024 per expert, as at T=8192 over 64)
    "w8a8": (160118016 + 29393152) / 96563200,
    "w4a8": (113460992 + 22359552) / 50425856,
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mxfp4_T4096")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU work for the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch the timed steps one by one instead of as a CUDA graph")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_workload(w, rank):
    """Rank r's replica: its own tokens (seed + 7919 r), the same expert weights."""
    return gen.Workload(w.name, w.scheme, w.T, w.H, w.E, w.k, w.I, w.routing, w.seed + 7919 * rank, w.wseed)


def max_over_ranks(value, world, device):
    """The largest of the ranks' values (every rank gets it); the value itself at world 1."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ algorithmic work

def weight_bytes_per_row(scheme, K):
    if scheme == "w4a16":
        return K // 2 + 2 * (K // 32)
    if scheme == "mxfp4":
        return K // 2 + K // 32
    if scheme == "w4a8":
        return K // 2 + 4
    return K + 4


def act_bytes_per_row(scheme, K):
    if scheme == "w4a16":
        return 2 * K
    if scheme == "mxfp4":
        return K + K // 32
    return K + 4


def touched_experts(ids, E):
    return int(np.count_nonzero(np.bincount(ids.reshape(-1), minlength=E)))


def algorithmic(w, ids):
    """Per-launch algorithmic bytes and flops of the two grouped GEMMs.
    Algorithmic bytes count what the method itself must move: the weights
    (with scales) of the experts the batch touches, plus the activations x
    read once (stage 1).  What the implementation moves on top (the
    expert-sorted copy of x read per routed pair, the intermediate h written
    and read, y written in slot order) is reported apart as overhead bytes."""
    Et = touched_experts(ids, w.E)
    P = w.P
    xa, ha = act_bytes_per_row(w.scheme, w.H), act_bytes_per_row(w.scheme, w.I)
    g1_bytes = Et * 2 * w.I * weight_bytes_per_row(w.scheme, w.H) + w.T * xa
    g2_bytes = Et * w.H * weight_bytes_per_row(w.scheme, w.I)
    g1_over = (P - w.T) * xa + P * ha  # per-pair activation rows beyond x once; h written
    g2_over = P * ha + P * w.H * 2     # h read; y written
    return dict(experts_touched=Et, gemm1_bytes=g1_bytes, gemm2_bytes=g2_bytes, gemm1_overhead_bytes=g1_over,
                gemm2_overhead_bytes=g2_over, gemm1_flops=4.0 * P * w.H * w.I, gemm2_flops=2.0 * P * w.H * w.I)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        # raw samples (the JSON line carries their summary); QMOE_CLOCKS_DIR keeps them elsewhere
        self.path = os.path.join(os.environ.get("QMOE_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"qmoe_clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=smax, reasons=sorted(reasons),
                    samples=len(sm))


# ------------------------------------------------------------------ CPU oracle baseline

def cpu_oracle_rate(w, d, seconds, rng_seed=0):
    """Times the oracle (as it stands) on a bounded sample of tokens of the
    same workload; returns (flops/s, tokens/s, cores, sample description)."""
    import oracle

    oracle.build()
    cores = oracle.num_threads()
    rng = np.random.default_rng(rng_seed)
    n = max(1, min(w.T, cores))
    toks = np.sort(rng.choice(w.T, n, replace=False))
    dims = (w.T, w.k, w.H, w.I, w.E)
    t0 = time.perf_counter()
    oracle.moe_forward(w.scheme, dims, d, tokens=toks)
    dt = time.perf_counter() - t0
    # grow the sample to about `seconds` of work
    want = int(min(w.T, max(n, n * seconds / max(dt, 1e-3))))
    if want > n:
        toks = np.sort(rng.choice(w.T, want, replace=False))
        t0 = time.perf_counter()
        oracle.moe_forward(w.scheme, dims, d, tokens=toks)
        dt = time.perf_counter() - t0
        n = want
    flops = 6.0 * n * w.k * w.H * w.I
    return flops / dt, n / dt, cores, f"{n} of {w.T} tokens (all k={w.k} pairs each), {dt:.1f} s wall"


# ------------------------------------------------------------------ reference arm (the CPU oracle)

def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    d = gen.make_all(w)
    import oracle

    oracle.build()
    cores = oracle.num_threads()
    rng = np.random.default_rng(1)
    dims = (w.T, w.k, w.H, w.I, w.E)
    # size each step to ~ (budget / (steps + warmup)) seconds of oracle work
    budget = 150.0
    per_step = budget / max(1, args.steps + args.warmup)
    probe = np.sort(rng.choice(w.T, max(1, min(w.T, cores)), replace=False))
    t0 = time.perf_counter()
    oracle.moe_forward(w.scheme, dims, d, tokens=probe)
    dt = time.perf_counter() - t0
    n = int(min(w.T, max(len(probe), len(probe) * per_step / max(dt, 1e-3))))
    times = []
    for i in range(args.warmup + args.steps):
        toks = np.sort(rng.choice(w.T, n, replace=False))
        t0 = time.perf_counter()
        oracle.moe_forward(w.scheme, dims, d, tokens=toks)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t = statistics.median(times)  # median step, as for our arm
    value = 6.0 * n * w.k * w.H * w.I / t / 1e12
    sample = f"{n} of {w.T} tokens per step (all k={w.k} pairs each)"
    line = dict(metric=METRIC, value=value, unit=UNIT, impl="reference", n_gpus=args.gpus, steps=args.steps,
                warmup=args.warmup, ms_per_step=t * 1e3, higher_is_better=True, scaling="weak", vs_baseline=None,
                dtype="f64", data="synthetic",
                config=dict(workload=w.name, scheme=w.scheme, T=w.T, H=w.H, E=w.E, k=w.k, I=w.I,
                            sample=sample),
                tokens_per_s=n / t,
                cpu_baseline=dict(value=value, unit=UNIT, cores=cores, kind="oracle", sample=sample),
                e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def run_ours(args, w):
    import torch

    from quantized_mixture_experts_moe_gb300 import binding as qb

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    qb.lib()

    # each rank: its own tokens (seed + rank), the same expert weights
    wr = rank_workload(w, rank)
    d = gen.make_all(wr)
    T, k, H, I, E, P = wr.T, wr.k, wr.H, wr.I, wr.E, wr.P

    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(dev)

    t = {key: to_dev(v) for key, v in d.items()}
    if w.scheme == "mxfp4":  # one-time weight preparation (not part of a step)
        t["w1"], t["w1_s"], t["w2"], t["w2_s"] = qb.prepack_mxfp4(t["w1"], t["w1_s"], t["w2"], t["w2_s"], H, I)
        torch.cuda.synchronize(dev)
    elif w.scheme == "w4a16":  # codes and scales pre-packed together
        t["w1"], t["w2"] = qb.prepack_w4a16(t["w1"], t["w1_s"], t["w2"], t["w2_s"], H, I)
        t["w1_s"] = t["w2_s"] = None
        torch.cuda.synchronize(dev)
    dims = qb.dims(T, k, H, I, E)

    # persistent buffers for the stage-by-stage step
    E_ = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
    counts, offsets = E_(E, torch.int32), E_(E + 1, torch.int32)
    sorted_ids, slot = E_(P, torch.int32), E_(P, torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = qb.alloc_workspace(qb.workspace_bytes(dims), dev)
    y = E_((P, H), torch.int16)  # bf16 bits
    out = E_((T, H), torch.int16)
    # MXFP4 stage 1 in the form the whole-layer call picks: token-major MX x gathered by the GEMM, or
    # the permuted MX tiles
    gathers = w.scheme == "mxfp4" and qb.mx_layer_gathers(dims)
    if w.scheme == "mxfp4":
        if gathers:
            xq, xs = E_((T, H), torch.uint8), E_((T, H // 32), torch.uint8)
        else:
            xt = E_(qb.mx_tiles_bytes(dims, H), torch.uint8)
        ht = E_(qb.mx_tiles_bytes(dims, I), torch.uint8)
    elif w.scheme in ("w8a8", "w4a8"):
        xt = E_(qb.w8a8_tiles_bytes(dims, H), torch.uint8)
        h32 = E_((P, I), torch.float32)
        ht = E_(qb.w8a8_tiles_bytes(dims, I), torch.uint8)
    else:
        xt = E_(qb.w4a16_x_tiles_bytes(dims), torch.uint8)
        ht = E_(qb.w4a16_h_tiles_bytes(dims), torch.uint8)
        h16 = E_(qb.w4a16_h16_tiles_bytes(dims), torch.uint8)

    ev = lambda: torch.cuda.Event(enable_timing=True)
    # Small batches touch fewer weight bytes than a few L2 capacities: the
    # timed steps then run behind an L2 flush (a 2xL2 write outside the
    # per-step events) so every step streams its weights from HBM.
    alg = algorithmic(wr, d["topk_ids"])
    touched = alg["gemm1_bytes"] + alg["gemm2_bytes"] + alg["gemm1_overhead_bytes"] + alg["gemm2_overhead_bytes"]
    flush = touched < 4 * L2_BYTES
    flush_buf = E_((2 * L2_BYTES,), torch.uint8) if flush else None

    def step(marks=None):
        qb.qmoe_align_sort(dims, t["topk_ids"], counts, offsets, sorted_ids, slot, status, ws)
        if gathers:
            qb.qmoe_quant_act_mxfp8(t["x"], xq, xs)
        elif w.scheme == "mxfp4":
            qb.qmoe_permute_quant_mxfp8(dims, t["x"], slot, offsets, xt, ws)
        elif w.scheme in ("w8a8", "w4a8"):
            qb.qmoe_permute_quant_int8(dims, t["x"], sorted_ids, offsets, xt, ws)
        else:
            qb.qmoe_permute_x_f16(dims, t["x"], sorted_ids, offsets, xt, ws)
        if marks:
            marks[0].record()
        if gathers:
            qb.qmoe_gemm1_swiglu_mxfp4_gather(dims, xq, xs, sorted_ids, t["w1"], t["w1_s"], offsets, ht, status, ws)
        elif w.scheme == "mxfp4":
            qb.qmoe_gemm1_swiglu_mxfp4(dims, xt, t["w1"], t["w1_s"], offsets, ht, status, ws)
        elif w.scheme == "w8a8":
            qb.qmoe_gemm1_swiglu_w8a8(dims, xt, t["w1"], t["w1_s"], offsets, h32, None, status, ws)
        elif w.scheme == "w4a8":
            qb.qmoe_gemm1_swiglu_w4a8(dims, xt, t["w1"], t["w1_s"], offsets, h32, None, status, ws)
        else:
            qb.qmoe_gemm1_swiglu_w4a16(dims, xt, t["w1"], offsets, ht, status, ws)
        if marks:
            marks[1].record()
        if w.scheme == "mxfp4":
            qb.qmoe_gemm2_mxfp4(dims, ht, t["w2"], t["w2_s"], offsets, y, status, ws)
        elif w.scheme == "w8a8":
            qb.qmoe_quant_tiles_int8_f32(dims, h32, offsets, ht, ws)
            qb.qmoe_gemm2_w8a8(dims, ht, t["w2"], t["w2_s"], offsets, y, None, status, ws)
        elif w.scheme == "w4a8":
            qb.qmoe_quant_tiles_int8_f32(dims, h32, offsets, ht, ws)
            qb.qmoe_gemm2_w4a8(dims, ht, t["w2"], t["w2_s"], offsets, y, None, status, ws)
        else:
            qb.qmoe_w4a16_h_to_f16(dims, ht, offsets, h16, ws)
            qb.qmoe_gemm2_w4a16(dims, h16, t["w2"], offsets, y, status, ws)
        if marks:
            marks[2].record()
        qb.qmoe_combine(dims, y, t["topk_w"], slot, out)

    # the kernels one timed step (one whole-layer call) launches, as the library counts them: routing
    # sort (one launch up to 2048 pairs, else two), activation quantisation, the two GEMMs, the
    # intermediate pass of the integer and W4A16 paths, and the combine
    launches_per_step = qb.forward_launches(dims, w.scheme)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    barrier()

    # The whole-layer call, as a user makes it (the GEMMs may then start
    # streaming weights before the kernel ahead of them completes).
    fws = qb.alloc_workspace(qb.forward_workspace_bytes(dims, w.scheme), dev)

    def fwd_step():
        qb.qmoe_moe_forward(w.scheme, dims, t["x"], t["topk_ids"], t["topk_w"], t["w1"], t["w1_s"], t["w2"], t["w2_s"],
                            out, status, fws)

    for _ in range(args.warmup):
        fwd_step()
    barrier()

    # Two replays of K steps, each one CUDA graph (a step is a handful of
    # dependent launches; at decode sizes launch gaps would otherwise cost as
    # much as the kernels):
    #   timed:  the K steps through qmoe_moe_forward, each step between two
    #           events -> ms_per_step, value;
    #   stages: the same K steps through the stage entry points with events
    #           around each GEMM -> the GEMMs' durations for the roofline.
    #           An event between two kernels costs a few microseconds (the
    #           next launch cannot overlap it), which is why the timed replay
    #           has none inside a step.
    K = args.steps
    ext = lambda: torch.cuda.Event(enable_timing=True, external=True)
    step_marks = [(ext(), ext()) for _ in range(K)]
    marks = [[ext() for _ in range(5)] for _ in range(K)]

    def timed_steps():
        for i in range(K):
            if flush:
                flush_buf.fill_(i & 0x7F)
            step_marks[i][0].record()
            fwd_step()
            step_marks[i][1].record()

    def stage_steps():
        for i in range(K):
            if flush:
                flush_buf.fill_(i & 0x7F)
            m = marks[i]
            m[0].record()
            step(m[1:4])
            m[4].record()

    def capture(body):
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream(dev)
        cs.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.graph(g, stream=cs):
            body()
        torch.cuda.current_stream(dev).wait_stream(cs)
        g.replay()  # uploads the graph: K more untimed warm-up steps
        barrier()
        return g

    graphs, launch = None, "eager"
    if not args.eager:
        try:
            graphs = (capture(timed_steps), capture(stage_steps))
            launch = ("one CUDA graph of the K timed steps (qmoe_moe_forward, dependent launches); GEMM times "
                      "from a second graph of the K steps through the stage calls with events around each GEMM")
        except Exception as ex:  # the eager loops below time the same launches
            torch.cuda.synchronize(dev)
            launch = f"eager (graph capture failed: {type(ex).__name__})"
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)
    barrier()
    if graphs is not None:
        graphs[0].replay()
    else:
        timed_steps()
    barrier()
    if graphs is not None:
        graphs[1].replay()
    else:
        stage_steps()
    barrier()
    clk = clocks.stop()
    # medians over the K timed steps
    ms = statistics.median(a_.elapsed_time(b_) for a_, b_ in step_marks)
    ms_stages = statistics.median(m[0].elapsed_time(m[4]) for m in marks)
    g1_ms = statistics.median(m[1].elapsed_time(m[2]) for m in marks)
    g2_ms = statistics.median(m[2].elapsed_time(m[3]) for m in marks)
    ms = max_over_ranks(ms, world, dev)
    assert int(status.item()) == 0, "device status flagged an error"
    pk = peaks()
    flops_step = wr.flops()
    value = flops_step * world / (ms * 1e-3) / 1e12
    tokens_per_s = T * world / (ms * 1e-3)
    # dominant kernel: the gate/up GEMM (2/3 of the weight bytes and flops)
    t_hbm = alg["gemm1_bytes"] / (pk["hbm"] * 1e9)
    fp8_peak = 2.0 * pk["bf16"]
    tensor_peak = fp8_peak if w.scheme == "mxfp4" else pk["bf16"]
    t_tc = alg["gemm1_flops"] / (tensor_peak * 1e12)
    # DRAM bytes per stage-1 launch from one ncu capture, scaled by units processed
    # (the capture's traffic / algorithmic bytes, times this launch's algorithmic bytes)
    ratio = TRAFFIC_RATIO_GEMM1.get(w.name)
    if ratio is None and not (w.scheme == "mxfp4" and (qb.tile_nmax(dims) == 16 or gathers)):
        ratio = TRAFFIC_RATIO_GEMM1.get(w.scheme)  # the scheme's capture: 112-row tiles, stage 1 from permuted tiles
    traffic = ratio * alg["gemm1_bytes"] if ratio else None
    if t_hbm >= t_tc:
        achieved = alg["gemm1_bytes"] / (g1_ms * 1e-3) / 1e9
        roof = dict(kernel="gemm1_swiglu", bound="hbm", achieved=achieved, peak=pk["hbm"], unit="GB/s",
                    frac=achieved / pk["hbm"], traffic=traffic,
                    peak_source=f"{pk['source']} (hbm_gbs, copy)")
    else:
        achieved = alg["gemm1_flops"] / (g1_ms * 1e-3) / 1e12
        src = "bf16 x2 (nominal fp8:bf16 ratio)" if w.scheme == "mxfp4" else "bf16"
        roof = dict(kernel="gemm1_swiglu", bound="tensor", achieved=achieved, peak=tensor_peak, unit="TFLOP/s",
                    frac=achieved / tensor_peak, traffic=traffic, peak_source=f"{pk['source']} {src}")
    roof["gemm1_ms"] = g1_ms
    roof["gemm2_ms"] = g2_ms
    roof["stage_calls_ms_per_step"] = ms_stages
    roof["gemm1_alg_bytes"] = alg["gemm1_bytes"]
    roof["gemm2_alg_bytes"] = alg["gemm2_bytes"]
    roof["overhead_bytes"] = dict(gemm1=alg["gemm1_overhead_bytes"], gemm2=alg["gemm2_overhead_bytes"])
    # stage 2 against HBM on its algorithmic bytes (W2 and scales), and with its overhead bytes added
    roof["gemm2_hbm_frac"] = alg["gemm2_bytes"] / (g2_ms * 1e-3) / 1e9 / pk["hbm"]
    roof["gemm2_hbm_frac_with_overhead"] = (alg["gemm2_bytes"] + alg["gemm2_overhead_bytes"]) / (g2_ms * 1e-3) / 1e9 / pk["hbm"]

    # end to end through the whole-layer entry point with host buffers
    e2e = None
    if not args.no_e2e:
        hx = t["x"].cpu().pin_memory()
        hid = t["topk_ids"].cpu().pin_memory()
        hw = t["topk_w"].cpu().pin_memory()
        # two slots of device inputs and outputs and of pinned results: step i
        # copies its inputs in and its result out on their own streams while
        # the neighbouring steps compute
        NSL = 2
        slots = [dict(x=torch.empty_like(t["x"]), ids=torch.empty_like(t["topk_ids"]), w=torch.empty_like(t["topk_w"]),
                      out=E_((T, H), torch.int16), hout=torch.empty((T, H), dtype=torch.int16).pin_memory())
                 for _ in range(NSL)]
        s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_done = [torch.cuda.Event() for _ in range(NSL)]
        comp_done = [torch.cuda.Event() for _ in range(NSL)]
        out_done = [torch.cuda.Event() for _ in range(NSL)]

        def e2e_step(i):
            b, j = slots[i % NSL], i % NSL
            with torch.cuda.stream(s_in):
                if i >= NSL:
                    s_in.wait_event(comp_done[j])  # step i - NSL has read this slot's inputs
                b["x"].copy_(hx, non_blocking=True)
                b["ids"].copy_(hid, non_blocking=True)
                b["w"].copy_(hw, non_blocking=True)
                in_done[j].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(in_done[j])
                if i >= NSL:
                    s_comp.wait_event(out_done[j])  # step i - NSL's result has left this slot
                qb.qmoe_moe_forward(w.scheme, dims, b["x"], b["ids"], b["w"], t["w1"], t["w1_s"], t["w2"], t["w2_s"],
                                    b["out"], status, fws)
                comp_done[j].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[j])
                b["hout"].copy_(b["out"], non_blocking=True)
                out_done[j].record(s_out)

        for i in range(args.warmup):
            e2e_step(i)
        barrier()
        if flush:
            # small steps: one step at a time behind an L2 flush, so no step finds its weights
            # in L2; the step (copies in, the forward call, copy out) replayed as a CUDA graph
            b = slots[0]

            def one_step():
                b["x"].copy_(hx, non_blocking=True)
                b["ids"].copy_(hid, non_blocking=True)
                b["w"].copy_(hw, non_blocking=True)
                qb.qmoe_moe_forward(w.scheme, dims, b["x"], b["ids"], b["w"], t["w1"], t["w1_s"], t["w2"], t["w2_s"],
                                    b["out"], status, fws)
                b["hout"].copy_(b["out"], non_blocking=True)

            run, how = one_step, "eager"
            if not args.eager:
                try:
                    g2 = torch.cuda.CUDAGraph()
                    cs = torch.cuda.Stream(dev)
                    cs.wait_stream(torch.cuda.current_stream(dev))
                    with torch.cuda.graph(g2, stream=cs):
                        one_step()
                    torch.cuda.current_stream(dev).wait_stream(cs)
                    g2.replay()
                    barrier()
                    run, how = g2.replay, "replayed as a CUDA graph"
                except Exception as ex:
                    torch.cuda.synchronize(dev)
                    how = f"eager (graph capture failed: {type(ex).__name__})"
            em = [(ev(), ev()) for _ in range(args.steps)]
            for i in range(args.steps):
                flush_buf.fill_(i & 0x7F)
                em[i][0].record()
                run()
                em[i][1].record()
            barrier()
            ems = statistics.median(a.elapsed_time(b_) for a, b_ in em)
            mode = f"one step at a time, L2 flushed between steps, {how}"
        else:
            s0, s1 = ev(), ev()
            s0.record(s_in)
            for i in range(args.steps):
                e2e_step(i)
            s1.record(s_out)
            barrier()
            ems = s0.elapsed_time(s1) / args.steps
            mode = "steps pipelined: copies on their own streams overlap the neighbouring steps' compute"
        barrier()
        ems = max_over_ranks(ems, world, dev)
        h2d = hx.numel() * 2 + hid.numel() * 4 + hw.numel() * 4
        e2e = dict(value=flops_step * world / (ems * 1e-3) / 1e12, unit=UNIT, ms_per_step=ems,
                   h2d_bytes_per_step=h2d, d2h_bytes_per_step=slots[0]["hout"].numel() * 2,
                   api=f"qmoe_moe_forward (C ABI) with pinned host buffers; {mode}")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        fl, tps, cores, sample = cpu_oracle_rate(wr, d, args.cpu_seconds)
        cpu = dict(value=fl / 1e12, unit=UNIT, cores=cores, kind="oracle", sample=sample, tokens_per_s=tps)

    if rank == 0:
        line = dict(metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps, warmup=args.warmup,
                    ms_per_step=ms, higher_is_better=True, scaling="weak", vs_baseline=None, dtype=dict(
                        mxfp4="e4m3 x e2m1 (fp32 accumulate)", w4a16="f16 x f16 (int4 dequantised on chip; fp32 accumulate)",
                        w8a8="int8 codes as exact f16 (exact int32 sums)",
                        w4a8="int4 x int8 codes as exact f16 (exact int32 sums)")[w.scheme], data="synthetic",
                    config=dict(workload=w.name, scheme=w.scheme, T=T, H=H, E=E, k=k, I=I,
                                experts_touched=alg["experts_touched"],
                                l2=(f"L2 flushed before every timed step (2 x L2 written outside the step's events): "
                                    f"the step touches only {touched / 1e9:.3f} GB"
                                    if flush else
                                    "inputs larger than L2: each step streams the touched experts' weights "
                                    f"({touched / 1e9:.2f} GB)"),
                                launch=launch,
                                stage1_input=("token-major MX x gathered by the GEMM" if gathers
                                              else "permuted MX tiles") if w.scheme == "mxfp4" else None,
                                parallelism=f"replicas x{world}"),
                    tokens_per_s=tokens_per_s, roofline=roof, cpu_baseline=cpu, e2e=e2e,
                    gpu_launches=launches_per_step * args.steps, clocks=clk)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def main():
    args = parse()
    w = gen.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
