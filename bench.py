"""Benchmark of the MoE expert-FFN forward on GB300.

One step = one moe_forward (route -> permute -> GEMM1+SwiGLU -> GEMM2 ->
combine) over one batch of synthetic tokens already resident in HBM.  The
default workload is the largest single-GPU one, the fine-grained skewed layer
(T=8192, H=7168, F=2048, E=256, top-8, bf16, Zipf(1.1) expert bias).  Its
22.5 GB of weights exceed the 129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload skewed|mixtral|decode|lowprec|tiny] [--T T] [--backward]

Roofline: the dominant kernel (GEMM1) against the tensor peak or HBM
bandwidth, whichever bounds it, and the whole layer against the slower of
6*T*k*H*F FLOPs at the tensor peak and its algorithmic bytes at HBM
bandwidth.  The tensor peak is the measured burst bf16 GEMM rate when the
timed region is shorter than SUSTAINED_AFTER_S seconds, else the measured
sustained rate; the fraction against the other peak is reported beside it.

Prints ONE JSON line on rank 0.  Under torchrun (N > 1) every rank runs its
own batch of T tokens with the same weights (weak scaling, no data-path
collective); the step time is the maximum over ranks.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload on this machine's host cores (rank 0 only).

--backward times moe_backward instead (dx, logit, dW1 and dW2 gradients of
the same workload, bf16), with its own metric line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import moe_inputs as mi  # noqa: E402

METRIC = "MoE layer fwd TFLOP/s & tokens/s at 1 GB300; % of tensor/HBM roofline"
METRIC_BWD = "MoE layer bwd TFLOP/s & tokens/s at 1 GB300; % of tensor roofline"
# Backward stages that are grouped GEMMs, with their algorithmic FLOPs in
# units of R*H*F (the pre-activation recompute is the backward's own choice:
# timed, but not counted in the layer's backward FLOPs)
BWD_GEMMS = {"gemm1_recompute": 4.0, "dgrad_h_swiglu": 2.0, "wgrad_w2": 2.0, "dgrad_x": 4.0,
             "wgrad_w1": 4.0}
BWD_KERNEL = ("grouped_gemm_bwd.cu", "grouped_gemm_bwd_kernel")
# GEMM kernel (file and instance) behind each moe_problem.kernel value
KERNEL_NAMES = {1: ("grouped_gemm.cu", "grouped_gemm_kernel<SwiGLU> (GEMM1, 1-CTA 128x256 tiles)"),
                2: ("grouped_gemm_swap.cu", "grouped_gemm_swap_kernel<SwiGLU,32> (GEMM1)"),
                6: ("grouped_gemm_swap2.cu",
                    "grouped_gemm_swap2_kernel<SwiGLU> (GEMM1, weight rows on M, cta_group::2)"),
                7: ("grouped_mlp_decode.cu",
                    "grouped_mlp_decode_kernel (GEMM1+SwiGLU, GEMM2 and combine in one launch)")}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# timed regions at least this long are compared with the sustained tensor peak
SUSTAINED_AFTER_S = 2.0
# dense FP8 over dense bf16 tensor rate (nominal GB300 figures, 4.5 / 2.25
# PFLOP/s): the FP8-activation layer's tensor peak is the measured bf16 peak
# times this
FP8_OVER_BF16 = 2.0
WORKLOADS = {
    "mixtral": (mi.MIXTRAL, "Mixtral-shaped MoE FFN layer: T=4096 H=4096 F=14336 E=8 top-2 bf16"),
    "skewed": (mi.SKEWED, "fine-grained skewed MoE FFN: T=8192 H=7168 F=2048 E=256 top-8 "
                          "bf16, Zipf(1.1) expert bias"),
    "decode": (mi.DECODE, "decode-sized MoE FFN: H=2048 F=768 E=128 top-8 bf16"),
    "tiny": (mi.TINY, "tiny MoE FFN: T=64 H=256 F=512 E=8 top-2 bf16"),
    "lowprec": (mi.LOWPREC, "low-precision MoE FFN: T=4096 H=7168 F=2048 E=256 top-8, FP8 "
                            "activations (fp32 scale / 128), NVFP4 weights, GLU interleave 32, "
                            "clamp 7, bf16 out"),
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="skewed")
    ap.add_argument("--T", type=int, default=0, help="override the token count")
    ap.add_argument("--E", type=int, default=0, help="override the expert count (profiling)")
    ap.add_argument("--k", type=int, default=0, help="override top-k (profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="time CUDA-graph replays of one forward (stage times from an eager pass)")
    ap.add_argument("--kernel", type=int, default=0,
                    help="moe_problem.kernel: 0 auto, 1 token-row tiles, 2 weight-row tiles")
    ap.add_argument("--wfmt", choices=["nvfp4", "mxfp4"], default="nvfp4",
                    help="FP4 weight format of the lowprec workload")
    ap.add_argument("--fusion", type=int, default=0,
                    help="moe_problem.fusion bits: 1 = TMA-gather A rows, 2 = combine in GEMM2")
    ap.add_argument("--backward", action="store_true",
                    help="time moe_backward (the layer's gradients) instead of the forward")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle sample")
    return ap.parse_args(argv)


def ncu_traffic(kernel_file: str, workload: str):
    """DRAM bytes (read + write) per GEMM1 launch from the committed ncu
    summary, if it was taken on the current source of the kernel's file."""
    import hashlib
    src = os.path.join(ROOT, "mixture_experts_ffn_permute_gb300", "csrc", kernel_file)
    table = os.path.join(ROOT, "profiles", "roofline_traffic.txt")
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        for line in open(table):
            f = line.split()
            if len(f) >= 5 and not line.startswith("#") and f[0] == sha and f[1] == workload:
                return float(f[3]) + float(f[4])
    except OSError:
        pass
    return None


def traffic_key(args) -> str:
    """Workload key of the ncu traffic table: the workload name, with -T<T>
    for a token-count override; other overrides have no entry."""
    if args.E or args.k:
        return "custom"
    return f"{args.workload}-T{args.T}" if args.T else args.workload


def gemm1_algorithmic_bytes(shape, used_experts: int, scale_block: int = 16) -> float:
    """HBM bytes GEMM1 cannot avoid: the gate/up weights of every expert that
    received tokens, the permuted activation rows read once and h written once.

    bf16: 2F*H*2 per expert, R*H*2 in, R*F*2 out.  FP8/FP4: 2F*H/2 packed
    E2M1 + 2F*H/scale_block scale bytes per expert (16 for NVFP4, 32 for MXFP4);
    the rows come in as f16 (the gather dequantises the E4M3 tokens), R*H*2,
    and h goes out as f16, R*F*2."""
    R, H, F = shape.R, shape.H, shape.F
    w = (2 * F * H / 2 + 2 * F * H / scale_block) if shape.lowprec else 2 * F * H * 2
    return used_experts * w + R * H * 2 + R * F * 2


def decode_mlp_algorithmic_bytes(shape, used_experts: int) -> float:
    """HBM bytes of the one-launch decode MLP: W1 (2F*H) and W2 (H*F) bf16 of
    every expert that received tokens, the permuted rows read once (R*H*2)
    and the combined output written once (T*H*2); h and y stay in L2."""
    R, H, F = shape.R, shape.H, shape.F
    return used_experts * 3 * F * H * 2 + R * H * 2 + shape.T * H * 2


def layer_algorithmic_bytes(shape, used_experts: int, scale_block: int = 16) -> float:
    """HBM bytes the whole layer cannot avoid: W1 and W2 of every expert that
    received tokens, x and the router logits read once, out written once.
    bf16 weights 3F*H*2 per expert and x T*H*2; FP8/FP4: 3F*H/2 packed E2M1 +
    3F*H/scale_block scale bytes + 2*4 bytes of expert scales per expert, x
    as E4M3 codes T*H plus fp32 scales T*H/128*4."""
    T, H, F, E = shape.T, shape.H, shape.F, shape.E
    if shape.lowprec:
        w = 3 * F * H / 2 + 3 * F * H / scale_block + 8
        xb = T * H + T * (H // 128) * 4
    else:
        w = 3 * F * H * 2
        xb = T * H * 2
    return used_experts * w + xb + T * E * 4 + T * H * 2


def tensor_peak(peaks, region_s: float, fp8: bool = False):
    """(peak TFLOP/s, its key, the other key) for a timed region of region_s
    seconds: burst below SUSTAINED_AFTER_S, sustained from there on; with fp8
    the bf16 figure times FP8_OVER_BF16 (keys prefixed "fp8=2x")."""
    if region_s < SUSTAINED_AFTER_S:
        key, other = "bf16_tflops", "bf16_tflops_sustained"
    else:
        key, other = "bf16_tflops_sustained", "bf16_tflops"
    if fp8:
        return peaks[key] * FP8_OVER_BF16, "fp8=2x" + key, "fp8=2x" + other
    return peaks[key], key, other


def peak_of(peaks, key: str) -> float:
    """The value of a key tensor_peak returned."""
    if key.startswith("fp8=2x"):
        return peaks[key[len("fp8=2x"):]] * FP8_OVER_BF16
    return peaks[key]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ distributed

def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, world: int, device) -> float:
    """Maximum of a per-rank scalar over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.sw_power_cap,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,power.limit")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.15)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.12)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons, power, limit = [], None, set(), [], None
        names = ["sw_power_cap", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            try:
                power.append(float(parts[2]))
            except ValueError:
                pass
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
            if len(parts) > 7:
                try:
                    limit = float(parts[7])
                except ValueError:
                    pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
               "samples": len(sm)}
        if power:
            out["power_w"] = round(statistics.median(power), 1)
        if limit is not None:
            out["power_limit_w"] = limit  # the board's enforced limit (sw_power_cap's bound)
        return out


# ------------------------------------------------------------------ CPU oracle

def oracle_sample(shape, inp_host, n_tokens: int):
    """Run the oracle on the first n tokens; returns (seconds, flops)."""
    import oracle
    lg = inp_host["logits"][:n_tokens]
    t0 = time.perf_counter()
    if shape.lowprec:
        h = inp_host
        oracle.moe_forward_lowprec(h["xq"][:n_tokens], h["xs"][:n_tokens], lg, h["w1q"], h["w1s"],
                                   h["w1g"], h["w2q"], h["w2s"], h["w2g"], shape.k,
                                   interleave=shape.glu_interleave, clamp=shape.swiglu_clamp,
                                   wfmt=h.get("_wfmt", oracle.WFMT_NVFP4))
    else:
        oracle.moe_forward(inp_host["x"][:n_tokens], lg, inp_host["w1"], inp_host["w2"], shape.k,
                           interleave=shape.glu_interleave, clamp=shape.swiglu_clamp)
    dt = time.perf_counter() - t0
    return dt, shape.with_T(n_tokens).flops()


def cpu_baseline(shape, inp_host, target_s: float):
    """Time the oracle on the first n tokens, n grown until the run takes about
    target_s seconds of wall time (capped at the whole batch)."""
    import oracle
    oracle.build()
    n = min(shape.T, 16)
    while True:
        dt, flops = oracle_sample(shape, inp_host, n)
        if dt >= target_s / 3 or n >= shape.T:
            break
        n = int(min(shape.T, max(2 * n, n * 0.8 * target_s / max(dt, 1e-6))))
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"first {n} of {shape.T} tokens of the same workload (fp64 oracle, "
                      f"{dt:.1f} s)"}


# ------------------------------------------------------------------ end to end

E2E_HOW = ("every step: inputs host->device from pinned memory, the layer call, its result "
           "device->host; the copies of step i+1 (in) and step i-1 (out) overlap step i's "
           "call (two buffer sets, separate copy streams), as a serving loop runs")


def timed_e2e(dev, stream, steps, warm, host_inputs, outs, run):
    """Milliseconds per step of a pipelined loop through the public API.  Step
    i's inputs go host->device on one stream while step i-1 computes, and its
    outputs come back on another while step i+1 computes; every step's bytes
    cross inside the timed region, which runs from an event before the first
    copy to the completion of the last read-back.  ``outs`` holds two sets of
    device output tensors; ``run(inputs, outs_set)`` enqueues one layer call on
    ``stream``."""
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dins = [[torch.empty(h.shape, dtype=h.dtype, device=dev) for h in host_inputs]
            for _ in range(2)]
    houts = [[torch.empty(o.shape, dtype=o.dtype, device="cpu").pin_memory() for o in outs[0]]
             for _ in range(2)]
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]

    def issue_h2d(i):
        b = i % 2
        with torch.cuda.stream(h2d):
            if i >= 2:
                h2d.wait_event(done[b])  # the call that read this buffer has finished
            for hs, dd in zip(host_inputs, dins[b]):
                dd.copy_(hs, non_blocking=True)
            copied[b].record(h2d)

    def step(i):
        b = i % 2
        stream.wait_event(copied[b])
        if i >= 2:
            stream.wait_event(read[b])  # this buffer's previous outputs are on the host
        run(dins[b], outs[b])
        done[b].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(done[b])
            for o, ho in zip(outs[b], houts[b]):
                ho.copy_(o, non_blocking=True)
            read[b].record(d2h)

    def loop(n, start=None):
        if start is not None:
            h2d.wait_event(start)
        issue_h2d(0)
        for i in range(n):
            if i + 1 < n:
                issue_h2d(i + 1)
            step(i)
        stream.wait_event(read[(n - 1) % 2])

    loop(max(warm, 2))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    loop(steps, start=e0)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


# ------------------------------------------------------------------ our arm

def bench_ours(args, shape, desc):
    import mixture_experts_ffn_permute_gb300 as moe
    from mixture_experts_ffn_permute_gb300 import _build

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    _build.build()
    moe.load()
    peaks, peak_src = load_peaks()

    # weights shared by all ranks (seed 0); each rank routes its own tokens
    p = moe.Problem.make(shape.T, shape.H, shape.F, shape.E, shape.k, True,
                         shape.glu_interleave, shape.swiglu_clamp, args.fusion, args.kernel,
                         moe.PREC_FP8_NVFP4 if shape.lowprec else moe.PREC_BF16)
    ws = moe.alloc_workspace(p, dev)
    out = torch.empty(shape.T, shape.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    mx = shape.lowprec and args.wfmt == "mxfp4"
    if shape.lowprec:
        lp = mi.make_lowprec_inputs(shape, 0, dev, wfmt=args.wfmt)
        if rank:
            lp.update({k: v for k, v in mi.make_lowprec_inputs(shape, rank, dev, weights=False).items()})
        prepared = torch.empty(moe.prepared_scales_size(p), dtype=torch.uint8, device=dev)
        if mx:  # MXFP4 scales re-encoded exactly, with per-expert fp32 scales
            lp["w1g"] = torch.empty(shape.E, dtype=torch.float32, device=dev)
            lp["w2g"] = torch.empty(shape.E, dtype=torch.float32, device=dev)
            moe.prepare_weights_mxfp4(p, lp["w1s"], lp["w2s"], prepared, lp["w1g"], lp["w2g"])
        else:
            moe.prepare_weights(p, lp["w1s"], lp["w2s"], prepared)
        x, logits = lp["xq"], lp["logits"]
        xs = lp["xs"]
        weight_bytes = sum(lp[n].numel() for n in ("w1q", "w1s", "w2q", "w2s"))

        def fwd(xx, ll):
            moe.forward_fp8_nvfp4(p, xx, xs, ll, lp["w1q"], lp["w1g"], lp["w2q"], lp["w2g"],
                                  prepared, out, ws)
    else:
        w1 = mi.make_w1(shape, 0, dev)
        w2 = mi.make_w2(shape, 0, dev)
        x = mi.make_x(shape, rank, dev)
        logits = mi.make_logits(shape, rank, dev)
        weight_bytes = 2 * (w1.numel() + w2.numel())

        def fwd(xx, ll):
            moe.forward(p, xx, ll, w1, w2, out, ws)

    def step():
        fwd(x, logits)

    moe.clear_device_status(ws)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    launches_per_step = moe.last_launch_count()
    K = args.steps

    # ---- device-resident timed region
    graph = None
    if args.graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        if graph is None:
            moe.stage_timing_begin(K)
        ev0.record(stream)
        for _ in range(K):
            if graph is None:
                step()
            else:
                graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        if graph is None:
            stages = moe.stage_timing_end()
        barrier(world)
    if graph is not None:  # per-stage times from an eager pass of the same call
        moe.stage_timing_begin(min(K, 200))
        for _ in range(min(K, 200)):
            step()
        stages = moe.stage_timing_end()
    ms_local = ev0.elapsed_time(ev1) / K
    status = moe.get_device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {moe.STATUS_NAMES.get(status, status)}")
    ms = reduce_max(ms_local, world, dev)
    sec = ms / 1e3

    # ---- end to end: pinned host inputs -> device -> forward -> host output
    # every per-step input (tokens, their scales when FP8, router logits) goes
    # host -> device each step; the weights are parameters and stay resident
    step_inputs = [x, logits] + ([xs] if shape.lowprec else [])
    hosts = [t.cpu().pin_memory() for t in step_inputs]
    outs2 = [[out], [torch.empty_like(out)]]

    def e2e_run(ins, o):
        if shape.lowprec:
            moe.forward_fp8_nvfp4(p, ins[0], ins[2], ins[1], lp["w1q"], lp["w1g"], lp["w2q"],
                                  lp["w2g"], prepared, o[0], ws)
        else:
            moe.forward(p, ins[0], ins[1], w1, w2, o[0], ws)

    K2 = max(3, K // 2)
    barrier(world)
    e2e_ms = reduce_max(timed_e2e(dev, stream, K2, 2, hosts, outs2, e2e_run), world, dev)
    barrier(world)

    # experts that received tokens (untimed extra call): their weights are the
    # bytes GEMM1 must stream
    tpe = torch.empty(shape.E, dtype=torch.int32, device=dev)
    if shape.lowprec:
        moe.forward_fp8_nvfp4(p, x, xs, logits, lp["w1q"], lp["w1g"], lp["w2q"], lp["w2g"],
                              prepared, out, ws, tokens_per_expert=tpe)
    else:
        moe.forward(p, x, logits, w1, w2, out, ws, tokens_per_expert=tpe)
    used_experts = int((tpe > 0).sum().item())

    flops = shape.flops()
    kid = moe.selected_kernel(p)
    kfile, kname = KERNEL_NAMES.get(kid, ("grouped_gemm_fp4.cu", "grouped_gemm_fp4_kernel<SwiGLU>"))
    if shape.lowprec:
        kfile, kname = "grouped_gemm_fp4.cu", "grouped_gemm_fp4_kernel<SwiGLU> (GEMM1, %s weights)" % (
            "MXFP4" if mx else "NVFP4")
    gemm1_ms = stages.get("gemm1_swiglu", float("nan"))
    gemm1_flops = 4.0 * shape.R * shape.H * shape.F
    gemm1_bytes = gemm1_algorithmic_bytes(shape, used_experts, 32 if mx else 16)
    if kid == 7 and not shape.lowprec:
        # one launch holds both GEMMs and the combine (its time is the
        # gemm1_swiglu stage; the gemm2 and combine stages read zero)
        gemm1_flops = 6.0 * shape.R * shape.H * shape.F
        gemm1_bytes = decode_mlp_algorithmic_bytes(shape, used_experts)
    region_s = K * sec
    # the FP8-activation layer against the FP8 tensor peak (its MMAs run
    # kind::f16 on exactly expanded operands, at the 16-bit rate)
    peak_val, peak_key, other_key = tensor_peak(peaks, region_s, fp8=shape.lowprec)
    gemm1_s = gemm1_ms / 1e3
    t_tensor = gemm1_flops / (peak_val * 1e12)
    t_hbm = gemm1_bytes / (peaks["hbm_gbs"] * 1e9)
    tensor_roof = {"bound": "tensor", "achieved": gemm1_flops / gemm1_s / 1e12,
                   "peak": peak_val, "unit": "TFLOP/s",
                   "peak_source": f"{peak_key} ({peak_src}; timed region {region_s:.2f} s)",
                   "frac_vs_" + other_key: gemm1_flops / gemm1_s / 1e12 / peak_of(peaks, other_key)}
    hbm_roof = {"bound": "hbm", "achieved": gemm1_bytes / gemm1_s / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "peak_source": f"hbm_gbs ({peak_src})"}
    for r in (tensor_roof, hbm_roof):
        r["frac"] = r["achieved"] / r["peak"]
    main, other = (hbm_roof, tensor_roof) if t_hbm > t_tensor else (tensor_roof, hbm_roof)
    # the whole layer: the slower of its FLOPs at the tensor peak and its
    # algorithmic bytes at HBM bandwidth, over the measured step time
    layer_bytes = layer_algorithmic_bytes(shape, used_experts, 32 if mx else 16)
    lt_tensor = flops / (peak_val * 1e12)
    lt_hbm = layer_bytes / (peaks["hbm_gbs"] * 1e9)
    layer_roof = {"bound": "tensor" if lt_tensor >= lt_hbm else "hbm",
                  "roof_ms": max(lt_tensor, lt_hbm) * 1e3, "ms_per_step": ms,
                  "frac": max(lt_tensor, lt_hbm) / sec,
                  "flops": flops, "bytes": layer_bytes,
                  "tensor_ms": lt_tensor * 1e3, "hbm_ms": lt_hbm * 1e3,
                  "peaks": {"tensor_tflops": peak_val, "tensor_key": peak_key,
                            "hbm_gbs": peaks["hbm_gbs"], "source": peak_src},
                  "frac_vs_" + other_key: max(flops / (peak_of(peaks, other_key) * 1e12),
                                              lt_hbm) / sec}
    line = {
        "metric": METRIC,
        "value": world * flops / sec / 1e12,
        "unit": "TFLOP/s",
        "tokens_per_s": world * shape.T / sec,
        "n_gpus": world,
        "steps": K,
        "warmup": max(args.warmup, 3),
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("fp8xmxfp4->f16 mma" if mx else "fp8xnvfp4->f16 mma") if shape.lowprec else "bf16",
        "data": "synthetic",
        "config": {"workload": desc, "T": shape.T, "H": shape.H, "F": shape.F, "E": shape.E,
                   "k": shape.k, "fusion": args.fusion, "kernel": args.kernel,
                   "precision": ("fp8-act/mxfp4-weight" if mx else "fp8-act/nvfp4-weight")
                   if shape.lowprec else "bf16",
                   "timing": "cuda-graph replay" if args.graph else "eager launches", "l2": "inputs larger than L2 (weights %.2f GB), no flush"
                   % (weight_bytes / 1e9)},
        "roofline": {"kernel": kname, "bound": main["bound"],
                     "achieved": main["achieved"], "peak": main["peak"], "unit": main["unit"],
                     "frac": main["frac"],
                     "traffic": ncu_traffic(kfile, traffic_key(args)),
                     "peak_source": main["peak_source"],
                     "algorithmic": {"flops": gemm1_flops, "bytes": gemm1_bytes,
                                     "experts_with_tokens": used_experts},
                     "other_roof": {k: other[k] for k in ("bound", "achieved", "peak", "unit",
                                                         "frac")}},
        "layer_roofline": layer_roof,
        "e2e": {"value": world * flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in step_inputs),
                "d2h_bytes_per_step": out.numel() * 2, "how": E2E_HOW},
        "gpu_launches": launches_per_step * K,
        "clocks": clk.summary(),
        "stages_ms": {k: round(v, 5) for k, v in stages.items() if not k.startswith("_")},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if shape.lowprec:
            host = {k: v.cpu() for k, v in lp.items()}
            host["_wfmt"] = 1 if mx else 0
        else:
            host = {"x": x.cpu(), "logits": logits.cpu(), "w1": w1.cpu(), "w2": w2.cpu()}
        line["cpu_baseline"] = cpu_baseline(shape, host, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ backward

def bwd_flops(shape) -> float:
    """Algorithmic FLOPs of the backward: dH 2RHF + dX 4RHF + dW2 2RHF + dW1 4RHF."""
    return 12.0 * shape.R * shape.H * shape.F


def oracle_bwd_sample(shape, host, n_tokens: int):
    """The oracle's per-token backward (recomputed forward, dh, dx and the
    route-weight gradients) on the first n tokens; returns (seconds, flops
    performed: 12 H F per route)."""
    import oracle
    idx, w = oracle.route_topk(host["logits"][:n_tokens], shape.k)
    t0 = time.perf_counter()
    oracle.backward_tokens(host["x"][:n_tokens], idx, w, host["w1"], host["w2"],
                           host["g"][:n_tokens], list(range(n_tokens)),
                           interleave=shape.glu_interleave, clamp=shape.swiglu_clamp)
    return time.perf_counter() - t0, 12.0 * n_tokens * shape.k * shape.H * shape.F


def cpu_baseline_bwd(shape, host, target_s: float):
    import oracle
    oracle.build()
    n = 1
    while True:
        dt, flops = oracle_bwd_sample(shape, host, n)
        if dt >= target_s / 3 or n >= shape.T:
            break
        n = int(min(shape.T, max(2 * n, n * 0.8 * target_s / max(dt, 1e-6))))
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"dx and route-weight gradients of the first {n} of {shape.T} tokens "
                      f"(fp64 oracle per-token backward, {dt:.1f} s)"}


def bench_backward(args, shape, desc):
    import mixture_experts_ffn_permute_gb300 as moe
    from mixture_experts_ffn_permute_gb300 import _build

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    _build.build()
    moe.load()
    peaks, peak_src = load_peaks()
    if shape.lowprec:
        raise SystemExit("the backward is bf16 only")
    p = moe.Problem.make(shape.T, shape.H, shape.F, shape.E, shape.k, True,
                         shape.glu_interleave, shape.swiglu_clamp)
    ws = moe.alloc_backward_workspace(p, dev)
    stream = torch.cuda.current_stream(dev)
    w1 = mi.make_w1(shape, 0, dev)
    w2 = mi.make_w2(shape, 0, dev)
    x = mi.make_x(shape, rank, dev)
    logits = mi.make_logits(shape, rank, dev)
    g = mi.make_grad_out(shape, rank, dev)
    dx = torch.empty_like(x)
    dl = torch.empty(shape.T, shape.E, dtype=torch.float32, device=dev)
    dw1 = torch.empty_like(w1)
    dw2 = torch.empty_like(w2)
    weight_bytes = 2 * (w1.numel() + w2.numel())

    def bwd(xx, ll, gg):
        moe.backward(p, xx, ll, w1, w2, gg, dx, dw1, dw2, ws, d_logits=dl)

    moe.clear_device_status(ws)
    for _ in range(max(args.warmup, 3)):
        bwd(x, logits, g)
    torch.cuda.synchronize()
    launches_per_step = moe.last_launch_count()
    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        moe.stage_timing_begin(K)
        ev0.record(stream)
        for _ in range(K):
            bwd(x, logits, g)
        ev1.record(stream)
        torch.cuda.synchronize()
        stages = moe.stage_timing_end()
        barrier(world)
    status = moe.get_device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {moe.STATUS_NAMES.get(status, status)}")
    ms = reduce_max(ev0.elapsed_time(ev1) / K, world, dev)
    sec = ms / 1e3

    # end to end: x, logits and dOut from pinned host memory each step, dx and
    # the logit gradient back; the weight gradients stay on the device (the
    # optimizer's input)
    step_inputs = [x, logits, g]
    hosts = [t.cpu().pin_memory() for t in step_inputs]
    outs = [dx, dl]
    outs2 = [outs, [torch.empty_like(dx), torch.empty_like(dl)]]

    def e2e_run(ins, o):
        moe.backward(p, ins[0], ins[1], w1, w2, ins[2], o[0], dw1, dw2, ws, d_logits=o[1])

    K2 = max(3, K // 2)
    barrier(world)
    e2e_ms = reduce_max(timed_e2e(dev, stream, K2, 2, hosts, outs2, e2e_run), world, dev)
    barrier(world)

    flops = bwd_flops(shape)
    rhf = float(shape.R) * shape.H * shape.F
    gemm_ms = {k: stages[k] for k in BWD_GEMMS if k in stages}
    top = max(gemm_ms, key=gemm_ms.get)
    top_flops = BWD_GEMMS[top] * rhf
    peak_val, peak_key, other_key = tensor_peak(peaks, K * sec)
    achieved = top_flops / (gemm_ms[top] / 1e3) / 1e12
    wl = ("backward-" + args.workload) if not args.T and not args.E and not args.k else "custom"
    line = {
        "metric": METRIC_BWD,
        "value": world * flops / sec / 1e12,
        "unit": "TFLOP/s",
        "tokens_per_s": world * shape.T / sec,
        "n_gpus": world,
        "steps": K,
        "warmup": max(args.warmup, 3),
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": desc + " -- backward (dx, d logits, dW1, dW2)", "T": shape.T,
                   "H": shape.H, "F": shape.F, "E": shape.E, "k": shape.k,
                   "timing": "eager launches",
                   "l2": "inputs larger than L2 (weights %.2f GB), no flush" % (weight_bytes / 1e9),
                   "flops": "12*R*H*F (dH 2, dX 4, dW2 2, dW1 4); the 4*R*H*F recompute of "
                            "the pre-activations is timed but not counted"},
        "roofline": {"kernel": f"{BWD_KERNEL[1]} ({top})", "bound": "tensor",
                     "achieved": achieved, "peak": peak_val, "unit": "TFLOP/s",
                     "frac": achieved / peak_val,
                     "frac_vs_" + other_key: achieved / peaks[other_key],
                     "traffic": ncu_traffic(BWD_KERNEL[0], wl + ":" + top),
                     "peak_source": f"{peak_key} ({peak_src})",
                     "algorithmic": {"flops": top_flops}},
        "e2e": {"value": world * flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in step_inputs),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in outs),
                "how": E2E_HOW},
        "gpu_launches": launches_per_step * K,
        "clocks": clk.summary(),
        "stages_ms": {k: round(v, 5) for k, v in stages.items() if not k.startswith("_")},
        "stage_tflops": {k: round(BWD_GEMMS[k] * rhf / (v / 1e3) / 1e12, 1)
                         for k, v in gemm_ms.items()},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = {"x": x.cpu(), "logits": logits.cpu(), "w1": w1.cpu(), "w2": w2.cpu(),
                "g": g.cpu()}
        line["cpu_baseline"] = cpu_baseline_bwd(shape, host, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def bench_reference_backward(args, shape, desc):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    import oracle
    oracle.build()
    n_max = 16
    logits = mi.make_logits(shape, 0)[:n_max]
    idx, _ = oracle.route_topk(logits, shape.k)
    used = sorted(set(idx.ravel().tolist()))
    w1 = [None] * shape.E
    w2 = [None] * shape.E
    for e in used:  # same distributions as moe_inputs, drawn per used expert
        gen = torch.Generator().manual_seed(1000 + e)
        w1[e] = torch.randn(2 * shape.F, shape.H, generator=gen).mul_(
            1 / math.sqrt(shape.H)).to(torch.bfloat16)
        w2[e] = torch.randn(shape.H, shape.F, generator=gen).mul_(
            1 / math.sqrt(shape.F)).to(torch.bfloat16)
    host = {"x": mi.make_x(shape.with_T(n_max), 0), "logits": logits, "w1": w1, "w2": w2,
            "g": mi.make_grad_out(shape.with_T(n_max), 0)}
    steps, warm = args.steps, max(args.warmup, 1)
    dt1, _ = oracle_bwd_sample(shape, host, 1)
    budget = 150.0 / (steps + warm)
    n = int(max(1, min(n_max, math.floor(budget / max(dt1, 1e-6)))))
    for _ in range(warm - 1):
        oracle_bwd_sample(shape, host, n)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(steps):
        _, flops = oracle_bwd_sample(shape, host, n)
    dt = (time.perf_counter() - t0) / steps
    val = flops / dt / 1e12
    line = {
        "metric": METRIC_BWD, "impl": "reference", "value": val, "unit": "TFLOP/s",
        "tokens_per_s": n / dt, "n_gpus": world, "steps": steps, "warmup": warm,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc + " -- backward (dx, d logits, dW1, dW2)", "T": shape.T,
                   "H": shape.H, "F": shape.F, "E": shape.E, "k": shape.k},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"dx and route-weight gradients of the first {n} of "
                                   f"{shape.T} tokens per step (fp64 oracle)"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ reference arm

def bench_reference(args, shape, desc):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    import oracle
    oracle.build()
    # Inputs of the same workload on the host; only the experts the sample
    # routes to are materialised (the oracle takes per-expert weights).
    logits = mi.make_logits(shape, 0)[:64]
    idx, _ = oracle.route_topk(logits, shape.k)
    used = sorted(set(idx.ravel().tolist()))
    if shape.lowprec:
        xq, xs = mi.quantize_fp8_rows(mi.make_x(shape.with_T(64), 0).float())
        host = {"logits": logits, "xq": xq, "xs": xs}
        for name, rows, cols in (("w1", 2 * shape.F, shape.H), ("w2", shape.H, shape.F)):
            qs, ss = [None] * shape.E, [None] * shape.E
            gs = torch.ones(shape.E)
            for e in used:  # same distributions as moe_inputs, drawn per used expert
                g = torch.Generator().manual_seed(1000 + e + (0 if name == "w1" else 5000))
                wf = torch.randn(rows, cols, generator=g).mul_(1 / math.sqrt(cols))
                qs[e], ss[e], gs[e] = mi.quantize_nvfp4(wf)
            host[name + "q"], host[name + "s"], host[name + "g"] = qs, ss, gs
    else:
        w1 = [None] * shape.E
        w2 = [None] * shape.E
        for e in used:  # same distributions as moe_inputs, drawn per used expert
            g = torch.Generator().manual_seed(1000 + e)
            w1[e] = torch.randn(2 * shape.F, shape.H, generator=g).mul_(
                1 / math.sqrt(shape.H)).to(torch.bfloat16)
            w2[e] = torch.randn(shape.H, shape.F, generator=g).mul_(
                1 / math.sqrt(shape.F)).to(torch.bfloat16)
        host = {"x": mi.make_x(shape.with_T(64), 0), "logits": logits, "w1": w1, "w2": w2}
    steps, warm = args.steps, max(args.warmup, 1)
    dt1, _ = oracle_sample(shape, host, 1)
    budget = 150.0 / (steps + warm)
    n = int(max(1, min(64, math.floor(budget / max(dt1, 1e-6)))))
    for _ in range(warm - 1):
        oracle_sample(shape, host, n)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_sample(shape, host, n)
    dt = (time.perf_counter() - t0) / steps
    flops = shape.with_T(n).flops()
    val = flops / dt / 1e12
    line = {
        "metric": METRIC, "impl": "reference", "value": val, "unit": "TFLOP/s",
        "tokens_per_s": n / dt, "n_gpus": world, "steps": steps, "warmup": warm,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, "T": shape.T, "H": shape.H, "F": shape.F, "E": shape.E,
                   "k": shape.k},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"first {n} of {shape.T} tokens per step (fp64 oracle)"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    shape, desc = WORKLOADS[args.workload]
    if args.E or args.k:
        import dataclasses
        shape = dataclasses.replace(shape, E=args.E or shape.E, k=args.k or shape.k)
        desc = desc + f" (E={shape.E}, k={shape.k})"
    if args.T:
        shape = shape.with_T(args.T)
        desc = desc + f" (T={args.T})"
    elif args.workload == "decode":
        desc = desc + f" T={shape.T}"
    if shape.lowprec and args.wfmt == "mxfp4":
        desc = desc.replace("NVFP4", "MXFP4")
    if args.backward:
        (bench_reference_backward if args.impl == "reference" else bench_backward)(
            args, shape, desc)
    elif args.impl == "reference":
        bench_reference(args, shape, desc)
    else:
        bench_ours(args, shape, desc)


if __name__ == "__main__":
    main()
