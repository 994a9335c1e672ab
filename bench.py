"""Benchmark: one training step of the dropless MoE expert layer (route + forward +
backward over one 16,384-token batch) on a GB300, through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

Prints one JSON line (rank 0).  `value` is whole-job tokens/s with inputs
resident in HBM; `e2e` is the same step with host buffers (pinned host ->
device copies of x, logits, dy and device -> host copies of out, dx, d_logits
inside the timed region).  Each timed step is bracketed by CUDA events on the
library's stream; an L2 flush (256 MiB write) runs between steps, outside the
events.  `roofline` covers the kernel with the largest share of step time, timed
live with per-kernel events.  `cpu_baseline` is the fp64 oracle timed on this
host's cores on a bounded sub-batch.  Also reported: `ckpt_2f_plus_b_ms`, the
activation-checkpointed step (route, a forward that keeps no activations, the
recompute of what the backward reads, the backward); `no_l2_flush`, the step
without the flush; `router_projection`, the router's linear layer in front of
the layer (logits = x . W_r and its backward), totals and per kernel.

--impl reference times that oracle alone (the only reference this method has:
the pages publish no runnable code), on bounded sub-batches of the same workload.

N > 1 (torchrun): every rank runs an independent replica of the workload on its
own GPU (the layer has no cross-GPU exchange on one GPU's worth of experts);
`value` sums tokens over ranks and divides by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
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

from dropless_mixture_experts_top_gb300 import synth  # noqa: E402

METRIC = "MoE layer fwd+bwd ms, TFLOPS & tokens/s on 1 GB300; % of dense tensor peak"
DEFAULT_WORKLOAD = "qwen3_30b_a3b_layer_t16384"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s) applied to the measured bf16 peak


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_work(shape):
    """Algorithmic work per launch: (bound, amount, unit) -- flops for the grouped
    GEMMs ("tensor" bf16, "tensor_fp8" MXFP8), bytes each memory-bound kernel must
    move at minimum (an MXFP8 quantiser reads bf16 and writes one code byte per
    element plus one scale byte per 32)."""
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    M = T * k
    MHI = float(M) * H * I
    q = lambda n: ("hbm", n * (2 + 1 + 1 / 32), "B")
    return {
        "mx_pad_offsets": ("hbm", (E + 1) * 8.0, "B"),
        "mx_pad_offsets_fwd": ("hbm", (E + 1) * 8.0, "B"),
        # mxfp8 forward: x along H; the weights along their middle axis (gate and up, down)
        # the dispatch with x quantised along H: reads x, writes its codes to every permuted row
        "permute_quant_x": ("hbm", T * H * 2 + M * H * (1 + 1 / 32) + M * 4, "B"),
        "mx_zero_pad_rows": ("hbm", 127 * E * H * (1 + 1 / 32) / 2, "B"),
        # each weight read once, written along both axes
        "mx_quant_W_gateup_fwd": ("hbm", 2 * E * H * I * (2 + 2 * (1 + 1 / 32)), "B"),
        "mx_quant_W_down_fwd": ("hbm", E * I * H * (2 + 2 * (1 + 1 / 32)), "B"),
        "mx_gemm_gateup_swiglu": ("tensor_fp8", 4 * MHI, "flop"),
        "mx_gemm_down": ("tensor_fp8", 2 * MHI, "flop"),
        # dy read once (through each permuted row's token), Y read for the router
        # gradient, codes and scales written along H and along tokens, g in partials
        "mx_dy_quant_gdot": ("hbm", T * H * 2 + M * H * 2 + 2 * M * H * (1 + 1 / 32) + M * 4 * 4.0, "B"),
        "mx_quantT_x": q(M * H),
        # fp8_bwd forward: x gathered into x_perm (bf16) and quantised along tokens, one pass
        "permute_rows_quantT_x": ("hbm", T * H * 2 + M * H * 2.0 + M * H * (1 + 1 / 32) + M * 4, "B"),
        "mx_gemm_dA_dswiglu": ("tensor_fp8", 2 * MHI, "flop"),
        "mx_gemm_dX": ("tensor_fp8", 4 * MHI, "flop"),
        "mx_gemm_dW_down": ("tensor_fp8", 2 * MHI, "flop"),
        "mx_gemm_dW_gateup": ("tensor_fp8", 4 * MHI, "flop"),
        "route_topk": ("hbm", T * E * 4 + T * k * 12.0, "B"),
        "route_index": ("hbm", T * k * 12.0 + M * 12.0, "B"),
        "permute_rows": ("hbm", T * H * 2 + M * H * 2.0 + M * 4, "B"),
        "gemm_gateup_swiglu": ("tensor", 4 * MHI, "flop"),
        "gemm_down": ("tensor", 2 * MHI, "flop"),
        "combine": ("hbm", M * H * 2 + T * H * 2.0 + M * 8, "B"),
        # bf16 backward: dy permuted (as x), the router gradient from the dA GEMM's partials
        "permute_dy": ("hbm", T * H * 2 + M * H * 2.0 + M * 4, "B"),
        "router_grad": ("hbm", M * 2 * ((I + 255) // 256) * 4.0 + T * E * 4 + M * 16, "B"),
        "gemm_dA_dswiglu": ("tensor", 2 * MHI, "flop"),
        "gemm_dX": ("tensor", 4 * MHI, "flop"),
        "unpermute_sum": ("hbm", M * H * 2 + T * H * 2.0 + M * 4, "B"),
        "gemm_dW_down": ("tensor", 2 * MHI, "flop"),
        "gemm_dW_gateup": ("tensor", 4 * MHI, "flop"),
    }


def gemm_bytes(shape, precision="bf16"):
    """Algorithmic HBM bytes per launch of each grouped GEMM: every operand read
    once and every output written once (bf16 2 B; MXFP8 one code byte per element
    plus one scale byte per 32).  Against the measured HBM bandwidth this gives a
    GEMM's second roof: the one that binds is the larger of flops / tensor peak and
    bytes / HBM bandwidth (the fused dSwiGLU GEMM, which reads G and U and writes
    dG and dU, is HBM-bound at the 30B shape).  Before an MXFP8 backward the two
    bf16 forward GEMMs also write the weights' codes, and GEMM1 w * A as codes
    along tokens instead of bf16."""
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    M = float(T * k)
    W = float(E) * H * I  # one expert weight tensor's elements
    c = 1 + 1 / 32
    np_ = 2 * ((I + 255) // 256)
    fp8b = precision == "fp8_bwd"
    return {
        "gemm_gateup_swiglu": M * H * 2 + 2 * W * 2 + (3 * M * I * 2 + M * I * c + 2 * W * c if fp8b else 4 * M * I * 2),
        "gemm_down": M * I * 2 + W * 2 + M * H * 2 + (W * c if fp8b else 0.0),
        "gemm_dA_dswiglu": M * H * 2 + W * 2 + 2 * M * I * 2 + 2 * M * I * 2 + M * np_ * 4,
        "gemm_dX": 2 * M * I * 2 + 2 * W * 2 + M * H * 2,
        "gemm_dW_down": M * I * 2 + M * H * 2 + W * 2,
        "gemm_dW_gateup": M * H * 2 + 2 * M * I * 2 + 2 * W * 2,
        "mx_gemm_gateup_swiglu": M * H * c + 2 * W * c + 4 * M * I * 2 + M * I * c,
        "mx_gemm_down": M * I * c + W * c + M * H * 2,
        # codes of dG and dU along I and along tokens
        "mx_gemm_dA_dswiglu": M * H * c + W * c + 2 * M * I * 2 + 4 * M * I * c,
        "mx_gemm_dX": 2 * M * I * c + 2 * W * c + M * H * 2,
        "mx_gemm_dW_down": M * I * c + M * H * c + W * 2,
        "mx_gemm_dW_gateup": M * H * c + 2 * M * I * c + 2 * W * 2,
    }


def launches_in_timed_region(labels, steps_hooked, steps):
    """Kernels the library launched in the timed region: the timing hook's labels of
    the hooked steps, scaled to all steps (every step launches the same kernels).
    Four labels cover two kernels each: the ragged-K GEMMs (their per-expert tensor
    maps, then the GEMM) and the mxfp8 forward's gate and up weight quantisers."""
    per_label = {"gemm_dW_down": 2, "gemm_dW_gateup": 2, "router_gemm_dW": 2, "mx_quant_W_gateup_fwd": 2}
    n = sum(per_label.get(lab, 1) for lab in labels)
    return n * steps // max(steps_hooked, 1)


def kernel_source(label):
    """The .cu file that defines the kernel behind a timing label."""
    if label.startswith("mx_gemm_"):
        return "gemm_mx.cu"
    if label.startswith("gemm_"):
        return "gemm.cu"
    if label.startswith("mx_"):
        return "mxfp8.cu"
    if label.startswith("route_"):
        return "route.cu"
    return "gather.cu"  # permute_rows, permute_dy, combine, router_grad, unpermute_sum


def source_hash(label):
    """Hash of a kernel's source and the headers it includes: a recorded traffic
    figure is valid only while this is unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dropless_mixture_experts_top_gb300", "csrc")
    for n in (kernel_source(label), "common.cuh", "epilogue.cuh", "internal.h", "mxfp8.cuh"):
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel, workload):
    """dram bytes per launch from a committed ncu summary, if taken on the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(workload, {}).get(kernel)
    if not ent or ent.get("source_hash") != source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [c.strip() for c in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- CPU oracle leg

def oracle_sub_batch_step(O, w, inp, S):
    """The oracle's whole step (route, forward, backward incl. weight gradients) on the
    first S tokens of the workload.  Returns seconds."""
    shape = w.shape
    sub = synth.MoEShape(T=S, H=shape.H, I=shape.I, E=shape.E, k=shape.k)
    t0 = time.perf_counter()
    idx, wts = O.route(inp["logits"][:S], shape.k)
    O.dispatch(idx, shape.E)
    O.forward(sub, inp["x"][:S], idx, wts, inp["W_gate"], inp["W_up"], inp["W_down"],
              fwd_quant=w.precision == "mxfp8")
    quant = w.precision in ("fp8_bwd", "mxfp8")
    fq = w.precision == "mxfp8"
    qW = O.quant_weights(inp["W_gate"], inp["W_up"], inp["W_down"]) if quant else None
    fW = O.quant_weights_fwd(inp["W_gate"], inp["W_up"], inp["W_down"]) if fq else None
    O.backward_tokens(sub, inp["x"][:S], inp["logits"][:S], idx, wts, inp["W_gate"], inp["W_up"],
                      inp["W_down"], inp["dy"][:S], quant=quant, qW=qW, fwd_quant=fq, fW=fW)
    O.dw_full(sub, inp["x"][:S], idx, wts, inp["W_gate"], inp["W_up"], inp["W_down"], inp["dy"][:S],
              quant=quant, qW=qW, fwd_quant=fq, fW=fW)
    return time.perf_counter() - t0


def size_oracle_sample(O, w, inp, target_s):
    """Tokens per sub-batch so that one oracle step takes about target_s seconds
    (two probes fit a fixed cost plus a per-token cost)."""
    p1, p2 = 16, 64
    t1 = oracle_sub_batch_step(O, w, inp, p1)
    t2 = oracle_sub_batch_step(O, w, inp, p2)
    per_tok = max((t2 - t1) / (p2 - p1), 1e-6)
    fixed = max(t1 - per_tok * p1, 0.0)
    S = int((target_s - fixed) / per_tok)
    return max(p2, min(w.shape.T, S)), per_tok


def cpu_cores():
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n else (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count())


def cpu_baseline(w, inp, target_s=15.0):
    from oracle import oracle as O
    S, _ = size_oracle_sample(O, w, inp, target_s)
    dt = oracle_sub_batch_step(O, w, inp, S)
    return {"value": S / dt, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"first {S} of {w.shape.T} tokens through the oracle's full step (route, forward, "
                      f"backward with weight gradients), {dt:.1f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from oracle import oracle as O
    O.build()
    w = workload_of(args)
    inp = synth.make_inputs(w)
    budget = 150.0 / max(1, args.steps + args.warmup)
    S, _ = size_oracle_sample(O, w, inp, budget)
    for _ in range(args.warmup):
        oracle_sub_batch_step(O, w, inp, S)
    times = [oracle_sub_batch_step(O, w, inp, S) for _ in range(args.steps)]
    sec = statistics.mean(times)
    value = S / sec
    shape = w.shape
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": shape.T, "H": shape.H, "I": shape.I, "E": shape.E, "k": shape.k,
                   "precision": w.precision, "sample_tokens_per_step": S},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"first {S} of {shape.T} tokens per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

def workload_of(args):
    """The named workload; --tokens shrinks T (small profiling cases only, never the bench line)."""
    import dataclasses
    w = synth.WORKLOADS[args.workload]
    if args.tokens:
        shape = dataclasses.replace(w.shape, T=args.tokens)
        w = dataclasses.replace(w, name=f"{w.name}_T{args.tokens}", shape=shape)
    return w


def ensure_built(rank, dist=None):
    """Rank 0 builds the in-tree library (a no-op when it is current); with
    several ranks (one process per GPU, one shared build) the others wait for
    it at a barrier."""
    from dropless_mixture_experts_top_gb300 import _build
    if rank == 0:
        _build.build()
    if dist is not None:
        dist.barrier()


def max_over_ranks(value, dist, device):
    """The largest of the ranks' values: every rank times its own replica, the
    whole job is as slow as the slowest (a no-op on one rank)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    ensure_built(rank, dist)
    from dropless_mixture_experts_top_gb300 import moe

    w = workload_of(args)
    shape = w.shape
    inp = synth.make_inputs(w)
    dev = torch.device("cuda", local)
    d = {n: torch.from_numpy(inp[n].view(np.int16)).to(dev) for n in ("x", "W_gate", "W_up", "W_down", "dy")}
    d["logits"] = torch.from_numpy(inp["logits"]).to(dev)
    layer = moe.MoELayer(shape, precision=w.precision, device=dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    grads = None

    def step():
        nonlocal grads
        layer.route(d["logits"], stream)
        layer.forward(d["x"], d["W_gate"], d["W_up"], d["W_down"], out=out, stream=stream)
        ev_mid.record(stream)
        grads = layer.backward(d["dy"], d["x"], d["W_gate"], d["W_up"], d["W_down"], grads=grads, stream=stream)

    out = torch.empty((shape.T, shape.H), dtype=torch.int16, device=dev)
    ev_mid = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            step()
    torch.cuda.synchronize()
    st = layer.status(stream)
    if any(st.values()):
        raise RuntimeError(f"device status after warm-up: {st}")

    # timed region: per-step events; per-kernel events through the library's
    # timing hook on the last KH steps only (two events around every kernel are
    # stream work a user does not pay for; the other steps run without them)
    K = args.steps
    KH = min(K, 2)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    cap = 64 * KH
    kev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * cap)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            for i in range(K):
                if i == K - KH:
                    moe.timing_attach(kev)
                flush.zero_()
                starts[i].record(stream)
                ev_mid = mids[i]
                step()
                ends[i].record(stream)
        torch.cuda.synchronize()
        nk = moe.timing_count()
        labels = [moe.timing_label(i) for i in range(nk)]
        moe.timing_attach(None)
    if dist:
        dist.barrier()
    fwd = [starts[i].elapsed_time(mids[i]) for i in range(K)]
    bwd = [mids[i].elapsed_time(ends[i]) for i in range(K)]
    tot = [starts[i].elapsed_time(ends[i]) for i in range(K)]
    ms = max_over_ranks(statistics.mean(tot), dist, dev)
    kern = {}
    for i, lab in enumerate(labels):
        kern.setdefault(lab, []).append(kev[2 * i].elapsed_time(kev[2 * i + 1]))

    # End to end through the public API with host buffers, as a training input
    # pipeline runs it: each step copies its inputs (x, dy, logits) from pinned
    # host memory and its results (out, dx, d_logits) back, on two copy streams
    # beside the compute stream, double-buffered so that step i+1's inputs
    # arrive and step i-1's results leave while step i computes; each phase of a
    # step waits only for the inputs it reads, and out leaves after the forward.  Every step
    # moves all of its bytes; the time is the whole run's (first input copy to
    # last result copy) over K steps.  Inputs and weights exceed L2, so no flush.
    pin = {n: torch.from_numpy(inp[n].view(np.int16)).pin_memory() for n in ("x", "dy")}
    pin["logits"] = torch.from_numpy(inp["logits"]).pin_memory()
    host_out = torch.empty((shape.T, shape.H), dtype=torch.int16).pin_memory()
    host_dx = torch.empty((shape.T, shape.H), dtype=torch.int16).pin_memory()
    host_dl = torch.empty((shape.T, shape.E), dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in (host_out, host_dx, host_dl))
    ins = [{n: torch.empty_like(d[n]) for n in ("x", "dy", "logits")} for _ in range(2)]
    outs = [{"out": torch.empty_like(out), "dx": torch.empty_like(grads["dx"]),
             "d_logits": torch.empty_like(grads["d_logits"]), "d_topk_w": torch.empty_like(grads["d_topk_w"])}
            for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    order = ("logits", "x", "dy")  # in the order the step reads them
    h2d_done = [{n: torch.cuda.Event() for n in order} for _ in range(K)]
    fwd_done = [torch.cuda.Event() for _ in range(K)]
    comp_done = [torch.cuda.Event() for _ in range(K)]
    d2h_done = [torch.cuda.Event() for _ in range(K)]
    e2e_start, e2e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def copy_in(i):
        with torch.cuda.stream(s_h2d):
            for n in order:
                ins[i % 2][n].copy_(pin[n], non_blocking=True)
                h2d_done[i][n].record(s_h2d)

    torch.cuda.synchronize()
    e2e_start.record(s_h2d)
    copy_in(0)
    for i in range(K):
        b_in, b_out = ins[i % 2], outs[i % 2]
        if i >= 2:
            stream.wait_event(d2h_done[i - 2])  # step i-2's results have left this buffer
        with torch.cuda.stream(stream):
            # each phase waits only for the input it reads: the first step's dy (and x)
            # still arriving while its route (and forward) run
            stream.wait_event(h2d_done[i]["logits"])
            layer.route(b_in["logits"], stream)
            stream.wait_event(h2d_done[i]["x"])
            layer.forward(b_in["x"], d["W_gate"], d["W_up"], d["W_down"], out=b_out["out"], stream=stream)
            fwd_done[i].record(stream)
            stream.wait_event(h2d_done[i]["dy"])
            g = dict(grads, dx=b_out["dx"], d_logits=b_out["d_logits"], d_topk_w=b_out["d_topk_w"])
            layer.backward(b_in["dy"], b_in["x"], d["W_gate"], d["W_up"], d["W_down"], grads=g, stream=stream)
            comp_done[i].record(stream)
        if i + 1 < K:
            if i >= 1:
                s_h2d.wait_event(comp_done[i - 1])  # step i-1 is done reading the other input buffer
            copy_in(i + 1)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(fwd_done[i])  # out leaves while the step's backward runs
            host_out.copy_(b_out["out"], non_blocking=True)
            s_d2h.wait_event(comp_done[i])
            host_dx.copy_(b_out["dx"], non_blocking=True)
            host_dl.copy_(b_out["d_logits"], non_blocking=True)
            d2h_done[i].record(s_d2h)
    e2e_end.record(s_d2h)
    torch.cuda.synchronize()
    # the last step's results are its own: the pipeline computed what the API promises
    if not torch.equal(host_dl.to(dev), grads["d_logits"]):
        raise RuntimeError("pipelined end-to-end step disagrees with the device-resident step")
    e2e_ms = max_over_ranks(e2e_start.elapsed_time(e2e_end) / K, dist, dev)
    # activation-checkpointed layer step (the pages' "2 fwd + bwd"): route, a forward
    # that keeps no activations (out only), then in the backward pass the recompute of
    # what the backward reads, followed by the backward
    c_starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    c_ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(K):
            flush.zero_()
            c_starts[i].record(stream)
            layer.route(d["logits"], stream)
            layer.forward(d["x"], d["W_gate"], d["W_up"], d["W_down"], out=out, stream=stream, save=False)
            layer.recompute(d["x"], d["W_gate"], d["W_up"], d["W_down"], stream=stream)
            grads = layer.backward(d["dy"], d["x"], d["W_gate"], d["W_up"], d["W_down"], grads=grads,
                                   stream=stream)
            c_ends[i].record(stream)
    torch.cuda.synchronize()
    ckpt_ms = statistics.mean(c_starts[i].elapsed_time(c_ends[i]) for i in range(K))
    # the same step without the L2 flush between steps (inputs still exceed L2)
    n_starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    n_ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(K):
            n_starts[i].record(stream)
            step()
            n_ends[i].record(stream)
    torch.cuda.synchronize()
    no_flush = [n_starts[i].elapsed_time(n_ends[i]) for i in range(K)]
    # the router projection in front of the layer (logits = x . W_r, and its backward)
    router_ms = None
    if shape.E % 8 == 0:
        rgen = np.random.default_rng(3300)
        W_r = torch.from_numpy((rgen.standard_normal((shape.H, shape.E), dtype=np.float32) * 0.02)
                               .astype(np.float32)).to(dev).to(torch.bfloat16).view(torch.int16)
        router = moe.Router(shape, device=dev)
        logits_r = torch.empty((shape.T, shape.E), dtype=torch.float32, device=dev)
        dW_r = torch.empty((shape.H, shape.E), dtype=torch.float32, device=dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3 * K)]
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for i in range(K):
                flush.zero_()
                ev[3 * i].record(stream)
                router.forward(d["x"], W_r, logits_r, stream=stream)
                ev[3 * i + 1].record(stream)
                router.backward(d["x"], W_r, grads["d_logits"], grads["dx"], dW_r, stream=stream)
                ev[3 * i + 2].record(stream)
        torch.cuda.synchronize()
        # a second pass with per-kernel events (they add gaps, so not in the totals above)
        rkev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * 8 * K)]
        moe.timing_attach(rkev)
        with torch.cuda.stream(stream):
            for i in range(K):
                flush.zero_()
                router.forward(d["x"], W_r, logits_r, stream=stream)
                router.backward(d["x"], W_r, grads["d_logits"], grads["dx"], dW_r, stream=stream)
        torch.cuda.synchronize()
        rlabels = [moe.timing_label(i) for i in range(moe.timing_count())]
        moe.timing_attach(None)
        rk = {}
        for i, lab in enumerate(rlabels):
            rk.setdefault(lab, []).append(rkev[2 * i].elapsed_time(rkev[2 * i + 1]))
        if any(router.status(stream).values()):
            raise RuntimeError(f"router status: {router.status(stream)}")
        router_ms = {"fwd_ms": statistics.mean(ev[3 * i].elapsed_time(ev[3 * i + 1]) for i in range(K)),
                     "bwd_ms": statistics.mean(ev[3 * i + 1].elapsed_time(ev[3 * i + 2]) for i in range(K)),
                     "flop_per_step": 3 * 2.0 * shape.T * shape.H * shape.E,
                     "kernels_avg_ms": {lab: statistics.mean(v) for lab, v in rk.items()}}
    st = layer.status(stream)
    if any(st.values()):
        raise RuntimeError(f"device status after timed steps: {st}")
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    work = kernel_work(shape)
    gbytes = gemm_bytes(shape, w.precision)
    fwd_fl, bwd_fl = shape.gemm_flops()
    kernels = {}
    for lab, ts in kern.items():
        bound, amount, unit = work.get(lab, ("?", 0.0, "?"))
        avg = statistics.mean(ts)
        if bound == "tensor":
            ach, pk, u = amount / (avg * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
        elif bound == "tensor_fp8":
            ach, pk, u = amount / (avg * 1e-3) / 1e12, peaks["bf16_tflops"] * FP8_OVER_BF16, "TFLOP/s"
        else:
            ach, pk, u = amount / (avg * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
        kernels[lab] = {"launches": len(ts), "avg_ms": avg, "share": sum(ts) / sum(sum(v) for v in kern.values()),
                        "bound": bound, "achieved": ach, "unit": u, "peak": pk, "frac": ach / pk}
        if lab in gbytes:  # a GEMM's HBM roof beside its tensor roof; the larger floor binds
            gb = gbytes[lab] / (avg * 1e-3) / 1e9
            t_tensor, t_hbm = amount / (pk * 1e12), gbytes[lab] / (peaks["hbm_gbs"] * 1e9)
            kernels[lab].update({"hbm_bytes": gbytes[lab], "hbm_achieved_gbs": gb, "hbm_frac": gb / peaks["hbm_gbs"],
                                 "binding_roof": "tensor" if t_tensor >= t_hbm else "hbm",
                                 "binding_frac": max(t_tensor, t_hbm) / (avg * 1e-3)})
    top = max(kernels, key=lambda n: kernels[n]["share"])
    kt = kernels[top]
    src = {"tensor": "bf16 burst", "tensor_fp8": f"bf16 burst x {FP8_OVER_BF16:g} (nominal fp8/bf16 ratio)",
           "hbm": "HBM copy"}[kt["bound"]]
    roofline = {"kernel": top, "bound": "tensor" if kt["bound"].startswith("tensor") else kt["bound"],
                "achieved": kt["achieved"], "peak": kt["peak"], "unit": kt["unit"], "frac": kt["frac"],
                "traffic": committed_traffic(top, w.name), "peak_source": f"{peak_src} ({src})"}
    world_tokens = shape.T * world
    fwd_ms, bwd_ms = statistics.mean(fwd), statistics.mean(bwd)
    line = {
        "metric": METRIC, "value": world_tokens / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"bf16": "bf16", "fp8_bwd": "bf16 fwd + mxfp8 bwd GEMMs",
                                            "mxfp8": "mxfp8 fwd + bwd GEMMs"}[w.precision],
        "data": "synthetic (seeded normals; Qwen3-shaped layer)",
        "config": {"workload": w.name, "T": shape.T, "H": shape.H, "I": shape.I, "E": shape.E, "k": shape.k,
                   "precision": w.precision, "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "256 MiB flush between steps; inputs (weights 1.1+ GiB) exceed L2",
                   "step": "route + forward + backward (all weight and data gradients)"},
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "fwd_bwd_ms": ms, "ms_per_step_median": statistics.median(tot),
        "no_l2_flush": {"ms_per_step": statistics.mean(no_flush), "median": statistics.median(no_flush)},
        "ckpt_2f_plus_b_ms": ckpt_ms,
        "tflops": (fwd_fl + bwd_fl) / (ms * 1e-3) / 1e12,
        "frac_of_bf16_peak": (fwd_fl + bwd_fl) / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
        "roofline": roofline, "kernels": kernels,
        "e2e": {"value": world_tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipeline": "K steps; inputs copied in on one stream, results out on another, "
                            "double-buffered around the compute stream (each phase waits for the inputs "
                            "it reads; out leaves after the forward); no L2 flush (inputs exceed L2)"},
        "gpu_launches": launches_in_timed_region(labels, KH, K), "clocks": clk.summary(),
        "router_projection": router_ms,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, inp)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=15)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0, help="override T (small profiling cases)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
