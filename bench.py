"""Benchmark of the routed MoE SwiGLU FFN forward pass on GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--T T]
                  [--impl ours|reference]

A step is one layer call (router, sort, both projections, combine) over one
batch of T fresh seeded tokens.  The default workload is the Qwen-3-style
decode layer (H=2048, I=768, E=128, top-8) at T=1.  Each rank (torchrun, one
per GPU) runs its own replica over its own token stream: the calls are
independent problems, so there is no data-path collective ("scaling": "weak").

Timing: the steps run back to back, as a model's layers do, over R layers'
weights (step j uses layer j % R; R is chosen so that the weights a step
reads have been streamed out of L2 by the steps in between, i.e. the inputs
are larger than L2).  W untimed warm-up steps and one untimed replay of the
timed graph (its first launch uploads it to the device), then the K timed
steps as one CUDA graph replay (--eager: launched one by one from Python),
bracketed by a barrier, cudaDeviceSynchronize and CUDA events on the
launching stream;
value = tokens of all ranks / max over ranks of that time.  A second replay
records the library's stage events between kernels for the roofline of the
dominant kernel.  cold_call times single calls after an L2 flush each.  e2e
repeats the steps through the host-buffer entry point, called step by step
from Python (pinned inputs copied in, output copied out, inside the region).

After the headline line's figures (at one GPU), every other configuration
of the layer the metric names (the 2048-hidden decode layer at T=2, the
4096-hidden one at T=1/4/16/64, the 7168-hidden one at T=1/8/32 and the
T=2048 training-size forward) is measured the same way, W warm-up and K
timed steps each over its own layers' weights drawn on the GPU, and reported
in the line's "supplementary" array: us per call, tokens/s, the whole
call's HBM fraction, the dominant kernel's roofline and the TFLOP/s against
dense BF16 peak and against min(peak, HBM peak x flop/byte).  Two of the
rows ("entry": moe_ffn_forward_router) run the 2048-hidden decode layer at
T=1 and 2 with the router projection inside the call (router weights and
bias passed instead of logits); nine ("entry": moe_ffn_forward_mxfp8) run
the 2048-hidden layer at T=1/2/4, the 4096-hidden one at T=1/16/64 and the
7168-hidden one at T=1/8/32 with MXFP8 expert weights (their bytes counted
at 1 + 1/32 per weight; T > 4 takes the grouped tensor-core path).  One row
("entry": moe_ffn_backward) runs the backward pass of the T=2048
training-size layer (dout ~ N(0,1) FP32 per call; all four gradients written
every call), with its own byte model (backward_bytes) and 16 H I T k flops.
One row ("entry": moe_ffn_forward_train + moe_ffn_backward_train) runs a
training step of that layer: the forward pass keeping g and u, then the
backward pass reading them (byte model train_bytes, 18 H I T k flops).

--impl reference times the FP64 CPU oracle on this machine's host cores on a
bounded sample of the same workload (it is the slow baseline, not a target).
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
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s; decode HBM TB/s vs peak; T=2048 TFLOPS vs BF16 peak"
DEFAULT_WORKLOAD = "decode_h2048_i768_e128_k8"
FLUSH_BYTES = 512 << 20
L2_BYTES = 129 << 20            # GB300 L2
LAYER_MEM_CAP = 72 << 30        # device memory for the layers' weights
BATCH_MEM_CAP = 2 << 30         # and for the token batches

# Kernel sources whose change voids a stored ncu traffic figure.
KERNEL_SOURCES = {
    "decode_fused": ["decode_fused.cu"],
    "decode_gate_up": ["decode.cu"],
    "decode_down": ["decode.cu"],
    "gemm_gate_up": ["grouped_gemm.cu"],
    "gemm_down": ["grouped_gemm.cu"],
    "gemm_q": ["grouped_gemm.cu"],
    "gemm_dx": ["grouped_gemm.cu"],
    "wgrad_down": ["grouped_bwd.cu"],
    "wgrad_gate_up": ["grouped_bwd.cu"],
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--T", type=int, default=None)
    p.add_argument("--E", type=int, default=None, help="fewer experts (profiling-size variant)")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--flush", choices=["write", "write+read"], default="write+read",
                   help="L2 flush between steps: a write larger than L2, optionally followed by a "
                        "read that makes the dirty lines' write-back happen before the next step")
    p.add_argument("--path", choices=["auto", "decode", "grouped"], default="auto",
                   help="force the library's execution path (default: its own choice)")
    p.add_argument("--skip-baseline", action="store_true", help="omit the CPU oracle timing")
    p.add_argument("--layers", type=int, default=None,
                   help="layers' weights cycled by the steps (default: enough that none is in L2)")
    p.add_argument("--eager", action="store_true",
                   help="launch every step from Python instead of replaying a CUDA graph of the steps")
    p.add_argument("--cold-steps", type=int, default=200,
                   help="single calls timed after an L2 flush each (secondary figure)")
    p.add_argument("--backward", action="store_true",
                   help="time the backward pass (moe_ffn_backward) as the step instead of the forward pass "
                        "(no e2e or CPU-baseline figures; e.g. with --E for a profiling-size variant)")
    p.add_argument("--train", action="store_true",
                   help="time a training step (moe_ffn_forward_train, then moe_ffn_backward_train) as the step "
                        "(no e2e or CPU-baseline figures)")
    p.add_argument("--no-supplementary", action="store_true",
                   help="omit the other configurations' rows (measured after the headline line)")
    p.add_argument("--weights", choices=["bf16", "mxfp8"], default="bf16",
                   help="expert weight format of the headline line (mxfp8: moe_ffn_forward_mxfp8, "
                        "one to four tokens; no e2e or CPU-baseline figures)")
    return p.parse_args()


def rank_calls(rank, W, K):
    """Call indices of the token stream that rank processes: disjoint per
    rank, so the replicas work on independent tokens."""
    return range(rank * (W + K), (rank + 1) * (W + K))


def max_over_ranks(values, world, device="cpu"):
    """Element-wise maximum of the per-rank values; every rank gets it."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def whole_job_tokens_per_s(T, K, world, max_ms):
    """Tokens of all ranks over the slowest rank's time (weak scaling)."""
    return T * K * world / (max_ms / 1e3)


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                "bf16_tflops_sustained": pk.get("bf16_tflops_sustained"), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def source_digest(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel, []):
        with open(os.path.join(ROOT, "mixture_experts_ffn_gate_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel, workload, T):
    """DRAM bytes per launch from a committed ncu summary, or None if absent
    or taken on a different version of the kernel's source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    rec = table.get(f"{kernel}@{workload}/T{T}")
    if not rec or rec.get("source_sha") != source_digest(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) >= 9 and f[1].replace(".", "").isdigit():
                rows.append(f)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows
                                                         if r[3].replace(".", "").isdigit())}


# bytes per expert-weight element: BF16, or MXFP8 (one E4M3 byte plus one
# E8M0 scale byte per 32 elements; the padding of the scale rows is not
# counted)
BPE = {"bf16": 2.0, "mxfp8": 1.0 + 1.0 / 32}


def algorithmic_bytes(wl, T, U, bpe=2.0):
    """Per-call algorithmic HBM bytes: each touched expert's weights once
    (U*3*H*I*bpe), x in (T*H*2), logits in (T*E*4), out written (T*H*4)."""
    return U * 3 * wl.H * wl.I * bpe + T * wl.H * 2 + T * wl.E * 4 + T * wl.H * 4


def kernel_bytes(kernel, wl, T, U, k, bpe=2.0):
    """Algorithmic bytes of one launch of a kernel."""
    H, I = wl.H, wl.I
    if kernel == "decode_fused":  # the whole layer in one kernel; act written and read back once
        return U * 3 * H * I * bpe + T * H * 2 + T * wl.E * 4 + T * H * 4 + 2 * T * k * I * 4
    if kernel == "decode_gate_up":
        return U * 2 * I * H * 2 + T * H * 2 + T * k * I * 4
    if kernel == "decode_down":
        return U * H * I * 2 + T * k * I * 4 + T * H * 4 + T * k * 4
    if kernel == "gemm_gate_up":  # x rows read by the sorted order (re-reads of a row come from L2)
        return U * 2 * I * H * bpe + T * H * 2 + 2 * T * k * I * 2
    if kernel == "gemm_down":
        return U * H * I * bpe + 2 * T * k * I * 2 + T * k * H * 4
    return None


def backward_bytes(wl, T, U):
    """Per-call algorithmic HBM bytes of the backward pass: the touched
    experts' W_gate_up read twice (the recomputation of gate/up, and dx) and
    W_down once; both weight gradients written once in FP32 (every expert,
    untouched ones as zeros); x, logits and dout read; dx and dlogits
    written."""
    H, I, E = wl.H, wl.I, wl.E
    return (U * (2 * 2 * I * H * 2 + H * I * 2) + E * 3 * H * I * 4
            + T * H * 2 + T * E * 4 + T * H * 4 + T * H * 4 + T * E * 4)


def backward_kernel_bytes(kernel, wl, T, U, k):
    """Algorithmic bytes of one launch of a backward-pass kernel (n = T k
    assignment rows; intermediates FP32 or BF16 hi/lo pairs)."""
    H, I, E = wl.H, wl.I, wl.E
    n = T * k
    return {
        "prep": T * H * 2 + T * H * 4 + n * H * 2 + 2 * n * H * 2 + n * 4,
        "gemm_gate_up": U * 2 * I * H * 2 + T * H * 2 + 2 * n * I * 4,
        "gemm_q": U * H * I * 2 + 2 * n * H * 2 + 2 * n * I * 4 + 2 * n * 2 * I * 2 + 2 * n * I * 2
        + n * (I // 32) * 4 + n * 4,
        "gemm_dx": U * 2 * I * H * 2 + 2 * n * 2 * I * 2 + n * H * 4,
        "combine": n * H * 4 + T * H * 4,
        "zero_grads": (E - U) * 3 * H * I * 4,
        "wgrad_down": U * H * I * 4 + 2 * n * H * 2 + 2 * n * I * 2,
        "wgrad_gate_up": U * 2 * I * H * 4 + 2 * n * 2 * I * 2 + n * H * 2,
    }.get(kernel)


def train_bytes(wl, T, U):
    """Per-step algorithmic HBM bytes of the training pair: the forward
    call's (algorithmic_bytes) plus g and u written for the backward, plus
    the backward call's (backward_bytes) without the recomputation's read of
    W_gate_up, which the pair does not repeat."""
    return (algorithmic_bytes(wl, T, U) + 2 * T * wl.k * wl.I * 4 + backward_bytes(wl, T, U)
            - U * 2 * wl.I * wl.H * 2)


def train_kernel_bytes(kernel, wl, T, U, k):
    """Algorithmic bytes of one launch of a kernel of the training pair
    (stage names "fwd:..." and "bwd:...")."""
    side, _, name = kernel.partition(":")
    if side == "fwd":
        b = kernel_bytes(name, wl, T, U, k)
        return b + 2 * T * k * wl.I * 4 if name == "gemm_gate_up" else b
    return backward_kernel_bytes(name, wl, T, U, k)


def reference_arm(args, wl, T):
    """The FP64 oracle on the host cores, on a bounded sample of the workload."""
    import numpy as np

    import oracle
    from mixture_experts_ffn_gate_gb300 import synth

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cores = len(os.sched_getaffinity(0))
    # weights of the experts the sampled tokens select, drawn on the host
    steps, warm = args.steps, args.warmup
    per_token = 6.0 * wl.H * wl.I * wl.k  # flops per token
    # cap the run at ~120 s of oracle time (measured rate ~1 GFLOP/s/thread)
    budget_tokens = max(1, int(120e9 * min(cores, max(T, 1)) / per_token))
    t_step = min(T, budget_tokens)
    steps_run = max(1, min(steps, budget_tokens // max(t_step, 1)))
    batches = [synth.make_tokens(wl, T, call=i) for i in range(warm + steps_run)]
    need = set()
    for x, L in batches:
        idx, _ = oracle.route(L[:t_step].numpy(), wl.k)
        need.update(np.unique(idx).tolist())
    need = sorted(need)
    emap = -np.ones(wl.E, np.int32)
    emap[need] = np.arange(len(need), dtype=np.int32)
    g, d = synth.make_weights(wl, device="cpu", experts=need)
    wgu, wd = synth.bf16_bits(g), synth.bf16_bits(d)
    del g, d
    for x, L in batches[:warm]:
        oracle.forward(synth.bf16_bits(x[:t_step]), L[:t_step].numpy(), wgu, wd, wl.k,
                       expert_map=emap, nthreads=cores)
    t0 = time.perf_counter()
    for x, L in batches[warm:]:
        oracle.forward(synth.bf16_bits(x[:t_step]), L[:t_step].numpy(), wgu, wd, wl.k,
                       expert_map=emap, nthreads=cores)
    dt = time.perf_counter() - t0
    tokens = t_step * steps_run
    value = tokens / dt
    sample = (f"{steps_run} steps of {t_step} of the {T} tokens per step (fresh seeded tokens), "
              f"weights of the {len(need)} experts they select drawn on the host")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": steps_run, "warmup": warm,
            "ms_per_step": 1e3 * dt / steps_run, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "T": T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": min(cores, t_step),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(wl, T, wgu_dev, wd_dev, bias):
    """The oracle as it stands on the host cores, on a bounded sample of the
    workload (~10-30 s of CPU work: the oracle does about 3 GFLOP/s per core
    on this layer); returns the cpu_baseline object."""
    import numpy as np

    import oracle
    from mixture_experts_ffn_gate_gb300 import synth
    import torch

    cores = len(os.sched_getaffinity(0))
    per_token = 6.0 * wl.H * wl.I * wl.k
    n_tok = max(1, min(int(45e9 * cores / per_token), 16384))
    xs, Ls = [], []
    got, call = 0, 0
    while got < n_tok:  # the first calls of the rank-0 token stream
        x, L = synth.make_tokens(wl, T, call=call, bias=bias)
        take = min(x.shape[0], n_tok - got)
        xs.append(x[:take])
        Ls.append(L[:take])
        got += take
        call += 1
    x = torch.cat(xs)
    L = torch.cat(Ls).numpy()
    idx, _ = oracle.route(L, wl.k)
    used = np.unique(idx)
    emap = -np.ones(wl.E, np.int32)
    emap[used] = np.arange(len(used), dtype=np.int32)
    sel = torch.as_tensor(used, dtype=torch.long, device=wgu_dev.device)
    wgu = synth.bf16_bits(wgu_dev.index_select(0, sel))
    wd = synth.bf16_bits(wd_dev.index_select(0, sel))
    xb = synth.bf16_bits(x)
    t0 = time.perf_counter()
    oracle.forward(xb, L, wgu, wd, wl.k, expert_map=emap, nthreads=cores)
    dt = time.perf_counter() - t0
    # the same oracle on one thread, on the first tokens of the sample (~5 s)
    n1 = max(1, min(got, int(15e9 / per_token)))
    t1 = time.perf_counter()
    oracle.forward(xb[:n1], L[:n1], wgu, wd, wl.k, expert_map=emap, nthreads=1)
    dt1 = time.perf_counter() - t1
    return {"value": got / dt, "unit": "tokens/s", "cores": min(cores, got), "kind": "oracle",
            "sample": f"{got} fresh seeded tokens of the workload in one oracle call "
                      f"({len(used)} experts), {dt:.1f} s",
            "cpu": cpu_model(),
            "single_thread": {"value": n1 / dt1, "unit": "tokens/s", "sample": f"the first {n1} tokens, {dt1:.1f} s"}}


def cpu_model():
    """The host CPU's name as /proc/cpuinfo or lscpu give it."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


# Every other configuration the metric names, measured by the same command
# after the headline line: a short timed run each (weights drawn on the GPU,
# no oracle timing), reported in the line's "supplementary" array.
SUPPLEMENTARY = [
    ("decode_h2048_i768_e128_k8", (2,)),
    ("decode_h2048_i768_e128_k8+router", (1, 2)),
    ("decode_h2048_i768_e128_k8+mxfp8", (1, 2, 4)),
    ("decode_h4096_i1536_e128_k8_bias+mxfp8", (1, 16, 64)),
    ("decode_h7168_i2048_e384_k8_bias+mxfp8", (1, 8, 32)),
    ("decode_h4096_i1536_e128_k8_bias", (1, 4, 16, 64)),
    ("decode_h7168_i2048_e384_k8_bias", (1, 8, 32)),
    ("fwd_t2048_h6144_i2048_e256_k8_bias", (2048,)),
    ("fwd_t2048_h6144_i2048_e256_k8_bias+backward", (2048,)),
    ("fwd_t2048_h6144_i2048_e256_k8_bias+train", (2048,)),
]


def layer_count(wl, T, layers_arg, bpe=2.0):
    """Layers' weights the steps cycle through: enough that the weights one
    step reads were streamed out of L2 by the steps in between."""
    touched = algorithmic_bytes(wl, T, min(wl.E, T * wl.k), bpe)
    R = max(2, math.ceil(3 * L2_BYTES / touched)) if layers_arg is None else layers_arg
    return max(1, min(R, int(LAYER_MEM_CAP // wl.weight_bytes()))), touched


class Measure:
    """One workload at one T on this rank: the steps cycle through the given
    layers' weights over fresh token batches on one workspace.  timed() runs
    W warm-up steps and times K steps as one CUDA-graph replay (or eager
    launches); stages() replays them with the library's stage events between
    kernels; summary() gives the figures of one line."""

    def __init__(self, wl, T, dev, K, W, path_code, layers, bias, rank, eager, routers=None, mx=False,
                 backward=False, train=False):
        import torch
        from mixture_experts_ffn_gate_gb300 import moe_ffn as m
        from mixture_experts_ffn_gate_gb300 import synth
        self.m, self.torch = m, torch
        self.wl, self.T, self.dev, self.K, self.W = wl, T, dev, K, W
        self.path_code, self.layers, self.R = path_code, layers, len(layers)
        self.eager = eager
        # routers: per layer W_r [E, H]; the calls then pass the router
        # weights and the bias instead of logits (moe_ffn_forward_router)
        self.routers = routers
        self.rbias = bias.to(dev) if routers is not None else None
        # mx: the layers hold MXFP8 weights (codes and scales, four tensors)
        # and the calls go through moe_ffn_forward_mxfp8
        self.mx = mx
        self.bpe = BPE["mxfp8" if mx else "bf16"]
        # backward: the steps are moe_ffn_backward calls, each with its own
        # upstream gradient, writing all four gradients
        self.backward = backward
        # train: a step is moe_ffn_forward_train and then moe_ffn_backward_train
        # on one state buffer (a training step of the layer)
        self.train = train
        batch_bytes = T * (wl.H * 2 + wl.E * 4 + (wl.H * 4 if backward or train else 0))
        self.NB = max(1, min(W + K, 256, int(BATCH_MEM_CAP // max(batch_bytes, 1))))
        calls = rank_calls(rank, W, K)   # rank r processes its own calls of the token stream
        self.batches = [synth.make_tokens(wl, T, call=calls[i], device=dev, bias=bias)
                        for i in range(self.NB)]
        if backward or train:
            self.douts = [synth.make_dout(wl, T, call=calls[i], device=dev) for i in range(self.NB)]
            self.ws = (m.new_train_state if train else m.new_backward_workspace)(T, wl.H, wl.I, wl.E, wl.k,
                                                                                  device=dev)
            self.grads = (torch.empty((T, wl.H), dtype=torch.float32, device=dev),
                          torch.empty((T, wl.E), dtype=torch.float32, device=dev),
                          torch.empty((wl.E, 2 * wl.I, wl.H), dtype=torch.float32, device=dev),
                          torch.empty((wl.E, wl.H, wl.I), dtype=torch.float32, device=dev))
        else:
            self.ws = (m.new_workspace(T, wl.H, wl.I, wl.E, wl.k, device=dev) if routers is None
                       else m.new_router_workspace(T, wl.H, wl.I, wl.E, wl.k, device=dev))
        self.out = torch.empty((T, wl.H), dtype=torch.float32, device=dev)
        self.stream = torch.cuda.current_stream()
        probe = self.new_opts()
        self.call(0, self.stream, probe)
        self.path, self.n_stages = probe.path_taken, probe.n_stages
        self.stage_names = [m.moe_ffn_stage_name(self.path, s) for s in range(self.n_stages)]
        if train:   # the forward call's stages, then the backward call's
            fwd = [m.moe_ffn_stage_name(m.MOE_PATH_TRAIN_FORWARD, s) for s in range(self.TRAIN_FWD_STAGES)]
            bwd = [m.moe_ffn_stage_name(m.MOE_PATH_TRAIN_BACKWARD, s) for s in range(self.n_stages)]
            self.path = "train"
            self.stage_names = ["fwd:" + n for n in fwd] + ["bwd:" + n for n in bwd]
        # unique experts touched per step (routing of each batch, untimed)
        idx_buf = torch.empty((T, wl.k), dtype=torch.int32, device=dev)
        U_of = {}
        for j in range(W, W + K):
            if j % self.NB not in U_of:
                if backward or train:   # the selection by torch.topk (ties aside, the same experts)
                    U_of[j % self.NB] = int(torch.unique(torch.topk(self.batches[j % self.NB][1], wl.k).indices)
                                            .numel())
                    continue
                self.call(j, self.stream, None, idx_buf)
                U_of[j % self.NB] = int(torch.unique(idx_buf).numel())
        self.U = [U_of[j % self.NB] for j in range(W, W + K)]
        torch.cuda.synchronize()
        if not eager:
            self.g_warm = self.capture(range(W))
            self.g_main = self.capture(range(W, W + K))

    TRAIN_FWD_STAGES = 5   # moe_ffn_forward_train's kernels

    def new_opts(self):
        o = self.m.moe_ffn_opts()
        o.path = self.path_code
        return o

    def call(self, j, stream, opts=None, idx=None):
        x, L = self.batches[j % self.NB]
        opts = opts if opts is not None else self.new_opts()
        if self.train:
            # the backward call records its stage events after the forward
            # call's (event TRAIN_FWD_STAGES is its start); opts reports the
            # backward call's path and stages
            lw_gu, lw_d = self.layers[j % self.R]
            of = self.new_opts()
            if opts.stage_events:
                of.stage_events = opts.stage_events
                opts.stage_events = opts.stage_events + self.TRAIN_FWD_STAGES * self.m.ctypes.sizeof(
                    self.m.ctypes.c_void_p)
            self.m.moe_ffn_forward_train(x, L, lw_gu, lw_d, self.wl.k, self.ws, out=self.out, opts=of,
                                         stream=stream)
            self.m.moe_ffn_backward_train(x, L, lw_gu, lw_d, self.douts[j % self.NB], self.wl.k, self.ws,
                                          *self.grads, opts=opts, stream=stream)
            return
        if self.backward:
            lw_gu, lw_d = self.layers[j % self.R]
            self.m.moe_ffn_backward(x, L, lw_gu, lw_d, self.douts[j % self.NB], self.wl.k, *self.grads,
                                    workspace=self.ws, opts=opts, stream=stream)
            return
        if self.mx:
            self.m.moe_ffn_forward_mxfp8(x, L, *self.layers[j % self.R], self.wl.k, out=self.out, workspace=self.ws,
                                         topk_idx=idx, opts=opts, stream=stream)
            return
        lw_gu, lw_d = self.layers[j % self.R]
        if self.routers is not None:
            self.m.moe_ffn_forward_router(x, self.routers[j % self.R], self.rbias, lw_gu, lw_d, self.wl.k,
                                          out=self.out, workspace=self.ws, topk_idx=idx, opts=opts, stream=stream)
            return
        self.m.moe_ffn_forward_ex(x, L, lw_gu, lw_d, self.wl.k, out=self.out, workspace=self.ws,
                                  topk_idx=idx, opts=opts, stream=stream)

    def capture(self, steps, events=None):
        """One CUDA graph holding the calls of `steps`, in order."""
        torch, m = self.torch, self.m
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            s = torch.cuda.current_stream()
            for n, j in enumerate(steps):
                o = self.new_opts()
                if events is not None:
                    o.stage_events = m.ctypes.cast(events[n], m.ctypes.c_void_p)
                self.call(j, s, o)
        return g

    def timed(self, world):
        """W untimed warm-up steps, then the K timed steps between a barrier,
        device synchronisation and CUDA events on the launching stream.  With
        CUDA graphs the graph of the K steps is also replayed once untimed
        first: its first launch uploads it to the device and runs about 1.5 us
        per call slower than every later one, which is what a serving loop
        replaying one graph sees (warm_steps counts both).
        Returns (ms for the K steps, host wall seconds)."""
        torch = self.torch
        import torch.distributed as dist
        W, K = self.W, self.K
        if self.eager:
            for j in range(W):
                self.call(j, self.stream)
            self.warm_steps = W
        else:
            self.g_warm.replay()
            self.g_main.replay()
            self.warm_steps = W + K
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        mark0 = torch.cuda.Event(enable_timing=True)
        mark1 = torch.cuda.Event(enable_timing=True)
        t_wall = time.perf_counter()
        mark0.record(self.stream)
        if self.eager:
            for j in range(W, W + K):
                self.call(j, self.stream)
        else:
            self.g_main.replay()
        mark1.record(self.stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_wall
        if world > 1:
            dist.barrier()
        return mark0.elapsed_time(mark1), wall

    def stages(self):
        """Mean ms of each kernel over the K steps, from the library's stage
        events (captured as event-record nodes when graphs are used)."""
        torch, m = self.torch, self.m
        K, W = self.K, self.W
        # a training step is two calls: the backward call's events follow
        # the forward call's TRAIN_FWD_STAGES
        n_ev = m.MOE_MAX_STAGES + 1 + (self.TRAIN_FWD_STAGES if self.train else 0)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(K)]
        arrs = []
        for j in range(K):
            for e in evs[j]:
                e.record(self.stream)
            arrs.append(m.stage_event_array(evs[j]))
        torch.cuda.synchronize()
        if self.eager:
            for j in range(K):
                o = self.new_opts()
                o.stage_events = m.ctypes.cast(arrs[j], m.ctypes.c_void_p)
                self.call(W + j, self.stream, o)
        else:
            g = self.capture(range(W, W + K), arrs)
            g.replay()   # uploads the graph; the second replay's events count
            g.replay()
        torch.cuda.synchronize()
        return {name: sum(evs[j][s].elapsed_time(evs[j][s + 1]) for j in range(K)) / K
                for s, name in enumerate(self.stage_names)}

    def summary(self, total_ms, kern_avg, peaks, world):
        """Throughput, the whole call's HBM fraction, the dominant kernel's
        roofline and the tensor figures of one workload line."""
        wl, T, K = self.wl, self.T, self.K
        if self.backward:
            return self.summary_backward(total_ms, kern_avg, peaks, world)
        if self.train:
            return self.summary_backward(total_ms, kern_avg, peaks, world, train=True)
        call_bytes = sum(algorithmic_bytes(wl, T, u, self.bpe) for u in self.U) / K
        # calls with the router projection inside also read W_r (E*H BF16)
        router_bytes = wl.E * wl.H * 2 if self.routers is not None else 0
        call_bytes += router_bytes
        flops = 6.0 * wl.H * wl.I * T * wl.k
        ms_call = total_ms / K
        # dominant kernel = largest share of the per-kernel pass.  When a step
        # is a single kernel, its launches are the timed region itself, so
        # their mean duration is at most the timed region / K; the
        # stage-event replay (event nodes between launches) would charge the
        # event overhead to it.
        dom = max(kern_avg, key=kern_avg.get)
        one_kernel = len(kern_avg) == 1
        dom_ms = ms_call if one_kernel else kern_avg[dom]
        dom_bytes = sum(kernel_bytes(dom, wl, T, u, wl.k, self.bpe) for u in self.U) / K
        if dom == "decode_fused":
            dom_bytes += router_bytes
        achieved = dom_bytes / (dom_ms / 1e3) / 1e9
        roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "traffic": stored_traffic(dom, wl.name + ("+mxfp8" if self.mx else "+router" if self.routers
                                                              is not None else ""), T),
                    "peak_source": f"{peaks['source']} HBM copy (burst)",
                    "algorithmic_bytes_per_launch": dom_bytes,
                    "kernel_time": ("timed region / K (one kernel per step)" if one_kernel
                                    else "stage events between kernels, CUDA-graph replay"),
                    "kernel_us": {n: round(1e3 * v, 3) for n, v in kern_avg.items()}}
        gbs = call_bytes / (ms_call / 1e3) / 1e9
        tflops = flops / (ms_call / 1e3) / 1e12
        intensity = flops / call_bytes
        attainable = min(peaks["bf16_tflops"], peaks["hbm_gbs"] * 1e9 * intensity / 1e12)
        return {
            "value": whole_job_tokens_per_s(T, K, world, total_ms),
            "ms_per_step": ms_call,
            "path": {1: "decode", 2: "grouped", 3: "decode_fused"}.get(self.path, self.path),
            "roofline": roofline,
            "call_hbm": {"achieved_gbs": gbs, "frac_of_measured": gbs / peaks["hbm_gbs"],
                         "frac_of_8tbs_spec": gbs / 8000.0, "bytes_per_call": call_bytes,
                         "unique_experts_mean": sum(self.U) / K},
            "tensor": {"tflops": tflops, "frac_of_dense_bf16_peak": tflops / peaks["bf16_tflops"],
                       "flop_per_byte": intensity, "attainable_tflops": attainable,
                       "frac_of_attainable": tflops / attainable,
                       "attainable": "min(dense BF16 peak, measured HBM copy peak x flop/byte)"},
        }


    def summary_backward(self, total_ms, kern_avg, peaks, world, train=False):
        """The figures of a backward-pass line (byte model backward_bytes,
        flops 16 H I T k: gate/up recomputed, q, dx and both weight
        gradients), or with train of a training-step line (train_bytes,
        flops 18 H I T k: the forward's 6 and the backward's 12)."""
        wl, T, K = self.wl, self.T, self.K
        step_bytes, kbytes = (train_bytes, train_kernel_bytes) if train else (backward_bytes, backward_kernel_bytes)
        call_bytes = sum(step_bytes(wl, T, u) for u in self.U) / K
        flops = (18.0 if train else 16.0) * wl.H * wl.I * T * wl.k
        ms_call = total_ms / K
        dom = max(kern_avg, key=kern_avg.get)
        dom_bytes = sum(kbytes(dom, wl, T, u, wl.k) for u in self.U) / K
        achieved = dom_bytes / (kern_avg[dom] / 1e3) / 1e9
        per_kernel = {}
        for n, v in kern_avg.items():
            b = kbytes(n, wl, T, sum(self.U) / K, wl.k)
            per_kernel[n] = {"us": round(1e3 * v, 3)}
            if b:
                per_kernel[n]["gbs"] = round(b / (v / 1e3) / 1e9, 1)
                per_kernel[n]["frac_of_hbm_peak"] = round(b / (v / 1e3) / 1e9 / peaks["hbm_gbs"], 3)
        roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "traffic": stored_traffic(dom.partition(":")[2] or dom, wl.name + "+backward", T),
                    "peak_source": f"{peaks['source']} HBM copy (burst)",
                    "algorithmic_bytes_per_launch": dom_bytes,
                    "kernel_time": "stage events between kernels, CUDA-graph replay",
                    "kernels": per_kernel}
        gbs = call_bytes / (ms_call / 1e3) / 1e9
        tflops = flops / (ms_call / 1e3) / 1e12
        intensity = flops / call_bytes
        attainable = min(peaks["bf16_tflops"], peaks["hbm_gbs"] * 1e9 * intensity / 1e12)
        return {
            "value": whole_job_tokens_per_s(T, K, world, total_ms),
            "ms_per_step": ms_call,
            "path": "train" if train else "backward",
            "roofline": roofline,
            "call_hbm": {"achieved_gbs": gbs, "frac_of_measured": gbs / peaks["hbm_gbs"],
                         "frac_of_8tbs_spec": gbs / 8000.0, "bytes_per_call": call_bytes,
                         "unique_experts_mean": sum(self.U) / K},
            "tensor": {"tflops": tflops, "frac_of_dense_bf16_peak": tflops / peaks["bf16_tflops"],
                       "flop_per_byte": intensity, "attainable_tflops": attainable,
                       "frac_of_attainable": tflops / attainable,
                       "attainable": "min(dense BF16 peak, measured HBM copy peak x flop/byte)"},
        }


def supplementary_rows(args, dev, peaks, skip):
    """The other configurations, one short timed run each (W warm-up and K
    timed steps as for the headline line); weights are shared by the T of a
    workload and freed before the next workload."""
    import gc

    import torch
    from mixture_experts_ffn_gate_gb300 import synth
    rows = []
    for entry, Ts in SUPPLEMENTARY:
        name, _, how = entry.partition("+")
        wl = synth.WORKLOADS[name]
        Ts = [T for T in Ts if (entry, T) != skip]
        if not Ts:
            continue
        R = max(layer_count(wl, T, args.layers, BPE["mxfp8" if how == "mxfp8" else "bf16"])[0] for T in Ts)
        make = synth.make_weights_mxfp8 if how == "mxfp8" else synth.make_weights
        layers = [make(wl, device=dev, layer=r) for r in range(R)]
        routers = [synth.make_router(wl, device=dev, layer=r) for r in range(R)] if how == "router" else None
        bias = synth.make_bias(wl)
        for T in Ts:
            # the training-size rows take ms per call: at most 100 timed steps
            # each, so that the default run (2000 steps) stays within minutes
            K = min(args.steps, 100) if T >= 2048 else args.steps
            run = Measure(wl, T, dev, K, max(3, args.warmup), {"auto": 0, "decode": 1, "grouped": 2}[
                args.path] if how not in ("backward", "train") else 0, layers, bias, 0, args.eager,
                routers=routers, mx=how == "mxfp8", backward=how == "backward", train=how == "train")
            with ClockSampler(dev.index or 0) as clocks:
                total_ms, _ = run.timed(1)
                kern = run.stages()
            row = {"workload": name, "T": T, "layers": R, "steps": K, "warmup": run.warm_steps}
            if how == "router":
                row["entry"] = ("moe_ffn_forward_router: router weights W_r [E,H] ~ N(0,1/H) and the "
                                "workload's bias passed instead of logits; the projection runs inside the call")
            if how == "backward":
                row["entry"] = ("moe_ffn_backward: dx, dlogits, dW_gate_up and dW_down (FP32) for dout ~ N(0,1) "
                                "FP32; gate/up recomputed from x inside the call")
                row["dtype"] = "bf16 inputs, f32 arithmetic and gradients"
            if how == "train":
                row["entry"] = ("moe_ffn_forward_train then moe_ffn_backward_train: a training step (output and "
                                "all four gradients for dout ~ N(0,1) FP32); the forward keeps g and u in a state "
                                "buffer, so the backward does not recompute gate/up")
                row["dtype"] = "bf16 inputs, f32 arithmetic and gradients"
            if how == "mxfp8":
                row["entry"] = ("moe_ffn_forward_mxfp8: the same seeded weights quantised to MXFP8 (E4M3 "
                                "codes, one E8M0 scale per 32 elements along K); bytes per weight 1 + 1/32")
                row["dtype"] = "mxfp8 weights, bf16 activations, f32 arithmetic"
            row.update(run.summary(total_ms, kern, peaks, 1))
            row["clocks"] = clocks.summary()
            rows.append(row)
            del run
        del layers
        gc.collect()
        torch.cuda.empty_cache()
    return rows


def main():
    args = parse()
    from mixture_experts_ffn_gate_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    if args.E is not None:   # a smaller variant of the shape, for profiler captures
        import dataclasses
        wl = dataclasses.replace(wl, E=args.E, name=f"{wl.name}_e{args.E}")
    T = args.T if args.T is not None else wl.T[0]
    if args.impl == "reference":
        reference_arm(args, wl, T)
        return

    import torch
    import torch.distributed as dist

    import __graft_entry__
    from mixture_experts_ffn_gate_gb300 import moe_ffn as m

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    __graft_entry__.build() if rank == 0 else None
    if world > 1:
        dist.barrier()
    m.lib()

    dev = torch.device("cuda", local)
    K, W = args.steps, max(3, args.warmup)
    bias = synth.make_bias(wl)
    mx = args.weights == "mxfp8"
    if mx or args.backward or args.train:   # no host-buffer form; the oracle baseline is the BF16 forward
        args.no_e2e = args.skip_baseline = True
    R, touched = layer_count(wl, T, args.layers, BPE[args.weights])
    make = synth.make_weights_mxfp8 if mx else synth.make_weights
    layers = [make(wl, device=dev, layer=r) for r in range(R)]
    wgu, wd = (None, None) if mx else layers[0]
    path_code = {"auto": m.MOE_PATH_AUTO, "decode": m.MOE_PATH_DECODE,
                 "grouped": m.MOE_PATH_GROUPED}[args.path]
    run = Measure(wl, T, dev, K, W, path_code if not (args.backward or args.train) else 0, layers, bias, rank,
                  args.eager, mx=mx, backward=args.backward, train=args.train)
    stream = run.stream
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sum = torch.empty((), dtype=torch.float32, device=dev)

    def do_flush(j):
        # write more than L2 holds; then read half of it back, so L2 ends up
        # full of clean lines and the write-back of the dirty ones happens
        # here, outside the step's events, not during the next step
        flush.fill_(float(j))
        if args.flush == "write+read":
            torch.sum(flush[: FLUSH_BYTES // 8], dim=0, out=flush_sum)

    with ClockSampler(local) as clocks:
        total_ms, wall = run.timed(world)
        kern_avg = run.stages()

        # cold single calls: L2 flushed before each, each between its own events
        n_cold = min(K, args.cold_steps)
        c_starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_cold)]
        c_ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_cold)]
        for j in range(n_cold):
            do_flush(j)
            c_starts[j].record(stream)
            run.call(W + j, stream)
            c_ends[j].record(stream)
        torch.cuda.synchronize()
        cold_ms = [s.elapsed_time(e) for s, e in zip(c_starts, c_ends)]

        # e2e: the host-buffer entry point, called step after step from Python
        # (pinned inputs copied in and the output copied out inside the region)
        e2e = None
        if not args.no_e2e:
            NB = run.NB
            xh = [b[0].cpu().pin_memory() for b in run.batches]
            lh = [b[1].cpu().pin_memory() for b in run.batches]
            oh = torch.empty((T, wl.H), dtype=torch.float32).pin_memory()
            wsh = m.new_workspace(T, wl.H, wl.I, wl.E, wl.k, device=dev, host=True)

            def host_call(j):
                lw_gu, lw_d = layers[j % R]
                m.moe_ffn_forward_host(xh[j % NB], lh[j % NB], lw_gu, lw_d, wl.k, oh, wsh,
                                       opts=run.new_opts(), stream=stream)
            mark0 = torch.cuda.Event(enable_timing=True)
            mark1 = torch.cuda.Event(enable_timing=True)
            for j in range(W):
                host_call(j)
            torch.cuda.synchronize()
            mark0.record(stream)
            for j in range(W, W + K):
                host_call(j)
            mark1.record(stream)
            torch.cuda.synchronize()
            e2e = {"ms": mark0.elapsed_time(mark1)}

    # max over ranks
    total_ms, e2e_max = max_over_ranks([total_ms, e2e["ms"] if e2e else 0.0], world, dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks = load_peaks()
    head = run.summary(total_ms, kern_avg, peaks, world)
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": run.warm_steps, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp8 weights, bf16 activations" if mx else "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "T": T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                   "path": head["path"],
                   "layers": R,
                   "l2": (f"inputs larger than L2: {R} layers' weights "
                          f"({R * wl.weight_bytes() * BPE[args.weights] / 2 / 1e9:.1f} GB) cycled step by step, "
                          f"{touched / 1e6:.0f} MB read per step at most, fresh tokens per step"),
                   "timing": ("the K steps launched from Python" if args.eager
                              else "CUDA graph of the K steps, replayed once untimed (its first launch "
                                   "uploads it) and once timed")
                             + ", CUDA events before and after on the launching stream",
                   "parallelism": f"replicas x{world} (independent token streams)"},
        "roofline": head["roofline"],
        "call_hbm": head["call_hbm"],
        "tensor": head["tensor"],
        "cold_call": {"us_median": 1e3 * statistics.median(cold_ms), "us_mean": 1e3 * sum(cold_ms) / n_cold,
                      "calls": n_cold,
                      "method": (f"L2 flushed before each call ({FLUSH_BYTES >> 20} MB write"
                                 + (f", then {FLUSH_BYTES >> 21} MB read" if args.flush == "write+read" else "")
                                 + "), each call between its own CUDA events")},
        "gpu_launches": run.n_stages * K,
        "stages": run.stage_names,
        "wall_s": wall,
    }
    if e2e is not None:
        line["e2e"] = {"value": whole_job_tokens_per_s(T, K, world, e2e_max), "unit": "tokens/s",
                       "h2d_bytes_per_step": T * wl.H * 2 + T * wl.E * 4,
                       "d2h_bytes_per_step": T * wl.H * 4}
    line["clocks"] = clocks.summary()
    if world == 1 and not args.skip_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, T, wgu, wd, bias)
    if world == 1 and not args.no_supplementary:
        del run, layers, wgu, wd, flush
        torch.cuda.empty_cache()
        line["supplementary"] = supplementary_rows(args, dev, peaks, skip=(wl.name, T))
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
