"""Per-CTA timeline of the fused decode kernel, from the instrumented build.

    python -m mixture_experts_ffn_gate_gb300.timeline [--workload NAME] [--T T]
                                                      [--steps K] [--reps N]
                                                      [--router | --mxfp8]

Builds the library with -DMOE_FUSED_TIMELINE (a separate build; the product
build carries no stamps), runs K calls of a decode workload back to back as
one CUDA-graph replay over fresh seeded tokens and enough layers' weights that
no call finds its weights in L2 (as the benchmark does), and reads the stamps
of the last call.  Each CTA records SM clock stamps of its phase boundaries
(the kernel source lists the slots); this prints, per event, the 0th, 50th
and 100th percentile over the CTAs in microseconds from the earliest CTA's
entry, aligned by the global timer each CTA also records.  Chunk arrivals are
the times consumer warp 0 passed each ring slot's full barrier.

The stamps are debugging evidence, not timing: the per-call time printed
beside them comes from CUDA events around the replay of the instrumented
build.  The compiler may move a clock read across a block barrier, so stamps
right after one are approximate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics

EVENTS = {1: "past_griddep_wait", 14: "router_slices_summed", 15: "router_logits_polled", 56: "route_start", 57: "route_end", 58: "flags_read", 2: "routed",
          3: "first_copy_issued", 4: "last_gate_up_copy_issued", 5: "last_w_down_copy_issued",
          6: "phase_a_done", 7: "exchange_done", 8: "act_staged", 9: "phase_b_done", 10: "out_written",
          11: "producer_drained"}


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--workload", default="decode_h2048_i768_e128_k8")
    p.add_argument("--T", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--reps", type=int, default=5)
    p.add_argument("--router", action="store_true",
                   help="pass router weights instead of logits (moe_ffn_forward_router)")
    p.add_argument("--mxfp8", action="store_true",
                   help="MXFP8 expert weights (moe_ffn_forward_mxfp8)")
    args = p.parse_args(argv)

    from . import _build
    os.environ["MOE_FFN_LIB"] = _build.build_timeline()
    import numpy as np
    import torch

    from . import moe_ffn as m
    from . import synth

    wl = synth.WORKLOADS[args.workload]
    T, K = args.T, args.steps
    touched = 6 * wl.H * wl.I * min(wl.E, T * wl.k)
    R = max(2, -(-3 * (129 << 20) // touched))
    R = min(R, max(1, int((72 << 30) // wl.weight_bytes())))
    dev = torch.device("cuda")
    make = synth.make_weights_mxfp8 if args.mxfp8 else synth.make_weights
    layers = [make(wl, device=dev, layer=r) for r in range(R)]
    bias = synth.make_bias(wl)
    batches = [synth.make_tokens(wl, T, call=i, device=dev, bias=bias) for i in range(K + 5)]
    routers = [synth.make_router(wl, device=dev, layer=r) for r in range(R)] if args.router else None
    ws = (m.new_router_workspace if args.router else m.new_workspace)(T, wl.H, wl.I, wl.E, wl.k)
    rbias = bias.to(dev)
    out = torch.empty((T, wl.H), dtype=torch.float32, device=dev)

    def call(j, s):
        x, L = batches[j % len(batches)]
        o = m.moe_ffn_opts()
        if args.mxfp8:
            m.moe_ffn_forward_mxfp8(x, L, *layers[j % R], wl.k, out=out, workspace=ws, opts=o, stream=s)
            return o
        g, d = layers[j % R]
        if routers is not None:
            m.moe_ffn_forward_router(x, routers[j % R], rbias, g, d, wl.k, out=out, workspace=ws, opts=o,
                                     stream=s)
        else:
            m.moe_ffn_forward_ex(x, L, g, d, wl.k, out=out, workspace=ws, opts=o, stream=s)
        return o

    o = call(0, torch.cuda.current_stream())
    if o.path_taken != m.MOE_PATH_DECODE_FUSED:
        raise SystemExit(f"{args.workload} at T={T} does not take the fused decode kernel")
    for j in range(5):
        call(j, torch.cuda.current_stream())
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        s = torch.cuda.current_stream()
        for j in range(K):
            call(5 + j, s)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    buf = np.zeros(n_sm * 64, dtype=np.uint64)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rows = []
    for _ in range(args.reps):
        torch.cuda.synchronize()
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        if m.lib().moe_ffn_debug_fused_timeline(buf.ctypes.data, n_sm) != 0:
            raise SystemExit("reading the timeline failed")
        tl = buf.reshape(n_sm, 64).astype(np.int64)
        gt0, gt1, c0 = tl[:, 63], tl[:, 62], tl[:, 0]
        mhz = float(np.median((tl[:, 10] - c0) / np.maximum(gt1 - gt0, 1) * 1e3))
        entry = (gt0 - gt0.min()) / 1e3

        def at(i):
            return (tl[:, i] - c0) / mhz + entry

        row = {"us_per_call_instrumented": e0.elapsed_time(e1) / K * 1e3, "sm_mhz": mhz,
               "kernel_us": float((gt1.max() - gt0.min()) / 1e3),
               "entry_spread_us": float(entry.max())}
        for i, name in EVENTS.items():
            row[name] = [round(float(np.percentile(at(i), q)), 2) for q in (0, 50, 100)]
        n_ch = min(40, int(np.median(tl[:, 12])))
        row["phase_a_chunks"] = int(np.median(tl[:, 13]))
        row["chunk_arrival_median"] = [round(float(np.median(at(16 + c))), 2) for c in range(n_ch)]
        rows.append(row)
    best = min(rows, key=lambda r: r["us_per_call_instrumented"])
    best["us_per_call_instrumented_median"] = statistics.median(r["us_per_call_instrumented"] for r in rows)
    print(json.dumps({"workload": args.workload, "T": T, "router": args.router, "mxfp8": args.mxfp8,
                      "steps": K, "layers": R,
                      **best}))


if __name__ == "__main__":
    main()
