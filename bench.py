"""Benchmark of the BitLinear hot path on B300 (one JSON line on stdout).

Workload (default): decode on 2B-shaped layers - hidden 2560, projections
q/k/v/o 2560x2560, gate/up 2560->6912, down 6912->2560 - for M = 1, 4 and
16 tokens.  One step runs, for each M, the seven projections of one layer
chained through the fused RMSNorm+int8 quantiser:
    h = quant(x); q,k,v = fwd(h); o = fwd(quant(v)); gate,up = fwd(quant(o));
    down = fwd(quant(up))
Every (M, projection) has its own packed weights, and steps rotate over
ROT distinct weight sets (535 MB in total, more than 4x the 126 MB L2), so
every weight byte is read from HBM.  Each step is one CUDA-graph replay of
the library's calls (the kernels chain with programmatic dependent launch).

value  = algorithmic bytes of the whole step (packed weights, int8 and bf16
         activations, scales, outputs) / device time, summed over ranks.
e2e    = the same bytes / time of a step that also copies the step's inputs
         from pinned host memory and reads its outputs back.
roofline: the decode GEMV (dominant kernel) timed per launch with CUDA events.
prefill: the 2B prefill chain at M = 4096 (int8-exact tensor-core GEMM), TOPS.
cpu_baseline: the CPU oracle on one full step (all three M), host cores.

--impl reference times the CPU oracle (the reference arm of this build) on
the same workload and prints the same kind of line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "BitLinear decode GB/s (% HBM peak) and prefill int8 TOPS, 2B-shape layers"
WORKLOAD = "decode_2b"
M_LIST = (1, 4, 16)
ROT = 9
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1400.0, "fallback"


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------ clocks ------

class ClockSampler:
    """nvidia-smi samples during the timed region (clocks, throttle reasons)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ workload ----

def algo_bytes_forward(M, N, K):
    Np, Kp = -(-N // 16) * 16, -(-K // 128) * 128
    return Np * Kp // 4 + M * K + 4 * M + 2 * M * N + 4


def algo_bytes_quant(M, K):
    return 2 * M * K + M * K + 4 * M


def chain_plan(shapes):
    """(kind, args) list for one layer: quant/forward with buffer names."""
    d = {n: (N, K) for n, N, K in shapes}
    return [
        ("quant", "x", "h0"),
        ("fwd", "h0", "q"), ("fwd", "h0", "k"), ("fwd", "h0", "v"),
        ("quant", "v", "h1"), ("fwd", "h1", "o"),
        ("quant", "o", "h2"), ("fwd", "h2", "gate"), ("fwd", "h2", "up"),
        ("quant", "up", "h3"), ("fwd", "h3", "down"),
    ], d


class DecodeBench:
    def __init__(self, torch, bl, inputs, dev):
        self.torch, self.bl, self.inputs, self.dev = torch, bl, inputs, dev
        wl = inputs.WORKLOADS[WORKLOAD]
        self.shapes = wl["shapes"]
        self.plan, self.dims = chain_plan(self.shapes)
        self.eps_w, self.eps_a = wl["eps_w"], wl["eps_a"]
        hidden = self.dims["q"][1]
        T = torch
        # weights: ROT sets x M x projection
        self.w = {}
        for r in range(ROT):
            for M in M_LIST:
                for i, (name, N, K) in enumerate(self.shapes):
                    seed = wl["seed"] * 100000 + r * 1000 + M * 10 + i
                    W = inputs.weights_fp32(N, K, seed=seed, device=dev)
                    self.w[(r, M, name)] = bl.pack_weights(W, self.eps_w)
                    del W
        # activation buffers per M
        self.buf = {}
        for M in M_LIST:
            b = {"x": inputs.activations_bf16(M, hidden, seed=wl["seed"] * 7 + M, device=dev)}
            for name, N, K in self.shapes:
                b[name] = T.empty(M, N, dtype=T.bfloat16, device=dev)
            for h, (src) in (("h0", "x"), ("h1", "v"), ("h2", "o"), ("h3", "up")):
                K = b[src].shape[1]
                b[h] = (T.empty(M, K, dtype=T.int8, device=dev), T.empty(M, dtype=T.float32, device=dev))
            self.buf[M] = b
        self.bytes_step = 0
        self.gemv_bytes = 0
        self.gemv_launches = 0
        self.launches = 0
        for M in M_LIST:
            for kind, a, b_ in self.plan:
                if kind == "quant":
                    self.bytes_step += algo_bytes_quant(M, self.buf[M][a].shape[1])
                else:
                    N, K = self.dims[b_]
                    self.bytes_step += algo_bytes_forward(M, N, K)
                    self.gemv_bytes += algo_bytes_forward(M, N, K)
                    self.gemv_launches += 1
                self.launches += 1
        torch.cuda.synchronize()

    def run_step(self, r, kinds=("quant", "fwd")):
        bl = self.bl
        for M in M_LIST:
            b = self.buf[M]
            for kind, a, o in self.plan:
                if kind == "quant" and "quant" in kinds:
                    q, s = b[o]
                    x = b[a]
                    bl.bitlinear_quant_act(x, None, M, x.shape[1], self.eps_a, q, s)
                elif kind == "fwd" and "fwd" in kinds:
                    q, s = b[a]
                    packed, gamma = self.w[(r, M, o)]
                    N, K = self.dims[o]
                    bl.bitlinear_forward(q, s, packed, gamma, M, N, K, b[o])

    def capture(self, stream, h2d=None, d2h=None):
        torch = self.torch
        with torch.cuda.stream(stream):  # one eager step: host-side set-up happens outside capture
            self.run_step(0)
        torch.cuda.synchronize()
        graphs = []
        for r in range(ROT):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                if h2d is not None:
                    for M in M_LIST:
                        self.buf[M]["x"].copy_(h2d[M], non_blocking=True)
                self.run_step(r)
                if d2h is not None:
                    for M in M_LIST:
                        d2h[M].copy_(self.buf[M]["down"], non_blocking=True)
            graphs.append(g)
        return graphs


def time_graphs(torch, graphs, steps, warmup, stream, barrier=None):
    for i in range(warmup):
        graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(steps):
            graphs[(warmup + i) % len(graphs)].replay()
        e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return e0.elapsed_time(e1)  # ms


def per_kernel_times(torch, db, stream, reps=20):
    """Average device duration of the decode GEMV and of the quantiser: each
    is captured alone (same launches, same rotating weights, PDL between
    kernels) and the replay time is divided by the number of launches."""
    def graph_of(kind):
        gs = []
        for r in range(ROT):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                db.run_step(r, kinds=(kind,))
            gs.append(g)
        return gs

    out = {}
    for kind in ("fwd", "quant"):
        gs = graph_of(kind)
        ms = time_graphs(torch, gs, reps * ROT, ROT, stream)
        n = sum(1 for M in M_LIST for k, _, _ in db.plan if k == kind) * reps * ROT
        out[kind + "_avg_us"] = 1000.0 * ms / n
        del gs
    out["gemv_avg_bytes"] = db.gemv_bytes / db.gemv_launches
    out["gemv_gbs"] = out["gemv_avg_bytes"] / (out["fwd_avg_us"] * 1e-6) / 1e9
    # per shape: a graph of 9 rotating launches of one (M, projection)
    per_shape = {}
    for M in M_LIST:
        b = db.buf[M]
        for kind, a, o in db.plan:
            if kind != "fwd" or o in ("k", "v", "up"):
                continue
            N, K = db.dims[o]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for r in range(ROT):
                    q, s = b[a]
                    packed, gamma = db.w[(r, M, o)]
                    db.bl.bitlinear_forward(q, s, packed, gamma, M, N, K, b[o])
            ms = time_graphs(torch, [g], reps, 3, stream)
            us = 1000.0 * ms / (reps * ROT)
            per_shape[f"M{M}_{N}x{K}"] = {"us": round(us, 3),
                                          "gbs": round(algo_bytes_forward(M, N, K) / (us * 1e-6) / 1e9, 1)}
            del g
    out["per_shape"] = per_shape
    return out


def prefill_bench(torch, bl, inputs, dev, stream, steps=5, warmup=3, M=4096):
    """2B prefill chain at M tokens: TOPS of the tensor-core GEMM (2*M*N*K per
    projection) and the whole chain."""
    wl = inputs.WORKLOADS["prefill_2b"]
    shapes = wl["shapes"]
    plan, dims = chain_plan(shapes)
    hidden = dims["q"][1]
    w = {}
    for i, (name, N, K) in enumerate(shapes):
        W = inputs.weights_fp32(N, K, seed=wl["seed"] * 100 + i, device=dev)
        w[name] = bl.pack_weights(W, wl["eps_w"])
        del W
    b = {"x": inputs.activations_bf16(M, hidden, seed=wl["seed"] * 1000 + M, outlier_frac=0.01,
                                      outlier_scale=20.0, device=dev)}
    for name, N, K in shapes:
        b[name] = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    for h, src in (("h0", "x"), ("h1", "v"), ("h2", "o"), ("h3", "up")):
        K = b[src].shape[1]
        b[h] = (torch.empty(M, K, dtype=torch.int8, device=dev), torch.empty(M, dtype=torch.float32, device=dev))
    ops = sum(2 * M * dims[o][0] * dims[o][1] for k, _, o in plan if k == "fwd")

    def step(kinds=("quant", "fwd")):
        for kind, a, o in plan:
            if kind == "quant" and "quant" in kinds:
                q, s = b[o]
                bl.bitlinear_quant_act(b[a], None, M, b[a].shape[1], wl["eps_a"], q, s)
            elif kind == "fwd" and "fwd" in kinds:
                q, s = b[a]
                N, K = dims[o]
                bl.bitlinear_forward(q, s, w[o][0], w[o][1], M, N, K, b[o])

    with torch.cuda.stream(stream):  # eager warm-up outside capture
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    ms = time_graphs(torch, [g], steps, warmup, stream)
    chain_tops = ops * steps / (ms * 1e-3) / 1e12
    # GEMM alone (quantised activations already in place)
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        step(kinds=("fwd",))
    ms2 = time_graphs(torch, [g2], steps, warmup, stream)
    gemm_tops = ops * steps / (ms2 * 1e-3) / 1e12
    del w, b, g, g2
    return {"workload": f"prefill_2b M={M}", "chain_tops": round(chain_tops, 1),
            "gemm_tops": round(gemm_tops, 1), "gemm_ms_per_chain": round(ms2 / steps, 4),
            "tokens_per_s": round(M * steps / (ms * 1e-3), 1)}


# ------------------------------------------------------------ CPU oracle --

def oracle_step_sample(budget_s=20.0):
    """The oracle on the decode workload: for each M, quantise, unpack the
    packed weights, matmul and rescale, for the seven projections of one
    layer.  Runs whole steps until `budget_s` is spent (at least one)."""
    import numpy as np
    import oracle
    from bitlinear_02_b300 import inputs
    wl = inputs.WORKLOADS[WORKLOAD]
    shapes = wl["shapes"]
    plan, dims = chain_plan(shapes)
    hidden = dims["q"][1]
    packed = {}
    gam = {}
    for i, (name, N, K) in enumerate(shapes):
        w = inputs.weights_fp32(N, K, seed=wl["seed"] * 100 + i).numpy()
        g = oracle.gamma(w)
        packed[name] = oracle.pack(oracle.ternarize(w, g, wl["eps_w"]))
        gam[name] = g
    xs = {M: inputs.bf16_bits(inputs.activations_bf16(M, hidden, seed=M)) for M in M_LIST}
    nbytes = 0
    t0 = time.perf_counter()
    steps = 0
    while True:
        for M in M_LIST:
            acts = {"x": xs[M]}
            for kind, a, o in plan:
                if kind == "quant":
                    acts[o] = oracle.quant_act(acts[a], None, wl["eps_a"])
                    nbytes += algo_bytes_quant(M, acts[a].shape[1])
                else:
                    q, s = acts[a]
                    N, K = dims[o]
                    wq, _ = oracle.unpack(packed[o], N, K)
                    acc = oracle.matmul(q, wq)
                    acts[o] = oracle.epilogue(acc, s, gam[o])
                    nbytes += algo_bytes_forward(M, N, K)
        steps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, steps, dt, oracle.threads()


# ------------------------------------------------------------ main --------

def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return 0
    gbs, steps, dt, cores = oracle_step_sample(budget_s=max(5.0, min(60.0, 10.0 * max(1, args.steps) / 10)))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * dt / steps, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8/int32 (fp32 scales)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": list(M_LIST), "hidden": 2560, "ffn": 6912,
                   "projections": 7, "sample": f"{steps} whole step(s)"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{steps} whole decode step(s) (M=1,4,16 x 7 projections) in {dt:.1f} s"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import bitlinear_02_b300 as bl
    from bitlinear_02_b300 import inputs

    ws, rank, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    barrier = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        barrier = lambda: dist.barrier()
    bl.load_library()
    hbm_peak, bf16_peak, bf16_sust, peak_kind = peaks()
    stream = torch.cuda.Stream()

    db = DecodeBench(torch, bl, inputs, dev)
    graphs = db.capture(stream)
    sampler = ClockSampler(local)
    with sampler:
        ms = time_graphs(torch, graphs, args.steps, args.warmup, stream, barrier)
    clocks = sampler.summary()
    if ws > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    total_bytes = db.bytes_step * args.steps * ws
    value = total_bytes / (ms * 1e-3) / 1e9
    del graphs

    # e2e: pinned host inputs copied in, outputs read back, every step
    h2d = {M: db.buf[M]["x"].cpu().pin_memory() for M in M_LIST}
    d2h = {M: torch.empty_like(db.buf[M]["down"], device="cpu").pin_memory() for M in M_LIST}
    g_e2e = db.capture(stream, h2d=h2d, d2h=d2h)
    for i in range(args.warmup):
        g_e2e[i % ROT].replay()
    torch.cuda.synchronize()
    n_e2e = max(10, args.steps // 2)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        g_e2e[i % ROT].replay()
        torch.cuda.current_stream().synchronize()
        stream.synchronize()
        _ = float(d2h[16][0, 0])  # read the result on the host
    e2e_s = time.perf_counter() - t0
    e2e_val = db.bytes_step * n_e2e * ws / e2e_s / 1e9
    h2d_bytes = sum(t.numel() * t.element_size() for t in h2d.values())
    d2h_bytes = sum(t.numel() * t.element_size() for t in d2h.values())
    del g_e2e

    kt = per_kernel_times(torch, db, stream)
    gemv_frac = kt["gemv_gbs"] / hbm_peak
    prefill = None
    if not args.no_prefill:
        prefill = prefill_bench(torch, bl, inputs, dev, stream)
        prefill["roofline"] = {"bound": "tensor", "achieved": prefill["gemm_tops"],
                               "peak": round(bf16_peak, 1), "unit": "TFLOP/s",
                               "frac": round(prefill["gemm_tops"] / bf16_peak, 4),
                               "peak_note": f"{peak_kind} cuBLAS bf16 burst; the GEMM runs f16 MMA (same rate); "
                                            "sm_103a has no int8 tcgen05 MMA"}
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        gbs, steps, dt, cores = oracle_step_sample(budget_s=15.0)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{steps} whole decode step(s) (M=1,4,16 x 7 projections, unpack+matmul+rescale) in {dt:.1f} s"}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 x ternary -> int32 (f16 tensor-core operands, exact), bf16 out",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": list(M_LIST), "hidden": 2560, "ffn": 6912,
                   "projections": "q,k,v,o 2560x2560; gate,up 2560->6912; down 6912->2560",
                   "l2": f"inputs larger than L2: {ROT} rotating weight sets "
                         f"({ROT * sum(db.w[(0, M, n)][0].numel() for M in M_LIST for n, _, _ in db.shapes) / 1e6:.0f} MB packed)",
                   "bytes_per_step": db.bytes_step, "graph": "one CUDA graph per step, PDL between kernels",
                   "parallelism": f"replicas x{ws}"},
        "hbm_frac_of_step": round(value / ws / hbm_peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(kt["gemv_gbs"], 1), "peak": round(hbm_peak, 1),
                     "unit": "GB/s", "frac": round(gemv_frac, 4), "traffic": None,
                     "kernel": "gemv_kernel (decode, M<=16)",
                     "launch_avg_us": round(kt["fwd_avg_us"], 3),
                     "algo_bytes_per_launch": round(kt["gemv_avg_bytes"]),
                     "peak_note": f"{peak_kind} HBM copy bandwidth",
                     "method": "GEMV launches alone in CUDA graphs (PDL chained), replay time / launches"},
        "kernels": {"quant_avg_us": round(kt["quant_avg_us"], 3), "gemv_per_shape": kt["per_shape"]},
        "prefill": prefill,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h_bytes,
                "mode": "graph replay of the public API calls incl. pinned H2D/D2H copies, host sync per step"},
        "gpu_launches": db.launches * args.steps,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
