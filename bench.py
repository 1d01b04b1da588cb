"""Benchmark of the BitLinear hot path on B300 (one JSON line on stdout).

Workload (default): one decode step of a stack of 2B-shaped layers, for
M = 1, 4 and 16 tokens.  A layer has the seven projections q/k/v/o
2560x2560, gate/up 2560->6912 and down 6912->2560, chained through the
fused RMSNorm + absmax int8 quantiser:
    h = x; q,k,v = f(h); o = f(v); gate,up = f(o); down = f(up); next x = down
The stack has LAYERS = 20 layers: 396 MB of packed 2-bit weights, the
0.4 GB the asi.tokyo write-up gives for the 2B model's weights, and more
than 3x the 126 MB L2, so every weight byte is read from HBM.  Each M runs
the whole stack; a step is all of it for the three M, replayed as one CUDA
graph.

The step runs the fused decode path: per M one bitlinear_act_stats of the
stack input, then per layer four bitlinear_forward_fused launches
(q,k,v | o | gate,up | down), each quantising its input on the fly.

value  = algorithmic bytes of the step (packed weights, activations in and
         out, scales; the same count as the unfused quant + forward calls)
         / device time, summed over ranks.
e2e    = the same bytes / wall time of steps that also copy each M's input
         from pinned host memory and read the last projection's output back.
roofline: the fused decode GEMV, bytes per launch / average launch time.
concurrent: the three M as independent decode streams (a graph branch per M,
         each with its own weight copy), the throughput when their dependent
         launches overlap.
chain, unfused: the same stack through the persistent fused-chain kernel
         (bitlinear_chain_run, one launch per M) and through separate
         bitlinear_quant_act + bitlinear_forward calls, for comparison.
sweep: the decode GEMV shape by shape (bitlinear_forward on a pre-quantised
         input, every launch reading its weights from HBM after an L2 flush),
         and bitlinear_quant_act on its own.
mid_m: batches of 32-256 tokens through the tensor-core GEMM, shape by shape
         (the crossover with the decode GEMV).
prefill: the 2B prefill chain at M = 4096 (int8-exact tensor-core GEMM), TOPS.
cpu_baseline: the CPU oracle on a bounded sample of the same workload.

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
LAYERS = 20
# DRAM bytes read per packed-weight byte by fused_gemv_kernel, from one ncu
# capture (profiles/fused_gemv_decode_2b_M16_full.md: 15.826 MB read over
# three launches holding 15.400 MB of packed weights).  Re-measure when the
# kernel changes.
FUSED_DRAM_PER_PACKED_BYTE = 1.0277
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


def replica_group(backend="nccl", device=None):
    """N > 1 (one process per GPU, torchrun environment): join the process
    group and return torch.distributed; None at N = 1.  The group carries
    only the barrier around the timed region and the max over ranks of its
    time: every rank runs its own replica of the whole workload."""
    ws, _, _ = dist_info()
    if ws == 1:
        return None
    import torch.distributed as dist
    if backend == "nccl" and device is not None:
        dist.init_process_group(backend, device_id=device)
    else:
        dist.init_process_group(backend)
    return dist


def max_over_ranks(torch, ms, device, dist):
    """The slowest rank's time of the timed region (ms)."""
    if dist is None:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_step, steps, ws, ms):
    """Whole-job GB/s: ws replicas each ran `steps` steps of bytes_step
    algorithmic bytes within the slowest rank's ms (weak scaling)."""
    return bytes_step * steps * ws / (ms * 1e-3) / 1e9


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


# projection inputs within a layer (chain slots relative to the layer):
# 0 = the layer input, i + 1 = output of the layer's projection i
LAYER_INPUTS = [0, 0, 0, 3, 4, 4, 6]


def layer_bytes(M, shapes):
    """Algorithmic bytes of one layer at M tokens (unfused-path count)."""
    plan, dims = chain_plan(shapes)
    width = {"x": dims["q"][1]}
    width.update({n: N for n, N, K in shapes})
    b = 0
    for kind, a, o in plan:
        if kind == "quant":
            b += algo_bytes_quant(M, width[a])
        else:
            N, K = dims[o]
            b += algo_bytes_forward(M, N, K)
    return b


class DecodeBench:
    """The decode stack: LAYERS x 7 packed projections shared by every M."""

    def __init__(self, torch, bl, inputs, dev, layers=LAYERS):
        self.torch, self.bl, self.inputs, self.dev = torch, bl, inputs, dev
        wl = inputs.WORKLOADS[WORKLOAD]
        self.shapes = wl["shapes"]
        self.layers = layers
        self.eps_w, self.eps_a = wl["eps_w"], wl["eps_a"]
        self.hidden = self.shapes[0][2]
        self.w = []  # (packed, gamma, N) per projection, layer-major
        for l in range(layers):
            for i, (name, N, K) in enumerate(self.shapes):
                W = inputs.weights_fp32(N, K, seed=wl["seed"] * 100000 + l * 10 + i, device=dev)
                packed, gamma = bl.pack_weights(W, self.eps_w)
                del W
                self.w.append((packed, gamma, N))
        self.packed_bytes = sum(p.numel() for p, _, _ in self.w)
        self.x = {M: inputs.activations_bf16(M, self.hidden, seed=wl["seed"] * 7 + M, device=dev)
                  for M in M_LIST}
        self.chains = {}
        for M in M_LIST:
            projs = []
            for l in range(layers):
                base = 7 * l
                for i, rel in enumerate(LAYER_INPUTS):
                    slot = (base if l > 0 else 0) if rel == 0 else base + rel
                    p, g, N = self.w[base + i]
                    projs.append(dict(packed=p, gamma=g, N=N, input=slot))
            self.chains[M] = bl.DecodeChain(M, self.hidden, projs, eps=self.eps_a)
        self.bytes_per_M = {M: layer_bytes(M, self.shapes) * layers for M in M_LIST}
        self.bytes_step = sum(self.bytes_per_M.values())
        self.launches = len(M_LIST)
        torch.cuda.synchronize()

    def run_step(self, stream, h2d=None, d2h=None):
        for M in M_LIST:
            if h2d is not None:
                self.x[M].copy_(h2d[M], non_blocking=True)
            self.chains[M].run(self.x[M], stream)
            if d2h is not None:
                d2h[M].copy_(self.chains[M].out[-1], non_blocking=True)

    def capture(self, stream, h2d=None, d2h=None):
        torch = self.torch
        with torch.cuda.stream(stream):  # one eager step: host-side set-up happens outside capture
            self.run_step(stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.run_step(stream, h2d, d2h)
        return g


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


def unfused_step_ms(torch, bl, db, stream, reps=5):
    """The same stack through the per-projection entry points: per layer
    h0 = quant(x); q,k,v = fwd(h0); h1 = quant(v); o = fwd(h1);
    h2 = quant(o); gate,up = fwd(h2); h3 = quant(up); down = fwd(h3),
    chained with programmatic dependent launch in one CUDA graph.  Returns
    ms per step (all M)."""
    T = torch
    bufs = {}
    for M in M_LIST:
        outs = [T.empty(M, N, dtype=T.bfloat16, device=db.dev) for _, N, _ in db.shapes]
        hs = [(T.empty(M, K, dtype=T.int8, device=db.dev), T.empty(M, dtype=T.float32, device=db.dev))
              for K in (db.hidden, db.shapes[2][1], db.shapes[3][1], db.shapes[5][1])]
        bufs[M] = (outs, hs)
    # (projection index, quantised input index) per layer; quant steps before them
    order = [("quant", 0, None), ("fwd", 0, 0), ("fwd", 1, 0), ("fwd", 2, 0), ("quant", 1, 2), ("fwd", 3, 1),
             ("quant", 2, 3), ("fwd", 4, 2), ("fwd", 5, 2), ("quant", 3, 5), ("fwd", 6, 3)]

    def step():
        for M in M_LIST:
            outs, hs = bufs[M]
            for l in range(db.layers):
                for kind, a, b in order:
                    if kind == "quant":
                        src = (db.x[M] if l == 0 else outs[6]) if a == 0 else outs[b]
                        q, sc = hs[a]
                        bl.bitlinear_quant_act(src, None, M, src.shape[1], db.eps_a, q, sc)
                    else:
                        packed, gamma, N = db.w[7 * l + a]
                        q, sc = hs[b]
                        bl.bitlinear_forward(q, sc, packed, gamma, M, N, q.shape[1], outs[a])

    with T.cuda.stream(stream):
        step()
    T.cuda.synchronize()
    g = T.cuda.CUDAGraph()
    with T.cuda.graph(g, stream=stream):
        step()
    ms = time_graphs(T, [g], reps, 2, stream)
    del g, bufs
    return ms / reps


class FusedDecode:
    """The decode stack through the fused path: per M one bitlinear_act_stats
    of the stack input, then per layer four bitlinear_forward_fused launches
    (q,k,v | o | gate,up | down), each quantising its input on the fly."""

    def __init__(self, torch, bl, db, m_list=M_LIST):
        self.torch, self.bl, self.db = torch, bl, db
        T = torch
        self.bufs = {}
        self.m_list = tuple(m_list)
        for M in self.m_list:
            outs = [[T.empty(M, N, dtype=T.bfloat16, device=db.dev) for _, N, _ in db.shapes]
                    for _ in range(db.layers)]
            stats = [[bl.new_stats(db.dev) for _ in range(4)] for _ in range(db.layers)]  # v, o, up, down
            x_stats = bl.new_stats(db.dev)
            self.bufs[M] = (outs, stats, x_stats)

    def run_step(self, stream, h2d=None, d2h=None):
        bl, db = self.bl, self.db
        for M in self.m_list:
            outs, stats, x_stats = self.bufs[M]
            if h2d is not None:
                db.x[M].copy_(h2d[M], non_blocking=True)
            bl.bitlinear_act_stats(db.x[M], M, db.hidden, db.eps_a, x_stats, stream)
            for l in range(db.layers):
                o = outs[l]
                st_v, st_o, st_up, st_down = stats[l]
                x = db.x[M] if l == 0 else outs[l - 1][6]
                xs = x_stats if l == 0 else stats[l - 1][3]

                def fp(i, st=None):
                    packed, gamma, N = db.w[7 * l + i]
                    return bl.FusedProj(packed.data_ptr(), gamma.data_ptr(), N, o[i].data_ptr(), None,
                                        st.data_ptr() if st is not None else None)

                K = db.hidden
                bl.bitlinear_forward_fused(x, xs, M, K, [fp(0), fp(1), fp(2, st_v)], db.eps_a, stream)
                bl.bitlinear_forward_fused(o[2], st_v, M, o[2].shape[1], [fp(3, st_o)], db.eps_a, stream)
                bl.bitlinear_forward_fused(o[3], st_o, M, o[3].shape[1], [fp(4), fp(5, st_up)], db.eps_a, stream)
                # the last layer's output feeds nothing here: no factors for it
                last = l == db.layers - 1
                bl.bitlinear_forward_fused(o[5], st_up, M, o[5].shape[1], [fp(6, None if last else st_down)],
                                           db.eps_a, stream)
            if d2h is not None:
                d2h[M].copy_(outs[-1][6], non_blocking=True)

    def capture(self, stream, h2d=None, d2h=None):
        torch = self.torch
        with torch.cuda.stream(stream):
            self.run_step(stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.run_step(stream, h2d, d2h)
        return g

    launches = len(M_LIST) * (1 + 4 * LAYERS)


def prefill_bench(torch, bl, inputs, dev, stream, steps=5, warmup=3, M=4096):
    """2B prefill chain at M tokens (the seven projections chained through the
    quantiser, f16-activation path: bitlinear_quant_act_f16 +
    bitlinear_forward_f16): TOPS of the tensor-core GEMMs (2*M*N*K per
    projection) and of the whole chain."""
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
        b[h] = (torch.empty(M, K, dtype=torch.float16, device=dev), torch.empty(M, dtype=torch.float32, device=dev))
    ops = sum(2 * M * dims[o][0] * dims[o][1] for k, _, o in plan if k == "fwd")

    def step(kinds=("quant", "fwd")):
        for kind, a, o in plan:
            if kind == "quant" and "quant" in kinds:
                q, s = b[o]
                bl.bitlinear_quant_act_f16(b[a], None, M, b[a].shape[1], wl["eps_a"], q, s)
            elif kind == "fwd" and "fwd" in kinds:
                q, s = b[a]
                N, K = dims[o]
                bl.bitlinear_forward_f16(q, s, w[o][0], w[o][1], M, N, K, b[o])

    with torch.cuda.stream(stream):  # eager warm-up outside capture
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    ms = time_graphs(torch, [g], steps, warmup, stream)
    chain_tops = ops * steps / (ms * 1e-3) / 1e12
    # GEMMs alone (quantised activations already in place)
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        step(kinds=("fwd",))
    ms2 = time_graphs(torch, [g2], steps, warmup, stream)
    gemm_tops = ops * steps / (ms2 * 1e-3) / 1e12
    del w, b, g, g2
    return {"workload": f"prefill_2b M={M}", "path": "quant_act_f16 + forward_f16 (tensor-map activations)",
            "chain_tops": round(chain_tops, 1), "gemm_tops": round(gemm_tops, 1),
            "gemm_ms_per_chain": round(ms2 / steps, 4), "gemm_launches_per_chain": 7,
            "gemm_us_per_launch": round(1000 * ms2 / steps / 7, 2),
            "tokens_per_s": round(M * steps / (ms * 1e-3), 1)}


# ------------------------------------------------------------ CPU oracle --

def oracle_step_sample(budget_s=20.0):
    """The oracle on a bounded sample of the decode workload: one layer of
    the 2B-shape stack for each M (quantise, unpack the packed weights,
    matmul, rescale, for the seven chained projections), repeated until
    `budget_s` is spent (at least once).  Returns GB/s of the same
    algorithmic bytes as the GPU line, steps, seconds, threads."""
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
    reps = 0
    while True:
        for M in M_LIST:
            acts = {"x": xs[M]}
            for kind, a, o in plan:
                if kind == "quant":
                    acts[o] = oracle.quant_act(acts[a], None, wl["eps_a"])
                else:
                    q, s = acts[a]
                    N, K = dims[o]
                    wq, _ = oracle.unpack(packed[o], N, K)
                    acc = oracle.matmul(q, wq)
                    acts[o] = oracle.epilogue(acc, s, gam[o])
            nbytes += layer_bytes(M, shapes)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, reps, dt, oracle.threads()


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
        "config": {"workload": WORKLOAD, "M": list(M_LIST), "layers": LAYERS, "hidden": 2560, "ffn": 6912,
                   "projections": 7, "sample": f"{steps} x one layer per M"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{steps} x one 2B-shape layer for each M=1,4,16 (7 chained projections) "
                                   f"in {dt:.1f} s"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def profile_gemm(spec):
    """--profile-gemm N,K,M[,int8]: one prefill GEMM shape, 3 warm-up + 20
    timed calls (the driver for ncu captures of the GEMM kernels)."""
    import torch
    import bitlinear_02_b300 as bl
    from bitlinear_02_b300 import inputs
    parts = spec.split(",")
    N, K, M = (int(v) for v in parts[:3])
    f16 = not (len(parts) > 3 and parts[3] == "int8")
    dev = torch.device("cuda:0")
    w = inputs.weights_fp32(N, K, seed=1, device=dev)
    packed, gamma = bl.pack_weights(w, 1e-5)
    x = inputs.activations_bf16(M, K, seed=2, device=dev)
    q, s = bl.quant_act_f16(x) if f16 else bl.quant_act(x)
    fwd = bl.forward_f16 if f16 else bl.forward
    out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        fwd(q, s, packed, gamma, N, out=out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(20):
        fwd(q, s, packed, gamma, N, out=out)
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / 20
    assert bl.bitlinear_check_status() == bl.OK
    print(json.dumps({"profile": "gemm", "N": N, "K": K, "M": M, "activations": "f16" if f16 else "int8",
                      "us": round(ms * 1000, 2), "tflops": round(2 * M * N * K / ms / 1e9, 1)}))
    return 0


def profile_fused(spec):
    """--profile-fused L,M: the fused decode path (act_stats + 4 fused GEMV
    launches per layer) on an L-layer 2B-shape stack at M tokens, eagerly
    launched: 3 warm-up + 5 timed passes (driver for ncu captures)."""
    import torch
    import bitlinear_02_b300 as bl
    from bitlinear_02_b300 import inputs
    L, M = (int(v) for v in spec.split(","))
    dev = torch.device("cuda:0")
    bl.load_library()
    db = DecodeBench(torch, bl, inputs, dev, layers=L)
    fd = FusedDecode(torch, bl, db, m_list=(M,))
    stream = torch.cuda.current_stream()
    for _ in range(3):
        fd.run_step(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        fd.run_step(stream)
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / 5
    assert bl.bitlinear_check_status() == bl.OK
    print(json.dumps({"profile": "fused", "layers": L, "M": M, "ms_per_pass": round(ms, 4),
                      "launches_per_pass": 1 + 4 * L}))
    return 0


def profile_chain(spec):
    """--profile-chain L,M: the decode chain on an L-layer 2B-shape stack at
    M tokens, 3 warm-up + 10 timed runs (driver for ncu captures)."""
    import torch
    import bitlinear_02_b300 as bl
    from bitlinear_02_b300 import inputs
    L, M = (int(v) for v in spec.split(","))
    dev = torch.device("cuda:0")
    shapes = inputs.WORKLOADS[WORKLOAD]["shapes"]
    hidden = shapes[0][2]
    projs = []
    for l in range(L):
        for i, rel in enumerate(LAYER_INPUTS):
            _, N, K = shapes[i]
            wq = inputs.ternary(N, K, seed=l * 10 + i, device=dev)
            packed = bl.pack_ternary(wq)
            slot = (7 * l if l > 0 else 0) if rel == 0 else 7 * l + rel
            projs.append(dict(packed=packed, gamma=torch.tensor([0.02], device=dev), N=N, input=slot))
    dc = bl.DecodeChain(M, hidden, projs)
    x = inputs.activations_bf16(M, hidden, seed=M, device=dev)
    for _ in range(3):
        dc.run(x)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(10):
        dc.run(x)
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / 10
    assert bl.bitlinear_check_status() == bl.OK
    wb = sum(p["packed"].numel() for p in projs)
    print(json.dumps({"profile": "chain", "layers": L, "M": M, "us": round(ms * 1000, 2),
                      "weight_gbs": round(wb / (ms * 1e-3) / 1e9, 1)}))
    return 0


def concurrent_step_ms(torch, bl, inputs, db, steps=300, warmup=5):
    """The three M of the step as independent decode streams: one CUDA graph
    with a branch per M, each branch on its own stream and with its OWN copy
    of the stack's weights (so no branch reads weights another just pulled
    into L2).  The branches' dependent launches overlap on the GPU; the
    algorithmic bytes are those of the sequential step.  Returns ms per step."""
    T = torch
    copies = [db] + [DecodeBench(T, bl, inputs, db.dev) for _ in range(len(M_LIST) - 1)]
    fds = [FusedDecode(T, bl, copies[i], m_list=(M,)) for i, M in enumerate(M_LIST)]
    streams = [T.cuda.Stream() for _ in M_LIST]
    main = T.cuda.Stream()

    def run():
        for f, s in zip(fds, streams):
            s.wait_stream(T.cuda.current_stream())
            with T.cuda.stream(s):
                f.run_step(s)
        for s in streams:
            T.cuda.current_stream().wait_stream(s)

    with T.cuda.stream(main):
        run()
    T.cuda.synchronize()
    g = T.cuda.CUDAGraph()
    with T.cuda.graph(g, stream=main):
        run()
    ms = time_graphs(T, [g], steps, warmup, main) / steps
    del g, fds, copies
    T.cuda.synchronize()
    return ms


def gemv_sweep(torch, bl, db, stream, reps=9):
    """The 2B decode GEMV sweep, shape by shape: bitlinear_forward on a
    pre-quantised input (the GEMV with its rescale epilogue), and
    bitlinear_quant_act reported on its own.  Per (M, shape) one CUDA graph
    of back-to-back launches over the stack's copies of that projection (20
    layers x the projections of that shape), replayed right after an L2
    flush (a 256 MB write, outside the timed events), so every launch reads
    its weights from HBM.  Per-launch time = median replay time / launches;
    GB/s = algorithmic bytes per launch / that time."""
    T = torch
    flush = T.empty(256 << 20, dtype=T.uint8, device=db.dev)
    kinds = [("q,k,v,o", [0, 1, 2, 3]), ("gate,up", [4, 5]), ("down", [6])]
    e0, e1 = T.cuda.Event(enable_timing=True), T.cuda.Event(enable_timing=True)

    def timed(graph, n):
        ts = []
        with T.cuda.stream(stream):
            for _ in range(reps):
                flush.zero_()
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts) / n  # ms per launch

    gemv, quant = [], []
    tot_b, tot_ms = 0, 0.0
    for M in M_LIST:
        for name, idxs in kinds:
            _, N, K = db.shapes[idxs[0]]
            x = db.inputs.activations_bf16(M, K, seed=900 + M, device=db.dev)
            q, sc = bl.quant_act(x, None, db.eps_a)
            out = T.empty(M, N, dtype=T.bfloat16, device=db.dev)
            mats = [db.w[7 * l + j] for l in range(db.layers) for j in idxs]

            def run():
                for packed, gamma, n in mats:
                    bl.bitlinear_forward(q, sc, packed, gamma, M, n, K, out)

            with T.cuda.stream(stream):
                run()
            T.cuda.synchronize()
            g = T.cuda.CUDAGraph()
            with T.cuda.graph(g, stream=stream):
                run()
            ms = timed(g, len(mats))
            b = algo_bytes_forward(M, N, K)
            gemv.append({"M": M, "proj": name, "N": N, "K": K, "us": round(ms * 1e3, 3),
                         "GB/s": round(b / (ms * 1e-3) / 1e9, 1), "launches": len(mats)})
            tot_b += b * len(mats)
            tot_ms += ms * len(mats)
            del g
        for K in sorted({k for _, _, k in db.shapes}):
            xs = [db.inputs.activations_bf16(M, K, seed=950 + M + i, device=db.dev) for i in range(20)]
            qo = T.empty(M, K, dtype=T.int8, device=db.dev)
            so = T.empty(M, dtype=T.float32, device=db.dev)

            def runq():
                for x in xs:
                    bl.bitlinear_quant_act(x, None, M, K, db.eps_a, qo, so)

            with T.cuda.stream(stream):
                runq()
            T.cuda.synchronize()
            g = T.cuda.CUDAGraph()
            with T.cuda.graph(g, stream=stream):
                runq()
            ms = timed(g, len(xs))
            quant.append({"M": M, "K": K, "us": round(ms * 1e3, 3),
                          "GB/s": round(algo_bytes_quant(M, K) / (ms * 1e-3) / 1e9, 2)})
            del g
    del flush
    return {"mode": "per (M, shape): a graph of bitlinear_forward launches over the stack's copies of that "
                    "projection on a pre-quantised input, replayed after a 256 MB L2 flush; median of "
                    f"{reps} replays / launches",
            "gemv": gemv, "quant_act": quant,
            "gemv_all": {"GB/s": round(tot_b / (tot_ms * 1e-3) / 1e9, 1),
                         "note": "all shapes and M: algorithmic bytes / summed launch times"}}


def midm_sweep(torch, bl, db, stream, reps=7, m_values=(32, 64, 128, 256)):
    """Mid-size batches (16 < M < 512) through the tensor-core GEMM
    (bitlinear_quant_act_f16 + bitlinear_forward_f16), measured like the
    GEMV sweep: per (M, shape) a graph of back-to-back launches over the
    stack's copies of that projection, replayed after an L2 flush.  Reports
    per launch us, TFLOP/s and packed-weight GB/s, to place the crossover
    with the decode GEMV (M <= 16)."""
    T = torch
    flush = T.empty(256 << 20, dtype=T.uint8, device=db.dev)
    kinds = [("q,k,v,o", [0, 1, 2, 3]), ("gate,up", [4, 5]), ("down", [6])]
    e0, e1 = T.cuda.Event(enable_timing=True), T.cuda.Event(enable_timing=True)
    rows = []
    for M in m_values:
        for name, idxs in kinds:
            _, N, K = db.shapes[idxs[0]]
            x = db.inputs.activations_bf16(M, K, seed=700 + M, device=db.dev)
            q, sc = bl.quant_act_f16(x, None, db.eps_a)
            out = T.empty(M, N, dtype=T.bfloat16, device=db.dev)
            mats = [db.w[7 * l + j] for l in range(db.layers) for j in idxs]

            def run():
                for packed, gamma, n in mats:
                    bl.forward_f16(q, sc, packed, gamma, n, out=out)

            with T.cuda.stream(stream):
                run()
            T.cuda.synchronize()
            g = T.cuda.CUDAGraph()
            with T.cuda.graph(g, stream=stream):
                run()
            ts = []
            with T.cuda.stream(stream):
                for _ in range(reps):
                    flush.zero_()
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                    e1.synchronize()
                    ts.append(e0.elapsed_time(e1))
            ms = statistics.median(ts) / len(mats)
            wbytes = (-(-N // 16) * 16) * (-(-K // 128) * 128) // 4
            rows.append({"M": M, "proj": name, "N": N, "K": K, "us": round(ms * 1e3, 3),
                         "TFLOP/s": round(2 * M * N * K / (ms * 1e-3) / 1e12, 1),
                         "weight_GB/s": round(wbytes / (ms * 1e-3) / 1e9, 1)})
            del g
    del flush
    return {"mode": "bitlinear_quant_act_f16 + bitlinear_forward_f16 (tcgen05 GEMM), per (M, shape) a graph of "
                    "launches over the stack's copies after a 256 MB L2 flush; median of "
                    f"{reps} replays / launches", "rows": rows}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--profile-gemm", default=None, help="N,K,M[,int8]: time one GEMM shape (ncu driver)")
    ap.add_argument("--profile-chain", default=None, help="L,M: time the decode chain (ncu driver)")
    ap.add_argument("--profile-fused", default=None, help="L,M: time the fused decode path (ncu driver)")
    args = ap.parse_args()
    if args.profile_gemm:
        return profile_gemm(args.profile_gemm)
    if args.profile_fused:
        return profile_fused(args.profile_fused)
    if args.profile_chain:
        return profile_chain(args.profile_chain)
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
    dist = replica_group("nccl", dev)
    barrier = (lambda: dist.barrier()) if dist is not None else None
    bl.load_library()
    hbm_peak, bf16_peak, bf16_sust, peak_kind = peaks()
    stream = torch.cuda.Stream()

    db = DecodeBench(torch, bl, inputs, dev)
    fd = FusedDecode(torch, bl, db)
    graph = fd.capture(stream)
    sampler = ClockSampler(local)
    with sampler:
        ms = time_graphs(torch, [graph], args.steps, args.warmup, stream, barrier)
    clocks = sampler.summary()
    ms = max_over_ranks(torch, ms, dev, dist)
    assert bl.bitlinear_check_status() == bl.OK, "a bounded wait expired during the timed steps"
    value = job_value(db.bytes_step, args.steps, ws, ms)
    ms_step = ms / args.steps
    del graph

    # e2e: each M's input copied from pinned host memory, the last output read back, every step
    h2d = {M: db.x[M].cpu().pin_memory() for M in M_LIST}
    d2h = {M: torch.empty_like(db.chains[M].out[-1], device="cpu").pin_memory() for M in M_LIST}
    g_e2e = fd.capture(stream, h2d=h2d, d2h=d2h)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            g_e2e.replay()
        stream.synchronize()
        n_e2e = max(10, args.steps // 4)
        t0 = time.perf_counter()
        for i in range(n_e2e):
            g_e2e.replay()            # replays on `stream`, the current stream here
            stream.synchronize()      # the step, copies included, has finished
            _ = float(d2h[16][0, 0])  # read the result on the host
        e2e_s = time.perf_counter() - t0
    e2e_val = db.bytes_step * n_e2e * ws / e2e_s / 1e9
    h2d_bytes = sum(t.numel() * t.element_size() for t in h2d.values())
    d2h_bytes = sum(t.numel() * t.element_size() for t in d2h.values())
    del g_e2e

    g_chain = db.capture(stream)
    chain_ms = time_graphs(torch, [g_chain], max(20, args.steps // 10), 3, stream) / max(20, args.steps // 10)
    del g_chain
    unf_ms = unfused_step_ms(torch, bl, db, stream)
    conc_ms = concurrent_step_ms(torch, bl, inputs, db)
    sweep = gemv_sweep(torch, bl, db, stream)
    midm = midm_sweep(torch, bl, db, stream)
    for r in sweep["gemv"]:
        r["frac"] = round(r["GB/s"] / hbm_peak, 4)
    n_fused = FusedDecode.launches  # act_stats + 4 fused GEMVs per layer, per M
    launch_us = 1000.0 * ms_step / n_fused
    bytes_launch = db.bytes_step / n_fused
    fused_gbs = bytes_launch / (launch_us * 1e-6) / 1e9
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
        gbs, reps, dt, cores = oracle_step_sample(budget_s=15.0)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{reps} x one 2B-shape layer for each M=1,4,16 (quantise, unpack, matmul, rescale; "
                         f"7 chained projections) in {dt:.1f} s"}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 x ternary -> int32 (f16 tensor-core operands, exact), bf16 out",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": list(M_LIST), "layers": db.layers, "hidden": 2560,
                   "ffn": 6912, "projections": "q,k,v,o 2560x2560; gate,up 2560->6912; down 6912->2560",
                   "packed_mb": round(db.packed_bytes / 1e6, 1),
                   "l2": "inputs larger than L2: the stack's packed weights are 3x the 126 MB L2",
                   "bytes_per_step": db.bytes_step,
                   "graph": "one CUDA graph per step: per M one act_stats + 4 fused GEMV launches per layer",
                   "parallelism": f"replicas x{ws}"},
        "hbm_frac_of_step": round(value / ws / hbm_peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(fused_gbs, 1), "peak": round(hbm_peak, 1),
                     "unit": "GB/s", "frac": round(fused_gbs / hbm_peak, 4),
                     "traffic": round(FUSED_DRAM_PER_PACKED_BYTE * db.packed_bytes * len(M_LIST) / n_fused),
                     "traffic_note": "bytes per average launch: ncu DRAM bytes per packed-weight byte "
                                     "(profiles/fused_gemv_decode_2b_M16_full.md) x packed bytes per launch",
                     "kernel": "fused_gemv_kernel (decode GEMV with the quantiser folded in)",
                     "launch_avg_us": round(launch_us, 2), "algo_bytes_per_launch": round(bytes_launch),
                     "peak_note": f"{peak_kind} HBM copy bandwidth",
                     "method": "CUDA events around the timed graph replays; launch time = step time / "
                               "launches in the step (3 of the 243 are act_stats)"},
        "chain": {"ms_per_step": round(chain_ms, 4),
                  "value": round(db.bytes_step / (chain_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                  "mode": "persistent fused-chain kernel, one launch per M through the whole stack"},
        "concurrent": {"ms_per_step": round(conc_ms, 4),
                       "value": round(db.bytes_step / (conc_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                       "mode": "the three M as independent decode streams: one graph, a branch per M on its own "
                               "stream, each branch with its own copy of the weights (3 x 396 MB, no shared L2 "
                               "reads); same kernels and algorithmic bytes as the step"},
        "unfused": {"ms_per_step": round(unf_ms, 4),
                    "value": round(db.bytes_step / (unf_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                    "mode": "bitlinear_quant_act + bitlinear_forward per projection, PDL-chained graph"},
        "sweep": sweep,
        "mid_m": midm,
        "prefill": prefill,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h_bytes,
                "mode": "graph replay of the public API calls incl. pinned H2D/D2H copies, host sync per step"},
        "gpu_launches": n_fused * args.steps,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
