"""Benchmark of the BitLinear hot path on B300 (one JSON line on stdout).

Headline workload (``value``): one decode step of a stack of 2B-shaped
layers, for M = 1, 4 and 16 tokens.  A layer has the seven projections
q/k/v/o 2560x2560, gate/up 2560->6912 and down 6912->2560, chained through
the fused RMSNorm + absmax int8 quantiser:
    h = x; q,k,v = f(h); o = f(v); gate,up = f(o); down = f(up); next x = down
The stack has LAYERS = 20 layers: 396 MB of packed 2-bit weights, the
0.4 GB the asi.tokyo write-up gives for the 2B model's weights, and more
than 3x the 126 MB L2, so every weight byte is read from HBM.  Each M runs
the whole stack; a step is all of it for the three M, replayed as one CUDA
graph.  The step runs the fused decode path: per M one bitlinear_act_stats
of the stack input, then per layer four bitlinear_forward_fused launches
(q,k,v | o | gate,up | down), each quantising its input on the fly.

value    = algorithmic bytes of the step (packed weights, activations in and
           out, scales; the count of the unfused quant + forward calls)
           / device time, summed over ranks.
e2e      = the same bytes / wall time of steps made of the public entry
           points called one by one from the host (their host cost
           included), with each M's input copied from pinned host memory and
           the last output read back every step; `e2e.graph` is the same
           step replayed as a CUDA graph.
roofline = the fused decode kernel: bytes per launch / average launch time.
configs  = every workload of the build: the small layer, the 2B decode
           stack per M, the 2B prefill GEMMs (M = 512, 2048, 4096, both
           activation entry points), and the 3B (26 layers) and 70B (80
           layers) stacks' decode steps at every M, with tokens/s and
           roofline fractions.  The stacks' ternary weights are drawn on the
           device by a counter-based generator.
sweep    = the decode GEMV shape by shape (2B, 3B and 70B shapes, every
           launch reading its weights from HBM after an L2 flush).
mid_m    = 32-256 tokens through bitlinear_forward and the f16 GEMM.
cpu_baseline = the CPU oracle on a bounded sample of the same workload,
           single-threaded and on all host cores.

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
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0
# DRAM bytes (read + write) per packed-weight byte of the fused decode
# kernel over the step's 240 launches, from an ncu capture of this kernel
# (profiles/fused_gemv_decode_2b_dram_traffic.md); None once the kernel
# changes after the capture.
FUSED_DRAM_PER_PACKED_BYTE = 1.0207


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
    """nvidia-smi samples while GPU work is timed (clocks, throttle reasons).
    `mark(True/False)` brackets timed regions; samples outside are dropped;
    `take()` returns (and forgets) the samples kept since the last take."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.all = []
        self.active = False

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

    def mark(self, on: bool):
        self.active = on

    def _read(self):
        for line in self.proc.stdout:
            if self.active:
                self.lines.append(line.strip())
                self.all.append(line.strip())

    def take(self):
        out, self.lines = self.lines, []
        return out

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    @staticmethod
    def summary(lines):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in lines:
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

def packed_bytes(N, K):
    return (-(-N // 16) * 16) * (-(-K // 128) * 128) // 4


def algo_bytes_forward(M, N, K):
    return packed_bytes(N, K) + M * K + 4 * M + 2 * M * N + 4


def algo_bytes_quant(M, K):
    return 2 * M * K + M * K + 4 * M


def chain_plan(shapes, o_from="v"):
    """(kind, input, output) list for one layer, with the shapes by name."""
    d = {n: (N, K) for n, N, K in shapes}
    return [
        ("quant", "x", "h0"),
        ("fwd", "h0", "q"), ("fwd", "h0", "k"), ("fwd", "h0", "v"),
        ("quant", o_from, "h1"), ("fwd", "h1", "o"),
        ("quant", "o", "h2"), ("fwd", "h2", "gate"), ("fwd", "h2", "up"),
        ("quant", "up", "h3"), ("fwd", "h3", "down"),
    ], d


def layer_bytes(M, shapes, o_from="v"):
    """Algorithmic bytes of one layer at M tokens (unfused-path count)."""
    plan, dims = chain_plan(shapes, o_from)
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


def time_graphs(torch, graphs, steps, warmup, stream, barrier=None, clock=None):
    for i in range(warmup):
        graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clock:
        clock.mark(True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(steps):
            graphs[(warmup + i) % len(graphs)].replay()
        e1.record(stream)
    e1.synchronize()
    if clock:
        clock.mark(False)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return e0.elapsed_time(e1)  # ms


def time_graph_flushed(torch, g, steps, warmup, stream, flush):
    """Mean ms per replay of graph g, each replay timed on its own with CUDA
    events on `stream`, after a write of `flush` (larger than L2) that stays
    outside the timed events, so no replay finds the previous one's data in
    L2."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tot = 0.0
        for _ in range(steps):
            flush.zero_()
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            tot += e0.elapsed_time(e1)
    return tot / steps


def capture(torch, fn, stream):
    """One eager run (host-side set-up happens outside capture), then a graph."""
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


class Stack:
    """A decode stack: `layers` x 7 packed projections shared by every M.

    Workloads with master weights (the 2B ones) draw W ~ N(0, 0.02^2) and
    absmean-pack it with bitlinear_pack_weights; the 3B and 70B stacks draw
    ternary weights on the device with the counter-based generator of the
    inputs module, pack them with bitlinear_pack_ternary, and take gamma ~
    U(0.01, 0.05) per matrix.  o_from: the projection whose output feeds o
    (v, or q where v is narrower than the hidden size)."""

    def __init__(self, torch, bl, inputs, dev, workload, layers=None):
        self.torch, self.bl, self.inputs, self.dev = torch, bl, inputs, dev
        wl = inputs.WORKLOADS[workload]
        self.workload = workload
        self.shapes = wl["shapes"]
        self.layers = layers or wl.get("layers", LAYERS)
        self.eps_a = wl["eps_a"]
        self.hidden = self.shapes[0][2]
        self.o_from = "v" if self.shapes[2][1] == self.hidden else "q"
        self.o_src = [n for n, _, _ in self.shapes].index(self.o_from)
        self.w = []  # (packed, gamma, N, K) per projection, layer-major
        for l in range(self.layers):
            for i, (name, N, K) in enumerate(self.shapes):
                if "eps_w" in wl:
                    W = inputs.weights_fp32(N, K, seed=wl["seed"] * 100000 + l * 10 + i, device=dev)
                    packed, gamma = bl.pack_weights(W, wl["eps_w"])
                    del W
                else:
                    wq = inputs.ternary_hash(N, K, inputs.stack_word(wl["seed"], l, i), device=dev)
                    packed = bl.pack_ternary(wq)
                    del wq
                    g = inputs.gamma_uniform(wl["seed"] * 100000 + l * 10 + i)
                    gamma = torch.tensor([g], dtype=torch.float32, device=dev)
                self.w.append((packed, gamma, N, K))
        torch.cuda.synchronize()
        self.packed_bytes = sum(p.numel() for p, _, _, _ in self.w)
        self.x = {}

    def input(self, M):
        if M not in self.x:
            self.x[M] = self.inputs.activations_bf16(M, self.hidden, seed=7 * M + 3, device=self.dev)
        return self.x[M]

    def bytes(self, M):
        return layer_bytes(M, self.shapes, self.o_from) * self.layers


class FusedRunner:
    """The stack through the fused decode path at M <= 16 tokens: one
    bitlinear_act_stats of the stack input, then per layer four
    bitlinear_forward_fused launches (q,k,v | o | gate,up | down), each
    quantising its input on the fly."""

    def __init__(self, st: Stack, M):
        T, bl = st.torch, st.bl
        self.st, self.M = st, M
        self.outs = [[T.empty(M, N, dtype=T.bfloat16, device=st.dev) for _, N, _ in st.shapes]
                     for _ in range(st.layers)]
        self.stats = [[bl.new_stats(st.dev) for _ in range(4)] for _ in range(st.layers)]  # o_src, o, up, down
        self.x_stats = bl.new_stats(st.dev)
        self.launches = 1 + 4 * st.layers

    def last_output(self):
        return self.outs[-1][6]

    def run(self, stream):
        st, bl, M = self.st, self.st.bl, self.M
        x0 = st.input(M)
        bl.bitlinear_act_stats(x0, M, st.hidden, st.eps_a, self.x_stats, stream)
        for l in range(st.layers):
            o = self.outs[l]
            s_src, s_o, s_up, s_down = self.stats[l]
            x = x0 if l == 0 else self.outs[l - 1][6]
            xs = self.x_stats if l == 0 else self.stats[l - 1][3]

            def fp(i, sb=None):
                packed, gamma, N, _ = st.w[7 * l + i]
                return bl.FusedProj(packed.data_ptr(), gamma.data_ptr(), N, o[i].data_ptr(), None,
                                    sb.data_ptr() if sb is not None else None)

            qkv = [fp(i, s_src if i == st.o_src else None) for i in range(3)]
            bl.bitlinear_forward_fused(x, xs, M, st.hidden, qkv, st.eps_a, stream)
            src = o[st.o_src]
            bl.bitlinear_forward_fused(src, s_src, M, src.shape[1], [fp(3, s_o)], st.eps_a, stream)
            bl.bitlinear_forward_fused(o[3], s_o, M, o[3].shape[1], [fp(4), fp(5, s_up)], st.eps_a, stream)
            last = l == st.layers - 1  # the last output feeds nothing here: no factors for it
            bl.bitlinear_forward_fused(o[5], s_up, M, o[5].shape[1], [fp(6, None if last else s_down)],
                                       st.eps_a, stream)


class UnfusedRunner:
    """The stack through the per-projection entry points at any M: per layer
    h0 = quant(x); q,k,v = fwd(h0); h1 = quant(o_src); o = fwd(h1);
    h2 = quant(o); gate,up = fwd(h2); h3 = quant(up); down = fwd(h3).
    bitlinear_forward runs the decode GEMV up to 64 tokens and the tcgen05
    GEMM above."""

    def __init__(self, st: Stack, M):
        T = st.torch
        self.st, self.M = st, M
        self.outs = [T.empty(M, N, dtype=T.bfloat16, device=st.dev) for _, N, _ in st.shapes]
        widths = (st.hidden, st.shapes[st.o_src][1], st.shapes[3][1], st.shapes[5][1])
        self.hs = [(T.empty(M, K, dtype=T.int8, device=st.dev), T.empty(M, dtype=T.float32, device=st.dev))
                   for K in widths]
        self.launches = 11 * st.layers

    def last_output(self):
        return self.outs[6]

    def run(self, stream):
        st, bl, M = self.st, self.st.bl, self.M
        order = [("quant", 0, None), ("fwd", 0, 0), ("fwd", 1, 0), ("fwd", 2, 0), ("quant", 1, st.o_src),
                 ("fwd", 3, 1), ("quant", 2, 3), ("fwd", 4, 2), ("fwd", 5, 2), ("quant", 3, 5), ("fwd", 6, 3)]
        for l in range(st.layers):
            for kind, a, b in order:
                if kind == "quant":
                    src = (st.input(M) if l == 0 else self.outs[6]) if a == 0 else self.outs[b]
                    q, sc = self.hs[a]
                    bl.bitlinear_quant_act(src, None, M, src.shape[1], st.eps_a, q, sc, stream)
                else:
                    packed, gamma, N, K = st.w[7 * l + a]
                    q, sc = self.hs[b]
                    bl.bitlinear_forward(q, sc, packed, gamma, M, N, K, self.outs[a], None, stream)


def runner(st, M):
    return FusedRunner(st, M) if M <= 16 else UnfusedRunner(st, M)


def stack_rows(torch, st, m_list, stream, hbm_peak, reps, clock=None):
    """Decode step per M through a stack: ms, GB/s, fraction, tokens/s."""
    rows = []
    for M in m_list:
        r = runner(st, M)
        g = capture(torch, lambda: r.run(stream), stream)
        ms = time_graphs(torch, [g], reps, 3, stream, clock=clock) / reps
        b = st.bytes(M)
        gbs = b / (ms * 1e-3) / 1e9
        rows.append({"M": M, "path": "fused" if M <= 16 else "quant_act + forward", "ms_per_step": round(ms, 4),
                     "GB/s": round(gbs, 1), "frac": round(gbs / hbm_peak, 4),
                     "tokens_per_s": round(M / (ms * 1e-3), 1), "launches": r.launches})
        del g, r
    return rows


def gemv_sweep(torch, bl, inputs, dev, stream, hbm_peak, reps=7, m_list=M_LIST):
    """The decode GEMV shape by shape: bitlinear_forward on a pre-quantised
    input (the GEMV with its rescale epilogue), for the distinct projection
    shapes of the 2B, 3B and 70B models.  Per (M, shape) one CUDA graph of
    back-to-back launches over distinct copies of the packed matrix (at least
    512 MB of them, so no launch finds its weights in L2), replayed right
    after an L2 flush (a 256 MB write, outside the timed events).  Per-launch
    time = median replay time / launches; GB/s = algorithmic bytes per
    launch / that time."""
    T = torch
    flush = T.empty(256 << 20, dtype=T.uint8, device=dev)
    e0, e1 = T.cuda.Event(enable_timing=True), T.cuda.Event(enable_timing=True)
    shapes = [("2b", "q,k,v,o", 2560, 2560), ("2b", "gate,up", 6912, 2560), ("2b", "down", 2560, 6912),
              ("3b", "q,k,v,o", 3200, 3200), ("3b", "gate,up", 8640, 3200), ("3b", "down", 3200, 8640),
              ("70b", "q,o", 8192, 8192), ("70b", "k,v", 1024, 8192), ("70b", "gate,up", 28672, 8192),
              ("70b", "down", 8192, 28672)]
    rows = []
    for si, (model, proj, N, K) in enumerate(shapes):
        pb = packed_bytes(N, K)
        ncopy = max(8, min(64, -(-(512 << 20) // pb)))
        wq = inputs.ternary_hash(N, K, inputs.stack_word(9, 0, si), device=dev)
        p0 = bl.pack_ternary(wq)
        del wq
        mats = [p0] + [p0.clone() for _ in range(ncopy - 1)]
        gam = T.tensor([0.02], dtype=T.float32, device=dev)
        for M in m_list:
            x = inputs.activations_bf16(M, K, seed=900 + M, device=dev)
            q, sc = bl.quant_act(x)
            out = T.empty(M, N, dtype=T.bfloat16, device=dev)

            def run():
                for p in mats:
                    bl.bitlinear_forward(q, sc, p, gam, M, N, K, out, None, stream)

            g = capture(T, run, stream)
            ts = []
            with T.cuda.stream(stream):
                for _ in range(reps):
                    flush.zero_()
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                    e1.synchronize()
                    ts.append(e0.elapsed_time(e1))
            ms = statistics.median(ts) / ncopy
            b = algo_bytes_forward(M, N, K)
            gbs = b / (ms * 1e-3) / 1e9
            rows.append({"model": model, "proj": proj, "N": N, "K": K, "M": M, "us": round(ms * 1e3, 3),
                         "GB/s": round(gbs, 1), "frac": round(gbs / hbm_peak, 4), "launches": ncopy})
            del g
        del mats, p0
    del flush
    T.cuda.empty_cache()
    return {"mode": "per (shape, M): a graph of bitlinear_forward launches over distinct copies of the packed "
                    "matrix on a pre-quantised input, replayed after a 256 MB L2 flush; median of "
                    f"{reps} replays / launches", "rows": rows}


def variants_sweep(torch, bl, inputs, dev, stream, hbm_peak, reps=7, m_list=(1, 16)):
    """The decode engines of the three weight formats on the same shapes:
    2-bit (bitlinear_forward), five ternary digits per byte
    (bitlinear_forward5) and the binary variant (bitlinear_forward_binary,
    8 row groups).  Same method as the GEMV sweep (a graph of launches over
    distinct copies, at least 512 MB, replayed after an L2 flush).  GB/s
    counts each format's own bytes; weights/s compares the formats."""
    T = torch
    flush = T.empty(256 << 20, dtype=T.uint8, device=dev)
    e0, e1 = T.cuda.Event(enable_timing=True), T.cuda.Event(enable_timing=True)
    shapes = [("2b", "q,k,v,o", 2560, 2560), ("2b", "gate,up", 6912, 2560), ("2b", "down", 2560, 6912),
              ("70b", "gate,up", 28672, 8192), ("70b", "down", 8192, 28672)]
    rows = []
    for si, (model, proj, N, K) in enumerate(shapes):
        w = inputs.weights_fp32(N, K, seed=700 + si, device=dev)
        p2, gam = bl.pack_weights(w, 1e-5)
        p5 = bl.repack5(p2, N, K)
        p1, beta = bl.pack_binary(w, 8)
        del w
        fmts = [("2bit", p2, lambda q, sc, p, out, M: bl.bitlinear_forward(q, sc, p, gam, M, N, K, out, None, stream)),
                ("5trit", p5, lambda q, sc, p, out, M: bl.bitlinear_forward5(q, sc, p, gam, M, N, K, out, None,
                                                                             stream)),
                ("binary", p1, lambda q, sc, p, out, M: bl.bitlinear_forward_binary(q, sc, p, beta, 8, M, N, K, out,
                                                                                    None, stream))]
        for name, p0, fn in fmts:
            pb = p0.numel()
            ncopy = max(8, min(64, -(-(512 << 20) // pb)))
            mats = [p0] + [p0.clone() for _ in range(ncopy - 1)]
            for M in m_list:
                x = inputs.activations_bf16(M, K, seed=900 + M, device=dev)
                q, sc = bl.quant_act(x)
                out = T.empty(M, N, dtype=T.bfloat16, device=dev)

                def run():
                    for p in mats:
                        fn(q, sc, p, out, M)

                g = capture(T, run, stream)
                ts = []
                with T.cuda.stream(stream):
                    for _ in range(reps):
                        flush.zero_()
                        e0.record(stream)
                        g.replay()
                        e1.record(stream)
                        e1.synchronize()
                        ts.append(e0.elapsed_time(e1))
                ms = statistics.median(ts) / ncopy
                b = pb + M * K + 4 * M + 2 * M * N + 4
                gbs = b / (ms * 1e-3) / 1e9
                rows.append({"model": model, "proj": proj, "N": N, "K": K, "M": M, "format": name,
                             "packed_bytes": pb, "us": round(ms * 1e3, 3), "GB/s": round(gbs, 1),
                             "frac": round(gbs / hbm_peak, 4),
                             "Gweights/s": round(N * K / (ms * 1e-3) / 1e9, 1), "launches": ncopy})
                del g
            del mats
        del p2, p5, p1
    del flush
    T.cuda.empty_cache()
    return {"mode": "per (shape, format, M): a graph of decode launches over distinct copies of the packed matrix "
                    f"on a pre-quantised input, replayed after a 256 MB L2 flush; median of {reps} replays / "
                    "launches; GB/s over each format's own bytes", "rows": rows}


def quant_sweep(torch, bl, inputs, dev, stream, reps=7):
    """bitlinear_quant_act on its own at the decode sizes (20 distinct inputs per graph)."""
    T = torch
    rows = []
    for M in M_LIST:
        for K in (2560, 6912):
            xs = [inputs.activations_bf16(M, K, seed=950 + M + i, device=dev) for i in range(20)]
            qo = T.empty(M, K, dtype=T.int8, device=dev)
            so = T.empty(M, dtype=T.float32, device=dev)

            def runq():
                for x in xs:
                    bl.bitlinear_quant_act(x, None, M, K, 1e-5, qo, so, stream)

            g = capture(T, runq, stream)
            ms = time_graphs(T, [g], reps, 2, stream) / reps / len(xs)
            rows.append({"M": M, "K": K, "us": round(ms * 1e3, 3),
                         "GB/s": round(algo_bytes_quant(M, K) / (ms * 1e-3) / 1e9, 2)})
            del g
    return rows


def midm_sweep(torch, bl, inputs, st, stream, reps=5, m_values=(32, 64, 65, 96, 128, 176, 256)):
    """Mid-size batches through bitlinear_forward (int8 activations: the
    decode GEMV in 16-token chunks up to 64, the tcgen05 GEMM above) and
    through bitlinear_forward_f16 (always the GEMM), per (M, shape) on the
    2B stack's matrices (20 copies per shape, 33-88 MB), after an L2 flush."""
    T = torch
    flush = T.empty(256 << 20, dtype=T.uint8, device=st.dev)
    kinds = [("q,k,v,o", [0, 1, 2, 3]), ("gate,up", [4, 5]), ("down", [6])]
    e0, e1 = T.cuda.Event(enable_timing=True), T.cuda.Event(enable_timing=True)
    rows = []
    for M in m_values:
        for name, idxs in kinds:
            _, N, K = st.shapes[idxs[0]]
            x = inputs.activations_bf16(M, K, seed=700 + M, device=st.dev)
            q, sc = bl.quant_act(x)
            q16, sc16 = bl.quant_act_f16(x)
            out = T.empty(M, N, dtype=T.bfloat16, device=st.dev)
            mats = [st.w[7 * l + j] for l in range(st.layers) for j in idxs]
            row = {"M": M, "proj": name, "N": N, "K": K}
            for tag in ("forward", "forward_f16"):
                def run():
                    for packed, gamma, n, k in mats:
                        if tag == "forward":
                            bl.bitlinear_forward(q, sc, packed, gamma, M, n, k, out, None, stream)
                        else:
                            bl.bitlinear_forward_f16(q16, sc16, packed, gamma, M, n, k, out, None, stream)

                g = capture(T, run, stream)
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
                row[tag + "_us"] = round(ms * 1e3, 3)
                row[tag + "_TFLOP/s"] = round(2 * M * N * K / (ms * 1e-3) / 1e12, 1)
                row[tag + "_weight_GB/s"] = round(packed_bytes(N, K) / (ms * 1e-3) / 1e9, 1)
                del g
            rows.append(row)
    del flush
    return {"mode": "per (M, shape): a graph of launches over the 2B stack's copies of that projection after a "
                    f"256 MB L2 flush; median of {reps} replays / launches", "rows": rows}


def prefill_bench(torch, bl, inputs, dev, stream, bf16_peak, steps=5, warmup=3, m_list=(512, 2048, 4096)):
    """The 2B prefill workload: the seven projections chained through the
    quantiser at M tokens.  Per M: the chain through the f16-activation path
    (bitlinear_quant_act_f16 + bitlinear_forward_f16) and through the int8
    entry points (bitlinear_quant_act + bitlinear_forward); TOPS of the
    tensor-core GEMMs alone (2*M*N*K per projection) and of the whole chain,
    and each distinct shape's f16 GEMM on its own.  Every replay is timed on
    its own after a 256 MB L2 flush (outside the timed events)."""
    wl = inputs.WORKLOADS["prefill_2b"]
    shapes = wl["shapes"]
    plan, dims = chain_plan(shapes)
    hidden = dims["q"][1]
    w = {}
    for i, (name, N, K) in enumerate(shapes):
        W = inputs.weights_fp32(N, K, seed=wl["seed"] * 100 + i, device=dev)
        w[name] = bl.pack_weights(W, wl["eps_w"])
        del W
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    res = []
    for M in m_list:
        b = {"x": inputs.activations_bf16(M, hidden, seed=wl["seed"] * 1000 + M, outlier_frac=0.01,
                                          outlier_scale=20.0, device=dev)}
        for name, N, K in shapes:
            b[name] = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        for h, src in (("h0", "x"), ("h1", "v"), ("h2", "o"), ("h3", "up")):
            K = b[src].shape[1]
            b[h] = (torch.empty(M, K, dtype=torch.float16, device=dev), torch.empty(M, dtype=torch.float32, device=dev))
            b[h + "i8"] = (torch.empty(M, K, dtype=torch.int8, device=dev),
                           torch.empty(M, dtype=torch.float32, device=dev))
        ops = sum(2 * M * dims[o][0] * dims[o][1] for k, _, o in plan if k == "fwd")

        def step(kinds=("quant", "fwd"), int8=False, only=None):
            for kind, a, o in plan:
                if kind == "quant" and "quant" in kinds:
                    q, s = b[o + ("i8" if int8 else "")]
                    if int8:
                        bl.bitlinear_quant_act(b[a], None, M, b[a].shape[1], wl["eps_a"], q, s, stream)
                    else:
                        bl.bitlinear_quant_act_f16(b[a], None, M, b[a].shape[1], wl["eps_a"], q, s, stream)
                elif kind == "fwd" and "fwd" in kinds and (only is None or o in only):
                    q, s = b[a + ("i8" if int8 else "")]
                    N, K = dims[o]
                    if int8:
                        bl.bitlinear_forward(q, s, w[o][0], w[o][1], M, N, K, b[o], None, stream)
                    else:
                        bl.bitlinear_forward_f16(q, s, w[o][0], w[o][1], M, N, K, b[o], None, stream)

        row = {"M": M}
        for path, int8 in (("f16", False), ("int8", True)):
            g = capture(torch, lambda: step(int8=int8), stream)
            ms = time_graph_flushed(torch, g, steps, warmup, stream, flush)
            g2 = capture(torch, lambda: step(kinds=("fwd",), int8=int8), stream)
            ms2 = time_graph_flushed(torch, g2, steps, warmup, stream, flush)
            row[path] = {"chain_ms": round(ms, 4), "chain_tops": round(ops / (ms * 1e-3) / 1e12, 1),
                         "gemm_ms": round(ms2, 4), "gemm_tops": round(ops / (ms2 * 1e-3) / 1e12, 1),
                         "gemm_frac": round(ops / (ms2 * 1e-3) / 1e12 / bf16_peak, 4),
                         "tokens_per_s": round(M / (ms * 1e-3), 1)}
            del g, g2
        per_shape = []
        for o in ("q", "gate", "down"):
            N, K = dims[o]
            g = capture(torch, lambda: step(kinds=("fwd",), only=(o,)), stream)
            ms = time_graph_flushed(torch, g, steps * 4, warmup, stream, flush)
            t = 2 * M * N * K / (ms * 1e-3) / 1e12
            per_shape.append({"proj": o, "N": N, "K": K, "us": round(ms * 1e3, 2), "TFLOP/s": round(t, 1),
                              "frac": round(t / bf16_peak, 4)})
            del g
        row["f16_per_shape"] = per_shape
        res.append(row)
        del b
    del w, flush
    torch.cuda.empty_cache()
    return {"shapes": "q,k,v,o 2560x2560; gate,up 2560->6912; down 6912->2560",
            "peak_note": "TOPS against the measured cuBLAS bf16 burst peak: the GEMM runs exact f16 tcgen05 "
                         "MMAs (sm_103a has no int8 tcgen05 MMA)", "rows": res}


def small_layer_row(torch, bl, inputs, dev, stream, hbm_peak, reps=50):
    """The small single-layer workload (M = 1, K = 256, N = 512): quantise +
    forward, back to back in a graph of 50 layers' worth of calls over 50
    distinct copies of the packed matrix, each replay timed after a 256 MB
    L2 flush (outside the timed events): every layer reads its weights from
    HBM."""
    wl = inputs.WORKLOADS["layer_small"]
    _, N, K = wl["shapes"][0]
    W = inputs.weights_fp32(N, K, seed=wl["seed"], device=dev)
    packed, gamma = bl.pack_weights(W, wl["eps_w"])
    mats = [packed] + [packed.clone() for _ in range(49)]
    x = inputs.activations_bf16(1, K, seed=1, device=dev)
    q = torch.empty(1, K, dtype=torch.int8, device=dev)
    s = torch.empty(1, dtype=torch.float32, device=dev)
    out = torch.empty(1, N, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def run():
        for p in mats:
            bl.bitlinear_quant_act(x, None, 1, K, wl["eps_a"], q, s, stream)
            bl.bitlinear_forward(q, s, p, gamma, 1, N, K, out, None, stream)

    g = capture(torch, run, stream)
    ms = time_graph_flushed(torch, g, reps, 5, stream, flush) / 50
    del g, flush
    b = algo_bytes_quant(1, K) + algo_bytes_forward(1, N, K)
    return {"M": 1, "K": K, "N": N, "us_per_layer": round(ms * 1e3, 3),
            "GB/s": round(b / (ms * 1e-3) / 1e9, 2), "frac": round(b / (ms * 1e-3) / 1e9 / hbm_peak, 5),
            "tokens_per_s": round(1 / (ms * 1e-3), 1),
            "note": "32 KB of packed weights: two dependent launches' latency, not bandwidth"}


def concurrent_step_ms(torch, bl, inputs, st0, stream_main, steps=300, warmup=5):
    """The three M of the step as independent decode streams: one CUDA graph
    with a branch per M, each branch on its own stream and with its OWN copy
    of the stack's weights (so no branch reads weights another just pulled
    into L2).  Returns ms per step."""
    T = torch
    copies = [st0] + [Stack(T, bl, inputs, st0.dev, WORKLOAD, layers=st0.layers) for _ in range(len(M_LIST) - 1)]
    runs = [FusedRunner(copies[i], M) for i, M in enumerate(M_LIST)]
    streams = [T.cuda.Stream() for _ in M_LIST]

    def run():
        for r, s in zip(runs, streams):
            s.wait_stream(T.cuda.current_stream())
            with T.cuda.stream(s):
                r.run(s)
        for s in streams:
            T.cuda.current_stream().wait_stream(s)

    g = capture(T, run, stream_main)
    ms = time_graphs(T, [g], steps, warmup, stream_main) / steps
    del g, runs, copies
    T.cuda.synchronize()
    return ms


# ------------------------------------------------------------ CPU oracle --

def oracle_step_sample(budget_s=20.0, threads=0):
    """The oracle on a bounded sample of the decode workload: one layer of
    the 2B-shape stack for each M (quantise, unpack the packed weights,
    matmul, rescale, for the seven chained projections), repeated until
    `budget_s` is spent (at least once).  threads: 1 = single-threaded, 0 =
    every host core.  Returns GB/s of the same algorithmic bytes as the GPU
    line, reps, seconds, threads used."""
    import oracle
    from bitlinear_02_b300 import inputs
    oracle.set_threads(threads)
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
    used = oracle.threads()
    oracle.set_threads(0)
    return nbytes / dt / 1e9, reps, dt, used


def oracle_configs(threads=0):
    """The oracle as it stands, on every host core, per config: the small
    layer in full (repeated for about a second); the 2B prefill chain with M
    capped at 64 tokens (TOPS; a full 4096-token run would take hours); one
    layer of the 3B and 70B stacks at M = 1 (their own counter-based
    weights, unpacked per call like every oracle call), scaled by the layer
    count and labelled extrapolated."""
    import numpy as np
    import oracle
    from bitlinear_02_b300 import inputs
    oracle.set_threads(threads)
    res = {}

    def run_chain(shapes, M, packed, gam, x, eps_a, o_from):
        plan, dims = chain_plan(shapes, o_from)
        acts = {"x": x}
        for kind, a, o in plan:
            if kind == "quant":
                acts[o] = oracle.quant_act(acts[a], None, eps_a)
            else:
                q, sc = acts[a]
                N, K = dims[o]
                wq, _ = oracle.unpack(packed[o], N, K)
                acts[o] = oracle.epilogue(oracle.matmul(q, wq), sc, gam[o])

    # config 1: quantise + forward, one 512 x 256 layer
    wl = inputs.WORKLOADS["layer_small"]
    _, N, K = wl["shapes"][0]
    w = inputs.weights_fp32(N, K, seed=wl["seed"]).numpy()
    g = oracle.gamma(w)
    pk = oracle.pack(oracle.ternarize(w, g, wl["eps_w"]))
    x = inputs.bf16_bits(inputs.activations_bf16(1, K, seed=1))
    reps, t0 = 0, time.perf_counter()
    while True:
        q, sc = oracle.quant_act(x, None, wl["eps_a"])
        wq, _ = oracle.unpack(pk, N, K)
        oracle.epilogue(oracle.matmul(q, wq), sc, g)
        reps += 1
        if time.perf_counter() - t0 >= 1.0:
            break
    dt = (time.perf_counter() - t0) / reps
    b = algo_bytes_quant(1, K) + algo_bytes_forward(1, N, K)
    res["layer_small"] = {"us_per_layer": round(dt * 1e6, 1), "GB/s": round(b / dt / 1e9, 4),
                          "tokens_per_s": round(1 / dt, 1), "sample": f"{reps} layers"}

    # config 3: the prefill chain at 64 tokens
    wl = inputs.WORKLOADS["prefill_2b"]
    shapes = wl["shapes"]
    packed, gam = {}, {}
    for i, (name, N, K) in enumerate(shapes):
        w = inputs.weights_fp32(N, K, seed=wl["seed"] * 100 + i).numpy()
        gam[name] = oracle.gamma(w)
        packed[name] = oracle.pack(oracle.ternarize(w, gam[name], wl["eps_w"]))
        del w
    M = 64
    x = inputs.bf16_bits(inputs.activations_bf16(M, shapes[0][2], seed=wl["seed"] * 1000 + M, outlier_frac=0.01,
                                                 outlier_scale=20.0))
    t0 = time.perf_counter()
    run_chain(shapes, M, packed, gam, x, wl["eps_a"], "v")
    dt = time.perf_counter() - t0
    _, dims = chain_plan(shapes)
    ops = sum(2 * M * dims[o][0] * dims[o][1] for k, _, o in chain_plan(shapes)[0] if k == "fwd")
    res["prefill_2b"] = {"M": M, "chain_ms": round(dt * 1e3, 1), "TOPS": round(ops / dt / 1e12, 5),
                         "tokens_per_s": round(M / dt, 1),
                         "sample": "one seven-projection chain at 64 tokens (M capped; 4096 would take hours)"}
    del packed

    # configs 4 and 5: one layer at M = 1, scaled by the layer count
    for name in ("stack_3b", "stack_70b"):
        wl = inputs.WORKLOADS[name]
        shapes, layers = wl["shapes"], wl["layers"]
        hidden = shapes[0][2]
        o_from = "v" if shapes[2][1] == hidden else "q"
        packed, gam = {}, {}
        for i, (pname, N, K) in enumerate(shapes):
            packed[pname] = oracle.pack(oracle.ternary_hash(inputs.stack_word(wl["seed"], 0, i), K, 0, N))
            gam[pname] = np.float32(inputs.gamma_uniform(wl["seed"] * 100000 + i))
        x = inputs.bf16_bits(inputs.activations_bf16(1, hidden, seed=3 + 7))
        t0 = time.perf_counter()
        run_chain(shapes, 1, packed, gam, x, wl["eps_a"], o_from)
        dt = time.perf_counter() - t0
        b = layer_bytes(1, shapes, o_from)
        res[name] = {"GB/s": round(b / dt / 1e9, 4), "tokens_per_s": round(1 / (dt * layers), 4),
                     "s_per_token": round(dt * layers, 2),
                     "sample": f"one layer at M = 1 in {dt:.2f} s, extrapolated to {layers} layers"}
        del packed
    used = oracle.threads()
    oracle.set_threads(0)
    for v in res.values():
        v["cores"] = used
    return res


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


def profile_gemv(spec):
    """--profile-gemv N,K,M[,copies]: the decode GEMV (bitlinear_forward) on
    `copies` distinct copies of one ternary matrix, 2 warm-up passes + 3
    timed passes (the driver for ncu captures of the decode kernel)."""
    import torch
    import bitlinear_02_b300 as bl
    from bitlinear_02_b300 import inputs
    parts = [int(v) for v in spec.split(",")]
    N, K, M = parts[:3]
    copies = parts[3] if len(parts) > 3 else 4
    dev = torch.device("cuda:0")
    wq = inputs.ternary_hash(N, K, inputs.stack_word(9, 0, 0), device=dev)
    mats = [bl.pack_ternary(wq) for _ in range(copies)]
    del wq
    gam = torch.tensor([0.02], dtype=torch.float32, device=dev)
    x = inputs.activations_bf16(M, K, seed=3, device=dev)
    q, s = bl.quant_act(x)
    out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)

    def rnd():
        for p in mats:
            bl.bitlinear_forward(q, s, p, gam, M, N, K, out)

    for _ in range(2):
        rnd()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        rnd()
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / (3 * copies)
    assert bl.bitlinear_check_status() == bl.OK
    print(json.dumps({"profile": "gemv", "N": N, "K": K, "M": M, "us": round(ms * 1000, 2),
                      "weight_GB/s": round(packed_bytes(N, K) / (ms * 1e-3) / 1e9, 1)}))
    return 0


def profile_format(spec):
    """--profile-format FMT,N,K,M[,copies]: the decode engine of one weight
    format (2bit, 5trit, binary) on `copies` distinct copies of one matrix,
    2 warm-up passes + 3 timed passes (the driver for ncu captures)."""
    import torch
    import bitlinear_02_b300 as bl
    from bitlinear_02_b300 import inputs
    parts = spec.split(",")
    fmt = parts[0]
    N, K, M = (int(v) for v in parts[1:4])
    copies = int(parts[4]) if len(parts) > 4 else 4
    dev = torch.device("cuda:0")
    w = inputs.weights_fp32(N, K, seed=5, device=dev)
    p2, gam = bl.pack_weights(w, 1e-5)
    if fmt == "5trit":
        p0 = bl.repack5(p2, N, K)
        fn = lambda q, s, p, out: bl.bitlinear_forward5(q, s, p, gam, M, N, K, out)
    elif fmt == "binary":
        p0, beta = bl.pack_binary(w, 8)
        fn = lambda q, s, p, out: bl.bitlinear_forward_binary(q, s, p, beta, 8, M, N, K, out)
    else:
        p0 = p2
        fn = lambda q, s, p, out: bl.bitlinear_forward(q, s, p, gam, M, N, K, out)
    del w
    mats = [p0] + [p0.clone() for _ in range(copies - 1)]
    x = inputs.activations_bf16(M, K, seed=3, device=dev)
    q, s = bl.quant_act(x)
    out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    for _ in range(2):
        for p in mats:
            fn(q, s, p, out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        for p in mats:
            fn(q, s, p, out)
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / (3 * copies)
    assert bl.bitlinear_check_status() == bl.OK
    print(json.dumps({"profile": "format", "format": fmt, "N": N, "K": K, "M": M, "us": round(ms * 1000, 2),
                      "weight_GB/s": round(p0.numel() / (ms * 1e-3) / 1e9, 1)}))
    return 0


def profile_fused(spec):
    """--profile-fused L,M[,WORKLOAD]: the fused decode path on an L-layer
    stack (the 2B shapes, or stack_3b / stack_70b) at M tokens, eagerly
    launched: 3 warm-up + 5 timed passes (driver for ncu captures)."""
    import torch
    import bitlinear_02_b300 as bl
    from bitlinear_02_b300 import inputs
    parts = spec.split(",")
    L, M = int(parts[0]), int(parts[1])
    workload = parts[2] if len(parts) > 2 else WORKLOAD
    dev = torch.device("cuda:0")
    bl.load_library()
    st = Stack(torch, bl, inputs, dev, workload, layers=L)
    fr = FusedRunner(st, M)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        fr.run(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        fr.run(stream)
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / 5
    assert bl.bitlinear_check_status() == bl.OK
    print(json.dumps({"profile": "fused", "workload": workload, "layers": L, "M": M, "ms_per_pass": round(ms, 4),
                      "launches_per_pass": fr.launches}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-stacks", action="store_true", help="skip the 3B and 70B stacks")
    ap.add_argument("--no-sweeps", action="store_true", help="skip the per-shape and mid-M sweeps")
    ap.add_argument("--profile-gemm", default=None, help="N,K,M[,int8]: time one GEMM shape (ncu driver)")
    ap.add_argument("--profile-gemv", default=None, help="N,K,M[,copies]: time the decode GEMV (ncu driver)")
    ap.add_argument("--profile-fused", default=None, help="L,M[,WORKLOAD]: time the fused decode path (ncu driver)")
    ap.add_argument("--profile-format", default=None,
                    help="FMT,N,K,M[,copies]: time one weight format's decode engine (ncu driver)")
    args = ap.parse_args()
    if args.profile_gemm:
        return profile_gemm(args.profile_gemm)
    if args.profile_gemv:
        return profile_gemv(args.profile_gemv)
    if args.profile_fused:
        return profile_fused(args.profile_fused)
    if args.profile_format:
        return profile_format(args.profile_format)
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

    st = Stack(torch, bl, inputs, dev, WORKLOAD, layers=LAYERS)
    runs = {M: FusedRunner(st, M) for M in M_LIST}
    bytes_step = sum(st.bytes(M) for M in M_LIST)
    n_launch = sum(r.launches for r in runs.values())

    def step():
        for M in M_LIST:
            runs[M].run(stream)

    graph = capture(torch, step, stream)
    sampler = ClockSampler(local)
    with sampler:
        ms = time_graphs(torch, [graph], args.steps, args.warmup, stream, barrier, clock=sampler)
        clocks = ClockSampler.summary(sampler.take())
        ms = max_over_ranks(torch, ms, dev, dist)
        assert bl.bitlinear_check_status() == bl.OK, "a bounded wait expired during the timed steps"
        value = job_value(bytes_step, args.steps, ws, ms)
        ms_step = ms / args.steps
        del graph

        # The fused decode kernel alone: the step less its three act_stats
        # launches (timed on their own) is 4 * LAYERS fused launches per M.
        stats_ms = 0.0
        for M in M_LIST:
            r = runs[M]
            g1 = capture(torch, lambda: bl.bitlinear_act_stats(st.input(M), M, st.hidden, st.eps_a, r.x_stats,
                                                               stream), stream)
            stats_ms += time_graphs(torch, [g1], 200, 5, stream) / 200
            del g1
        n_fused = n_launch - len(M_LIST)
        launch_us = 1000.0 * max(1e-9, ms_step - stats_ms) / n_fused
        fused_bytes = bytes_step - sum(algo_bytes_quant(M, st.hidden) for M in M_LIST)
        bytes_launch = fused_bytes / n_fused
        fused_gbs = bytes_launch / (launch_us * 1e-6) / 1e9

        # e2e: each M's input from pinned host memory, the public entry points
        # called one by one from the host, the last output read back, every step
        h2d = {M: st.input(M).cpu().pin_memory() for M in M_LIST}
        d2h = {M: torch.empty_like(runs[M].last_output(), device="cpu").pin_memory() for M in M_LIST}

        def e2e_step():
            for M in M_LIST:
                st.x[M].copy_(h2d[M], non_blocking=True)
                runs[M].run(stream)
                d2h[M].copy_(runs[M].last_output(), non_blocking=True)

        n_e2e = max(10, args.steps // 4)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                e2e_step()
            stream.synchronize()
            sampler.mark(True)
            t0 = time.perf_counter()
            for _ in range(n_e2e):
                e2e_step()
                stream.synchronize()
                _ = float(d2h[16][0, 0])  # read the result on the host
            e2e_s = time.perf_counter() - t0
            sampler.mark(False)
        e2e_val = bytes_step * n_e2e * ws / e2e_s / 1e9
        h2d_bytes = sum(t.numel() * t.element_size() for t in h2d.values())
        d2h_bytes = sum(t.numel() * t.element_size() for t in d2h.values())
        g_e2e = capture(torch, e2e_step, stream)
        with torch.cuda.stream(stream):
            t0 = time.perf_counter()
            for _ in range(n_e2e):
                g_e2e.replay()
                stream.synchronize()
                _ = float(d2h[16][0, 0])
            e2e_graph_s = time.perf_counter() - t0
        del g_e2e
        e2e_graph = bytes_step * n_e2e * ws / e2e_graph_s / 1e9

        unf = {M: UnfusedRunner(st, M) for M in M_LIST}
        g_unf = capture(torch, lambda: [unf[M].run(stream) for M in M_LIST], stream)
        unf_ms = time_graphs(torch, [g_unf], 20, 3, stream, clock=sampler) / 20
        del g_unf, unf
        conc_ms = concurrent_step_ms(torch, bl, inputs, st, stream)

        configs = {"layer_small": small_layer_row(torch, bl, inputs, dev, stream, hbm_peak)}
        rows2b = stack_rows(torch, st, M_LIST, stream, hbm_peak, reps=50, clock=sampler)
        configs["decode_2b"] = {"layers": st.layers, "packed_mb": round(st.packed_bytes / 1e6, 1), "rows": rows2b}
        sweep = midm = None
        if not args.no_sweeps:
            sweep = gemv_sweep(torch, bl, inputs, dev, stream, hbm_peak)
            sweep["quant_act"] = quant_sweep(torch, bl, inputs, dev, stream)
            sweep["formats"] = variants_sweep(torch, bl, inputs, dev, stream, hbm_peak)
            midm = midm_sweep(torch, bl, inputs, st, stream)
        del runs
        if not args.no_prefill:
            sampler.mark(True)
            configs["prefill_2b"] = prefill_bench(torch, bl, inputs, dev, stream, bf16_peak)
            sampler.mark(False)
        if not args.no_stacks:
            for wl, m_list in (("stack_3b", (1, 2, 4, 8, 16, 32, 64)),
                               ("stack_70b", (1, 2, 4, 8, 16, 32, 64, 128, 256))):
                t0 = time.perf_counter()
                stk = Stack(torch, bl, inputs, dev, wl)
                gen_s = time.perf_counter() - t0
                rows = stack_rows(torch, stk, m_list, stream, hbm_peak, reps=10, clock=sampler)
                configs[wl] = {"layers": stk.layers, "packed_gb": round(stk.packed_bytes / 1e9, 3),
                               "weights": "ternary from the on-device counter-based generator, "
                                          f"generated and packed in {gen_s:.1f} s", "o_from": stk.o_from,
                               "rows": rows}
                del stk
                torch.cuda.empty_cache()
        assert bl.bitlinear_check_status() == bl.OK, "a bounded wait expired during the measurements"
        clocks_all = ClockSampler.summary(sampler.all)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        gbs1, reps1, dt1, c1 = oracle_step_sample(budget_s=8.0, threads=1)
        gbs, reps, dt, cores = oracle_step_sample(budget_s=12.0, threads=0)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{reps} x one 2B-shape layer for each M=1,4,16 (quantise, unpack, matmul, rescale; "
                         f"7 chained projections) in {dt:.1f} s",
               "single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "cores": c1,
                                 "sample": f"{reps1} x the same sample in {dt1:.1f} s"},
               "configs": oracle_configs()}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 x ternary -> int32 (f16 tensor-core operands, exact), bf16 out",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": list(M_LIST), "layers": st.layers, "hidden": 2560,
                   "ffn": 6912, "projections": "q,k,v,o 2560x2560; gate,up 2560->6912; down 6912->2560",
                   "packed_mb": round(st.packed_bytes / 1e6, 1),
                   "l2": "inputs larger than L2: the stack's packed weights are 3x the 126 MB L2",
                   "bytes_per_step": bytes_step,
                   "graph": "one CUDA graph per step: per M one act_stats + 4 fused decode launches per layer",
                   "parallelism": f"replicas x{ws}"},
        "hbm_frac_of_step": round(value / ws / hbm_peak, 4),
        "tokens_per_s": {str(r["M"]): r["tokens_per_s"] for r in rows2b},
        "roofline": {"bound": "hbm", "achieved": round(fused_gbs, 1), "peak": round(hbm_peak, 1),
                     "unit": "GB/s", "frac": round(fused_gbs / hbm_peak, 4),
                     "traffic": (round(FUSED_DRAM_PER_PACKED_BYTE * st.packed_bytes * len(M_LIST) / n_fused)
                                 if FUSED_DRAM_PER_PACKED_BYTE else None),
                     "kernel": "fused_gemv_kernel<NT> (the fused decode path: quantiser folded into the GEMV)",
                     "launch_avg_us": round(launch_us, 3), "algo_bytes_per_launch": round(bytes_launch),
                     "peak_note": f"{peak_kind} HBM copy bandwidth",
                     "method": "CUDA events on the launching stream around the timed graph replays; the three "
                               "act_stats launches timed on their own and subtracted; average over the step's "
                               f"{n_fused} fused launches"},
        "concurrent": {"ms_per_step": round(conc_ms, 4),
                       "value": round(bytes_step / (conc_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                       "mode": "the three M as independent decode streams: one graph, a branch per M on its own "
                               "stream, each branch with its own copy of the weights; same kernels and bytes"},
        "unfused": {"ms_per_step": round(unf_ms, 4),
                    "value": round(bytes_step / (unf_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                    "mode": "bitlinear_quant_act + bitlinear_forward per projection, PDL-chained graph"},
        "configs": configs,
        "sweep": sweep,
        "mid_m": midm,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h_bytes,
                "mode": "the public entry points called one by one from Python (ctypes) every step, with the "
                        "pinned H2D input copies and D2H output reads inside, host sync per step",
                "graph": {"value": round(e2e_graph, 2), "unit": "GB/s",
                          "mode": "the same step (copies included) replayed as one CUDA graph"}},
        "gpu_launches": n_launch * args.steps,
        "clocks": clocks,
        "clocks_all_timed_regions": clocks_all,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
