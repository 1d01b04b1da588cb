"""Seeded synthetic inputs for the BitLinear workloads.

This module only draws random numbers and names shapes; it holds none of the
method's arithmetic (no quantisation, packing or matmul), so both the CUDA
path and the CPU oracle can be fed from it.

Workloads (shapes follow the model sizes the BitNet b1.58 pages discuss: the
2B4T model of the asi.tokyo write-up and the 3B / 70B rows of the
cheatsheet.md tables):

* ``layer_small``   M=1, K=256, N=512; W ~ N(0, 0.02^2) fp32, x ~ N(0, 1) bf16.
* ``decode_2b``     hidden 2560, projections q/k/v/o 2560x2560, gate/up
                    2560->6912, down 6912->2560; M in {1, 4, 16}.
* ``prefill_2b``    the same six shapes, M in {512, 2048, 4096}; x ~ N(0, 1)
                    with 1% of the K channels (seeded choice) scaled by 20.
* ``stack_3b``      26 layers, hidden 3200, FFN 8640; ternary weights drawn
                    directly (P(-1)=P(0)=P(+1)=1/3), per-tensor gamma ~ U(0.01, 0.05);
                    M in {1, 2, 4, ..., 64}.
* ``stack_70b``     80 layers, hidden 8192, FFN 28672, K/V 8192->1024;
                    ternary weights as above; M in {1, 2, 4, ..., 256}.

The two stacks' weights (0.8 GB and 17.1 GB packed) are drawn on the device
by ``ternary_hash``, a counter-based generator (SplitMix64), so that any row
can be regenerated on the host and no weight crosses the PCIe bus.
"""
from __future__ import annotations

import torch

# (name, N out, K in) per projection
SHAPES_2B = [
    ("q", 2560, 2560),
    ("k", 2560, 2560),
    ("v", 2560, 2560),
    ("o", 2560, 2560),
    ("gate", 6912, 2560),
    ("up", 6912, 2560),
    ("down", 2560, 6912),
]


def shapes_stack(hidden: int, ffn: int, kv: int):
    return [
        ("q", hidden, hidden),
        ("k", kv, hidden),
        ("v", kv, hidden),
        ("o", hidden, hidden),
        ("gate", ffn, hidden),
        ("up", ffn, hidden),
        ("down", hidden, ffn),
    ]


SHAPES_3B = shapes_stack(3200, 8640, 3200)
SHAPES_70B = shapes_stack(8192, 28672, 1024)

WORKLOADS = {
    "layer_small": dict(M=[1], shapes=[("proj", 512, 256)], seed=0, eps_w=1e-5, eps_a=1e-5),
    "decode_2b": dict(M=[1, 4, 16], shapes=SHAPES_2B, seed=2, eps_w=1e-5, eps_a=1e-5),
    "prefill_2b": dict(M=[512, 2048, 4096], shapes=SHAPES_2B, seed=3, eps_w=1e-5, eps_a=1e-5,
                       outlier_frac=0.01, outlier_scale=20.0),
    "stack_3b": dict(M=[1, 2, 4, 8, 16, 32, 64], shapes=SHAPES_3B, layers=26, seed=4, eps_a=1e-5),
    "stack_70b": dict(M=[1, 2, 4, 8, 16, 32, 64, 128, 256], shapes=SHAPES_70B, layers=80, seed=5,
                      eps_a=1e-5),
}


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def weights_fp32(N: int, K: int, seed: int, std: float = 0.02, device="cpu") -> torch.Tensor:
    """Master weights W[N, K] ~ N(0, std^2), fp32, row-major (K contiguous)."""
    g = generator(seed, device)
    return torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * std


def ternary(N: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """Ternary weights drawn directly: int8 in {-1, 0, +1}, each with p = 1/3."""
    g = generator(seed, device)
    return torch.randint(-1, 2, (N, K), generator=g, device=device, dtype=torch.int8)


def gamma_uniform(seed: int, lo: float = 0.01, hi: float = 0.05) -> float:
    g = generator(seed, "cpu")
    return float(torch.rand(1, generator=g).item() * (hi - lo) + lo)


def activations_bf16(M: int, K: int, seed: int, outlier_frac: float = 0.0,
                     outlier_scale: float = 20.0, device="cpu") -> torch.Tensor:
    """x[M, K] ~ N(0, 1) rounded to bf16; optionally a seeded set of
    round(outlier_frac * K) channels (at least one) scaled by outlier_scale."""
    g = generator(seed, device)
    x = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    if outlier_frac > 0.0:
        n_out = max(1, int(round(outlier_frac * K)))
        gc = generator(seed + 7919, "cpu")
        ch = torch.randperm(K, generator=gc)[:n_out].to(device)
        x[:, ch] *= outlier_scale
    return x.to(torch.bfloat16)


def gain_bf16(K: int, seed: int, device="cpu") -> torch.Tensor:
    """An RMSNorm gain vector ~ U(0.5, 1.5), bf16 (used by the gain tests)."""
    g = generator(seed, device)
    return (torch.rand(K, generator=g, device=device) + 0.5).to(torch.bfloat16)


def bf16_bits(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")


# ---------------------------------------------------------------- SplitMix64 ---
# Counter-based ternary weights for the stacked workloads.  SplitMix64
# (Steele, Lea and Flood, OOPSLA 2014): the i-th output (i = 0, 1, ...) of
# the generator seeded with s is mix(s + (i + 1) * 0x9E3779B97F4A7C15), with
#   mix(z): z = (z ^ z >> 30) * 0xBF58476D1CE4E5B9;
#           z = (z ^ z >> 27) * 0x94D049BB133111EB;  z ^ z >> 31
# (64-bit wrap-around, logical shifts).  A matrix keyed by `word` takes
# s = the first output of SplitMix64 seeded with `word`; its element (n, k)
# is output n*K + k of SplitMix64 seeded with s, mapped to {-1, 0, +1} as
# floor(hi32 * 3 / 2^32) - 1, hi32 being the output's upper 32 bits.
# Written here with torch int64 tensors (two's-complement wrap-around), so
# it runs on the GPU; the oracle has its own C version of the definition.

_GOLDEN = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB


def _i64(u: int) -> int:
    """A uint64 constant as the int64 with the same bits."""
    u &= (1 << 64) - 1
    return u - (1 << 64) if u >= (1 << 63) else u


def _srl(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _i64(_MIX1)
    z = (z ^ _srl(z, 27)) * _i64(_MIX2)
    return z ^ _srl(z, 31)


def _mix_int(z: int) -> int:
    m = (1 << 64) - 1
    z &= m
    z = ((z ^ (z >> 30)) * _MIX1) & m
    z = ((z ^ (z >> 27)) * _MIX2) & m
    return z ^ (z >> 31)


def stack_word(seed: int, layer: int, proj: int) -> int:
    """Key of one matrix of a stacked workload (its seed, layer, projection)."""
    return (int(seed) << 40) | (int(layer) << 8) | int(proj)


def ternary_hash(N: int, K: int, word: int, device="cpu", rows_per_chunk: int = 4096) -> torch.Tensor:
    """The [N, K] ternary matrix keyed by `word`, int8 in {-1, 0, +1}
    (P = 1/3 each up to 2^-32), computed on `device`."""
    s = _mix_int(int(word) + _GOLDEN)  # first output of SplitMix64 seeded with word
    out = torch.empty(N, K, dtype=torch.int8, device=device)
    col = torch.arange(K, dtype=torch.int64, device=device)
    for n0 in range(0, N, rows_per_chunk):
        n1 = min(N, n0 + rows_per_chunk)
        rows = torch.arange(n0, n1, dtype=torch.int64, device=device)
        i1 = rows[:, None] * K + col[None, :] + 1          # i + 1
        v = _mix(i1 * _i64(_GOLDEN) + _i64(s))
        out[n0:n1] = ((_srl(v, 32) * 3) >> 32).to(torch.int8) - 1
    return out
