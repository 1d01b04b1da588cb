"""CPU oracle for the BitNet b1.58 BitLinear hot path (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never loads it, and it
shares no code with the CUDA path: it is a plain C restatement of the
method's definitions (``bitlinear_oracle.c``) behind a ctypes wrapper.

Pages cited by the C source: the asi.tokyo "BitNet B1.58 2B4T" write-up, the
cheatsheet.md BitNet b1.58 summary (section "BitNet b1.58とは？"), the
lumen-it.ai BitNet article, and the vi.news.hada.io topic 20406 comments on
ternary packing (five ternary digits per byte).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bitlinear_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-fopenmp"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        L.bl_oracle_sum_abs.argtypes = [P, I64]
        L.bl_oracle_sum_abs.restype = ctypes.c_double
        L.bl_oracle_gamma.argtypes = [P, I64, I64]
        L.bl_oracle_gamma.restype = ctypes.c_float
        L.bl_oracle_ternarize.argtypes = [P, I64, ctypes.c_float, ctypes.c_float, P]
        L.bl_oracle_packed_bytes.argtypes = [I64, I64]
        L.bl_oracle_packed_bytes.restype = I64
        L.bl_oracle_position.argtypes = [I64, I64, I64, ctypes.POINTER(I64), ctypes.POINTER(ctypes.c_int)]
        L.bl_oracle_pack.argtypes = [P, I64, I64, P]
        L.bl_oracle_unpack.argtypes = [P, I64, I64, P]
        L.bl_oracle_unpack.restype = I64
        L.bl_oracle_quant_act.argtypes = [P, P, I64, I64, ctypes.c_float, P, P]
        L.bl_oracle_matmul.argtypes = [P, P, I64, I64, I64, P]
        L.bl_oracle_splitmix64.argtypes = [ctypes.c_uint64, I64, P]
        L.bl_oracle_ternary_hash.argtypes = [ctypes.c_uint64, I64, I64, I64, P]
        L.bl_oracle_matmul.restype = ctypes.c_int
        L.bl_oracle_matmul_pairs.argtypes = [P, P, I64, P, P, I64, P]
        L.bl_oracle_epilogue.argtypes = [P, P, ctypes.c_float, I64, I64, P]
        L.bl_oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.bl_oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.bl_oracle_threads.restype = ctypes.c_int
        L.bl_oracle_set_threads.argtypes = [ctypes.c_int]
        L.bl_oracle_set_threads.restype = None
        L.bl_oracle_packed5_bytes.argtypes = [I64, I64]
        L.bl_oracle_packed5_bytes.restype = I64
        L.bl_oracle_position5.argtypes = [I64, I64, I64, ctypes.POINTER(I64), ctypes.POINTER(ctypes.c_int)]
        L.bl_oracle_encode5.argtypes = [P]
        L.bl_oracle_encode5.restype = ctypes.c_uint8
        L.bl_oracle_decode5.argtypes = [ctypes.c_uint8, P]
        L.bl_oracle_decode5.restype = ctypes.c_int
        L.bl_oracle_pack5.argtypes = [P, I64, I64, P]
        L.bl_oracle_unpack5.argtypes = [P, I64, I64, P]
        L.bl_oracle_unpack5.restype = I64
        L.bl_oracle_beta.argtypes = [P, I64, I64, I64, P]
        L.bl_oracle_binarize.argtypes = [P, I64, P]
        L.bl_oracle_packed1_bytes.argtypes = [I64, I64]
        L.bl_oracle_packed1_bytes.restype = I64
        L.bl_oracle_position1.argtypes = [I64, I64, I64, ctypes.POINTER(I64), ctypes.POINTER(ctypes.c_int)]
        L.bl_oracle_pack1.argtypes = [P, I64, I64, P]
        L.bl_oracle_unpack1.argtypes = [P, I64, I64, P]
        L.bl_oracle_unpack1.restype = I64
        L.bl_oracle_epilogue_groups.argtypes = [P, P, P, I64, I64, I64, P]
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def sum_abs(w: np.ndarray) -> float:
    w = np.ascontiguousarray(w, dtype=np.float32)
    return lib().bl_oracle_sum_abs(_ptr(w), w.size)


def gamma(w: np.ndarray) -> np.float32:
    """Absmean scale of an [N, K] fp32 weight matrix."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    return np.float32(lib().bl_oracle_gamma(_ptr(w), N, K))


def ternarize(w: np.ndarray, g: float, eps: float) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty(w.shape, dtype=np.int8)
    lib().bl_oracle_ternarize(_ptr(w), w.size, float(np.float32(g)), float(np.float32(eps)), _ptr(out))
    return out


def packed_bytes(N: int, K: int) -> int:
    return int(lib().bl_oracle_packed_bytes(N, K))


def position(n: int, k: int, K: int) -> tuple[int, int]:
    b = ctypes.c_int64()
    s = ctypes.c_int()
    lib().bl_oracle_position(n, k, K, ctypes.byref(b), ctypes.byref(s))
    return b.value, s.value


def pack(wq: np.ndarray) -> np.ndarray:
    wq = np.ascontiguousarray(wq, dtype=np.int8)
    N, K = wq.shape
    out = np.empty(packed_bytes(N, K), dtype=np.uint8)
    lib().bl_oracle_pack(_ptr(wq), N, K, _ptr(out))
    return out


def unpack(packed: np.ndarray, N: int, K: int) -> tuple[np.ndarray, int]:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    assert packed.size == packed_bytes(N, K)
    out = np.zeros((N, K), dtype=np.int8)
    bad = lib().bl_oracle_unpack(_ptr(packed), N, K, _ptr(out))
    return out, int(bad)


def quant_act(x_bf16: np.ndarray, gain_bf16: np.ndarray | None, eps: float):
    """x_bf16: uint16 [M, K] holding bf16 bit patterns.  Returns (q int8, s_tok fp32)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    q = np.empty((M, K), dtype=np.int8)
    s = np.empty(M, dtype=np.float32)
    g = None if gain_bf16 is None else np.ascontiguousarray(gain_bf16, dtype=np.uint16)
    lib().bl_oracle_quant_act(_ptr(x), None if g is None else _ptr(g), M, K, float(np.float32(eps)), _ptr(q), _ptr(s))
    return q, s


def matmul(q: np.ndarray, wq: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int8)
    wq = np.ascontiguousarray(wq, dtype=np.int8)
    M, K = q.shape
    N, K2 = wq.shape
    assert K == K2
    acc = np.empty((M, N), dtype=np.int32)
    if lib().bl_oracle_matmul(_ptr(q), _ptr(wq), M, N, K, _ptr(acc)):
        raise OverflowError("accumulator exceeds int32")
    return acc


def matmul_pairs(q: np.ndarray, wq: np.ndarray, ms: np.ndarray, ns: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int8)
    wq = np.ascontiguousarray(wq, dtype=np.int8)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    acc = np.empty(ms.size, dtype=np.int32)
    lib().bl_oracle_matmul_pairs(_ptr(q), _ptr(wq), q.shape[1], _ptr(ms), _ptr(ns), ms.size, _ptr(acc))
    return acc


def epilogue(acc: np.ndarray, s_tok: np.ndarray, g: float) -> np.ndarray:
    """Returns uint16 [M, N] bf16 bit patterns."""
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    s_tok = np.ascontiguousarray(s_tok, dtype=np.float32)
    M, N = acc.shape
    out = np.empty((M, N), dtype=np.uint16)
    lib().bl_oracle_epilogue(_ptr(acc), _ptr(s_tok), float(np.float32(g)), M, N, _ptr(out))
    return out


def f32_to_bf16(f: float) -> int:
    return int(lib().bl_oracle_f32_to_bf16(float(np.float32(f))))


def threads() -> int:
    return int(lib().bl_oracle_threads())


def set_threads(n: int) -> None:
    """Threads of the oracle's parallel loops (n <= 0: all cores)."""
    lib().bl_oracle_set_threads(int(n))


def forward(x_bf16: np.ndarray, w: np.ndarray, eps_w: float, eps_a: float, gain_bf16=None):
    """The whole path on the CPU: (gamma, packed, q, s_tok, acc, out_bf16)."""
    g = gamma(w)
    wq = ternarize(w, g, eps_w)
    packed = pack(wq)
    q, s = quant_act(x_bf16, gain_bf16, eps_a)
    acc = matmul(q, wq)
    out = epilogue(acc, s, g)
    return g, packed, q, s, acc, out


def splitmix64(seed: int, n: int) -> np.ndarray:
    """The first n outputs of SplitMix64 seeded with `seed` (uint64)."""
    out = np.empty(n, dtype=np.uint64)
    lib().bl_oracle_splitmix64(ctypes.c_uint64(seed & (2**64 - 1)), n, _ptr(out))
    return out


def ternary_hash(word: int, K: int, n0: int, n1: int) -> np.ndarray:
    """Rows [n0, n1) of the ternary matrix keyed by `word` (int8, {-1,0,1}):
    the synthetic weights of the stacked workloads, from SplitMix64."""
    out = np.empty((n1 - n0, K), dtype=np.int8)
    lib().bl_oracle_ternary_hash(ctypes.c_uint64(word & (2**64 - 1)), K, n0, n1, _ptr(out))
    return out


# ----------------------------------------------- five digits per byte ---

def packed5_bytes(N: int, K: int) -> int:
    return int(lib().bl_oracle_packed5_bytes(N, K))


def position5(n: int, k: int, K: int) -> tuple[int, int]:
    b = ctypes.c_int64()
    d = ctypes.c_int()
    lib().bl_oracle_position5(n, k, K, ctypes.byref(b), ctypes.byref(d))
    return b.value, d.value


def encode5(digits) -> int:
    e = np.ascontiguousarray(digits, dtype=np.int32)
    assert e.shape == (5,)
    return int(lib().bl_oracle_encode5(_ptr(e)))


def decode5(b: int):
    """The five digits of byte b, or None if b encodes nothing."""
    e = np.zeros(5, dtype=np.int32)
    return e if lib().bl_oracle_decode5(ctypes.c_uint8(b), _ptr(e)) else None


def pack5(wq: np.ndarray) -> np.ndarray:
    wq = np.ascontiguousarray(wq, dtype=np.int8)
    N, K = wq.shape
    out = np.empty(packed5_bytes(N, K), dtype=np.uint8)
    lib().bl_oracle_pack5(_ptr(wq), N, K, _ptr(out))
    return out


def unpack5(packed: np.ndarray, N: int, K: int) -> tuple[np.ndarray, int]:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    assert packed.size == packed5_bytes(N, K)
    wq = np.empty((N, K), dtype=np.int8)
    bad = int(lib().bl_oracle_unpack5(_ptr(packed), N, K, _ptr(wq)))
    return wq, bad


# ------------------------------------------------ original binary BitNet ---

def beta(w: np.ndarray, G: int) -> np.ndarray:
    """Mean |W| of each of G equal blocks of consecutive rows (float32 [G])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    assert N % G == 0
    out = np.empty(G, dtype=np.float32)
    lib().bl_oracle_beta(_ptr(w), N, K, G, _ptr(out))
    return out


def binarize(w: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty(w.shape, dtype=np.int8)
    lib().bl_oracle_binarize(_ptr(w), w.size, _ptr(out))
    return out


def packed1_bytes(N: int, K: int) -> int:
    return int(lib().bl_oracle_packed1_bytes(N, K))


def position1(n: int, k: int, K: int) -> tuple[int, int]:
    b = ctypes.c_int64()
    s = ctypes.c_int()
    lib().bl_oracle_position1(n, k, K, ctypes.byref(b), ctypes.byref(s))
    return b.value, s.value


def pack1(wb: np.ndarray) -> np.ndarray:
    wb = np.ascontiguousarray(wb, dtype=np.int8)
    N, K = wb.shape
    out = np.empty(packed1_bytes(N, K), dtype=np.uint8)
    lib().bl_oracle_pack1(_ptr(wb), N, K, _ptr(out))
    return out


def unpack1(packed: np.ndarray, N: int, K: int) -> tuple[np.ndarray, int]:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    assert packed.size == packed1_bytes(N, K)
    wb = np.empty((N, K), dtype=np.int8)
    bad = int(lib().bl_oracle_unpack1(_ptr(packed), N, K, _ptr(wb)))
    return wb, bad


def epilogue_groups(acc: np.ndarray, s_tok: np.ndarray, beta_g: np.ndarray) -> np.ndarray:
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    s_tok = np.ascontiguousarray(s_tok, dtype=np.float32)
    beta_g = np.ascontiguousarray(beta_g, dtype=np.float32)
    M, N = acc.shape
    out = np.empty((M, N), dtype=np.uint16)
    lib().bl_oracle_epilogue_groups(_ptr(acc), _ptr(s_tok), _ptr(beta_g), beta_g.size, M, N, _ptr(out))
    return out
