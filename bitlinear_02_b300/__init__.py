"""BitNet b1.58 BitLinear on one B300: thin Python binding of ``libbitlinear.so``.

The functions named ``bitlinear_*`` mirror the C ABI in ``include/bitlinear.h``
one to one: they only turn torch tensors into device pointers, pass the
current CUDA stream and raise on a non-zero status.  Every step of the path
runs in the library's CUDA kernels; there is no CPU fallback.  If the
library is missing (not built) every call raises ``RuntimeError``.

Convenience wrappers (``pack_weights``, ``quant_act``, ``forward``,
``bitlinear``) allocate the outputs with torch and call the same entry points.

With ``BITLINEAR_DEBUG=1`` in the environment the binding loads the debug
build, ``libbitlinear_debug.so`` (device-side bounds checks; see
``include/bitlinear.h``), instead.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "BitLinearError", "library_path", "load_library",
    "bitlinear_packed_bytes", "bitlinear_pack_weights", "bitlinear_pack_weights_noalloc",
    "bitlinear_pack_ternary",
    "bitlinear_quant_act", "bitlinear_forward", "bitlinear_check_status",
    "bitlinear_quant_act_f16", "bitlinear_forward_f16", "quant_act_f16", "forward_f16",
    "bitlinear_set_wait_limit", "bitlinear_set_engine", "bitlinear_status_string",
    "bitlinear_packed5_bytes", "bitlinear_repack5", "bitlinear_forward5", "repack5", "forward5",
    "bitlinear_packed1_bytes", "bitlinear_pack_binary", "bitlinear_forward_binary", "pack_binary", "forward_binary", "bitlinear_version",
    "pack_weights", "pack_ternary", "quant_act", "forward", "bitlinear",
    "FusedProj", "bitlinear_fused_stats_bytes", "bitlinear_act_stats", "bitlinear_forward_fused",
    "bitlinear_fused_factors", "fused_factors", "new_stats",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libbitlinear_debug.so" if os.environ.get("BITLINEAR_DEBUG") == "1" else "libbitlinear.so"

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_CUDA = 3
ERR_TIMEOUT = 4
ERR_STATE = 5
ERR_BOUNDS = 6


class FusedProj(ctypes.Structure):
    """bitlinear_fused_proj_t: one projection of a fused decode GEMV launch."""
    _fields_ = [("packed", ctypes.c_void_p), ("gamma", ctypes.c_void_p), ("N", ctypes.c_int64),
                ("out_bf16", ctypes.c_void_p), ("acc_out", ctypes.c_void_p), ("stats", ctypes.c_void_p)]


class BitLinearError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {bitlinear_status_string(status)} (status {status})")


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


_lib = None


def load_library():
    """Load the in-tree CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python bitlinear_02_b300/build.py` "
            "(or __graft_entry__.build()); there is no CPU fallback")
    L = ctypes.CDLL(path)
    P, I64, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
    L.bitlinear_status_string.argtypes = [ctypes.c_int]
    L.bitlinear_status_string.restype = ctypes.c_char_p
    L.bitlinear_version.restype = ctypes.c_int
    L.bitlinear_packed_bytes.argtypes = [I64, I64]
    L.bitlinear_packed_bytes.restype = ctypes.c_size_t
    L.bitlinear_pack_weights.argtypes = [P, I64, I64, F, P, P, P]
    L.bitlinear_pack_ternary.argtypes = [P, I64, I64, P, P]
    L.bitlinear_pack_weights_noalloc.argtypes = [P, I64, I64, F, P, P, P]
    L.bitlinear_quant_act.argtypes = [P, P, I64, I64, F, P, P, P]
    L.bitlinear_forward.argtypes = [P, P, P, P, I64, I64, I64, P, P, P]
    L.bitlinear_check_status.argtypes = [P]
    L.bitlinear_set_wait_limit.argtypes = [ctypes.c_uint32]
    L.bitlinear_set_wait_limit.restype = None
    L.bitlinear_set_engine.argtypes = [ctypes.c_int32, ctypes.c_int32]
    L.bitlinear_packed5_bytes.argtypes = [I64, I64]
    L.bitlinear_packed5_bytes.restype = ctypes.c_size_t
    L.bitlinear_repack5.argtypes = [P, I64, I64, P, P]
    L.bitlinear_forward5.argtypes = [P, P, P, P, I64, I64, I64, P, P, P]
    L.bitlinear_packed1_bytes.argtypes = [I64, I64]
    L.bitlinear_packed1_bytes.restype = ctypes.c_size_t
    L.bitlinear_pack_binary.argtypes = [P, I64, I64, I64, P, P, P]
    L.bitlinear_forward_binary.argtypes = [P, P, P, P, I64, I64, I64, I64, P, P, P]
    L.bitlinear_quant_act_f16.argtypes = [P, P, I64, I64, F, P, P, P]
    L.bitlinear_fused_stats_bytes.argtypes = []
    L.bitlinear_fused_stats_bytes.restype = ctypes.c_size_t
    L.bitlinear_act_stats.argtypes = [P, I64, I64, F, P, P]
    L.bitlinear_forward_fused.argtypes = [P, P, I64, I64, ctypes.c_int32, ctypes.POINTER(FusedProj), F, P]
    L.bitlinear_fused_factors.argtypes = [P, I64, I64, F, ctypes.c_int32, P, P, P]
    L.bitlinear_forward_f16.argtypes = [P, P, P, P, I64, I64, I64, P, P, P]
    L.bitlinear_set_fused_prepass.argtypes = [I64]
    L.bitlinear_debug_selftest.argtypes = [P]
    for name in ("bitlinear_pack_weights", "bitlinear_pack_weights_noalloc", "bitlinear_pack_ternary", "bitlinear_quant_act",
                 "bitlinear_forward", "bitlinear_check_status",
                 "bitlinear_quant_act_f16", "bitlinear_forward_f16", "bitlinear_act_stats",
                 "bitlinear_forward_fused", "bitlinear_fused_factors", "bitlinear_set_engine",
                 "bitlinear_repack5", "bitlinear_forward5", "bitlinear_pack_binary", "bitlinear_forward_binary",
                 "bitlinear_set_fused_prepass", "bitlinear_debug_selftest"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, what: str):
    if status != OK:
        raise BitLinearError(status, what)


# ---------------------------------------------------------------- C names ---

def bitlinear_status_string(status: int) -> str:
    return load_library().bitlinear_status_string(int(status)).decode()


def bitlinear_version() -> int:
    return int(load_library().bitlinear_version())


def bitlinear_packed_bytes(N: int, K: int) -> int:
    return int(load_library().bitlinear_packed_bytes(int(N), int(K)))


def bitlinear_pack_weights(W, N: int, K: int, eps: float, packed, gamma, stream=None) -> None:
    _check(load_library().bitlinear_pack_weights(_ptr(W), int(N), int(K), float(eps), _ptr(packed),
                                                 _ptr(gamma), _stream(stream)),
           "bitlinear_pack_weights")


def bitlinear_pack_weights_noalloc(W, N: int, K: int, eps: float, packed, gamma,
                                   stream=None) -> None:
    """bitlinear_pack_weights for callers that cannot allocate: its scratch
    is a fixed array inside the library (see include/bitlinear.h)."""
    _check(load_library().bitlinear_pack_weights_noalloc(_ptr(W), int(N), int(K), float(eps),
                                                         _ptr(packed), _ptr(gamma), _stream(stream)),
           "bitlinear_pack_weights_noalloc")


def bitlinear_pack_ternary(Wq, N: int, K: int, packed, stream=None) -> None:
    _check(load_library().bitlinear_pack_ternary(_ptr(Wq), int(N), int(K), _ptr(packed),
                                                 _stream(stream)),
           "bitlinear_pack_ternary")


def bitlinear_quant_act(x, gain, M: int, K: int, eps: float, q, tok_scale, stream=None) -> None:
    _check(load_library().bitlinear_quant_act(_ptr(x), _ptr(gain), int(M), int(K), float(eps),
                                              _ptr(q), _ptr(tok_scale), _stream(stream)),
           "bitlinear_quant_act")


def bitlinear_forward(q, tok_scale, packed, gamma, M: int, N: int, K: int, out, acc_out=None,
                      stream=None) -> None:
    _check(load_library().bitlinear_forward(_ptr(q), _ptr(tok_scale), _ptr(packed), _ptr(gamma),
                                            int(M), int(N), int(K), _ptr(out), _ptr(acc_out),
                                            _stream(stream)),
           "bitlinear_forward")


def bitlinear_quant_act_f16(x, gain, M: int, K: int, eps: float, q_f16, tok_scale, stream=None) -> None:
    _check(load_library().bitlinear_quant_act_f16(_ptr(x), _ptr(gain), int(M), int(K), float(eps),
                                                  _ptr(q_f16), _ptr(tok_scale), _stream(stream)),
           "bitlinear_quant_act_f16")


def bitlinear_forward_f16(q_f16, tok_scale, packed, gamma, M: int, N: int, K: int, out, acc_out=None,
                          stream=None) -> None:
    _check(load_library().bitlinear_forward_f16(_ptr(q_f16), _ptr(tok_scale), _ptr(packed), _ptr(gamma),
                                                int(M), int(N), int(K), _ptr(out), _ptr(acc_out),
                                                _stream(stream)),
           "bitlinear_forward_f16")


def bitlinear_fused_stats_bytes() -> int:
    return int(load_library().bitlinear_fused_stats_bytes())


def bitlinear_act_stats(x, M: int, K: int, eps: float, stats, stream=None) -> None:
    _check(load_library().bitlinear_act_stats(_ptr(x), int(M), int(K), float(eps), _ptr(stats),
                                              _stream(stream)),
           "bitlinear_act_stats")


def bitlinear_forward_fused(x, x_stats, M: int, K: int, projs, eps: float = 1e-5, stream=None) -> None:
    """projs: list of FusedProj (up to 4) sharing the input x."""
    arr = (FusedProj * len(projs))(*projs)
    _check(load_library().bitlinear_forward_fused(_ptr(x), _ptr(x_stats), int(M), int(K), len(projs), arr,
                                                  float(eps), _stream(stream)),
           "bitlinear_forward_fused")


def bitlinear_fused_factors(stats, M: int, K: int, eps: float, consume: bool, c_out, ts_out,
                            stream=None) -> None:
    _check(load_library().bitlinear_fused_factors(_ptr(stats), int(M), int(K), float(eps), 1 if consume else 0,
                                                  _ptr(c_out), _ptr(ts_out), _stream(stream)),
           "bitlinear_fused_factors")


def fused_factors(stats, M: int, K: int, eps: float = 1e-5, consume: bool = False, stream=None):
    """(c, tok_scale) of a factor buffer as device fp32 [M] tensors."""
    c = torch.empty(M, dtype=torch.float32, device=stats.device)
    ts = torch.empty(M, dtype=torch.float32, device=stats.device)
    bitlinear_fused_factors(stats, M, K, eps, consume, c, ts, stream)
    return c, ts


def new_stats(device="cuda"):
    """A zeroed factor buffer for the fused decode path."""
    return torch.zeros(bitlinear_fused_stats_bytes(), dtype=torch.uint8, device=device)


def bitlinear_check_status(stream=None) -> int:
    """Returns the status code (OK, ERR_STATE or ERR_TIMEOUT); does not raise."""
    return int(load_library().bitlinear_check_status(_stream(stream)))


def bitlinear_set_wait_limit(iterations: int) -> None:
    load_library().bitlinear_set_wait_limit(int(iterations))


def bitlinear_packed5_bytes(N: int, K: int) -> int:
    return int(load_library().bitlinear_packed5_bytes(int(N), int(K)))


def bitlinear_repack5(packed, N: int, K: int, packed5, stream=None) -> None:
    _check(load_library().bitlinear_repack5(_ptr(packed), int(N), int(K), _ptr(packed5), _stream(stream)),
           "bitlinear_repack5")


def bitlinear_forward5(q, tok_scale, packed5, gamma, M: int, N: int, K: int, out, acc_out=None,
                       stream=None) -> None:
    _check(load_library().bitlinear_forward5(_ptr(q), _ptr(tok_scale), _ptr(packed5), _ptr(gamma), int(M), int(N),
                                             int(K), _ptr(out), _ptr(acc_out), _stream(stream)),
           "bitlinear_forward5")


def bitlinear_packed1_bytes(N: int, K: int) -> int:
    return int(load_library().bitlinear_packed1_bytes(int(N), int(K)))


def bitlinear_pack_binary(W, N: int, K: int, groups: int, packed1, beta, stream=None) -> None:
    _check(load_library().bitlinear_pack_binary(_ptr(W), int(N), int(K), int(groups), _ptr(packed1), _ptr(beta),
                                                _stream(stream)),
           "bitlinear_pack_binary")


def bitlinear_forward_binary(q, tok_scale, packed1, beta, groups: int, M: int, N: int, K: int, out,
                             acc_out=None, stream=None) -> None:
    _check(load_library().bitlinear_forward_binary(_ptr(q), _ptr(tok_scale), _ptr(packed1), _ptr(beta),
                                                   int(groups), int(M), int(N), int(K), _ptr(out), _ptr(acc_out),
                                                   _stream(stream)),
           "bitlinear_forward_binary")


def bitlinear_debug_selftest(stream=None) -> int:
    """Debug build: records one failed bounds check (no memory access);
    returns the status (ERR_UNSUPPORTED in a release build), does not raise."""
    return int(load_library().bitlinear_debug_selftest(_stream(stream)))


def bitlinear_set_fused_prepass(min_weight_bytes: int = -1) -> None:
    """Pre-pass threshold of bitlinear_forward_fused (-1 restores the default)."""
    _check(load_library().bitlinear_set_fused_prepass(int(min_weight_bytes)), "bitlinear_set_fused_prepass")


def bitlinear_set_engine(gemv_max_tokens: int = -1, split_k: int = 0) -> None:
    """Engine choice of the forward calls (-1 / 0 restore the defaults)."""
    _check(load_library().bitlinear_set_engine(int(gemv_max_tokens), int(split_k)), "bitlinear_set_engine")


# ------------------------------------------------------------ convenience ---

def pack_weights(W: torch.Tensor, eps: float = 1e-5):
    """fp32 [N, K] CUDA tensor -> (packed uint8 tensor, gamma float32 [1] tensor)."""
    N, K = W.shape
    packed = torch.empty(bitlinear_packed_bytes(N, K), dtype=torch.uint8, device=W.device)
    gamma = torch.empty(1, dtype=torch.float32, device=W.device)
    bitlinear_pack_weights(W, N, K, eps, packed, gamma)
    return packed, gamma


def pack_ternary(Wq: torch.Tensor) -> torch.Tensor:
    N, K = Wq.shape
    packed = torch.empty(bitlinear_packed_bytes(N, K), dtype=torch.uint8, device=Wq.device)
    bitlinear_pack_ternary(Wq, N, K, packed)
    return packed


def quant_act(x: torch.Tensor, gain: torch.Tensor | None = None, eps: float = 1e-5):
    """bf16 [M, K] -> (q int8 [M, K], tok_scale float32 [M])."""
    M, K = x.shape
    q = torch.empty(M, K, dtype=torch.int8, device=x.device)
    s = torch.empty(M, dtype=torch.float32, device=x.device)
    bitlinear_quant_act(x, gain, M, K, eps, q, s)
    return q, s


def quant_act_f16(x: torch.Tensor, gain: torch.Tensor | None = None, eps: float = 1e-5):
    """bf16 [M, K] -> (q as f16 [M, K], tok_scale float32 [M])."""
    M, K = x.shape
    q = torch.empty(M, K, dtype=torch.float16, device=x.device)
    s = torch.empty(M, dtype=torch.float32, device=x.device)
    bitlinear_quant_act_f16(x, gain, M, K, eps, q, s)
    return q, s


def forward_f16(q: torch.Tensor, tok_scale: torch.Tensor, packed: torch.Tensor, gamma: torch.Tensor,
                N: int, out: torch.Tensor | None = None, acc_out: torch.Tensor | None = None):
    M, K = q.shape
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=q.device)
    bitlinear_forward_f16(q, tok_scale, packed, gamma, M, N, K, out, acc_out)
    return out


def forward(q: torch.Tensor, tok_scale: torch.Tensor, packed: torch.Tensor, gamma: torch.Tensor,
            N: int, out: torch.Tensor | None = None, acc_out: torch.Tensor | None = None):
    M, K = q.shape
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=q.device)
    bitlinear_forward(q, tok_scale, packed, gamma, M, N, K, out, acc_out)
    return out


def repack5(packed: torch.Tensor, N: int, K: int) -> torch.Tensor:
    """2-bit packed matrix -> the five-digits-per-byte layout (uint8 tensor)."""
    p5 = torch.empty(bitlinear_packed5_bytes(N, K), dtype=torch.uint8, device=packed.device)
    bitlinear_repack5(packed, N, K, p5)
    return p5


def forward5(q: torch.Tensor, tok_scale: torch.Tensor, packed5: torch.Tensor, gamma: torch.Tensor,
             N: int, out: torch.Tensor | None = None, acc_out: torch.Tensor | None = None):
    M, K = q.shape
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=q.device)
    bitlinear_forward5(q, tok_scale, packed5, gamma, M, N, K, out, acc_out)
    return out


def pack_binary(W: torch.Tensor, groups: int = 1):
    """fp32 [N, K] CUDA tensor -> (packed sign bits uint8, beta float32 [groups])."""
    N, K = W.shape
    p1 = torch.empty(bitlinear_packed1_bytes(N, K), dtype=torch.uint8, device=W.device)
    beta = torch.empty(groups, dtype=torch.float32, device=W.device)
    bitlinear_pack_binary(W, N, K, groups, p1, beta)
    return p1, beta


def forward_binary(q: torch.Tensor, tok_scale: torch.Tensor, packed1: torch.Tensor, beta: torch.Tensor,
                   N: int, out: torch.Tensor | None = None, acc_out: torch.Tensor | None = None):
    M, K = q.shape
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=q.device)
    bitlinear_forward_binary(q, tok_scale, packed1, beta, beta.numel(), M, N, K, out, acc_out)
    return out


def bitlinear(x: torch.Tensor, packed: torch.Tensor, gamma: torch.Tensor, N: int,
              gain: torch.Tensor | None = None, eps: float = 1e-5) -> torch.Tensor:
    """One BitLinear layer: RMSNorm + int8 quantisation, then the ternary matmul."""
    q, s = quant_act(x, gain, eps)
    return forward(q, s, packed, gamma, N)
