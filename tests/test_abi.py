"""The C ABI library builds, loads and exports every declared symbol; argument
validation works without a GPU (it runs before any CUDA call)."""
import ctypes
import os
import re

import pytest

import bitlinear_02_b300 as bl
from bitlinear_02_b300 import build as blbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bitlinear.h")


@pytest.fixture(scope="module")
def lib():
    blbuild.build()
    return bl.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bitlinear_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("bitlinear_pack_weights", "bitlinear_pack_ternary", "bitlinear_quant_act",
                 "bitlinear_forward", "bitlinear_packed_bytes", "bitlinear_status_string",
                 "bitlinear_check_status"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def exported_abi(path):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    return {s for s in exported if s.startswith("bitlinear_")}


def test_only_abi_symbols_are_exported(lib):
    # the build hides everything that is not declared extern "C" in the header
    assert exported_abi(bl.library_path()) == set(declared_functions())


def test_debug_build_exports_the_same_boundary(lib):
    """The -DBITLINEAR_DEBUG build (device-side bounds checks) has the same
    ABI; in the release build the self-test reports that it has no checks."""
    path = blbuild.build(debug=True)
    assert os.path.basename(path) == "libbitlinear_debug.so"
    assert exported_abi(path) == set(declared_functions())
    assert lib.bitlinear_debug_selftest(None) == bl.ERR_UNSUPPORTED  # release: nothing enqueued
    assert lib.bitlinear_status_string(bl.ERR_BOUNDS) == b"a device bounds check failed (debug build)"


def test_packed_bytes(lib):
    assert bl.bitlinear_packed_bytes(512, 256) == 512 * 256 // 4
    assert bl.bitlinear_packed_bytes(17, 144) == 32 * 256 // 4
    assert bl.bitlinear_packed_bytes(0, 16) == 0
    assert bl.bitlinear_packed_bytes(16, 0) == 0


def test_status_strings(lib):
    assert bl.bitlinear_status_string(0) == "ok"
    assert "invalid" in bl.bitlinear_status_string(1)
    assert "bounded wait" in bl.bitlinear_status_string(4)
    assert bl.bitlinear_status_string(99) == "unknown status"
    assert bl.bitlinear_version() == 101


FAKE = 1 << 20  # an aligned non-null address: never dereferenced, checks fail first


def test_forward_rejects_bad_arguments(lib):
    L = lib
    P = ctypes.c_void_p
    ok = dict(q=P(FAKE), s=P(FAKE), p=P(FAKE), g=P(FAKE), o=P(FAKE))

    def call(M=4, N=32, K=64, **kw):
        a = dict(ok, **kw)
        return L.bitlinear_forward(a["q"], a["s"], a["p"], a["g"], M, N, K, a["o"], None, None)

    assert call(K=10) == bl.ERR_INVALID_ARG       # K not a multiple of 16
    assert call(K=0) == bl.ERR_INVALID_ARG
    assert call(K=65536 + 16) == bl.ERR_INVALID_ARG
    assert call(N=0) == bl.ERR_INVALID_ARG
    assert call(M=-1) == bl.ERR_INVALID_ARG
    assert call(q=None) == bl.ERR_INVALID_ARG
    assert call(o=P(FAKE + 2)) == bl.ERR_INVALID_ARG  # misaligned output
    assert call(g=P(FAKE + 2)) == bl.ERR_INVALID_ARG  # misaligned gamma
    assert call(M=0) == bl.OK                         # empty batch: nothing to do


def test_quant_and_pack_reject_bad_arguments(lib):
    L = lib
    P = ctypes.c_void_p
    assert L.bitlinear_quant_act(P(FAKE), None, 3, 24, 1e-5, P(FAKE), P(FAKE), None) == bl.ERR_INVALID_ARG
    assert L.bitlinear_quant_act(None, None, 3, 32, 1e-5, P(FAKE), P(FAKE), None) == bl.ERR_INVALID_ARG
    assert L.bitlinear_quant_act(P(FAKE + 8), None, 3, 32, 1e-5, P(FAKE), P(FAKE), None) == bl.ERR_INVALID_ARG
    assert L.bitlinear_quant_act(P(FAKE), None, 0, 32, 1e-5, P(FAKE), P(FAKE), None) == bl.OK
    assert L.bitlinear_pack_weights(P(FAKE), 0, 32, 1e-5, P(FAKE), P(FAKE), None) == bl.ERR_INVALID_ARG
    assert L.bitlinear_pack_weights(P(FAKE), 4, 33, 1e-5, P(FAKE), P(FAKE), None) == bl.ERR_INVALID_ARG
    assert L.bitlinear_pack_weights(None, 4, 32, 1e-5, P(FAKE), P(FAKE), None) == bl.ERR_INVALID_ARG
    assert L.bitlinear_pack_ternary(P(FAKE), 4, 32, P(FAKE + 4), None) == bl.ERR_INVALID_ARG


def test_fused_entry_points_reject_bad_arguments(lib):
    L = lib
    P = ctypes.c_void_p
    assert L.bitlinear_fused_stats_bytes() == 2304
    assert "pending factor buffer" in bl.bitlinear_status_string(bl.ERR_STATE)
    # bitlinear_act_stats(x, M, K, eps, stats, stream)
    assert L.bitlinear_act_stats(P(FAKE), 0, 64, 1e-5, P(FAKE), None) == bl.ERR_INVALID_ARG
    assert L.bitlinear_act_stats(P(FAKE), 17, 64, 1e-5, P(FAKE), None) == bl.ERR_INVALID_ARG
    assert L.bitlinear_act_stats(P(FAKE), 4, 72 + 4, 1e-5, P(FAKE), None) == bl.ERR_INVALID_ARG
    assert L.bitlinear_act_stats(None, 4, 64, 1e-5, P(FAKE), None) == bl.ERR_INVALID_ARG
    assert L.bitlinear_act_stats(P(FAKE), 4, 64, 1e-5, P(FAKE + 4), None) == bl.ERR_INVALID_ARG
    # bitlinear_fused_factors(stats, M, K, eps, consume, c_out, ts_out, stream)
    assert L.bitlinear_fused_factors(P(FAKE), 0, 64, 1e-5, 0, None, None, None) == bl.ERR_INVALID_ARG
    assert L.bitlinear_fused_factors(P(FAKE), 17, 64, 1e-5, 0, None, None, None) == bl.ERR_INVALID_ARG
    assert L.bitlinear_fused_factors(None, 4, 64, 1e-5, 0, None, None, None) == bl.ERR_INVALID_ARG
    assert L.bitlinear_fused_factors(P(FAKE), 4, 64, 1e-5, 0, P(FAKE + 2), None, None) == bl.ERR_INVALID_ARG

    # bitlinear_forward_fused(x, x_stats, M, K, nproj, projs, eps, stream)
    def proj(N=64, packed=FAKE, gamma=FAKE, out=FAKE, acc=None, stats=None):
        return bl.FusedProj(packed, gamma, N, out, acc, stats)

    def call(projs, M=4, K=256, x=FAKE, xs=FAKE + 4096):
        arr = (bl.FusedProj * max(1, len(projs)))(*projs)
        return L.bitlinear_forward_fused(P(x) if x else None, P(xs) if xs else None, M, K, len(projs), arr,
                                         1e-5, None)

    good = proj(stats=FAKE + 8192)
    assert call([good], M=0) == bl.ERR_INVALID_ARG
    assert call([good], M=17) == bl.ERR_INVALID_ARG
    assert call([good], K=250) == bl.ERR_INVALID_ARG
    assert call([good], x=0) == bl.ERR_INVALID_ARG
    assert call([good], xs=FAKE + 8) == bl.ERR_INVALID_ARG                  # misaligned factor buffer
    assert call([]) == bl.ERR_INVALID_ARG                                   # no projection
    assert call([good] * 5) == bl.ERR_INVALID_ARG                           # more than four
    assert call([proj(N=0)]) == bl.ERR_INVALID_ARG
    assert call([proj(packed=0)]) == bl.ERR_INVALID_ARG
    assert call([proj(out=FAKE + 2)]) == bl.ERR_INVALID_ARG                 # misaligned output
    assert call([proj(stats=FAKE + 4096)]) == bl.ERR_INVALID_ARG            # output factors = input factors
    assert call([good, good]) == bl.ERR_INVALID_ARG                         # two outputs, one factor buffer


def test_python_binding_raises_on_error(lib):
    with pytest.raises(bl.BitLinearError) as ei:
        bl._check(bl.ERR_INVALID_ARG, "bitlinear_forward")
    assert ei.value.status == bl.ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import importlib
    monkeypatch.setattr(bl, "_lib", None)
    monkeypatch.setattr(bl, "_HERE", str(tmp_path))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        bl.load_library()


def test_set_engine_validates_without_a_gpu(lib):
    assert lib.bitlinear_set_engine(65, 0) == bl.ERR_INVALID_ARG   # the GEMV takes at most 64 tokens
    assert lib.bitlinear_set_engine(-2, 0) == bl.ERR_INVALID_ARG
    assert lib.bitlinear_set_engine(0, 17) == bl.ERR_INVALID_ARG   # clusters of at most 16 CTAs
    assert lib.bitlinear_set_engine(0, -1) == bl.ERR_INVALID_ARG
    assert lib.bitlinear_set_engine(0, 16) == bl.OK
    assert lib.bitlinear_set_engine(-1, 0) == bl.OK                # the defaults again


def test_set_fused_prepass_validates_without_a_gpu(lib):
    assert lib.bitlinear_set_fused_prepass(-2) == bl.ERR_INVALID_ARG
    for v in (0, 1, 1 << 40, -1):                                  # -1 last: the default again
        assert lib.bitlinear_set_fused_prepass(v) == bl.OK


def test_variant_sizes_and_argument_checks(lib):
    assert bl.bitlinear_packed5_bytes(16, 160) == 512
    assert bl.bitlinear_packed5_bytes(17, 336) == 32 * 480 // 5
    assert bl.bitlinear_packed5_bytes(0, 16) == 0
    assert bl.bitlinear_packed1_bytes(16, 256) == 512
    assert bl.bitlinear_packed1_bytes(17, 272) == 32 * 512 // 8
    P = ctypes.c_void_p
    f = P(FAKE)
    assert lib.bitlinear_repack5(f, 16, 10, f, None) == bl.ERR_INVALID_ARG          # K % 16
    assert lib.bitlinear_repack5(None, 16, 16, f, None) == bl.ERR_INVALID_ARG
    assert lib.bitlinear_forward5(f, f, f, f, 65, 32, 64, f, None, None) == bl.ERR_UNSUPPORTED  # decode only
    assert lib.bitlinear_forward5(f, f, f, f, 4, 32, 60, f, None, None) == bl.ERR_INVALID_ARG
    assert lib.bitlinear_forward5(f, f, f, f, 0, 32, 64, f, None, None) == bl.OK     # empty batch
    assert lib.bitlinear_pack_binary(f, 32, 64, 0, f, f, None) == bl.ERR_INVALID_ARG  # no groups
    assert lib.bitlinear_pack_binary(f, 30, 64, 4, f, f, None) == bl.ERR_INVALID_ARG  # N % G
    assert lib.bitlinear_forward_binary(f, f, f, f, 3, 4, 32, 64, f, None, None) == bl.ERR_INVALID_ARG
    assert lib.bitlinear_forward_binary(f, f, f, f, 2, 65, 32, 64, f, None, None) == bl.ERR_UNSUPPORTED
