"""Guard bytes around every output (needs a B300): each engine route writes
exactly its M x N outputs and nothing around them.

Outputs are views into larger buffers filled with a canary pattern; after
the call the canary regions before and after the view must be intact, and
the view itself fully written.  Ragged shapes put partial row groups, row
tiles and token tiles at the edges, where the tensor-map stores (which clip
at the tensor's extent) and the split-K reductions write last.
"""
import numpy as np
import pytest
import torch

import bitlinear_02_b300 as bl
from bitlinear_02_b300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
PAD = 4096  # elements of canary on each side (a multiple of 8: the view stays 16-byte aligned)
C16 = 0x7FC1  # a bf16 NaN: no output takes it (outputs are finite)
C32 = 0x5A5A5A5A


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from bitlinear_02_b300 import build as blbuild
    blbuild.build()
    bl.load_library()
    torch.cuda.init()


@pytest.fixture(autouse=True)
def _default_engine():
    yield
    bl.bitlinear_set_engine(-1, 0)


def guarded(M, N):
    ob = torch.full((PAD + M * N + PAD,), C16, dtype=torch.int16, device=DEV)
    ab = torch.full((PAD + M * N + PAD,), C32, dtype=torch.int32, device=DEV)
    out = ob[PAD:PAD + M * N].view(torch.bfloat16).view(M, N)
    acc = ab[PAD:PAD + M * N].view(M, N)
    return ob, ab, out, acc


def check(ob, ab, M, N, with_acc=True):
    o = ob.cpu().numpy().view(np.uint16)
    a = ab.cpu().numpy().view(np.uint32)
    assert (o[:PAD] == C16).all() and (o[PAD + M * N:] == C16).all(), "bf16 output guard overwritten"
    assert (o[PAD:PAD + M * N] != C16).all(), "bf16 output not fully written"
    if with_acc:
        assert (a[:PAD] == C32).all() and (a[PAD + M * N:] == C32).all(), "int32 output guard overwritten"
        assert (a[PAD:PAD + M * N] != C32).all(), "int32 output not fully written"


# (route, gemv_max_tokens, split_k, M, N, K)
ROUTES = [
    ("gemv", -1, 0, 5, 300, 1040),
    ("gemv_chunks", -1, 0, 40, 1000, 6912),
    ("gemm_whole_tiles", 0, 1, 100, 300, 1040),
    ("gemm_split", 0, 0, 100, 1000, 6912),
    ("gemm_split_16", 0, 16, 65, 136, 8192),
    ("gemm_widened", -1, 0, 300, 4104, 4096),
    ("gemm_big_tiles", -1, 0, 700, 2568, 1040),
]


@pytest.mark.parametrize("route,gmax,split,M,N,K", ROUTES, ids=[r[0] for r in ROUTES])
def test_forward_writes_only_its_outputs(route, gmax, split, M, N, K):
    bl.bitlinear_set_engine(gmax, split)
    packed = bl.pack_ternary(inputs.ternary(N, K, seed=N + K, device=DEV))
    gam = torch.tensor([0.02], dtype=torch.float32, device=DEV)
    x = inputs.activations_bf16(M, K, seed=M, device=DEV)
    q, s = bl.quant_act(x)
    ob, ab, out, acc = guarded(M, N)
    bl.forward(q, s, packed, gam, N, out=out, acc_out=acc)
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    check(ob, ab, M, N)
    # without the int32 copy (the staged and persistent epilogues)
    ob2, _, out2, _ = guarded(M, N)
    bl.forward(q, s, packed, gam, N, out=out2)
    torch.cuda.synchronize()
    check(ob2, ab, M, N, with_acc=False)
    assert torch.equal(out2, out)


@pytest.mark.parametrize("M,N,K", [(1900, 2568, 1040), (600, 6400, 256), (17, 300, 1040), (300, 4104, 512)])
def test_forward_f16_writes_only_its_outputs(M, N, K):
    """The f16 entry point, including the persistent kernel (the first two
    shapes) and the split-K kernel (the third)."""
    packed = bl.pack_ternary(inputs.ternary(N, K, seed=N * K, device=DEV))
    gam = torch.tensor([0.02], dtype=torch.float32, device=DEV)
    x = inputs.activations_bf16(M, K, seed=M + 1, device=DEV)
    q16, s16 = bl.quant_act_f16(x)
    ob, ab, out, acc = guarded(M, N)
    bl.forward_f16(q16, s16, packed, gam, N, out=out)
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    check(ob, ab, M, N, with_acc=False)


@pytest.mark.parametrize("M,N,K", [(1, 300, 1040), (16, 1000, 6912), (37, 136, 320)])
def test_variant_formats_write_only_their_outputs(M, N, K):
    w = inputs.weights_fp32(N, K, seed=M + N, device=DEV)
    packed, gamma = bl.pack_weights(w, 1e-5)
    p5 = bl.repack5(packed, N, K)
    p1, beta = bl.pack_binary(w, 4 if N % 4 == 0 else 1)
    x = inputs.activations_bf16(M, K, seed=M, device=DEV)
    q, s = bl.quant_act(x)
    for fn in (lambda o, a: bl.forward5(q, s, p5, gamma, N, out=o, acc_out=a),
               lambda o, a: bl.forward_binary(q, s, p1, beta, N, out=o, acc_out=a)):
        ob, ab, out, acc = guarded(M, N)
        fn(out, acc)
        torch.cuda.synchronize()
        assert bl.bitlinear_check_status() == bl.OK
        check(ob, ab, M, N)


def test_packers_write_only_their_bytes():
    """The 2-bit, five-digit and binary packers write exactly their buffers."""
    N, K = 300, 1040
    w = inputs.weights_fp32(N, K, seed=9, device=DEV)
    for nbytes, run in (
            (bl.bitlinear_packed_bytes(N, K),
             lambda p: bl.bitlinear_pack_weights(w, N, K, 1e-5, p, torch.empty(1, device=DEV))),
            (bl.bitlinear_packed1_bytes(N, K),
             lambda p: bl.bitlinear_pack_binary(w, N, K, 3, p, torch.empty(3, device=DEV)))):
        buf = torch.full((256 + nbytes + 256,), 0xA5, dtype=torch.uint8, device=DEV)
        run(buf[256:256 + nbytes])
        torch.cuda.synchronize()
        b = buf.cpu().numpy()
        assert (b[:256] == 0xA5).all() and (b[256 + nbytes:] == 0xA5).all()
    packed, _ = bl.pack_weights(w, 1e-5)
    n5 = bl.bitlinear_packed5_bytes(N, K)
    buf = torch.full((256 + n5 + 256,), 0xA5, dtype=torch.uint8, device=DEV)
    bl.bitlinear_repack5(packed, N, K, buf[256:256 + n5])
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert (b[:256] == 0xA5).all() and (b[256 + n5:] == 0xA5).all()
