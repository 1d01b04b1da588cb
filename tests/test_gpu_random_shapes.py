"""Seeded random shapes through every engine route, against the oracle (needs
a B300).

Each case draws M, N, K (K a multiple of 16) and a route - the default
choice, the decode GEMV forced, the GEMM forced (whole tiles, planner split
or a forced split), the f16-activation GEMM, or the fused decode path with
or without its quantising pre-pass - packs fp32 weights on the GPU, quantises
bf16 activations on the GPU and compares packed bytes, int8 activations,
int32 accumulators and bf16 outputs with the oracle, bit for bit.  The
shapes are kept small enough for the oracle's int64 matmul (at most a few
hundred million multiply-adds a case).  Edge cases (N = 1, K = 16, N = 15,
M at chunk and tile boundaries) are listed explicitly beside them.
"""
import numpy as np
import pytest
import torch

import oracle
import bitlinear_02_b300 as bl
from bitlinear_02_b300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
S_TOK_RTOL = 1e-6
ROUTES = ("default", "gemv", "gemm_whole", "gemm_planned", "gemm_split", "f16", "fused", "fused_prepass")


def bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from bitlinear_02_b300 import build as blbuild
    blbuild.build()
    bl.load_library()
    oracle.build()
    torch.cuda.init()


@pytest.fixture(autouse=True)
def _defaults():
    yield
    bl.bitlinear_set_engine(-1, 0)
    bl.bitlinear_set_fused_prepass(-1)


def random_cases(n=28, seed=20261203):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        route = ROUTES[i % len(ROUTES)]
        if route.startswith("fused"):
            M = int(rng.integers(1, 17))
        elif route == "gemv":
            M = int(rng.integers(1, 65))
        else:
            M = int(rng.choice([rng.integers(1, 65), rng.integers(65, 301)]))
        N = int(rng.integers(1, 1200 if M <= 64 else 700))
        K = 16 * int(rng.integers(1, 161))
        split = int(rng.integers(2, 17))
        cases.append((route, M, N, K, split))
    return cases


EDGE = [("default", 1, 1, 16, 0), ("default", 5, 1, 16, 0), ("default", 300, 1, 16, 0), ("gemv", 64, 15, 32, 0),
        ("gemm_whole", 65, 17, 16, 0), ("gemm_split", 129, 1, 4096, 16), ("f16", 1, 1, 16, 0),
        ("fused", 16, 1, 16, 0), ("fused_prepass", 9, 33, 48, 0), ("default", 48, 2064, 16, 0),
        ("gemv", 33, 1, 65536, 0)]


def run_case(route, M, N, K, split, seed):
    w = inputs.weights_fp32(N, K, seed=seed)
    x = inputs.activations_bf16(M, K, seed=seed + 1, outlier_frac=0.01)
    wn = w.numpy()
    g_ref = oracle.gamma(wn)
    wq = oracle.ternarize(wn, g_ref, 1e-5)
    xb = inputs.bf16_bits(x)
    q_ref, s_ref = oracle.quant_act(xb, None, 1e-5)
    acc_ref = oracle.matmul(q_ref, wq)
    packed, gamma = bl.pack_weights(w.to(DEV), 1e-5)
    acc = torch.full((M, N), -7, dtype=torch.int32, device=DEV)
    if route.startswith("fused"):
        bl.bitlinear_set_fused_prepass(0 if route == "fused_prepass" else 1 << 40)
        xs = bl.new_stats(DEV)
        xd = x.to(DEV)
        bl.bitlinear_act_stats(xd, M, K, 1e-5, xs)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        bl.bitlinear_forward_fused(xd, xs, M, K, [bl.FusedProj(packed.data_ptr(), gamma.data_ptr(), N,
                                                              out.data_ptr(), acc.data_ptr(), None)])
        _, s = bl.fused_factors(xs, M, K)
    else:
        engine = {"default": (-1, 0), "gemv": (64, 0), "gemm_whole": (0, 1), "gemm_planned": (0, 0),
                  "gemm_split": (0, split), "f16": (-1, 0)}[route]
        bl.bitlinear_set_engine(*engine)
        if route == "f16":
            q16, s = bl.quant_act_f16(x.to(DEV))
            out = bl.forward_f16(q16, s, packed, gamma, N, acc_out=acc)
        else:
            q, s = bl.quant_act(x.to(DEV))
            out = bl.forward(q, s, packed, gamma, N, acc_out=acc)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    np.testing.assert_array_equal(packed.cpu().numpy(), oracle.pack(wq))
    s = s.cpu().numpy()
    np.testing.assert_allclose(s, s_ref, rtol=S_TOK_RTOL, atol=0)
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
    np.testing.assert_array_equal(bits16(out), oracle.epilogue(acc_ref, s, g_ref))


@pytest.mark.parametrize("i,case", list(enumerate(random_cases())), ids=lambda v: str(v))
def test_random_shape(i, case):
    run_case(*case, seed=4000 + 17 * i)


@pytest.mark.parametrize("case", EDGE, ids=lambda v: "-".join(map(str, v)))
def test_edge_shape(case):
    run_case(*case, seed=5000 + sum(case[1:4]))
