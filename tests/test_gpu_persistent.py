"""The persistent tcgen05 GEMM (token tile 192, more tiles than SMs, K <=
4096, no int32 copy asked) against the oracle (needs a B300).

The shapes take the persistent kernel (token tile 192 in the one-tile plan
too) and leave ragged row groups, row tiles and token tiles.  The persistent kernel writes bf16
only, so the accumulators are checked through the outputs: with activations
in {-1, 0, +1}, all scales 1 and K = 256, every accumulator is an integer of
magnitude <= 256, which bf16 holds exactly.  A second test runs realistic
activations (f16 entry point and the int8 one, which widens first) and
compares the bf16 outputs bit for bit with the oracle's epilogue.
"""
import numpy as np
import pytest
import torch

import oracle
import bitlinear_02_b300 as bl
from bitlinear_02_b300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
# (N, M), all with 192-token tiles and more tiles than 148 SMs
SHAPES = [(6400, 600), (2568, 1900), (4104, 2050), (2560, 4096)]


def bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from bitlinear_02_b300 import build as blbuild
    blbuild.build()
    bl.load_library()
    oracle.build()
    torch.cuda.init()


@pytest.mark.parametrize("N,M", SHAPES)
def test_persistent_accumulators_exact(N, M):
    K = 256
    wq = inputs.ternary(N, K, seed=N + M)
    g = torch.Generator().manual_seed(M)
    q = torch.randint(-1, 2, (M, K), generator=g, dtype=torch.int8)
    packed = bl.pack_ternary(wq.to(DEV))
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    s = torch.ones(M, dtype=torch.float32, device=DEV)
    out = bl.forward_f16(q.to(DEV).to(torch.float16), s, packed, one, N)
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    acc_ref = oracle.matmul(q.numpy(), wq.numpy())
    assert np.abs(acc_ref).max() <= 256
    np.testing.assert_array_equal(out.float().cpu().numpy().astype(np.int64), acc_ref)


@pytest.mark.parametrize("N,M", SHAPES)
@pytest.mark.parametrize("K", [1040])
def test_persistent_outputs_bit_exact(N, M, K):
    w = inputs.weights_fp32(N, K, seed=3 * N + M)
    x = inputs.activations_bf16(M, K, seed=5 * M + N, outlier_frac=0.01)
    wn = w.numpy()
    g_ref = oracle.gamma(wn)
    wq = oracle.ternarize(wn, g_ref, 1e-5)
    q_ref, s_ref = oracle.quant_act(inputs.bf16_bits(x), None, 1e-5)
    acc_ref = oracle.matmul(q_ref, wq)
    packed, gamma = bl.pack_weights(w.to(DEV), 1e-5)
    q16, s16 = bl.quant_act_f16(x.to(DEV))
    out16 = bl.forward_f16(q16, s16, packed, gamma, N)
    q8, s8 = bl.quant_act(x.to(DEV))
    out8 = bl.forward(q8, s8, packed, gamma, N)
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    np.testing.assert_array_equal(bits16(out16), oracle.epilogue(acc_ref, s16.cpu().numpy(), g_ref))
    np.testing.assert_array_equal(bits16(out8), oracle.epilogue(acc_ref, s8.cpu().numpy(), g_ref))
