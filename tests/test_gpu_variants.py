"""The two variant formats on the GPU against the oracle (needs a B300).

Five ternary digits per byte: bitlinear_repack5 gives the oracle's bytes
(oracle.pack5 of the unpacked 2-bit matrix), and bitlinear_forward5 gives
the oracle's int32 accumulators and bf16 outputs bit for bit (the same as
bitlinear_forward on the 2-bit layout).

The original binary BitNet: bitlinear_pack_binary gives the oracle's sign
bits and group scales (bits of beta), bitlinear_forward_binary the oracle's
accumulators and grouped rescale bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import bitlinear_02_b300 as bl
from bitlinear_02_b300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


def bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from bitlinear_02_b300 import build as blbuild
    blbuild.build()
    bl.load_library()
    oracle.build()
    torch.cuda.init()


# ------------------------------------------------------ five per byte ---

@pytest.mark.parametrize("N,K", [(17, 336), (100, 1040), (48, 16), (2560, 2560), (6912, 2560), (2560, 6912)])
def test_repack5_bytes(N, K):
    wq = inputs.ternary(N, K, seed=N + K)
    packed = bl.pack_ternary(wq.to(DEV))
    p5 = bl.repack5(packed, N, K)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(p5.cpu().numpy(), oracle.pack5(wq.numpy()))


@pytest.mark.parametrize("M", [1, 3, 8, 9, 16, 17, 40, 64])
@pytest.mark.parametrize("N,K", [(300, 1040), (2560, 2560), (1000, 6912), (17, 160), (64, 16)])
def test_forward5_bit_exact(M, N, K):
    w = inputs.weights_fp32(N, K, seed=3 * N + K + M)
    x = inputs.activations_bf16(M, K, seed=5 * M + K, outlier_frac=0.01)
    g_ref = oracle.gamma(w.numpy())
    wq = oracle.ternarize(w.numpy(), g_ref, 1e-5)
    packed, gamma = bl.pack_weights(w.to(DEV), 1e-5)
    p5 = bl.repack5(packed, N, K)
    q, s = bl.quant_act(x.to(DEV))
    acc = torch.full((M, N), -7, dtype=torch.int32, device=DEV)
    out = bl.forward5(q, s, p5, gamma, N, acc_out=acc)
    acc2 = torch.empty(M, N, dtype=torch.int32, device=DEV)
    out2 = bl.forward(q, s, packed, gamma, N, acc_out=acc2)
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    acc_ref = oracle.matmul(q.cpu().numpy(), wq)
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
    np.testing.assert_array_equal(bits16(out), oracle.epilogue(acc_ref, s.cpu().numpy(), g_ref))
    # the same bits as the 2-bit engine
    assert torch.equal(acc, acc2) and torch.equal(out, out2)


@pytest.mark.parametrize("M", [1, 16])
def test_forward5_70b_down_projection_sampled(M):
    N, K = 8192, 28672
    wq = inputs.ternary_hash(N, K, inputs.stack_word(5, 0, 6), device=DEV)
    p5 = bl.repack5(bl.pack_ternary(wq), N, K)
    gam = torch.tensor([0.02], dtype=torch.float32, device=DEV)
    x = inputs.activations_bf16(M, K, seed=M, device=DEV)
    q, s = bl.quant_act(x)
    acc = torch.empty(M, N, dtype=torch.int32, device=DEV)
    bl.forward5(q, s, p5, gam, N, acc_out=acc)
    torch.cuda.synchronize()
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 24)]))
    w_rows = np.concatenate([oracle.ternary_hash(inputs.stack_word(5, 0, 6), K, int(n), int(n) + 1) for n in rows])
    want = oracle.matmul(q.cpu().numpy(), w_rows)
    np.testing.assert_array_equal(acc.cpu().numpy()[:, rows], want)


def test_forward5_rejects_prefill_batches():
    N, K = 64, 160
    p5 = bl.repack5(bl.pack_ternary(inputs.ternary(N, K, seed=1).to(DEV)), N, K)
    q = torch.zeros(65, K, dtype=torch.int8, device=DEV)
    s = torch.ones(65, dtype=torch.float32, device=DEV)
    with pytest.raises(bl.BitLinearError):
        bl.forward5(q, s, p5, torch.ones(1, device=DEV), N)


# ------------------------------------------------------- binary BitNet ---

@pytest.mark.parametrize("N,K,G", [(17, 272, 1), (64, 1040, 4), (2560, 2560, 1), (2560, 2560, 8), (6912, 2560, 4)])
def test_pack_binary_bytes_and_group_scales(N, K, G):
    if N % G:
        pytest.skip("groups must divide N")
    w = inputs.weights_fp32(N, K, seed=N * 3 + K)
    p1, beta = bl.pack_binary(w.to(DEV), G)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(p1.cpu().numpy(), oracle.pack1(oracle.binarize(w.numpy())))
    np.testing.assert_array_equal(beta.cpu().numpy().view(np.uint32), oracle.beta(w.numpy(), G).view(np.uint32))


def test_pack_binary_special_values():
    N, K = 16, 32
    w = torch.zeros(N, K, dtype=torch.float32)
    w[0, :6] = torch.tensor([0.0, -0.0, 1e-45, -1e-45, 3e38, -3e38])
    w[1] = 1.0
    w[2] = -1.0
    p1, beta = bl.pack_binary(w.to(DEV), 2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(p1.cpu().numpy(), oracle.pack1(oracle.binarize(w.numpy())))
    np.testing.assert_array_equal(beta.cpu().numpy().view(np.uint32), oracle.beta(w.numpy(), 2).view(np.uint32))


@pytest.mark.parametrize("M", [1, 4, 9, 16, 33, 64])
@pytest.mark.parametrize("N,K,G", [(300, 1040, 3), (2560, 2560, 1), (1024, 6912, 8), (16, 16, 1)])
def test_forward_binary_bit_exact(M, N, K, G):
    w = inputs.weights_fp32(N, K, seed=7 * N + K + M)
    x = inputs.activations_bf16(M, K, seed=11 * M + K, outlier_frac=0.01)
    wb = oracle.binarize(w.numpy())
    beta_ref = oracle.beta(w.numpy(), G)
    p1, beta = bl.pack_binary(w.to(DEV), G)
    q, s = bl.quant_act(x.to(DEV))
    acc = torch.full((M, N), -7, dtype=torch.int32, device=DEV)
    out = bl.forward_binary(q, s, p1, beta, N, acc_out=acc)
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    acc_ref = oracle.matmul(q.cpu().numpy(), wb)
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
    np.testing.assert_array_equal(bits16(out), oracle.epilogue_groups(acc_ref, s.cpu().numpy(), beta_ref))
