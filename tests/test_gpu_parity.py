"""Parity of the CUDA path with the CPU oracle (needs a B300).

Bit-exact: gamma bits, packed bytes, int8 activations, int32 accumulators,
and the bf16 output when the oracle's epilogue is fed the GPU's token
scales.  The token scale itself is a float reduction and is held to 1e-6
relative (in practice almost all are bit-identical).  Inputs are seeded and
synthetic, drawn from bitlinear_02_b300.inputs (shared by both sides).
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


def bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from bitlinear_02_b300 import build as blbuild
    blbuild.build()
    bl.load_library()
    oracle.build()
    torch.cuda.init()


def gpu_pack(w_cpu, eps=1e-5):
    packed, gamma = bl.pack_weights(w_cpu.to(DEV), eps)
    return packed, gamma


def check_quant(x_cpu, gain_cpu=None, eps=1e-5):
    xb = inputs.bf16_bits(x_cpu)
    gb = None if gain_cpu is None else inputs.bf16_bits(gain_cpu)
    q_ref, s_ref = oracle.quant_act(xb, gb, eps)
    q, s = bl.quant_act(x_cpu.to(DEV), None if gain_cpu is None else gain_cpu.to(DEV), eps)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    s_np = s.cpu().numpy()
    np.testing.assert_allclose(s_np, s_ref, rtol=S_TOK_RTOL, atol=0)
    return q, s, q_ref, s_ref


def run_chain(w_cpu, x_cpu, eps_w=1e-5, eps_a=1e-5, gain_cpu=None):
    """Full path on the GPU, returned as numpy (gamma, packed, q, s, acc, out)."""
    packed, gamma = gpu_pack(w_cpu, eps_w)
    q, s = bl.quant_act(x_cpu.to(DEV), None if gain_cpu is None else gain_cpu.to(DEV), eps_a)
    M, K = x_cpu.shape
    N = w_cpu.shape[0]
    acc = torch.empty(M, N, dtype=torch.int32, device=DEV)
    out = bl.forward(q, s, packed, gamma, N, acc_out=acc)
    torch.cuda.synchronize()
    return (np.float32(gamma.item()), packed.cpu().numpy(), q.cpu().numpy(), s.cpu().numpy(),
            acc.cpu().numpy(), bits16(out))


def check_full(w_cpu, x_cpu, eps_w=1e-5, eps_a=1e-5, gain_cpu=None):
    w = w_cpu.numpy()
    xb = inputs.bf16_bits(x_cpu)
    gb = None if gain_cpu is None else inputs.bf16_bits(gain_cpu)
    g_ref = oracle.gamma(w)
    wq = oracle.ternarize(w, g_ref, eps_w)
    p_ref = oracle.pack(wq)
    q_ref, s_ref = oracle.quant_act(xb, gb, eps_a)
    acc_ref = oracle.matmul(q_ref, wq)
    g, p, q, s, acc, out = run_chain(w_cpu, x_cpu, eps_w, eps_a, gain_cpu)
    assert g.view(np.uint32) == np.float32(g_ref).view(np.uint32)
    np.testing.assert_array_equal(p, p_ref)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_allclose(s, s_ref, rtol=S_TOK_RTOL, atol=0)
    np.testing.assert_array_equal(acc, acc_ref)
    np.testing.assert_array_equal(out, oracle.epilogue(acc_ref, s, g_ref))
    # with the oracle's own token scales the bf16 output stays within 1e-3
    # relative wherever the scales agree bit for bit
    same = s.view(np.uint32) == s_ref.view(np.uint32)
    ref_own = oracle.epilogue(acc_ref, s_ref, g_ref)
    np.testing.assert_array_equal(out[same], ref_own[same])
    return same.mean()


# ------------------------------------------------------------------ pack ---

@pytest.mark.parametrize("N,K", [(512, 256), (17, 144), (200, 8640), (2560, 2560), (6912, 2560),
                                 (2560, 6912), (16, 16), (1, 32)])
def test_pack_weights_bit_exact(N, K):
    w = inputs.weights_fp32(N, K, seed=N * 7 + K)
    g_ref = oracle.gamma(w.numpy())
    p_ref = oracle.pack(oracle.ternarize(w.numpy(), g_ref, 1e-5))
    packed, gamma = gpu_pack(w)
    torch.cuda.synchronize()
    assert np.float32(gamma.item()).view(np.uint32) == np.float32(g_ref).view(np.uint32)
    np.testing.assert_array_equal(packed.cpu().numpy(), p_ref)


def test_pack_weights_special_values():
    # wide dynamic range incl. subnormals; ties exactly at 1/2; constant rows
    rng = np.random.default_rng(1)
    N, K = 64, 256
    w = (rng.standard_normal((N, K)) * np.exp2(rng.integers(-140, 40, (N, K)))).astype(np.float32)
    w[3, :] = 0.0
    w[5, :] = 7.25
    for eps in (1e-5, 0.0):
        g_ref = oracle.gamma(w)
        p_ref = oracle.pack(oracle.ternarize(w, g_ref, eps))
        packed, gamma = gpu_pack(torch.from_numpy(w), eps)
        torch.cuda.synchronize()
        assert np.float32(gamma.item()).view(np.uint32) == np.float32(g_ref).view(np.uint32)
        np.testing.assert_array_equal(packed.cpu().numpy(), p_ref)
    # a matrix with gamma a power of two and entries at +-gamma/2: exact ties
    w2 = np.tile(np.array([0.5, -0.5, 1.5, -1.5, 0.25, -2.0, 1.0, 0.0], np.float32) * 0.125, (16, 4))
    g_ref = oracle.gamma(w2)
    p_ref = oracle.pack(oracle.ternarize(w2, g_ref, 0.0))
    packed, gamma = gpu_pack(torch.from_numpy(w2), 0.0)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(packed.cpu().numpy(), p_ref)


@pytest.mark.parametrize("N,K", [(512, 256), (33, 144), (3200, 8640)])
def test_pack_ternary_bit_exact(N, K):
    wq = inputs.ternary(N, K, seed=N + K)
    p_ref = oracle.pack(wq.numpy())
    packed = bl.pack_ternary(wq.to(DEV))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(packed.cpu().numpy(), p_ref)


# ----------------------------------------------------------------- quant ---

@pytest.mark.parametrize("M,K", [(1, 256), (3, 144), (16, 2560), (17, 6912), (300, 2560),
                                 (65, 8640), (4, 28672), (1, 16)])
def test_quant_act(M, K):
    x = inputs.activations_bf16(M, K, seed=M * 31 + K, outlier_frac=0.01)
    check_quant(x)


def test_quant_act_gain_zero_token_and_integers():
    M, K = 9, 512
    x = inputs.activations_bf16(M, K, seed=77)
    x[2] = 0
    x[4] = torch.arange(K, dtype=torch.float32).remainder(255).sub(127).to(torch.bfloat16)
    g = inputs.gain_bf16(K, seed=78)
    check_quant(x, g)
    q, s, _, _ = check_quant(x)
    assert (q[2] == 0).all()


# ------------------------------------------------------------ full chain ---

@pytest.mark.parametrize("M", [1, 2, 7, 8, 9, 15, 16])
@pytest.mark.parametrize("N,K", [(512, 256), (200, 8640), (17, 144), (1024, 1152)])
def test_decode_gemv_parity(M, N, K):
    w = inputs.weights_fp32(N, K, seed=3 * N + K)
    x = inputs.activations_bf16(M, K, seed=5 * M + K)
    check_full(w, x)


@pytest.mark.parametrize("M", [17, 18, 33, 48, 63, 64])
@pytest.mark.parametrize("N,K", [(512, 256), (200, 8640), (2560, 2560)])
def test_chunked_gemv_parity(M, N, K):
    # 16 < M <= 64: the decode GEMV in 16-token chunks (a partial last chunk included)
    w = inputs.weights_fp32(N, K, seed=17 * N + K)
    x = inputs.activations_bf16(M, K, seed=19 * M + K)
    check_full(w, x)


@pytest.mark.parametrize("M", [65, 80, 128, 129, 200, 256, 300])
@pytest.mark.parametrize("N,K", [(512, 256), (200, 8640), (144, 144), (1040, 1280)])
def test_prefill_gemm_parity(M, N, K):
    # bitlinear_forward above 64 tokens: the tcgen05 GEMM with int8 activations
    w = inputs.weights_fp32(N, K, seed=11 * N + K)
    x = inputs.activations_bf16(M, K, seed=13 * M + K, outlier_frac=0.01)
    check_full(w, x)


@pytest.mark.parametrize("M", [1, 17, 64, 65, 200, 300])
@pytest.mark.parametrize("N,K", [(512, 256), (200, 8640), (144, 144), (1040, 1280)])
def test_prefill_f16_path_parity(M, N, K):
    """quant_act_f16 + forward_f16: the same q values, bit-exact accumulators
    and outputs as the oracle (and the int8 path)."""
    w = inputs.weights_fp32(N, K, seed=17 * N + K)
    x = inputs.activations_bf16(M, K, seed=19 * M + K, outlier_frac=0.01)
    wn = w.numpy()
    g_ref = oracle.gamma(wn)
    wq = oracle.ternarize(wn, g_ref, 1e-5)
    q_ref, s_ref = oracle.quant_act(inputs.bf16_bits(x), None, 1e-5)
    packed, gamma = gpu_pack(w)
    q16, s = bl.quant_act_f16(x.to(DEV))
    acc = torch.empty(M, N, dtype=torch.int32, device=DEV)
    out = bl.forward_f16(q16, s, packed, gamma, N, acc_out=acc)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q16.cpu().to(torch.int32).numpy(), q_ref.astype(np.int32))
    np.testing.assert_allclose(s.cpu().numpy(), s_ref, rtol=S_TOK_RTOL, atol=0)
    acc_ref = oracle.matmul(q_ref, wq)
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
    np.testing.assert_array_equal(bits16(out), oracle.epilogue(acc_ref, s.cpu().numpy(), g_ref))


def test_prefill_f16_2b_full_size_sampled():
    M = 4096
    wl = inputs.WORKLOADS["prefill_2b"]
    for i, (name, N, K) in enumerate(wl["shapes"]):
        if name not in ("gate", "down"):
            continue
        w = inputs.weights_fp32(N, K, seed=wl["seed"] * 100 + i)
        x = inputs.activations_bf16(M, K, seed=wl["seed"] * 1000 + M + i, outlier_frac=0.01,
                                    outlier_scale=20.0)
        wn = w.numpy()
        g_ref = oracle.gamma(wn)
        wq = oracle.ternarize(wn, g_ref, 1e-5)
        packed, gamma = gpu_pack(w)
        q16, s = bl.quant_act_f16(x.to(DEV))
        acc = torch.empty(M, N, dtype=torch.int32, device=DEV)
        out = bl.forward_f16(q16, s, packed, gamma, N, acc_out=acc)
        torch.cuda.synchronize()
        q_ref, _ = oracle.quant_act(inputs.bf16_bits(x), None, 1e-5)
        np.testing.assert_array_equal(q16.cpu().to(torch.int32).numpy(), q_ref.astype(np.int32))
        rng = np.random.default_rng(i)
        ms = rng.integers(0, M, 4096)
        ns = rng.integers(0, N, 4096)
        accn = acc.cpu().numpy()
        np.testing.assert_array_equal(accn[ms, ns], oracle.matmul_pairs(q_ref, wq, ms, ns))
        np.testing.assert_array_equal(bits16(out), oracle.epilogue(accn, s.cpu().numpy(), g_ref))


def test_layer_small_workload():
    wl = inputs.WORKLOADS["layer_small"]
    _, N, K = wl["shapes"][0]
    w = inputs.weights_fp32(N, K, seed=wl["seed"])
    x = inputs.activations_bf16(1, K, seed=wl["seed"] + 1)
    check_full(w, x, wl["eps_w"], wl["eps_a"])


@pytest.mark.parametrize("M", [1, 4, 16])
def test_decode_2b_full_shapes(M):
    wl = inputs.WORKLOADS["decode_2b"]
    for i, (name, N, K) in enumerate(wl["shapes"]):
        if name in ("k", "v"):
            continue  # same shape as q
        w = inputs.weights_fp32(N, K, seed=wl["seed"] * 100 + i)
        x = inputs.activations_bf16(M, K, seed=wl["seed"] * 1000 + 10 * M + i)
        check_full(w, x)


def sampled_check(w_cpu, x_cpu, n_samples=4096, seed=0):
    """Full-size shapes: bit-exact packed bytes and quantised activations,
    and the exact accumulator on a random sample of (m, n) outputs."""
    w = w_cpu.numpy()
    g_ref = oracle.gamma(w)
    wq = oracle.ternarize(w, g_ref, 1e-5)
    g, p, q, s, acc, out = run_chain(w_cpu, x_cpu)
    assert g.view(np.uint32) == np.float32(g_ref).view(np.uint32)
    np.testing.assert_array_equal(p, oracle.pack(wq))
    q_ref, s_ref = oracle.quant_act(inputs.bf16_bits(x_cpu), None, 1e-5)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_allclose(s, s_ref, rtol=S_TOK_RTOL, atol=0)
    M, N = acc.shape
    rng = np.random.default_rng(seed)
    ms = rng.integers(0, M, n_samples)
    ns = rng.integers(0, N, n_samples)
    ms[:4] = [0, M - 1, 0, M - 1]
    ns[:4] = [0, N - 1, N - 1, 0]
    want = oracle.matmul_pairs(q_ref, wq, ms, ns)
    np.testing.assert_array_equal(acc[ms, ns], want)
    ep = oracle.epilogue(acc, s, g_ref)
    np.testing.assert_array_equal(out, ep)


@pytest.mark.parametrize("M", [512, 4096])
def test_prefill_2b_full_size_sampled(M):
    wl = inputs.WORKLOADS["prefill_2b"]
    for i, (name, N, K) in enumerate(wl["shapes"]):
        if name in ("k", "v", "o", "up"):
            continue
        w = inputs.weights_fp32(N, K, seed=wl["seed"] * 100 + i)
        x = inputs.activations_bf16(M, K, seed=wl["seed"] * 1000 + M + i, outlier_frac=0.01,
                                    outlier_scale=20.0)
        sampled_check(w, x, seed=i)


@pytest.mark.parametrize("M", [1, 16, 256])
def test_70b_shapes_sampled(M):
    # one projection of each 70B shape (the 80-layer stack repeats them)
    for i, (name, N, K) in enumerate(inputs.SHAPES_70B):
        if name in ("q", "v", "up"):
            continue
        wq = inputs.ternary(N, K, seed=500 + i)
        gam = np.float32(inputs.gamma_uniform(600 + i))
        packed = bl.pack_ternary(wq.to(DEV))
        x = inputs.activations_bf16(M, K, seed=700 + M + i)
        q, s = bl.quant_act(x.to(DEV))
        acc = torch.empty(M, N, dtype=torch.int32, device=DEV)
        gdev = torch.tensor([gam], dtype=torch.float32, device=DEV)
        out = bl.forward(q, s, packed, gdev, N, acc_out=acc)
        torch.cuda.synchronize()
        q_ref, s_ref = oracle.quant_act(inputs.bf16_bits(x), None, 1e-5)
        np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
        rng = np.random.default_rng(i)
        ms = rng.integers(0, M, 2048)
        ns = rng.integers(0, N, 2048)
        wq_np = wq.numpy()
        want = oracle.matmul_pairs(q_ref, wq_np, ms, ns)
        accn = acc.cpu().numpy()
        np.testing.assert_array_equal(accn[ms, ns], want)
        np.testing.assert_array_equal(bits16(out), oracle.epilogue(accn, s.cpu().numpy(), gam))


# ------------------------------------------------------- edge and errors ---

def test_empty_batch_is_noop():
    packed, gamma = gpu_pack(inputs.weights_fp32(32, 64, seed=1))
    q = torch.empty(0, 64, dtype=torch.int8, device=DEV)
    s = torch.empty(0, dtype=torch.float32, device=DEV)
    out = bl.forward(q, s, packed, gamma, 32)
    assert out.shape == (0, 32)


def test_invalid_arguments_raise():
    packed, gamma = gpu_pack(inputs.weights_fp32(32, 64, seed=1))
    q = torch.zeros(2, 64, dtype=torch.int8, device=DEV)
    s = torch.ones(2, dtype=torch.float32, device=DEV)
    out = torch.empty(2, 32, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(bl.BitLinearError):
        bl.bitlinear_forward(q, s, packed, gamma, 2, 32, 60, out)
