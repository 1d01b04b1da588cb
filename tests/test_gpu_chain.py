"""Parity of the fused decode chain (bitlinear_chain_*) with the CPU oracle.

Every projection of a chain is checked layer by layer: the oracle quantises
the projection's input as the GPU saw it (the chain input, or the GPU's bf16
output of the projection feeding it), multiplies with the ternary weights
and rescales.  Bit-exact: the int32 accumulators (which pins the int8
activations too), and the bf16 outputs when the oracle's epilogue is fed the
GPU's token scales.  The token scales are a float reduction and are held to
1e-6 relative.  The chain is also compared with the unfused path
(bitlinear_quant_act + bitlinear_forward).
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from bitlinear_02_b300 import build as blbuild
    blbuild.build()
    bl.load_library()
    oracle.build()
    torch.cuda.init()
    yield
    bl.bitlinear_chain_set_split(0)


def bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def make_weights(shapes, seed, ternary=False):
    """shapes: list of (N, K).  Returns per projection (packed, gamma, wq numpy, gamma float)."""
    out = []
    for i, (N, K) in enumerate(shapes):
        if ternary:
            wq = inputs.ternary(N, K, seed=seed + i)
            g = np.float32(inputs.gamma_uniform(seed + 100 + i))
            packed = bl.pack_ternary(wq.to(DEV))
            gamma = torch.tensor([g], dtype=torch.float32, device=DEV)
            out.append((packed, gamma, wq.numpy(), g))
        else:
            w = inputs.weights_fp32(N, K, seed=seed + i)
            g = oracle.gamma(w.numpy())
            wq = oracle.ternarize(w.numpy(), g, 1e-5)
            packed, gamma = bl.pack_weights(w.to(DEV), 1e-5)
            out.append((packed, gamma, wq, np.float32(g)))
    return out


def run_chain(M, K0, chain, weights, x, split=0):
    """chain: list of (N, input slot).  Returns the DecodeChain after one run."""
    bl.bitlinear_chain_set_split(split)
    projs = [dict(packed=weights[j][0], gamma=weights[j][1], N=N, input=inp)
             for j, (N, inp) in enumerate(chain)]
    dc = bl.DecodeChain(M, K0, projs, eps=1e-5, keep_acc=True, keep_scales=True)
    bl.bitlinear_chain_set_split(0)
    dc.run(x.to(DEV))
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    return dc


def check_chain(dc, chain, weights, x, sample=None):
    slots = [inputs.bf16_bits(x)]
    for j, (N, inp) in enumerate(chain):
        src = slots[inp]
        q_ref, s_ref = oracle.quant_act(src, None, 1e-5)
        s = dc.tok_scale[j].cpu().numpy()
        np.testing.assert_allclose(s, s_ref, rtol=S_TOK_RTOL, atol=0, err_msg=f"proj {j} scales")
        acc = dc.acc[j].cpu().numpy()
        wq = weights[j][2]
        if sample is None:
            acc_ref = oracle.matmul(q_ref, wq)
            np.testing.assert_array_equal(acc, acc_ref, err_msg=f"proj {j} accumulators")
        else:
            rng = np.random.default_rng(j)
            ms = rng.integers(0, acc.shape[0], sample)
            ns = rng.integers(0, acc.shape[1], sample)
            np.testing.assert_array_equal(acc[ms, ns], oracle.matmul_pairs(q_ref, wq, ms, ns),
                                          err_msg=f"proj {j} accumulators")
        out = bits16(dc.out[j])
        np.testing.assert_array_equal(out, oracle.epilogue(acc, s, weights[j][3]),
                                      err_msg=f"proj {j} outputs")
        slots.append(out)


# chain of the decode bench: h = x; q,k,v = f(h); o = f(v); gate,up = f(o); down = f(up)
def layer_chain(hidden, ffn, kv):
    shapes = [(hidden, hidden), (kv, hidden), (kv, hidden), (hidden, kv), (ffn, hidden),
              (ffn, hidden), (hidden, ffn)]
    chain = [(hidden, 0), (kv, 0), (kv, 0), (hidden, 3), (ffn, 4), (ffn, 4), (hidden, 6)]
    return shapes, chain


@pytest.mark.parametrize("split", [0, 1, 2, 3])
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_small_chain(M, split):
    # two projections with ragged tiles (K = 272 is not a multiple of 128)
    K0 = 272
    shapes = [(400, 272), (144, 400), (48, 144)]
    chain = [(400, 0), (144, 1), (48, 2)]
    w = make_weights(shapes, seed=1000 + M)
    x = inputs.activations_bf16(M, K0, seed=17 + M, outlier_frac=0.01)
    dc = run_chain(M, K0, chain, w, x, split)
    check_chain(dc, chain, w, x)


@pytest.mark.parametrize("M", [1, 4, 16])
def test_2b_layer_chain(M):
    shapes, chain = layer_chain(2560, 6912, 2560)
    w = make_weights(shapes, seed=2000)
    x = inputs.activations_bf16(M, 2560, seed=2100 + M)
    dc = run_chain(M, 2560, chain, w, x)
    check_chain(dc, chain, w, x)


@pytest.mark.parametrize("M", [2, 16])
def test_two_layers_and_runs_in_a_row(M):
    # two 3B-shaped layers chained (the second layer reads the first's down
    # projection), run twice with different inputs on the same plan
    shapes, chain = layer_chain(3200, 8640, 3200)
    chain2 = chain + [(N, inp + 7 if inp else 7) for N, inp in chain]
    shapes2 = shapes + shapes
    w = make_weights(shapes2, seed=3000, ternary=True)
    projs = [dict(packed=w[j][0], gamma=w[j][1], N=N, input=inp) for j, (N, inp) in enumerate(chain2)]
    dc = bl.DecodeChain(M, 3200, projs, keep_acc=True, keep_scales=True)
    for r in range(2):
        x = inputs.activations_bf16(M, 3200, seed=3100 + 10 * r + M)
        dc.run(x.to(DEV))
        torch.cuda.synchronize()
        assert bl.bitlinear_check_status() == bl.OK
        check_chain(dc, chain2, w, x, sample=4096)


def test_chain_matches_unfused_path():
    M, K0 = 5, 2560
    shapes, chain = layer_chain(2560, 6912, 2560)
    w = make_weights(shapes, seed=4000)
    x = inputs.activations_bf16(M, K0, seed=4100)
    dc = run_chain(M, K0, chain, w, x)
    slots = [x.to(DEV)]
    for j, (N, inp) in enumerate(chain):
        q, s = bl.quant_act(slots[inp], None, 1e-5)
        acc = torch.empty(M, N, dtype=torch.int32, device=DEV)
        bl.forward(q, s, w[j][0], w[j][1], N, acc_out=acc)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(dc.acc[j].cpu().numpy(), acc.cpu().numpy())
        np.testing.assert_allclose(dc.tok_scale[j].cpu().numpy(), s.cpu().numpy(), rtol=S_TOK_RTOL)
        slots.append(dc.out[j])


def test_70b_shapes_one_layer_sampled():
    shapes, chain = layer_chain(8192, 28672, 1024)
    # 70B: o reads q (v is only 1024 wide)
    chain = [(8192, 0), (1024, 0), (1024, 0), (8192, 1), (28672, 4), (28672, 4), (8192, 6)]
    shapes = [(8192, 8192), (1024, 8192), (1024, 8192), (8192, 8192), (28672, 8192),
              (28672, 8192), (8192, 28672)]
    w = make_weights(shapes, seed=5000, ternary=True)
    for M in (1, 16):
        x = inputs.activations_bf16(M, 8192, seed=5100 + M)
        dc = run_chain(M, 8192, chain, w, x)
        check_chain(dc, chain, w, x, sample=2048)


def test_chain_timeout_is_reported_and_recovers():
    M, K0 = 4, 256
    shapes = [(512, 256), (256, 512)]
    chain = [(512, 0), (256, 1)]
    w = make_weights(shapes, seed=6000)
    x = inputs.activations_bf16(M, K0, seed=6100)
    projs = [dict(packed=w[j][0], gamma=w[j][1], N=N, input=inp) for j, (N, inp) in enumerate(chain)]
    dc = bl.DecodeChain(M, K0, projs, keep_acc=True, keep_scales=True)
    assert bl.bitlinear_check_status() == bl.OK
    try:
        bl.bitlinear_set_wait_limit(1)
        dc.run(x.to(DEV))
        st = bl.bitlinear_check_status()
    finally:
        bl.bitlinear_set_wait_limit(0)
    assert st == bl.ERR_TIMEOUT
    dc.run(x.to(DEV))
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    check_chain(dc, chain, w, x)


def test_chain_rejects_bad_descriptions():
    w = make_weights([(512, 256)], seed=7000)
    P = bl.ChainProj
    good = P(w[0][0].data_ptr(), w[0][1].data_ptr(), 512, 0, 0, None, None, None)
    assert bl.bitlinear_chain_workspace_bytes(4, 256, [good]) > 0
    assert bl.bitlinear_chain_workspace_bytes(17, 256, [good]) == 0          # M > 16
    assert bl.bitlinear_chain_workspace_bytes(4, 250, [good]) == 0           # K0 % 16
    bad_slot = P(w[0][0].data_ptr(), w[0][1].data_ptr(), 512, 1, 0, None, None, None)
    assert bl.bitlinear_chain_workspace_bytes(4, 256, [bad_slot]) == 0      # reads its own output
    odd = P(w[0][0].data_ptr(), w[0][1].data_ptr(), 500, 0, 0, None, None, None)
    reader = P(w[0][0].data_ptr(), w[0][1].data_ptr(), 16, 1, 0, None, None, None)
    assert bl.bitlinear_chain_workspace_bytes(4, 256, [odd, reader]) == 0   # read output N % 16
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    with pytest.raises(bl.BitLinearError):
        bl.bitlinear_chain_prepare(4, 256, [good], 1e-5, ws, 16)            # workspace too small
