"""Parity of the fused decode path (bitlinear_act_stats + bitlinear_forward_fused)
with the CPU oracle.

Layer by layer: the oracle quantises each projection's input as the GPU saw
it (the layer input, or the GPU's bf16 output of the projection feeding it),
multiplies with the ternary weights and rescales.  Bit-exact: the int32
accumulators (which pins the int8 activations), and the bf16 outputs when the
oracle's epilogue is fed the token scales the GPU used (read back from the
input's factor buffer).  The token scales and the factors c = 127/max are
held to the oracle's within 1e-6 and bit for bit respectively.  Also the
factor buffer's protocol: pending until consumed, published by the consumer,
a second production into a pending buffer reported, a reset by
bitlinear_act_stats.
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


@pytest.fixture(autouse=True)
def _default_prepass():
    yield
    bl.bitlinear_set_fused_prepass(-1)


# bitlinear_set_fused_prepass thresholds: the default (in-kernel quantisation
# for these small launches) and 0 (every launch through the quantising
# pre-pass and the GEMV on int8 input)
PREPASS = [-1, 0]


def bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def factors(stats, M, K):
    c, ts = bl.fused_factors(stats, M, K)
    return c.cpu().numpy(), ts.cpu().numpy()


def make_weights(shapes, seed):
    out = []
    for i, (N, K) in enumerate(shapes):
        w = inputs.weights_fp32(N, K, seed=seed + i)
        g = oracle.gamma(w.numpy())
        wq = oracle.ternarize(w.numpy(), g, 1e-5)
        packed, gamma = bl.pack_weights(w.to(DEV), 1e-5)
        out.append((packed, gamma, wq, np.float32(g)))
    return out


def check_proj(x_bits, stats_in, M, w, acc, out):
    """One projection: the oracle on the GPU's input bits and token scales."""
    q_ref, s_ref = oracle.quant_act(x_bits, None, 1e-5)
    c, ts = factors(stats_in, M, x_bits.shape[1])
    mx = np.maximum(np.abs(x_bits_to_f32(x_bits)).max(axis=1), np.float32(1e-5))
    np.testing.assert_array_equal(c, np.float32(127.0) / mx.astype(np.float32))
    np.testing.assert_allclose(ts, s_ref, rtol=S_TOK_RTOL, atol=0)
    acc_ref = oracle.matmul(q_ref, w[2])
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
    np.testing.assert_array_equal(bits16(out), oracle.epilogue(acc_ref, ts, w[3]))


def x_bits_to_f32(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def run_layer(M, hidden, ffn, kv, w, x, stats, check=True):
    """h = x; q,k,v = f(h); o = f(v); gate,up = f(o); down = f(up)."""
    dev_out = {}
    N = {"q": hidden, "k": kv, "v": kv, "o": hidden, "gate": ffn, "up": ffn, "down": hidden}
    for name in N:
        dev_out[name] = (torch.empty(M, N[name], dtype=torch.bfloat16, device=DEV),
                         torch.empty(M, N[name], dtype=torch.int32, device=DEV))
    names = ["q", "k", "v", "o", "gate", "up", "down"]
    W = dict(zip(names, w))

    def fp(name, st=None):
        o, a = dev_out[name]
        p, g = W[name][0], W[name][1]
        return bl.FusedProj(p.data_ptr(), g.data_ptr(), N[name], o.data_ptr(), a.data_ptr(),
                            st.data_ptr() if st is not None else None)

    bl.bitlinear_act_stats(x, M, hidden, 1e-5, stats["x"])
    bl.bitlinear_forward_fused(x, stats["x"], M, hidden, [fp("q"), fp("k"), fp("v", stats["v"])])
    bl.bitlinear_forward_fused(dev_out["v"][0], stats["v"], M, kv, [fp("o", stats["o"])])
    bl.bitlinear_forward_fused(dev_out["o"][0], stats["o"], M, hidden, [fp("gate"), fp("up", stats["up"])])
    bl.bitlinear_forward_fused(dev_out["up"][0], stats["up"], M, ffn, [fp("down", stats["down"])])
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    if check:
        xb = inputs.bf16_bits(x)
        for name, src, st in [("q", xb, "x"), ("k", xb, "x"), ("v", xb, "x")]:
            check_proj(src, stats[st], M, W[name], dev_out[name][1], dev_out[name][0])
        check_proj(bits16(dev_out["v"][0]), stats["v"], M, W["o"], dev_out["o"][1], dev_out["o"][0])
        ob = bits16(dev_out["o"][0])
        for name in ("gate", "up"):
            check_proj(ob, stats["o"], M, W[name], dev_out[name][1], dev_out[name][0])
        check_proj(bits16(dev_out["up"][0]), stats["up"], M, W["down"], dev_out["down"][1], dev_out["down"][0])
        # the down projection's factors, for the next layer (still pending)
        check_factors(bits16(dev_out["down"][0]), stats["down"], M)
    # nothing consumes them here: consume them so the buffer can be produced again
    bl.fused_factors(stats["down"], M, hidden, consume=True)
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    return dev_out


def check_factors(x_bits, stats, M):
    _, s_ref = oracle.quant_act(x_bits, None, 1e-5)
    c, ts = factors(stats, M, x_bits.shape[1])
    mx = np.maximum(np.abs(x_bits_to_f32(x_bits)).max(axis=1), np.float32(1e-5))
    np.testing.assert_array_equal(c, np.float32(127.0) / mx.astype(np.float32))
    np.testing.assert_allclose(ts, s_ref, rtol=S_TOK_RTOL, atol=0)


def new_stats():
    return {k: bl.new_stats(DEV) for k in ("x", "v", "o", "up", "down")}


@pytest.mark.parametrize("prepass", PREPASS)
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_fused_small_ragged_layer(M, prepass):
    bl.bitlinear_set_fused_prepass(prepass)
    # ragged: N not a multiple of 64, K not a multiple of 128
    hidden, ffn, kv = 272, 400, 144
    shapes = [(hidden, hidden), (kv, hidden), (kv, hidden), (hidden, kv), (ffn, hidden), (ffn, hidden),
              (hidden, ffn)]
    w = make_weights(shapes, seed=8000 + M)
    x = inputs.activations_bf16(M, hidden, seed=8100 + M, outlier_frac=0.01).to(DEV)
    stats = new_stats()
    run_layer(M, hidden, ffn, kv, w, x, stats)
    # the factor buffers are reusable: a second layer pass with another input
    x2 = inputs.activations_bf16(M, hidden, seed=8200 + M).to(DEV)
    run_layer(M, hidden, ffn, kv, w, x2, stats)


@pytest.mark.parametrize("prepass", PREPASS)
@pytest.mark.parametrize("M", [1, 4, 16])
def test_fused_2b_layer(M, prepass):
    bl.bitlinear_set_fused_prepass(prepass)
    hidden, ffn, kv = 2560, 6912, 2560
    shapes = [(hidden, hidden), (kv, hidden), (kv, hidden), (hidden, kv), (ffn, hidden), (ffn, hidden),
              (hidden, ffn)]
    w = make_weights(shapes, seed=9000)
    x = inputs.activations_bf16(M, hidden, seed=9100 + M).to(DEV)
    run_layer(M, hidden, ffn, kv, w, x, new_stats())


@pytest.mark.parametrize("prepass", PREPASS)
def test_fused_matches_unfused_path(prepass):
    bl.bitlinear_set_fused_prepass(prepass)
    M, K, N = 5, 2560, 6912
    w = make_weights([(N, K)], seed=9500)[0]
    x = inputs.activations_bf16(M, K, seed=9600).to(DEV)
    st = bl.new_stats(DEV)
    bl.bitlinear_act_stats(x, M, K, 1e-5, st)
    out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    acc = torch.empty(M, N, dtype=torch.int32, device=DEV)
    bl.bitlinear_forward_fused(x, st, M, K, [bl.FusedProj(w[0].data_ptr(), w[1].data_ptr(), N, out.data_ptr(),
                                                          acc.data_ptr(), None)])
    q, s = bl.quant_act(x)
    acc2 = torch.empty(M, N, dtype=torch.int32, device=DEV)
    bl.forward(q, s, w[0], w[1], N, acc_out=acc2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(acc.cpu().numpy(), acc2.cpu().numpy())
    _, ts = factors(st, M, K)
    np.testing.assert_allclose(ts, s.cpu().numpy(), rtol=S_TOK_RTOL)


@pytest.mark.parametrize("prepass", PREPASS)
def test_factor_buffer_protocol(prepass):
    """Pending until consumed; every consumer sees the same factors; a second
    production into a pending buffer is reported; act_stats resets.  (With
    the pre-pass, the pre-pass kernel is the consumer.)"""
    bl.bitlinear_set_fused_prepass(prepass)
    M, K, N, N2 = 7, 512, 640, 384
    w1 = make_weights([(N, K)], seed=9800)[0]
    w2 = make_weights([(N2, N)], seed=9801)[0]
    x = inputs.activations_bf16(M, K, seed=9802).to(DEV)
    sx, sh = bl.new_stats(DEV), bl.new_stats(DEV)
    h = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)

    def produce():
        bl.bitlinear_act_stats(x, M, K, 1e-5, sx)
        bl.bitlinear_forward_fused(x, sx, M, K, [bl.FusedProj(w1[0].data_ptr(), w1[1].data_ptr(), N, h.data_ptr(),
                                                              None, sh.data_ptr())])

    def consume():
        out = torch.empty(M, N2, dtype=torch.bfloat16, device=DEV)
        acc = torch.empty(M, N2, dtype=torch.int32, device=DEV)
        bl.bitlinear_forward_fused(h, sh, M, N, [bl.FusedProj(w2[0].data_ptr(), w2[1].data_ptr(), N2,
                                                              out.data_ptr(), acc.data_ptr(), None)])
        return out, acc

    produce()
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    state = lambda: int(sh.view(torch.int32)[32].item())
    assert state() == 1                                   # pending
    c0, ts0 = factors(sh, M, N)                           # read without consuming
    assert state() == 1
    out1, acc1 = consume()
    torch.cuda.synchronize()
    assert state() == 0                                   # published, accumulator cleared
    f = sh.view(torch.float32).cpu().numpy()
    np.testing.assert_array_equal(f[0:M], c0)
    np.testing.assert_array_equal(f[16:16 + M], ts0)
    assert not sh.view(torch.int32)[64:64 + 512].any().item()
    out2, acc2 = consume()                                # a second consumer: the published factors
    torch.cuda.synchronize()
    np.testing.assert_array_equal(acc1.cpu().numpy(), acc2.cpu().numpy())
    np.testing.assert_array_equal(bits16(out1), bits16(out2))
    check_proj(bits16(h), sh, M, w2, acc1, out1)
    assert bl.bitlinear_check_status() == bl.OK
    # produce twice without consuming: reported, and act_stats makes it usable again
    produce()
    produce()
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.ERR_STATE
    assert bl.bitlinear_check_status() == bl.OK           # the status word was cleared
    bl.bitlinear_act_stats(h, M, N, 1e-5, sh)
    torch.cuda.synchronize()
    assert state() == 0
    produce()
    out3, acc3 = consume()
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    np.testing.assert_array_equal(acc1.cpu().numpy(), acc3.cpu().numpy())
    check_proj(bits16(h), sh, M, w2, acc3, out3)   # the sum order of the token scale may differ


def test_fused_rejects_bad_arguments():
    w = make_weights([(64, 256)], seed=9700)[0]
    x = torch.zeros(2, 256, dtype=torch.bfloat16, device=DEV)
    st = bl.new_stats(DEV)
    out = torch.empty(2, 64, dtype=torch.bfloat16, device=DEV)
    p = bl.FusedProj(w[0].data_ptr(), w[1].data_ptr(), 64, out.data_ptr(), None, None)
    with pytest.raises(bl.BitLinearError):
        bl.bitlinear_forward_fused(x, st, 17, 256, [p])          # M > 16
    with pytest.raises(bl.BitLinearError):
        bl.bitlinear_forward_fused(x, st, 2, 250, [p])           # K % 16
    with pytest.raises(bl.BitLinearError):
        bl.bitlinear_forward_fused(x, st, 2, 256, [p] * 5)       # more than 4 projections
    with pytest.raises(bl.BitLinearError):
        bl.bitlinear_act_stats(x, 0, 256, 1e-5, st)
    ps = bl.FusedProj(w[0].data_ptr(), w[1].data_ptr(), 64, out.data_ptr(), None, st.data_ptr())
    with pytest.raises(bl.BitLinearError):
        bl.bitlinear_forward_fused(x, st, 2, 256, [ps])          # reads and writes one factor buffer
    st2 = bl.new_stats(DEV)
    ps2 = bl.FusedProj(w[0].data_ptr(), w[1].data_ptr(), 64, out.data_ptr(), None, st2.data_ptr())
    with pytest.raises(bl.BitLinearError):
        bl.bitlinear_forward_fused(x, st, 2, 256, [ps2, ps2])    # two outputs into one factor buffer
