"""The stacked workloads (3B: 26 layers, 70B: 80 layers) on the GPU, layer by
layer against the CPU oracle, on sampled output rows.

Their ternary weights are drawn on the device by the counter-based generator
of the inputs module (SplitMix64, torch int64 arithmetic); the oracle
regenerates any row with its own C version of the same published generator,
so a sampled check needs no copy of the 17 GB of weights.  Per layer and
projection the oracle quantises the input the GPU saw (the stack input, or
the GPU's bf16 output feeding it) and multiplies it with the regenerated
rows.  Bit-exact: the int32 accumulators and the bf16 outputs (with the
token scales the GPU used); the token scales within 1e-6.
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


def bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def test_device_generator_matches_oracle_rows():
    N, K = 28672, 8192  # a 70B gate/up matrix, generated whole on the device
    word = inputs.stack_word(5, 41, 4)
    wq = inputs.ternary_hash(N, K, word, device=DEV)
    rng = np.random.default_rng(0)
    rows = np.concatenate([[0, N - 1], rng.integers(0, N, 30)])
    got = wq[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    want = np.concatenate([oracle.ternary_hash(word, K, int(n), int(n) + 1) for n in rows])
    np.testing.assert_array_equal(got, want)
    frac = torch.bincount((wq[:4096].flatten().to(torch.int64) + 1), minlength=3).cpu().numpy() / (4096 * K)
    assert np.all(np.abs(frac - 1 / 3) < 0.002)


class StackLayers:
    """The first `layers` layers of a stacked workload, generated on the device."""

    def __init__(self, workload, layers):
        wl = inputs.WORKLOADS[workload]
        self.seed = wl["seed"]
        self.shapes = wl["shapes"]
        self.hidden = self.shapes[0][2]
        self.o_src = 2 if self.shapes[2][1] == self.hidden else 0  # o reads v, or q where v is narrow
        self.w = []
        for l in range(layers):
            row = []
            for i, (_, N, K) in enumerate(self.shapes):
                word = inputs.stack_word(self.seed, l, i)
                packed = bl.pack_ternary(inputs.ternary_hash(N, K, word, device=DEV))
                g = np.float32(inputs.gamma_uniform(self.seed * 100000 + l * 10 + i))
                row.append((packed, torch.tensor([g], device=DEV), N, K, word, g))
            self.w.append(row)
        torch.cuda.synchronize()


def check_rows(x_bits, ts, proj, acc, out, rows):
    """Sampled rows of one projection against the oracle, from the GPU's input bits."""
    _, _, N, K, word, g = proj
    q_ref, s_ref = oracle.quant_act(x_bits, None, 1e-5)
    np.testing.assert_allclose(ts, s_ref, rtol=S_TOK_RTOL, atol=0)
    wq = np.concatenate([oracle.ternary_hash(word, K, int(n), int(n) + 1) for n in rows])
    acc_ref = oracle.matmul(q_ref, wq)  # [M, len(rows)]
    np.testing.assert_array_equal(acc.cpu().numpy()[:, rows], acc_ref)
    np.testing.assert_array_equal(bits16(out)[:, rows], oracle.epilogue(acc_ref, ts, g))


def sample_rows(N, rng, n=24):
    return np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, n)]))


# prepass: the threshold of bitlinear_set_fused_prepass (-1: the default,
# 16 MiB, under which every 70B launch quantises its input in a pre-pass and
# every 3B launch in its CTAs; 0: all launches; 2^40: none)
@pytest.mark.parametrize("workload,layers,M,prepass", [("stack_70b", 2, 1, -1), ("stack_70b", 2, 16, -1),
                                                       ("stack_70b", 1, 5, -1), ("stack_70b", 1, 8, -1),
                                                       ("stack_70b", 1, 11, -1),
                                                       ("stack_70b", 1, 4, 1 << 40), ("stack_3b", 2, 4, -1),
                                                       ("stack_3b", 1, 9, 0)])
def test_stack_fused_path_sampled(workload, layers, M, prepass):
    """The fused decode path (act_stats + 4 launches per layer), as the
    benchmark runs it, through the first layers of the stack."""
    bl.bitlinear_set_fused_prepass(prepass)
    S = StackLayers(workload, layers)
    rng = np.random.default_rng(M)
    x0 = inputs.activations_bf16(M, S.hidden, seed=7 * M + 3, device=DEV)
    xs = bl.new_stats(DEV)
    bl.bitlinear_act_stats(x0, M, S.hidden, 1e-5, xs)
    x, x_stats = x0, xs
    for l in range(layers):
        outs = [torch.empty(M, N, dtype=torch.bfloat16, device=DEV) for _, N, _ in S.shapes]
        accs = [torch.empty(M, N, dtype=torch.int32, device=DEV) for _, N, _ in S.shapes]
        st = [bl.new_stats(DEV) for _ in range(4)]  # o_src, o, up, down

        def fp(i, sb=None):
            p = S.w[l][i]
            return bl.FusedProj(p[0].data_ptr(), p[1].data_ptr(), p[2], outs[i].data_ptr(), accs[i].data_ptr(),
                                sb.data_ptr() if sb is not None else None)

        bl.bitlinear_forward_fused(x, x_stats, M, S.hidden,
                                   [fp(i, st[0] if i == S.o_src else None) for i in range(3)])
        src = outs[S.o_src]
        bl.bitlinear_forward_fused(src, st[0], M, src.shape[1], [fp(3, st[1])])
        bl.bitlinear_forward_fused(outs[3], st[1], M, outs[3].shape[1], [fp(4), fp(5, st[2])])
        bl.bitlinear_forward_fused(outs[5], st[2], M, outs[5].shape[1], [fp(6, st[3])])
        torch.cuda.synchronize()
        assert bl.bitlinear_check_status() == bl.OK
        ins = [(x, x_stats)] * 3 + [(src, st[0]), (outs[3], st[1]), (outs[3], st[1]), (outs[5], st[2])]
        for i, (xi, si) in enumerate(ins):
            _, ts = bl.fused_factors(si, M, xi.shape[1])
            check_rows(bits16(xi), ts.cpu().numpy(), S.w[l][i], accs[i], outs[i], sample_rows(S.w[l][i][2], rng))
        x, x_stats = outs[6], st[3]
    bl.fused_factors(x_stats, M, S.hidden, consume=True)
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK


@pytest.mark.parametrize("M", [32, 100, 256])
def test_70b_layer_unfused_large_batch_sampled(M):
    """Above 16 tokens the stacks run quant_act + forward per projection (the
    decode GEMV in 16-token chunks up to 64 tokens, the tcgen05 GEMM above)."""
    S = StackLayers("stack_70b", 1)
    rng = np.random.default_rng(100 + M)
    x = inputs.activations_bf16(M, S.hidden, seed=M, device=DEV)
    outs = [torch.empty(M, N, dtype=torch.bfloat16, device=DEV) for _, N, _ in S.shapes]
    accs = [torch.empty(M, N, dtype=torch.int32, device=DEV) for _, N, _ in S.shapes]
    srcs = {0: x, 1: x, 2: x}
    for i in range(7):
        if i == 3:
            srcs[3] = outs[S.o_src]
        elif i in (4, 5):
            srcs[i] = outs[3]
        elif i == 6:
            srcs[6] = outs[5]
        xi = srcs[i]
        q, s = bl.quant_act(xi)
        p = S.w[0][i]
        bl.forward(q, s, p[0], p[1], p[2], out=outs[i], acc_out=accs[i])
        torch.cuda.synchronize()
        check_rows(bits16(xi), s.cpu().numpy(), p, accs[i], outs[i], sample_rows(p[2], rng))
    assert bl.bitlinear_check_status() == bl.OK
