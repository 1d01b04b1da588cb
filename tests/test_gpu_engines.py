"""Engine choice of bitlinear_forward / bitlinear_forward_f16 against the
oracle (needs a B300).

The same inputs go through every route the library has around the switch
from the decode GEMV to the tensor-core GEMM: the default choice, the GEMV
and the GEMM at the same batch sizes, and the GEMM with its k range split
across a cluster of CTAs (the planner's size and forced sizes).  Every route
must give the oracle's int32 accumulators and bf16 outputs bit for bit.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import bitlinear_02_b300 as bl
from bitlinear_02_b300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
S_TOK_RTOL = 1e-6

# name -> (gemv_max_tokens, split_k) for bitlinear_set_engine
ROUTES = {
    "default": (-1, 0),
    "gemv_up_to_16": (16, 0),
    "gemm_unsplit": (0, 1),
    "gemm_planned": (0, 0),
    "gemm_split2": (0, 2),
    "gemm_split5": (0, 5),
    "gemm_split16": (0, 16),
}


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
def _default_engine():
    yield
    bl.bitlinear_set_engine(-1, 0)
    bl.bitlinear_set_wait_limit(0)


class Case:
    """Weights packed on the GPU, activations quantised on the GPU, and the
    oracle's accumulators for them."""

    def __init__(self, N, K, M, seed):
        w = inputs.weights_fp32(N, K, seed=seed)
        x = inputs.activations_bf16(M, K, seed=seed + 1, outlier_frac=0.01)
        wn = w.numpy()
        self.g_ref = oracle.gamma(wn)
        wq = oracle.ternarize(wn, self.g_ref, 1e-5)
        self.q_ref, self.s_ref = oracle.quant_act(inputs.bf16_bits(x), None, 1e-5)
        self.acc_ref = oracle.matmul(self.q_ref, wq)
        self.packed, self.gamma = bl.pack_weights(w.to(DEV), 1e-5)
        self.q, self.s = bl.quant_act(x.to(DEV))
        self.q16, self.s16 = bl.quant_act_f16(x.to(DEV))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(self.q.cpu().numpy(), self.q_ref)
        np.testing.assert_allclose(self.s.cpu().numpy(), self.s_ref, rtol=S_TOK_RTOL, atol=0)
        self.N, self.K, self.M = N, K, M

    def check(self, f16=False):
        acc = torch.full((self.M, self.N), -7, dtype=torch.int32, device=DEV)
        if f16:
            out = bl.forward_f16(self.q16, self.s16, self.packed, self.gamma, self.N, acc_out=acc)
            s = self.s16
        else:
            out = bl.forward(self.q, self.s, self.packed, self.gamma, self.N, acc_out=acc)
            s = self.s
        torch.cuda.synchronize()
        assert bl.bitlinear_check_status() == bl.OK
        np.testing.assert_array_equal(acc.cpu().numpy(), self.acc_ref)
        np.testing.assert_array_equal(bits16(out), oracle.epilogue(self.acc_ref, s.cpu().numpy(), self.g_ref))


@pytest.mark.parametrize("M", [1, 16, 40, 64, 65, 100, 176, 256])
@pytest.mark.parametrize("N,K", [(300, 1040), (2560, 2560), (1000, 6912), (4112, 4096)])
def test_every_route_bit_exact(N, K, M):
    # 4112 x 4096 holds 2^24 + 2^16 weights: above 64 tokens the int8 input
    # is widened to f16 first (and 4112 rows leave a ragged last row tile)
    case = Case(N, K, M, seed=31 * N + K + M)
    for route, (gmax, split) in ROUTES.items():
        bl.bitlinear_set_engine(gmax, split)
        case.check()
        if route.startswith("gemm"):
            case.check(f16=True)


@pytest.mark.parametrize("M", [65, 130, 256])
def test_split_on_narrow_70b_projection(M):
    """k/v of the 70B shapes (N = 1024, K = 8192): 8 row tiles, so the planner
    splits k across up to 16 CTAs; sampled outputs against the oracle."""
    N, K = 1024, 8192
    wq = inputs.ternary(N, K, seed=900 + M)
    gam = np.float32(inputs.gamma_uniform(901 + M))
    packed = bl.pack_ternary(wq.to(DEV))
    gdev = torch.tensor([gam], dtype=torch.float32, device=DEV)
    x = inputs.activations_bf16(M, K, seed=902 + M)
    q, s = bl.quant_act(x.to(DEV))
    q_ref, _ = oracle.quant_act(inputs.bf16_bits(x), None, 1e-5)
    acc_ref = oracle.matmul(q_ref, wq.numpy())
    for split in (0, 1, 3, 8, 16):
        bl.bitlinear_set_engine(0, split)
        acc = torch.empty(M, N, dtype=torch.int32, device=DEV)
        out = bl.forward(q, s, packed, gdev, N, acc_out=acc)
        torch.cuda.synchronize()
        assert bl.bitlinear_check_status() == bl.OK
        np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
        np.testing.assert_array_equal(bits16(out), oracle.epilogue(acc_ref, s.cpu().numpy(), gam))


@pytest.mark.parametrize("M", [33, 48])
def test_mid_batch_default_route_on_deep_matrix(M):
    """33-48 tokens on a matrix with K >= 8192, N <= K and N*K >= 2^24 (2064
    x 8192, a ragged last row tile): the default route is the split GEMM on
    widened activations; it gives the GEMV's bits, and sampled accumulators
    match the oracle."""
    N, K = 2064, 8192
    wq = inputs.ternary(N, K, seed=950 + M)
    gdev = torch.tensor([0.03], dtype=torch.float32, device=DEV)
    packed = bl.pack_ternary(wq.to(DEV))
    x = inputs.activations_bf16(M, K, seed=951 + M)
    q, s = bl.quant_act(x.to(DEV))
    runs = {}
    for route, gmax in (("default", -1), ("gemv", 64)):
        bl.bitlinear_set_engine(gmax, 0)
        acc = torch.empty(M, N, dtype=torch.int32, device=DEV)
        out = bl.forward(q, s, packed, gdev, N, acc_out=acc)
        torch.cuda.synchronize()
        assert bl.bitlinear_check_status() == bl.OK
        runs[route] = (acc.cpu().numpy(), bits16(out))
    np.testing.assert_array_equal(runs["default"][0], runs["gemv"][0])
    np.testing.assert_array_equal(runs["default"][1], runs["gemv"][1])
    rng = np.random.default_rng(M)
    ms, ns = rng.integers(0, M, 512), rng.integers(0, N, 512)
    want = oracle.matmul_pairs(q.cpu().numpy(), wq.numpy(), ms, ns)
    np.testing.assert_array_equal(runs["default"][0][ms, ns], want)


def test_set_engine_rejects_out_of_range():
    for args in ((65, 0), (-2, 0), (0, 17), (0, -1)):
        with pytest.raises(bl.BitLinearError):
            bl.bitlinear_set_engine(*args)


def _time_forward(fn, reps=3):
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(reps):
        ev0.record()
        fn()
        ev1.record()
        torch.cuda.synchronize()
        best = min(best, ev0.elapsed_time(ev1))
    return best


@pytest.mark.parametrize("M,N,split", [(4096, 2560, 0), (64, 240, 4)])
def test_expired_wait_ends_the_gemm_promptly(M, N, split):
    """One expired wait ends every role's waits (a flag in shared memory):
    with a wait limit of one try the GEMM over K = 65536 reports ERR_TIMEOUT
    and ends well before its normal time, and the next call computes the same
    bits as before.  Without the flag every stage would still run (each
    role's failed tries only set its own bit), so the call would take at
    least its normal time.  When the first one-try wait expires depends on
    how long the hardware suspends a try, hence the bound of half the normal
    time; the best of two aborted calls is taken.  (4096 tokens: the
    f16-operand kernel after the widening pass; 64 tokens on 240 rows - two
    row tiles - through the GEMM, below 2^24 weights, so not widened: the
    int8-operand kernel split across clusters of 4.)"""
    K = 65536
    bl.bitlinear_set_engine(0, split)
    wq = inputs.ternary(N, K, seed=77, device=DEV)
    packed = bl.pack_ternary(wq)
    gdev = torch.tensor([0.5], dtype=torch.float32, device=DEV)
    x = inputs.activations_bf16(M, K, seed=78, device=DEV)
    q, s = bl.quant_act(x)
    out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    acc = torch.empty(M, N, dtype=torch.int32, device=DEV)

    def run():
        bl.forward(q, s, packed, gdev, N, out=out, acc_out=acc)

    assert bl.bitlinear_check_status() == bl.OK
    t_norm = _time_forward(run)
    assert bl.bitlinear_check_status() == bl.OK
    ref_acc, ref_out = acc.clone(), out.clone()
    try:
        bl.bitlinear_set_wait_limit(1)
        t0 = time.perf_counter()
        t_abort = _time_forward(run, reps=2)
        wall = time.perf_counter() - t0
        st = bl.bitlinear_check_status()
    finally:
        bl.bitlinear_set_wait_limit(0)
    assert st == bl.ERR_TIMEOUT
    assert t_abort < 0.5 * t_norm, (t_abort, t_norm)
    assert wall < 5.0
    # recovery: the same bits as before the timeout
    assert bl.bitlinear_check_status() == bl.OK
    run()
    torch.cuda.synchronize()
    assert bl.bitlinear_check_status() == bl.OK
    assert torch.equal(acc, ref_acc) and torch.equal(out, ref_out)
    # and right: sampled accumulators against the oracle
    q_ref = q.cpu().numpy()
    rng = np.random.default_rng(5)
    ms, ns = rng.integers(0, M, 256), rng.integers(0, N, 256)
    wq_cpu = wq.cpu().numpy()
    want = oracle.matmul_pairs(q_ref, wq_cpu, ms, ns)
    np.testing.assert_array_equal(acc.cpu().numpy()[ms, ns], want)


def test_failing_allocation_is_err_cuda_and_recovers():
    """Host-side failure injection: a prefill call whose f16 widening buffer
    cannot exist (4e6 tokens x 65536 x 2 bytes = 512 GB, above the 288 GB of
    HBM) returns ERR_CUDA before any kernel runs and leaves no error behind;
    the next calls compute the right bits.  (The activation buffers are
    small: nothing reads them, the allocation fails first.)"""
    M, N, K = 4_000_000, 16, 65536
    # only where the buffer cannot fit in the device's memory at all
    assert torch.cuda.mem_get_info()[1] < M * K * 2
    q = torch.zeros(16, K, dtype=torch.int8, device=DEV)
    s = torch.ones(16, dtype=torch.float32, device=DEV)
    packed = bl.pack_ternary(inputs.ternary(N, K, seed=3).to(DEV))
    gam = torch.ones(1, dtype=torch.float32, device=DEV)
    out = torch.empty(16, N, dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    L = bl.load_library()
    st = L.bitlinear_forward(bl._ptr(q), bl._ptr(s), bl._ptr(packed), bl._ptr(gam), M, N, K, bl._ptr(out), None,
                             bl._stream(None))
    assert st == bl.ERR_CUDA
    torch.cuda.synchronize()  # no error left in the context or the runtime
    assert bl.bitlinear_check_status() == bl.OK
    # a normal prefill call afterwards is right
    case = Case(300, 1040, 300, seed=41)
    case.check()
