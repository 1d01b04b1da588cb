"""The packing entry point that allocates nothing gives the same result as the
regular one.

bitlinear_pack_weights_noalloc exists for callers that cannot call
cudaMalloc (their device memory is owned by another allocator, or they must
not take the driver's allocation lock).  Its scratch is a fixed array inside
the library that every call clears and reuses, so this test calls it twice
in a row on different matrices (a leftover sum from the first call would
change the second call's gamma) and compares each call, through the C ABI,
with bitlinear_pack_weights: gamma bits and packed bytes must be identical,
the same bit-exact bar the other packing tests use.  It lives in its own file
so that it runs after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import bitlinear_02_b300 as bl
from bitlinear_02_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from bitlinear_02_b300 import build as blbuild
    blbuild.build()
    L = bl.load_library()
    L.bitlinear_pack_weights_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                                 ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_void_p]
    L.bitlinear_pack_weights_noalloc.restype = ctypes.c_int
    return L


def pack_both(L, w):
    N, K = w.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    nbytes = L.bitlinear_packed_bytes(N, K)
    p_ref = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    g_ref = torch.empty(1, dtype=torch.float32, device="cuda")
    p_new = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")
    g_new = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    st = L.bitlinear_pack_weights(ctypes.c_void_p(w.data_ptr()), N, K, 1e-5,
                                  ctypes.c_void_p(p_ref.data_ptr()), ctypes.c_void_p(g_ref.data_ptr()),
                                  stream)
    assert st == 0
    st = L.bitlinear_pack_weights_noalloc(ctypes.c_void_p(w.data_ptr()), N, K, 1e-5,
                                          ctypes.c_void_p(p_new.data_ptr()),
                                          ctypes.c_void_p(g_new.data_ptr()), stream)
    assert st == 0
    torch.cuda.synchronize()
    return p_ref.cpu().numpy(), g_ref.cpu().numpy(), p_new.cpu().numpy(), g_new.cpu().numpy()


def test_noalloc_pack_matches_pack_on_two_calls_in_a_row(lib):
    shapes = [(2560, 2560), (200, 8640)]
    for i, (N, K) in enumerate(shapes):  # two calls in a row, different sizes and sums
        w = inputs.weights_fp32(N, K, seed=4242 + i, std=0.02 * (i + 1), device="cuda")
        p_ref, g_ref, p_new, g_new = pack_both(lib, w)
        assert g_new.view(np.uint32)[0] == g_ref.view(np.uint32)[0]
        np.testing.assert_array_equal(p_new, p_ref)


def test_noalloc_pack_rejects_bad_sizes(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)
    # beyond the scratch's limit of 2^40 weights
    assert lib.bitlinear_pack_weights_noalloc(fake, 1 << 21, 1 << 20, 1e-5, fake, fake, None) == \
        bl.ERR_UNSUPPORTED
    assert lib.bitlinear_pack_weights_noalloc(fake, 4, 33, 1e-5, fake, fake, None) == bl.ERR_INVALID_ARG
