"""Concurrent use of the library (needs a B300): several engine routes at
once on separate CUDA streams, issued from separate host threads, give the
bits each route gives alone.

The routes share the library's host-side state - the tensor-map cache, the
memory pool behind the widening pass and the fused path's pre-pass scratch,
the device status word - and the device itself.  Each thread repeats its
route on its own buffers; afterwards every output is compared with the same
route run alone on one stream beforehand.
"""
import threading

import pytest
import torch

import bitlinear_02_b300 as bl
from bitlinear_02_b300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from bitlinear_02_b300 import build as blbuild
    blbuild.build()
    bl.load_library()
    torch.cuda.init()


def make_routes():
    """(name, run(stream) -> output tensor) for each route, on its own
    weights and buffers."""
    routes = []

    def forward_route(name, M, N, K, seed):
        w = inputs.weights_fp32(N, K, seed=seed, device=DEV)
        packed, gamma = bl.pack_weights(w, 1e-5)
        x = inputs.activations_bf16(M, K, seed=seed + 1, device=DEV)
        q, s = bl.quant_act(x)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)

        def run(st):
            bl.bitlinear_forward(q, s, packed, gamma, M, N, K, out, None, st)
            return out
        routes.append((name, run))

    def f16_route(name, M, N, K, seed):
        w = inputs.weights_fp32(N, K, seed=seed, device=DEV)
        packed, gamma = bl.pack_weights(w, 1e-5)
        x = inputs.activations_bf16(M, K, seed=seed + 1, device=DEV)
        q16, s = bl.quant_act_f16(x)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)

        def run(st):
            bl.bitlinear_forward_f16(q16, s, packed, gamma, M, N, K, out, None, st)
            return out
        routes.append((name, run))

    def fused_route(name, M, N, K, seed):
        w = inputs.weights_fp32(N, K, seed=seed, device=DEV)
        packed, gamma = bl.pack_weights(w, 1e-5)
        x = inputs.activations_bf16(M, K, seed=seed + 1, device=DEV)
        xs = bl.new_stats(DEV)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)

        def run(st):
            bl.bitlinear_act_stats(x, M, K, 1e-5, xs, st)
            bl.bitlinear_forward_fused(x, xs, M, K, [bl.FusedProj(packed.data_ptr(), gamma.data_ptr(), N,
                                                                  out.data_ptr(), None, None)], 1e-5, st)
            return out
        routes.append((name, run))

    forward_route("gemm_widened", 300, 4104, 4096, 11)     # widening pass + f16 GEMM (pool memory)
    forward_route("gemm_split", 100, 1000, 6912, 21)       # int8 GEMM split across a cluster
    forward_route("gemv", 5, 2560, 2560, 31)               # decode GEMV
    forward_route("gemv_chunks", 40, 1000, 6912, 41)       # decode GEMV, 16-token chunks
    f16_route("persistent", 1900, 2568, 1040, 51)          # persistent f16 GEMM
    fused_route("fused_prepass", 9, 2064, 8192, 61)        # fused path through the pre-pass (scratch memory)
    return routes


def test_concurrent_routes_match_their_solo_bits():
    bl.bitlinear_set_fused_prepass(0)  # every fused launch through the pre-pass and its scratch
    try:
        routes = make_routes()
        torch.cuda.synchronize()  # the inputs were made on torch's current stream
        solo = {}
        st0 = torch.cuda.Stream()
        for name, run in routes:
            o = run(st0)
            st0.synchronize()  # before the copy, which runs on torch's current stream
            solo[name] = o.clone()
        assert bl.bitlinear_check_status() == bl.OK
        for _ in range(3):
            streams = {name: torch.cuda.Stream() for name, _ in routes}
            outs, errors = {}, []

            def worker(name, run):
                try:
                    for _ in range(4):
                        o = run(streams[name])
                    outs[name] = o
                except Exception as e:  # reported below
                    errors.append((name, e))

            threads = [threading.Thread(target=worker, args=(n, r)) for n, r in routes]
            for t in threads:
                t.start()
            for t in threads:
                t.join()
            assert not errors, errors
            torch.cuda.synchronize()
            assert bl.bitlinear_check_status() == bl.OK
            for name, _ in routes:
                assert torch.equal(outs[name], solo[name]), name
    finally:
        bl.bitlinear_set_fused_prepass(-1)
