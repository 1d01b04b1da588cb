"""The benchmark's algorithmic byte counts (the numerators of its GB/s and
roofline figures), checked against the sizes written out by hand."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SHAPES_2B = [("q", 2560, 2560), ("k", 2560, 2560), ("v", 2560, 2560), ("o", 2560, 2560),
             ("gate", 6912, 2560), ("up", 6912, 2560), ("down", 2560, 6912)]


def test_forward_bytes_are_packed_weights_plus_activations():
    # packed weights N*K/4 (padded to 16 rows, 128 k), int8 input M*K, scales 4M,
    # bf16 output 2MN, gamma 4
    assert bench.algo_bytes_forward(1, 2560, 2560) == 2560 * 2560 // 4 + 2560 + 4 + 2 * 2560 + 4
    assert bench.algo_bytes_forward(16, 6912, 2560) == 6912 * 2560 // 4 + 16 * 2560 + 64 + 2 * 16 * 6912 + 4
    # ragged: N = 100 pads to 112 rows, K = 272 pads to 384
    assert bench.algo_bytes_forward(3, 100, 272) == 112 * 384 // 4 + 3 * 272 + 12 + 2 * 3 * 100 + 4


def test_quant_bytes():
    assert bench.algo_bytes_quant(4, 2560) == 2 * 4 * 2560 + 4 * 2560 + 16


def test_layer_bytes_match_the_chain():
    # h0 = quant(x); q,k,v = f(h0); h1 = quant(v); o = f(h1); h2 = quant(o);
    # gate,up = f(h2); h3 = quant(up); down = f(h3)
    for M in (1, 4, 16):
        expect = (bench.algo_bytes_quant(M, 2560) * 3 + bench.algo_bytes_quant(M, 6912)
                  + sum(bench.algo_bytes_forward(M, N, K) for _, N, K in SHAPES_2B))
        assert bench.layer_bytes(M, SHAPES_2B) == expect
    # one 2B layer: 19.8 MB of packed weights dominate
    w = sum(N * K // 4 for _, N, K in SHAPES_2B)
    assert w == 4 * 2560 * 2560 // 4 + 3 * 6912 * 2560 // 4 == 19_824_640
    # M = 1: forwards 4 x (2560 + 4 + 2*2560 + 4) + 2 x (2560 + 4 + 2*6912 + 4) + (6912 + 4 + 2*2560 + 4),
    # quantisers 3 x (3*2560 + 4) + (3*6912 + 4)
    assert bench.layer_bytes(1, SHAPES_2B) - w == 30_752 + 32_784 + 12_040 + 23_052 + 20_740


def test_whole_job_value():
    # 3 replicas x 10 steps x 1 GB in 2 s of the slowest rank: 15 GB/s
    assert bench.job_value(1e9, 10, 3, 2000.0) == 15.0
