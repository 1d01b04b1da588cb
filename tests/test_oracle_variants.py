"""Pins of the oracle's two variant formats (no GPU).

Five ternary digits per byte (vi.news.hada.io topic 20406, the Hacker News
comments on ternary packing: 3^5 = 243 <= 256, so a b1.58 weight needs
log2(3) = 1.585 bits): byte values worked out by hand, the bijection onto 243
byte values, the digit-by-multiplication property of the scaled encoding,
the index formula on hand cases, and round trips.

The original binary BitNet (lumen-it.ai BitNet article: signum weights,
absmax activations, group quantisation): binarisation and group scales on
hand values, the bit index formula on hand cases, round trips, and the
grouped rescale against the single-scale one.
"""
import itertools
import math

import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module", autouse=True)
def _build():
    oracle.build()


# ------------------------------------------------------ five per byte ---

def test_encode5_hand_values():
    # v = 2*81 + 1*27 + 0*9 + 1*3 + 2 = 194; 256 * 194 / 243 = 204.378 -> 205
    assert oracle.encode5([2, 1, 0, 1, 2]) == 205
    # v = 0 -> 0;  v = 242 -> 254.95 -> 255;  v = 121 (all zero weights) -> 127.47 -> 128
    assert oracle.encode5([0, 0, 0, 0, 0]) == 0
    assert oracle.encode5([2, 2, 2, 2, 2]) == 255
    assert oracle.encode5([1, 1, 1, 1, 1]) == 128
    # most significant digit first: (1,0,0,0,0) is v = 81 -> 85.33 -> 86, (0,0,0,0,1) is v = 1 -> 1.05 -> 2
    assert oracle.encode5([1, 0, 0, 0, 0]) == 86
    assert oracle.encode5([0, 0, 0, 0, 1]) == 2


def test_encode5_is_a_bijection_onto_243_bytes():
    seen = {}
    for e in itertools.product(range(3), repeat=5):
        b = oracle.encode5(list(e))
        assert 0 <= b <= 255
        assert b not in seen
        seen[b] = e
        assert list(oracle.decode5(b)) == list(e)
    assert len(seen) == 243
    others = [b for b in range(256) if b not in seen]
    assert len(others) == 13
    assert all(oracle.decode5(b) is None for b in others)


def test_scaled_encoding_gives_digits_by_multiplying_by_three():
    # b = ceil(256 v / 243): multiplying by 3 and taking the byte above the
    # low eight bits yields the digits from the most significant one.
    for e in itertools.product(range(3), repeat=5):
        x = oracle.encode5(list(e))
        got = []
        for _ in range(5):
            x *= 3
            got.append(x >> 8)
            x &= 255
        assert tuple(got) == e


def test_position5_hand_cases():
    K = 320
    assert oracle.position5(0, 0, K) == (0, 0)
    assert oracle.position5(0, 4, K) == (0, 4)       # fifth digit of the first byte
    assert oracle.position5(0, 5, K) == (1, 0)       # next byte of the same row
    assert oracle.position5(0, 39, K) == (7, 4)      # last byte of lane 0, row g
    assert oracle.position5(0, 40, K) == (16, 0)     # t = 1: lane 1
    assert oracle.position5(8, 0, K) == (8, 0)       # row g + 8: second half of the lane's 16 bytes
    assert oracle.position5(1, 0, K) == (64, 0)      # g = 1: lane 4
    assert oracle.position5(0, 160, K) == (512, 0)   # next 160-k tile
    assert oracle.position5(16, 0, K) == (1024, 0)   # next row group: KT5 = 2 tiles later


@pytest.mark.parametrize("N,K", [(16, 160), (17, 336), (48, 1000), (3, 16)])
def test_pack5_round_trip(N, K):
    rng = np.random.default_rng(N * 1000 + K)
    wq = rng.integers(-1, 2, (N, K), dtype=np.int8)
    p = oracle.pack5(wq)
    assert p.size == oracle.packed5_bytes(N, K)
    back, bad = oracle.unpack5(p, N, K)
    assert bad == 0
    np.testing.assert_array_equal(back, wq)


def test_pack5_padding_is_weight_zero_and_checked():
    N, K = 5, 170
    wq = -np.ones((N, K), dtype=np.int8)
    p = oracle.pack5(wq)
    # row 15 of the row group is padding: every byte of it encodes digits 1
    b, _ = oracle.position5(15, 0, K)
    assert p[b] == 128
    p2 = p.copy()
    p2[b] = oracle.encode5([1, 1, 0, 1, 1])  # a padding weight of -1
    assert oracle.unpack5(p2, N, K)[1] == 1
    p3 = p.copy()
    p3[0] = next(x for x in range(256) if oracle.decode5(x) is None)  # a byte that encodes nothing
    assert oracle.unpack5(p3, N, K)[1] == 1


def test_packed5_size_is_1_6_bits_per_weight():
    assert oracle.packed5_bytes(16, 160) == 512
    assert oracle.packed5_bytes(16, 160) * 8 / (16 * 160) == 1.6
    # 20 % fewer bytes than the 2-bit layout where both tile sizes divide K
    for K in (640, 1280, 2560):
        assert oracle.packed_bytes(2560, K) / oracle.packed5_bytes(2560, K) == 1.25
    assert math.log2(3) < 1.6 < 2


# ------------------------------------------------------- binary BitNet ---

def test_binarize_hand_values():
    w = np.array([0.5, -0.5, 0.0, -0.0, 1e-30, -1e-30, 3.0e38], dtype=np.float32)
    np.testing.assert_array_equal(oracle.binarize(w), [1, -1, -1, -1, 1, -1, 1])


def test_beta_hand_values_and_fsum():
    w = np.array([[1.0, -2.0], [3.0, -4.0]], dtype=np.float32)
    assert oracle.beta(w, 1)[0] == np.float32(2.5)
    np.testing.assert_array_equal(oracle.beta(w, 2), np.array([1.5, 3.5], dtype=np.float32))
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((64, 300)) * 0.02).astype(np.float32)
    b = oracle.beta(w, 4)
    for g in range(4):
        blk = w[16 * g:16 * (g + 1)]
        want = np.float32(math.fsum(abs(float(v)) for v in blk.ravel()) / blk.size)
        assert b[g] == want


def test_position1_hand_cases():
    K = 512
    assert oracle.position1(0, 0, K) == (0, 0)
    assert oracle.position1(0, 1, K) == (2, 0)      # h = 1: high 16-bit half
    assert oracle.position1(0, 2, K) == (0, 1)      # sb = 1: next bit position
    assert oracle.position1(0, 4, K) == (0, 2)      # s = 1: the next 16-k step
    assert oracle.position1(0, 31, K) == (3, 7)     # s = 7, sb = 1, h = 1: bit 31 of word 0
    assert oracle.position1(0, 32, K) == (8, 0)     # P = 1: word 2 (row g, second half)
    assert oracle.position1(8, 0, K) == (4, 0)      # row g + 8: word 1
    assert oracle.position1(0, 64, K) == (16, 0)    # t = 1: lane 1
    assert oracle.position1(1, 0, K) == (64, 0)     # g = 1: lane 4
    assert oracle.position1(0, 256, K) == (512, 0)  # next 256-k tile


@pytest.mark.parametrize("N,K", [(16, 256), (17, 272), (40, 1040), (1, 16)])
def test_pack1_round_trip(N, K):
    rng = np.random.default_rng(N + 7 * K)
    wb = np.where(rng.random((N, K)) < 0.5, 1, -1).astype(np.int8)
    p = oracle.pack1(wb)
    assert p.size == oracle.packed1_bytes(N, K) == (N + 15) // 16 * 16 * ((K + 255) // 256 * 256) // 8
    back, bad = oracle.unpack1(p, N, K)
    assert bad == 0
    np.testing.assert_array_equal(back, wb)
    # exactly the +1 weights are set bits
    assert int(np.unpackbits(p).sum()) == int((wb > 0).sum())


def test_binary_matmul_brute_force():
    rng = np.random.default_rng(11)
    wb = np.where(rng.random((5, 48)) < 0.5, 1, -1).astype(np.int8)
    q = rng.integers(-128, 128, (3, 48), dtype=np.int8)
    acc = oracle.matmul(q, wb)
    for m in range(3):
        for n in range(5):
            assert acc[m, n] == sum(int(q[m, k]) * int(wb[n, k]) for k in range(48))


def test_epilogue_groups():
    rng = np.random.default_rng(5)
    acc = rng.integers(-5000, 5000, (3, 32), dtype=np.int32)
    s = np.array([0.01, 0.02, 0.5], dtype=np.float32)
    one = oracle.epilogue_groups(acc, s, np.array([0.03], dtype=np.float32))
    np.testing.assert_array_equal(one, oracle.epilogue(acc, s, np.float32(0.03)))
    two = oracle.epilogue_groups(acc, s, np.array([0.03, 0.07], dtype=np.float32))
    np.testing.assert_array_equal(two[:, :16], oracle.epilogue(acc[:, :16], s, np.float32(0.03)))
    np.testing.assert_array_equal(two[:, 16:], oracle.epilogue(acc[:, 16:], s, np.float32(0.07)))
