"""The device-side weight generator (bitlinear_02_b300.inputs.ternary_hash,
torch int64 arithmetic) against the oracle's own C version of the same
published generator, on the CPU.  The GPU copy is compared in
tests/test_gpu_stacks.py."""
import numpy as np
import pytest

import oracle
from bitlinear_02_b300 import inputs


@pytest.mark.parametrize("N,K,seed,layer,proj", [(300, 1040, 5, 79, 6), (64, 28672, 5, 0, 6),
                                                 (17, 16, 4, 25, 0), (1024, 8192, 5, 3, 1)])
def test_torch_generator_matches_oracle(N, K, seed, layer, proj):
    w = inputs.stack_word(seed, layer, proj)
    t = inputs.ternary_hash(N, K, w, rows_per_chunk=100).numpy()
    np.testing.assert_array_equal(t, oracle.ternary_hash(w, K, 0, N))


def test_stack_words_are_distinct():
    words = {inputs.stack_word(s, l, p) for s in (4, 5) for l in range(80) for p in range(7)}
    assert len(words) == 2 * 80 * 7
