"""The chunk-parallel use of the oracle that the full-size GPU parity tests
compare against gives exactly the single-call oracle's stream (Section III-A
"Stream format": chunks are coded on their own; all sizes come first, then
all payloads)."""
import numpy as np
import pytest

import oracle
from lossless_bit_plane_gb300 import workloads as W
from tests import oracle_parallel


@pytest.mark.parametrize("ew", [4, 2])
@pytest.mark.parametrize("threads", [1, 2, 3, 8])
def test_parallel_oracle_equals_the_single_call(ew, threads):
    rng = np.random.default_rng(17)
    data = np.concatenate([
        W.relu_values(4096 * 5 + 333, rng).view(np.uint8), rng.integers(0, 256, 4096 * 2 + 5, dtype=np.uint8),
        np.zeros(4096 + 64, np.uint8), W.f32_to_bf16_rne(W.gelu_values(4096 * 3 + 11, rng)).view(np.uint8)])
    want = oracle.compress(data, ew)
    for cand in (oracle.CAND_ALL, 0x1 | 0x10, 0x2 | 0x10):
        want = oracle.compress(data, ew, cand)
        assert oracle_parallel.compress(data, ew, cand, threads=threads) == want


def test_parallel_oracle_on_tiny_and_empty_inputs():
    for n in (0, 1, 4095, 4096, 4097):
        data = np.arange(n, dtype=np.uint32).astype(np.uint8)
        assert oracle_parallel.compress(data, 4, threads=4) == oracle.compress(data, 4)
