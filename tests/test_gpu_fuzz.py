"""Randomised parity through the C ABI: seeded inputs of random length (a
ragged tail in most cases), element width and candidate mask, each built
from a mix of the workload recipes (ReLU, GELU, conv fields, causal softmax
rows, layer-norm outputs, uniform bytes, a few-symbol alphabet, the edge
blocks) cut into random stretches, so that chunks and blocks mix kinds at
random boundaries. Every stream must equal the oracle's byte for byte
(Section III-A "Codec" and "Stream format") and decode back exactly.

Integer work: exact, no tolerance.
"""
import numpy as np
import pytest

import oracle
from lossless_bit_plane_gb300 import _lib, build
from lossless_bit_plane_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    _lib.load()


from tests.gpu_util import explain_mismatch, gpu_decompress, to_device  # noqa: E402


def _piece(rng, kind: str, nbytes: int, dtype: str) -> np.ndarray:
    """About nbytes of one recipe as raw bytes of the given dtype."""
    n32 = max(1, nbytes // 4)
    if kind == "relu":
        v = W.relu_values(n32, rng)
    elif kind == "gelu":
        v = W.gelu_values(n32, rng)
    elif kind == "conv":
        v = W.conv_fields(1, 32, 32, np.array([float(rng.uniform(0.1, 4))]), rng).reshape(-1)
    elif kind == "softmax":
        v = W.causal_softmax_rows(1, 64, rng).reshape(-1)
    elif kind == "layernorm":
        v = W.layernorm_values(max(1, n32 // 64), 64, rng).reshape(-1)
    elif kind == "uniform":
        return rng.integers(0, 256, nbytes, dtype=np.uint8)
    elif kind == "alphabet":
        return W.tiny_alphabet_blocks(max(1, nbytes // 128), dtype).view(np.uint8).reshape(-1)
    else:  # edge blocks
        e = W.edge_blocks_bf16() if dtype == "bf16" else W.edge_blocks_fp32()
        return np.ascontiguousarray(e).view(np.uint8).reshape(-1)
    v = np.asarray(v, dtype=np.float32).reshape(-1)
    return (W.f32_to_bf16_rne(v) if dtype == "bf16" else v).view(np.uint8).reshape(-1)


KINDS = ("relu", "gelu", "conv", "softmax", "layernorm", "uniform", "alphabet", "edge")
MASKS = (_lib.PZ_CAND_ALL, _lib.PZ_CAND_ALL, _lib.PZ_CAND_ZVC, _lib.PZ_CAND_DBX, _lib.PZ_CAND_BX, _lib.PZ_CAND_ZBX,
         _lib.PZ_CAND_ZVC | _lib.PZ_CAND_ZBX, _lib.PZ_CAND_DBX | _lib.PZ_CAND_BX)


def _case(seed: int):
    rng = np.random.default_rng(1000 + seed)
    dtype = "bf16" if rng.random() < 0.5 else "fp32"
    ew = 2 if dtype == "bf16" else 4
    if rng.random() < 0.2:  # BF16 bytes coded with 32-bit symbols, or FP32 bytes with 16-bit ones
        ew = 6 - ew
    target = int(rng.integers(1, 160_000))
    parts, size = [], 0
    while size < target:
        p = _piece(rng, KINDS[int(rng.integers(len(KINDS)))], int(rng.integers(64, 40_000)), dtype)
        cut = int(rng.integers(1, p.size + 1))
        parts.append(p[:cut])
        size += cut
    data = np.concatenate(parts)[:target]
    mask = MASKS[int(rng.integers(len(MASKS)))]
    return data.tobytes(), ew, mask


@pytest.mark.parametrize("seed", range(48))
def test_random_mixtures_equal_the_oracle(seed):
    data, ew, mask = _case(seed)
    x = to_device(data)
    out, total = _lib.compress_tensor(x, ew, candidates=mask)
    torch.cuda.synchronize()
    got = out[: int(total.item())].cpu().numpy().tobytes()
    want = oracle.compress(data, ew, mask | _lib.PZ_CAND_RAW)
    assert got == want, explain_mismatch(data, ew, got, want)
    st, back = gpu_decompress(got, len(data), ew)
    assert st == _lib.PZ_OK and back == data
