"""GPU parity of the two entry points that widen the codec, through the C ABI:

- pz_compress_candidates: block selection restricted to a candidate mask
  (the single-encoding comparisons of Section V-A, Fig. 3). Streams must be
  byte-identical to the oracle's restricted streams and decode back.
- pz_compressed_size: sizes only (Section III-B's profiling pass) and every
  s-th chunk (Section IV, "Tensor capture": every fourth 4 KB chunk). The
  sizes must equal the oracle's chunk headers and the total the sum of 2 + L.

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


from tests import oracle_parallel  # noqa: E402
from tests.gpu_util import chunk_table, gpu_decompress, to_device  # noqa: E402

MASKS = {
    "zvc": _lib.PZ_CAND_ZVC,
    "dbx": _lib.PZ_CAND_DBX,
    "bx": _lib.PZ_CAND_BX,
    "zbx": _lib.PZ_CAND_ZBX,
    "raw": _lib.PZ_CAND_RAW,
    "zvc+zbx": _lib.PZ_CAND_ZVC | _lib.PZ_CAND_ZBX,
    "all": _lib.PZ_CAND_ALL,
}


def survivors_every_count(ew: int, seed: int) -> np.ndarray:
    """Blocks with n non-zero symbols of random value for every n from 0 to
    the block's symbol count, twice each: restricted to ZBX (or DBX, BX) the
    verbatim plane codes then come in every plane width, and whole groups of
    four verbatim planes in every width (the encoder writes those in one
    step: as pairs of codes up to 31 bits, as five or nine words at 32 and
    64 bits, as four codes of up to 64 bits for BF16 ZBX)."""
    rng = np.random.default_rng(seed)
    nsym, dt = (32, np.uint32) if ew == 4 else (64, np.uint16)
    blocks = []
    for n in range(nsym + 1):
        for _ in range(2):
            b = np.zeros(nsym, dtype=dt)
            b[rng.choice(nsym, n, replace=False)] = rng.integers(1, 1 << (8 * ew), n, dtype=np.uint64).astype(dt)
            blocks.append(b)
    return np.concatenate(blocks)


def _data():
    rng = np.random.default_rng(21)
    relu = W.relu_values(3 * 32768 + 1000, rng)                            # ~388 KB FP32, ragged tail
    conv = W.f32_to_bf16_rne(W.conv_fields(2, 56, 56, np.array([0.5, 3.0]), rng)).reshape(-1)
    att = W.f32_to_bf16_rne(W.causal_softmax_rows(1, 256, rng)).reshape(-1)  # 128 KB BF16
    return [
        ("edge_fp32", W.edge_blocks_fp32(), 4),
        ("edge_fp32_as16", W.edge_blocks_fp32(), 2),
        ("edge_bf16", W.edge_blocks_bf16(), 2),
        ("relu_fp32", relu, 4),
        ("conv_bf16", conv, 2),
        ("attention_bf16", att, 2),
        ("tiny_bf16", W.tiny_alphabet_blocks(256, "bf16"), 2),
        ("survivors_fp32", survivors_every_count(4, 31), 4),
        ("survivors_bf16", survivors_every_count(2, 32), 2),
    ]


DATA = _data()


def gpu_compress_candidates(data: bytes, ew: int, mask: int) -> bytes:
    x = to_device(data)
    out, total = _lib.compress_tensor(x, ew, candidates=mask)
    torch.cuda.synchronize()
    return out[: int(total.item())].cpu().numpy().tobytes()


@pytest.mark.parametrize("mask_name", list(MASKS))
@pytest.mark.parametrize("name,arr,ew", DATA, ids=[d[0] for d in DATA])
def test_restricted_streams_match_the_oracle(name, arr, ew, mask_name):
    data = np.ascontiguousarray(arr).view(np.uint8).reshape(-1).tobytes()
    mask = MASKS[mask_name]
    got = gpu_compress_candidates(data, ew, mask)
    want = oracle.compress(data, ew, mask | (1 << oracle.TAG_RAW))
    assert len(got) == len(want)
    assert got == want
    st, back = gpu_decompress(got, len(data), ew)
    assert st == _lib.PZ_OK and back == data


def gpu_sizes(data: bytes, ew: int, stride: int, mask: int = _lib.PZ_CAND_ALL, with_sizes: bool = True):
    x = to_device(data)
    sizes, total = _lib.compressed_size_tensor(x, ew, stride, mask, with_sizes)
    torch.cuda.synchronize()
    return (sizes.cpu().numpy().astype(np.int64) if sizes is not None else None), int(total.item())


@pytest.mark.parametrize("stride", [1, 3, 4])
@pytest.mark.parametrize("mask_name", ["all", "zvc", "dbx"])
@pytest.mark.parametrize("name,arr,ew", DATA, ids=[d[0] for d in DATA])
def test_sizes_equal_the_oracle_headers(name, arr, ew, mask_name, stride):
    data = np.ascontiguousarray(arr).view(np.uint8).reshape(-1).tobytes()
    mask = MASKS[mask_name]
    stream = oracle.compress(data, ew, mask | (1 << oracle.TAG_RAW))
    lens, _ = chunk_table(stream, len(data))
    want = lens[::stride]
    sizes, total = gpu_sizes(data, ew, stride, mask)
    assert sizes.tolist() == want.tolist()
    assert total == int((2 + want).sum())
    if stride == 1:
        assert total == len(stream)  # the stream length pz_compress reports
    _, total_only = gpu_sizes(data, ew, stride, mask, with_sizes=False)
    assert total_only == total


def test_sizes_of_an_empty_input_and_a_stride_past_the_end():
    x = torch.empty(16, dtype=torch.uint8, device="cuda")
    total = torch.full((1,), 7, dtype=torch.int64, device="cuda")
    rc = _lib.pz_compressed_size(x.data_ptr(), 0, 4, _lib.PZ_CAND_ALL, 1, 0, total.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == _lib.PZ_OK and int(total.item()) == 0
    data = W.relu_values(5000, np.random.default_rng(2)).view(np.uint8).tobytes()  # 5 chunks
    sizes, total = gpu_sizes(data, 4, 1000)
    want = oracle.compress(data[:4096], 4)
    assert sizes.tolist() == [int.from_bytes(want[:2], "little")]
    assert total == len(want)


def test_sampled_sizes_at_full_size_attention_bf16_192mib():
    # the 192 MiB causal-attention tensor: every fourth chunk, as the paper
    # samples tensors above 32 MB. Every sampled size equals the oracle's
    # header of that chunk (the oracle's whole stream, computed chunk-parallel
    # on the host) and the header of the full GPU stream.
    t = W.attention_bf16()
    x = torch.from_numpy(t.data.view(np.uint8).reshape(-1)).cuda()
    sizes, total = _lib.compressed_size_tensor(x, 2, 4)
    out, full_total = _lib.compress_tensor(x, 2)
    torch.cuda.synchronize()
    C = (x.numel() + 4095) // 4096
    headers = out[: 2 * C].cpu().numpy().view("<u2").astype(np.int64)
    want = np.frombuffer(oracle_parallel.compress(t.data, 2)[: 2 * C], "<u2").astype(np.int64)
    s = sizes.cpu().numpy().astype(np.int64)
    assert s.tolist() == want[::4].tolist()
    assert headers.tolist() == want.tolist()
    assert int(total.item()) == int((2 + want[::4]).sum())
    # the sampled ratio estimate tracks the exact ratio
    sampled_raw = 4096 * s.size
    est, exact = sampled_raw / int(total.item()), x.numel() / int(full_total.item())
    assert abs(est / exact - 1) < 0.02
