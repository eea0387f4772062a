"""The compressed swap path through the C ABI (pz_swap_out / pz_swap_in):
a tensor leaves the device as PlaneZip streams in pinned host memory and
comes back bit-exact. Each piece of the container must be exactly the
oracle's stream of that piece's bytes (Section III-A "Stream format"), and a
malformed piece must surface in the device status.
"""
import struct

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


def parse(container: bytes):
    magic, n, nbytes, piece, ew, zero = struct.unpack_from("<IIQQII", container, 0)
    assert magic == 0x57535A50 and zero == 0
    lens = struct.unpack_from(f"<{n}Q", container, 32)
    off = (32 + 8 * n + 15) // 16 * 16
    pieces = []
    for L in lens:
        pieces.append(container[off: off + L])
        off += (L + 15) // 16 * 16
    return nbytes, piece, ew, pieces, off


def roundtrip(arr: np.ndarray, ew: int, piece: int):
    raw = np.ascontiguousarray(arr).view(np.uint8).reshape(-1)
    x = torch.from_numpy(raw.copy()).cuda()
    bufs = _lib.SwapBuffers(max(raw.size, 1), piece)
    length = bufs.swap_out(x, ew)
    container = bufs.host[:length].numpy().tobytes()
    out = torch.empty_like(x)
    st = bufs.swap_in(length, out)
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.PZ_OK
    assert torch.equal(out, x)
    return raw, container


CASES = [
    ("relu_fp32_ragged", lambda: W.relu_values(300_001, np.random.default_rng(1)), 4, 64 * 1024),
    ("conv_bf16", lambda: W.f32_to_bf16_rne(W.conv_fields(4, 56, 56, np.array([0.3, 1, 2, 4.0]),
                                                          np.random.default_rng(2))), 2, 16 * 1024),
    ("edge_fp32_one_piece", W.edge_blocks_fp32, 4, 1 << 20),
    ("edge_bf16", W.edge_blocks_bf16, 2, 4096),
]


@pytest.mark.parametrize("name,make,ew,piece", CASES, ids=[c[0] for c in CASES])
def test_swap_round_trip_and_pieces_equal_the_oracle(name, make, ew, piece):
    raw, container = roundtrip(make(), ew, piece)
    nbytes, p, w, pieces, end = parse(container)
    assert (nbytes, p, w) == (raw.size, piece, ew)
    assert len(pieces) == (raw.size + piece - 1) // piece
    assert end == len(container)
    for k, s in enumerate(pieces):
        want = oracle.compress(raw[k * piece: (k + 1) * piece].tobytes(), ew)
        assert s == want, f"piece {k}"


def test_swap_64mib_attention_bf16_in_16mib_pieces():
    t = W.sweep_segment("attention", "bf16", seg_bytes=64 << 20)
    x = torch.from_numpy(t.data.view(np.uint8).reshape(-1)).cuda()
    bufs = _lib.SwapBuffers(x.numel(), 16 << 20)
    length = bufs.swap_out(x, 2)
    out = torch.empty_like(x)
    st = bufs.swap_in(length, out)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.equal(out, x)
    # each piece's length is the total pz_compress reports for that piece
    _, piece, _, pieces, _ = parse(bufs.host[:length].numpy().tobytes())
    for k, s in enumerate(pieces):
        o, tot = _lib.compress_tensor(x[k * piece: (k + 1) * piece], 2)
        torch.cuda.synchronize()
        assert len(s) == int(tot.item())


def test_swap_in_reports_a_malformed_piece():
    arr = W.relu_values(40_000, np.random.default_rng(3))  # 160 KB: 3 pieces of 64 KB
    raw = arr.view(np.uint8)
    x = torch.from_numpy(raw.copy()).cuda()
    bufs = _lib.SwapBuffers(raw.size, 64 * 1024)
    length = bufs.swap_out(x, 4)
    _, _, _, pieces, _ = parse(bufs.host[:length].numpy().tobytes())
    n = len(pieces)
    off = (32 + 8 * n + 15) // 16 * 16 + (len(pieces[0]) + 15) // 16 * 16  # piece 1's stream
    bufs.host[off: off + 2] = 0  # chunk 0 of piece 1 claims L = 0
    out = torch.empty_like(x)
    st = bufs.swap_in(length, out)
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.PZ_ERR_CORRUPT
