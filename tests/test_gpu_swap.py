"""The compressed swap path through the C ABI (pz_swap_out / pz_swap_in and
the host slot pool pz_pool_*): a tensor leaves the device as PlaneZip
streams in pinned host memory and comes back bit-exact. Each coded piece of
the container must be exactly the oracle's stream of that piece's bytes
(Section III-A "Stream format"); a piece whose stream would not be shorter
than its bytes is stored raw (Section III-C, Equation 2: the engine is
bypassed when compression would not shorten the transfer); a malformed piece
must surface in the device status.
"""
import struct

import numpy as np
import pytest

import oracle
from lossless_bit_plane_gb300 import _lib, build
from lossless_bit_plane_gb300 import workloads as W
from tests.test_abi import piece_schedule

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

RAW_FLAG = 1 << 63


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    _lib.load()


def parse(container: bytes):
    magic, n, nbytes, piece, ew, zero = struct.unpack_from("<IIQQII", container, 0)
    assert magic == 0x33535A50 and zero == 0
    entries = struct.unpack_from(f"<{2 * n}Q", container, 32)
    off = (32 + 16 * n + 127) // 128 * 128  # pieces at 128-byte boundaries
    pieces = []
    for k in range(n):
        raw, stored = entries[2 * k], entries[2 * k + 1]
        L = stored & ~RAW_FLAG
        pieces.append((raw, bool(stored & RAW_FLAG), container[off: off + L]))
        off += (L + 127) // 128 * 128
    return nbytes, piece, ew, pieces, off


def check_pieces(raw_bytes: np.ndarray, ew: int, piece: int, pieces):
    assert [p[0] for p in pieces] == piece_schedule(raw_bytes.size, piece)
    at = 0
    for k, (n, is_raw, body) in enumerate(pieces):
        src = raw_bytes[at: at + n].tobytes()
        want = oracle.compress(src, ew)
        if is_raw:  # only where the stream would not be shorter than the bytes
            assert body == src and len(want) >= n, f"piece {k}"
        else:
            assert body == want and len(want) < n, f"piece {k}"
        at += n
    assert at == raw_bytes.size


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
    ("random_then_zeros", lambda: np.concatenate([np.random.default_rng(5).integers(0, 256, 200_000, dtype=np.uint8),
                                                  np.zeros(100_000, np.uint8)]), 4, 32 * 1024),
]


@pytest.mark.parametrize("name,make,ew,piece", CASES, ids=[c[0] for c in CASES])
def test_swap_round_trip_and_pieces_equal_the_oracle(name, make, ew, piece):
    raw, container = roundtrip(make(), ew, piece)
    nbytes, p, w, pieces, end = parse(container)
    assert (nbytes, p, w) == (raw.size, piece, ew)
    assert end == len(container)
    check_pieces(raw, ew, piece, pieces)


def test_swap_through_pageable_host_memory():
    # a pageable container: the pieces' lengths reach the host by copies
    # instead of the kernel stores used for pinned memory; same container,
    # same round trip
    arr = W.relu_values(200_000, np.random.default_rng(23))
    raw = arr.view(np.uint8)
    x = torch.from_numpy(raw.copy()).cuda()
    piece = 256 * 1024
    work_bytes = _lib.pz_swap_work_bytes(piece)
    work = torch.empty(work_bytes, dtype=torch.uint8, device="cuda")
    cap = _lib.pz_swap_capacity(raw.size, piece)
    host = np.zeros(cap + 128, dtype=np.uint8)  # pageable
    h = (host.ctypes.data + 127) // 128 * 128
    rc, length = _lib.pz_swap_out(x.data_ptr(), raw.size, 4, piece, work.data_ptr(), work_bytes, h, cap)
    assert rc == _lib.PZ_OK
    off = h - host.ctypes.data
    container = host[off: off + length].tobytes()
    _, _, _, pieces, end = parse(container)
    assert end == length
    check_pieces(raw, 4, piece, pieces)
    _, pinned_container = roundtrip(arr, 4, piece)
    assert container == pinned_container
    out = torch.empty_like(x)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _lib.pz_swap_in(h, length, work.data_ptr(), work_bytes, out.data_ptr(), raw.size, st.data_ptr()) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.equal(out, x)


def test_incompressible_tensor_is_moved_raw():
    rng = np.random.default_rng(7)
    raw, container = roundtrip(rng.integers(0, 256, 3 << 20, dtype=np.uint8), 4, 1 << 20)
    _, _, _, pieces, _ = parse(container)
    assert all(is_raw for _, is_raw, _ in pieces)
    check_pieces(raw, 4, 1 << 20, pieces)


def test_swap_64mib_attention_bf16_in_16mib_pieces():
    t = W.sweep_segment("attention", "bf16", seg_bytes=64 << 20)
    x = torch.from_numpy(t.data.view(np.uint8).reshape(-1)).cuda()
    bufs = _lib.SwapBuffers(x.numel(), 16 << 20)
    length = bufs.swap_out(x, 2)
    out = torch.empty_like(x)
    st = bufs.swap_in(length, out)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.equal(out, x)
    # each coded piece's length is the total pz_compress reports for that piece
    _, piece, _, pieces, _ = parse(bufs.host[:length].numpy().tobytes())
    at = 0
    for n, is_raw, s in pieces:
        assert not is_raw
        o, tot = _lib.compress_tensor(x[at: at + n], 2)
        torch.cuda.synchronize()
        assert len(s) == int(tot.item())
        at += n


def test_swap_in_reports_a_malformed_piece():
    arr = W.relu_values(40_000, np.random.default_rng(3))  # 160 KB: 3 pieces of at most 64 KB
    raw = arr.view(np.uint8)
    x = torch.from_numpy(raw.copy()).cuda()
    bufs = _lib.SwapBuffers(raw.size, 64 * 1024)
    length = bufs.swap_out(x, 4)
    _, _, _, pieces, _ = parse(bufs.host[:length].numpy().tobytes())
    n = len(pieces)
    assert n == 3 and not pieces[1][1]
    off = (32 + 16 * n + 127) // 128 * 128 + (len(pieces[0][2]) + 127) // 128 * 128  # piece 1's stream
    bufs.host[off: off + 2] = 0  # chunk 0 of piece 1 claims L = 0
    out = torch.empty_like(x)
    st = bufs.swap_in(length, out)
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.PZ_ERR_CORRUPT


def test_pool_round_trips_releases_and_runs_out():
    rng = np.random.default_rng(11)
    slot = 256 * 1024
    pool = _lib.SwapPool(16 * slot + 8192, slot_bytes=slot, piece_bytes=1 << 20)
    nslots = pool.free_slots()
    assert nslots == 16
    arrays = [(W.relu_values(700_000, rng).view(np.uint8), 4),                       # 2.8 MB, ~1.4 MB stored
              (W.f32_to_bf16_rne(W.gelu_values(300_001, rng)).view(np.uint8), 2),
              (rng.integers(0, 256, 100_000, dtype=np.uint8), 4)]                     # stored raw
    held = []
    for a, ew in arrays:
        x = torch.from_numpy(a.copy()).cuda()
        t, stored = pool.swap_out(x, ew)
        held.append((t, stored, x, a, ew))
    used = nslots - pool.free_slots()
    assert used == sum((s + slot - 1) // slot for _, s, _, _, _ in held)
    for t, stored, x, a, ew in held:
        # the container laid over the tensor's slot chain reads back as pieces
        # equal to the oracle's streams
        out = torch.empty_like(x)
        st = pool.swap_in(t, out)
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and torch.equal(out, x)
    for t, _, _, _, _ in held:
        pool.release(t)
    assert pool.free_slots() == nslots
    # a tensor larger than the pool: PZ_ERR_CAPACITY, every slot given back
    big = torch.from_numpy(rng.integers(0, 256, 8 << 20, dtype=np.uint8)).cuda()
    with pytest.raises(_lib.PlaneZipError) as e:
        pool.swap_out(big, 4)
    assert e.value.status == _lib.PZ_ERR_CAPACITY
    assert pool.free_slots() == nslots


def test_pool_container_spans_slots_and_equals_the_buffer_container():
    # small slots: pieces continue from one slot into the next; the pooled
    # container has the same length as the one-buffer container of the same
    # tensor (whose pieces equal the oracle's streams) and reads back exactly
    rng = np.random.default_rng(13)
    slot = 64 * 1024
    pool = _lib.SwapPool(64 * slot + 8192, slot_bytes=slot, piece_bytes=256 * 1024)
    a = W.relu_values(250_000, rng).view(np.uint8)  # 1 MB
    x = torch.from_numpy(a.copy()).cuda()
    t, stored = pool.swap_out(x, 4)
    assert stored > 4 * slot
    raw, container = roundtrip(a, 4, 256 * 1024)
    assert stored == len(container)
    check_pieces(raw, 4, 256 * 1024, parse(container)[3])
    out = torch.empty_like(x)
    st = pool.swap_in(t, out)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.equal(out, x)
    pool.release(t)
    assert pool.free_slots() == 64
