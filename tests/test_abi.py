"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
entry point that the headers under include/ declare, and rejects bad arguments on
the host before touching the device."""
import re
from pathlib import Path

import pytest

from lossless_bit_plane_gb300 import _lib, build

INCLUDE = Path(__file__).resolve().parents[1] / "include"
HEADERS = sorted(INCLUDE.glob("*.h"))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        names |= set(re.findall(r"\b(pz_\w+)\s*\(", text))
    return sorted(names)


def test_test_hooks_stay_out_of_the_codec_header():
    text = re.sub(r"/\*.*?\*/", "", (INCLUDE / "planezip.h").read_text(), flags=re.S)
    assert "pz_test_" not in text
    assert [h.name for h in HEADERS] == ["planezip.h", "planezip_testing.h"]


def test_header_declares_every_entry_point():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_max_compressed_bytes_closed_form(lib):
    for n in (0, 1, 127, 128, 4095, 4096, 4097, 12845056, 1 << 30):
        C = (n + 4095) // 4096
        assert _lib.pz_max_compressed_bytes(n) == ((2 * C + n + 15) // 16) * 16 + 8 * C + 64


FAKE_IN, FAKE_OUT, FAKE_WORD = 0x100000, 0x200000, 0x300000  # never dereferenced


def test_compress_argument_errors_are_host_side(lib):
    n = 8192
    cap = _lib.pz_max_compressed_bytes(n)
    assert _lib.pz_compress(FAKE_IN, n, 0, FAKE_OUT, cap, FAKE_WORD) == _lib.PZ_ERR_ARG
    assert _lib.pz_compress(FAKE_IN, n, -4, FAKE_OUT, cap, FAKE_WORD) == _lib.PZ_ERR_ARG
    assert _lib.pz_compress(FAKE_IN, n, 4, FAKE_OUT, cap, 0) == _lib.PZ_ERR_ARG
    assert _lib.pz_compress(0, n, 4, FAKE_OUT, cap, FAKE_WORD) == _lib.PZ_ERR_ARG
    assert _lib.pz_compress(FAKE_IN, n, 4, 0, cap, FAKE_WORD) == _lib.PZ_ERR_ARG
    assert _lib.pz_compress(FAKE_IN + 4, n, 4, FAKE_OUT, cap, FAKE_WORD) == _lib.PZ_ERR_ARG
    assert _lib.pz_compress(FAKE_IN, n, 4, FAKE_OUT + 8, cap, FAKE_WORD) == _lib.PZ_ERR_ARG
    assert _lib.pz_compress(FAKE_IN, n, 4, FAKE_OUT, cap - 1, FAKE_WORD) == _lib.PZ_ERR_CAPACITY


def test_candidates_and_size_argument_errors_are_host_side(lib):
    n = 8192
    cap = _lib.pz_max_compressed_bytes(n)
    # mask bits outside PZ_CAND_ALL
    assert _lib.pz_compress_candidates(FAKE_IN, n, 4, 0x20, FAKE_OUT, cap, FAKE_WORD) == _lib.PZ_ERR_ARG
    assert _lib.pz_compress_candidates(FAKE_IN, n, 0, _lib.PZ_CAND_ZVC, FAKE_OUT, cap, FAKE_WORD) == _lib.PZ_ERR_ARG
    assert _lib.pz_compress_candidates(FAKE_IN, n, 4, _lib.PZ_CAND_DBX, FAKE_OUT, cap - 1,
                                       FAKE_WORD) == _lib.PZ_ERR_CAPACITY
    size = _lib.pz_compressed_size
    assert size(FAKE_IN, n, 4, _lib.PZ_CAND_ALL, 0, 0, FAKE_WORD) == _lib.PZ_ERR_ARG      # stride 0
    assert size(FAKE_IN, n, 4, _lib.PZ_CAND_ALL, 1, 0, 0) == _lib.PZ_ERR_ARG              # no total
    assert size(FAKE_IN, n, 0, _lib.PZ_CAND_ALL, 1, 0, FAKE_WORD) == _lib.PZ_ERR_ARG      # width
    assert size(FAKE_IN, n, 4, 0x40, 1, 0, FAKE_WORD) == _lib.PZ_ERR_ARG                  # mask
    assert size(0, n, 4, _lib.PZ_CAND_ALL, 1, 0, FAKE_WORD) == _lib.PZ_ERR_ARG            # no input
    assert size(FAKE_IN + 4, n, 4, _lib.PZ_CAND_ALL, 1, 0, FAKE_WORD) == _lib.PZ_ERR_ARG  # misaligned


def piece_schedule(n, P):
    """The documented piece schedule: a first piece of half of P (rounded
    down to 4096, at least 4096), then pieces of P, the last possibly
    shorter."""
    out, rem, s = [], n, max(4096, (P // 2) // 4096 * 4096)
    while rem:
        out.append(min(s, rem))
        rem -= out[-1]
        s = P
    return out


def test_piece_schedule_examples():
    M = 1 << 20
    assert piece_schedule(128 * M, 64 * M) == [32 * M, 64 * M, 32 * M]
    assert piece_schedule(10 * M, 64 * M) == [10 * M]
    assert piece_schedule(3 << 20, 1 << 20) == [M // 2, M, M, M // 2]
    assert piece_schedule(12288, 4096) == [4096] * 3
    assert sum(piece_schedule(300_001, 65536)) == 300_001


def test_swap_sizes_closed_forms(lib):
    assert _lib.pz_swap_work_bytes(0) == 0 and _lib.pz_swap_work_bytes(4097) == 0
    for piece in (4096, 1 << 20, 16 << 20):
        stage = (_lib.pz_max_compressed_bytes(piece) + 15) // 16 * 16
        assert _lib.pz_swap_work_bytes(piece) == 2 * stage + 32
    for n, piece in ((0, 4096), (1, 4096), (4096, 4096), (4097, 4096), (10 << 20, 1 << 20), (3 << 20, 2 << 20),
                     (128 << 20, 32 << 20), (300_001, 65536), (10 << 20, 64 << 20)):
        sizes = piece_schedule(n, piece)
        # the head and table, then every piece at a 128-byte boundary
        cap = (32 + 16 * len(sizes) + 127) // 128 * 128 + sum((r + 127) // 128 * 128 for r in sizes)
        assert _lib.pz_swap_capacity(n, piece) == cap


def test_swap_argument_and_container_errors_are_host_side(lib):
    import ctypes
    import struct

    piece, n = 1 << 20, 3 << 20
    work = _lib.pz_swap_work_bytes(piece)
    host = ctypes.create_string_buffer(_lib.pz_swap_capacity(n, piece))
    h = ctypes.addressof(host)
    cap = len(host)
    assert _lib.pz_swap_out(FAKE_IN, n, 4, 4095, FAKE_OUT, work, h, cap)[0] == _lib.PZ_ERR_ARG
    assert _lib.pz_swap_out(FAKE_IN, n, 0, piece, FAKE_OUT, work, h, cap)[0] == _lib.PZ_ERR_ARG
    assert _lib.pz_swap_out(FAKE_IN + 4, n, 4, piece, FAKE_OUT, work, h, cap)[0] == _lib.PZ_ERR_ARG
    assert _lib.pz_swap_out(FAKE_IN, n, 4, piece, FAKE_OUT, work - 1, h, cap)[0] == _lib.PZ_ERR_CAPACITY
    assert _lib.pz_swap_out(FAKE_IN, n, 4, piece, FAKE_OUT, work, h, cap - 1)[0] == _lib.PZ_ERR_CAPACITY
    # an empty tensor needs no device at all: the container is its head
    rc, total = _lib.pz_swap_out(0, 0, 4, piece, 0, 0, h, cap)
    assert rc == _lib.PZ_OK and total == 128  # the head, rounded up to the pieces' 128-byte boundary
    assert struct.unpack_from("<IIQQII", host.raw, 0) == (0x33535A50, 0, 0, piece, 4, 0)
    # swap-in rejects a container that does not match, before any device work:
    # a well-formed container of three 1 MiB pieces, each a 1 KB stream
    head = struct.pack("<IIQQII", 0x33535A50, 3, n, piece, 4, 0) + struct.pack("<6Q", piece, 1024, piece, 1024,
                                                                               piece, 1024)
    ctypes.memmove(h, head, len(head))
    ok_len = 128 + 3 * 1024  # pieces from the table's end rounded up to 128
    assert _lib.pz_swap_in(h, ok_len, FAKE_OUT, work, FAKE_IN, n + 1, FAKE_WORD) == _lib.PZ_ERR_ARG   # nbytes
    assert _lib.pz_swap_in(h, 40, FAKE_OUT, work, FAKE_IN, n, FAKE_WORD) == _lib.PZ_ERR_ARG          # truncated
    bad = struct.pack("<IIQQII", 0x57535A50, 3, n, piece, 4, 0)
    ctypes.memmove(h, bad, len(bad))
    assert _lib.pz_swap_in(h, ok_len, FAKE_OUT, work, FAKE_IN, n, FAKE_WORD) == _lib.PZ_ERR_ARG      # magic
    ctypes.memmove(h, head, len(head))
    for entry in ((piece, 1 << 40), (piece, 511), (piece, piece), (piece + 4096, 1024), (0, 1024),
                  (piece, (1 << 63) | 1024), (piece - 4096, 1024)):
        ctypes.memmove(h + 32, struct.pack("<2Q", *entry), 16)                         # bad lengths or sizes
        assert _lib.pz_swap_in(h, ok_len, FAKE_OUT, work, FAKE_IN, n, FAKE_WORD) == _lib.PZ_ERR_ARG, entry
    ctypes.memmove(h + 32, struct.pack("<2Q", piece, 1024), 16)
    assert _lib.pz_swap_in(h, ok_len - 1, FAKE_OUT, work, FAKE_IN, n, FAKE_WORD) == _lib.PZ_ERR_ARG  # past the end
    assert _lib.pz_swap_in(h, ok_len, FAKE_OUT, work - 1, FAKE_IN, n, FAKE_WORD) == _lib.PZ_ERR_CAPACITY


def test_pool_layout_and_host_side_errors(lib):
    import ctypes

    S = 1 << 20
    assert _lib.pz_pool_bytes(S, 0) == 0 and _lib.pz_pool_bytes(4095, 4) == 0
    # the head (40 bytes of fields and a mutex) and 4-byte slot links, then the
    # slots from a 4096-byte boundary
    assert _lib.pz_pool_bytes(S, 3) == 4096 + 3 * S
    assert _lib.pz_pool_bytes(S, 1024) == 8192 + 1024 * S
    mem = ctypes.create_string_buffer(_lib.pz_pool_bytes(65536, 5) + 64)
    base = (ctypes.addressof(mem) + 63) // 64 * 64
    assert _lib.pz_pool_init(base + 8, len(mem) - 64, 65536)[0] == _lib.PZ_ERR_ARG       # alignment
    assert _lib.pz_pool_init(base, 4096 + 65535, 65536)[0] == _lib.PZ_ERR_CAPACITY        # no slot fits
    rc, pool = _lib.pz_pool_init(base, len(mem) - 64, 65536)
    assert rc == _lib.PZ_OK and pool == base
    assert _lib.pz_pool_free_slots(pool) == 5
    assert _lib.pz_pool_release(pool, 5) == _lib.PZ_ERR_ARG                               # no such slot
    assert _lib.pz_pool_swap_out(pool, FAKE_IN, 4096, 0, 65536, FAKE_OUT, 1 << 30)[0] == _lib.PZ_ERR_ARG
    assert _lib.pz_pool_swap_in(pool, 7, FAKE_OUT, 1 << 30, FAKE_IN, 4096, FAKE_WORD) == _lib.PZ_ERR_ARG
    # an empty tensor takes one slot (its head) and gives it back
    rc, t, stored = _lib.pz_pool_swap_out(pool, 0, 0, 4, 65536, 0, 0)
    assert rc == _lib.PZ_OK and stored == 128 and _lib.pz_pool_free_slots(pool) == 4
    assert _lib.pz_pool_release(pool, t) == _lib.PZ_OK and _lib.pz_pool_free_slots(pool) == 5
    assert _lib.pz_pool_release(pool, t) == _lib.PZ_ERR_ARG and _lib.pz_pool_free_slots(pool) == 5  # twice
    ts = [_lib.pz_pool_swap_out(pool, 0, 0, 2, 65536, 0, 0)[1] for _ in range(5)]
    assert sorted(ts) == list(range(5)) and _lib.pz_pool_free_slots(pool) == 0
    assert _lib.pz_pool_swap_out(pool, 0, 0, 2, 65536, 0, 0)[0] == _lib.PZ_ERR_CAPACITY  # no slot left
    for t in ts:
        assert _lib.pz_pool_release(pool, t) == _lib.PZ_OK
    assert _lib.pz_pool_free_slots(pool) == 5


def test_timeout_hook_argument_errors_are_host_side(lib):
    cap = _lib.pz_max_compressed_bytes(4096)
    assert _lib.pz_test_lookback_timeout(FAKE_IN, 4096, 4, FAKE_OUT, cap, FAKE_WORD) == _lib.PZ_ERR_ARG  # 1 chunk
    n = 4097 * 4096
    assert _lib.pz_test_lookback_timeout(FAKE_IN, n, 4, FAKE_OUT, _lib.pz_max_compressed_bytes(n),
                                         FAKE_WORD) == _lib.PZ_ERR_ARG  # over 4096 chunks
    n = 8192
    assert _lib.pz_test_lookback_timeout(FAKE_IN, n, 4, FAKE_OUT, _lib.pz_max_compressed_bytes(n) - 1,
                                         FAKE_WORD) == _lib.PZ_ERR_CAPACITY


def test_decompress_argument_errors_are_host_side(lib):
    n = 3 * 4096 + 5  # 4 chunks -> the stream has at least 8 bytes
    assert _lib.pz_decompress(FAKE_IN, 100, 0, FAKE_OUT, n, FAKE_WORD) == _lib.PZ_ERR_ARG
    assert _lib.pz_decompress(FAKE_IN, 100, 4, FAKE_OUT, n, 0) == _lib.PZ_ERR_ARG
    assert _lib.pz_decompress(FAKE_IN, 7, 4, FAKE_OUT, n, FAKE_WORD) == _lib.PZ_ERR_ARG
    assert _lib.pz_decompress(FAKE_IN + 2, 100, 4, FAKE_OUT, n, FAKE_WORD) == _lib.PZ_ERR_ARG
    assert _lib.pz_decompress(FAKE_IN, 100, 4, FAKE_OUT + 1, n, FAKE_WORD) == _lib.PZ_ERR_ARG
    assert _lib.pz_decompress(0, 100, 4, FAKE_OUT, n, FAKE_WORD) == _lib.PZ_ERR_ARG


def test_product_package_never_imports_the_oracle():
    pkg = Path(_lib.__file__).resolve().parent
    for f in list(pkg.rglob("*.py")) + list(pkg.rglob("*.cu")) + list(pkg.rglob("*.cuh")) + list(pkg.rglob("*.h")):
        text = f.read_text()
        assert "import oracle" not in text and "from oracle" not in text and "pz_oracle" not in text, f
