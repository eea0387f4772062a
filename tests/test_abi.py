"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
entry point that include/planezip.h declares, and rejects bad arguments on
the host before touching the device."""
import re
from pathlib import Path

import pytest

from lossless_bit_plane_gb300 import _lib, build

HEADER = Path(__file__).resolve().parents[1] / "include" / "planezip.h"


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(pz_\w+)\s*\(", text)))


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
