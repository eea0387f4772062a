"""CPU oracle of the PlaneZip block codec (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product library under
``lossless_bit_plane_gb300/`` never imports, links or calls it.

The codec itself is plain C in ``pz_oracle.c`` (single-threaded, one bit at a
time). This module compiles it with gcc and wraps it with ctypes: argument
marshalling only.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "pz_oracle.c"
_LIB = _HERE / "libpzoracle.so"

OK, ERR_ARG, ERR_CAPACITY, ERR_CORRUPT = 0, 1, 2, 3
TAG_ZVC, TAG_DBX, TAG_BX, TAG_ZBX, TAG_RAW = 0, 1, 2, 3, 4
TAG_NAMES = ("ZVC", "DBX", "BX", "ZBX", "RAW")
CAND_ALL = 0x1F  # candidate mask: bit t = tag t; the raw block is always allowed

_lib = None


def build(force: bool = False) -> Path:
    """Compile the oracle into ``oracle/libpzoracle.so`` (plain -O2, no SIMD flags)."""
    deps = [_SRC, _HERE / "pz_oracle.h"]
    if not force and _LIB.exists() and all(_LIB.stat().st_mtime >= d.stat().st_mtime for d in deps):
        return _LIB
    tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
    subprocess.check_call(
        ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-shared", "-fPIC", "-o", str(tmp), str(_SRC)]
    )
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(str(_LIB))
        sz, u8p, i32p = ctypes.c_size_t, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)
        L.pzo_max_stream_bytes.argtypes = [sz]
        L.pzo_max_stream_bytes.restype = sz
        L.pzo_compress.argtypes = [u8p, sz, ctypes.c_int, u8p, sz, ctypes.POINTER(sz)]
        L.pzo_compress.restype = ctypes.c_int
        L.pzo_decompress.argtypes = [u8p, sz, ctypes.c_int, u8p, sz]
        L.pzo_decompress.restype = ctypes.c_int
        L.pzo_block_candidates.argtypes = [u8p, ctypes.c_int, i32p, i32p, i32p]
        L.pzo_block_candidates.restype = ctypes.c_int
        L.pzo_encode_candidate.argtypes = [u8p, ctypes.c_int, ctypes.c_int, u8p, sz]
        L.pzo_encode_candidate.restype = ctypes.c_int
        L.pzo_analyze.argtypes = [u8p, sz, ctypes.c_int, u8p, u8p, u8p]
        L.pzo_analyze.restype = ctypes.c_int
        L.pzo_compress_candidates.argtypes = [u8p, sz, ctypes.c_int, ctypes.c_uint, u8p, sz, ctypes.POINTER(sz)]
        L.pzo_compress_candidates.restype = ctypes.c_int
        L.pzo_analyze_candidates.argtypes = [u8p, sz, ctypes.c_int, ctypes.c_uint, u8p, u8p, u8p]
        L.pzo_analyze_candidates.restype = ctypes.c_int
        _lib = L
    return _lib


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(np.frombuffer(bytes(a), dtype=np.uint8) if isinstance(a, (bytes, bytearray)) else np.asarray(a).view(np.uint8).reshape(-1))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a.size else None


def max_stream_bytes(nbytes: int) -> int:
    return int(lib().pzo_max_stream_bytes(nbytes))


def compress(data, elem_width: int, candidates: int = CAND_ALL) -> bytes:
    """Compress a byte buffer (bytes or numpy array); returns the stream.
    ``candidates`` restricts block selection (bit t = tag t; raw always)."""
    src = _u8(data)
    cap = max_stream_bytes(src.size)
    out = np.zeros(max(cap, 1), dtype=np.uint8)
    total = ctypes.c_size_t(0)
    rc = lib().pzo_compress_candidates(_ptr(src), src.size, elem_width, candidates, _ptr(out), cap,
                                       ctypes.byref(total))
    if rc != OK:
        raise RuntimeError(f"pzo_compress failed with status {rc}")
    return out[: total.value].tobytes()


def decompress_status(stream, nbytes: int, elem_width: int):
    src = _u8(stream)
    out = np.zeros(max(nbytes, 1), dtype=np.uint8)
    rc = lib().pzo_decompress(_ptr(src), src.size, elem_width, _ptr(out), nbytes)
    return rc, out[:nbytes].tobytes()


def decompress(stream, nbytes: int, elem_width: int) -> bytes:
    rc, out = decompress_status(stream, nbytes, elem_width)
    if rc != OK:
        raise RuntimeError(f"pzo_decompress failed with status {rc}")
    return out


def block_candidates(block, elem_width: int):
    """(encoder bits[5], size-model bits[5], chosen tag) for one 128-byte block."""
    b = _u8(block)
    assert b.size == 128
    enc = (ctypes.c_int * 5)()
    mod = (ctypes.c_int * 5)()
    tag = ctypes.c_int(-1)
    rc = lib().pzo_block_candidates(_ptr(b), elem_width, enc, mod, ctypes.byref(tag))
    assert rc == OK
    return list(enc), list(mod), tag.value


def encode_candidate(block, elem_width: int, tag: int) -> tuple[int, bytes]:
    """Bit-exact payload of one candidate (no tag): (bit count, bytes)."""
    b = _u8(block)
    buf = np.zeros(512, dtype=np.uint8)
    n = lib().pzo_encode_candidate(_ptr(b), elem_width, tag, _ptr(buf), buf.size)
    assert n >= 0
    return n, buf[: (n + 7) // 8].tobytes()


def analyze(data, elem_width: int, candidates: int = CAND_ALL):
    """Per-block tags and bit counts and per-chunk L for a whole buffer."""
    src = _u8(data)
    nb = (src.size + 127) // 128
    nc = (src.size + 4095) // 4096
    tags = np.zeros(max(nc * 32, 1), dtype=np.uint8)
    bits = np.zeros(max(nc * 32, 1), dtype=np.uint16)
    lens = np.zeros(max(nc, 1), dtype=np.uint16)
    rc = lib().pzo_analyze_candidates(_ptr(src), src.size, elem_width, candidates, _ptr(tags), _ptr(bits),
                                      _ptr(lens))
    assert rc == OK
    return tags[:nb], bits[:nb], lens[:nc]
