"""ctypes binding of ``libplanezip.so`` — argument marshalling only.

The functions mirror the C ABI in ``include/planezip.h`` one to one
(``pz_max_compressed_bytes``, ``pz_compress``, ``pz_decompress``,
``pz_compress_candidates``, ``pz_compressed_size``, the swap path ``pz_swap_*``, the
host slot pool ``pz_pool_*`` and ``pz_compress_noalloc``); every step
of the codec runs in the library's CUDA kernels. The ``*_tensor`` helpers
below use PyTorch only to allocate device memory and to name the current
stream. There is no fallback: if the library is missing or cannot be loaded,
these calls raise.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

LIB_PATH = Path(__file__).resolve().parent / "libplanezip.so"

PZ_OK, PZ_ERR_ARG, PZ_ERR_CAPACITY, PZ_ERR_CORRUPT, PZ_ERR_CUDA, PZ_ERR_TIMEOUT = range(6)
STATUS_NAMES = {0: "PZ_OK", 1: "PZ_ERR_ARG", 2: "PZ_ERR_CAPACITY", 3: "PZ_ERR_CORRUPT",
                4: "PZ_ERR_CUDA", 5: "PZ_ERR_TIMEOUT"}
EXPORTS = ("pz_max_compressed_bytes", "pz_compress", "pz_decompress", "pz_compress_candidates",
           "pz_compressed_size", "pz_swap_work_bytes", "pz_swap_capacity", "pz_swap_out", "pz_swap_in",
           "pz_pool_bytes", "pz_pool_init", "pz_pool_free_slots", "pz_pool_swap_out", "pz_pool_swap_in",
           "pz_pool_release", "pz_test_lookback_timeout", "pz_compress_noalloc")
# candidate masks (bit t = tag t: ZVC 0, DBX 1, BX 2, ZBX 3, raw 4; raw is always allowed)
PZ_CAND_ZVC, PZ_CAND_DBX, PZ_CAND_BX, PZ_CAND_ZBX, PZ_CAND_RAW = 0x01, 0x02, 0x04, 0x08, 0x10
PZ_CAND_ALL = 0x1F
NOALLOC_MAX_BYTES = 256 << 20  # PZ_NOALLOC_MAX_BYTES

_lib = None


class PlaneZipError(RuntimeError):
    def __init__(self, where: str, status: int):
        super().__init__(f"{where} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


def load() -> ctypes.CDLL:
    """Load libplanezip.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH} is missing: build it with lossless_bit_plane_gb300.build.build()")
        L = ctypes.CDLL(str(LIB_PATH))
        sz, vp = ctypes.c_size_t, ctypes.c_void_p
        L.pz_max_compressed_bytes.argtypes = [sz]
        L.pz_max_compressed_bytes.restype = sz
        L.pz_compress.argtypes = [vp, sz, ctypes.c_int, vp, sz, vp, vp]
        L.pz_compress.restype = ctypes.c_int
        L.pz_decompress.argtypes = [vp, sz, ctypes.c_int, vp, sz, vp, vp]
        L.pz_decompress.restype = ctypes.c_int
        L.pz_compress_noalloc.argtypes = [vp, sz, ctypes.c_int, vp, sz, vp, vp]
        L.pz_compress_noalloc.restype = ctypes.c_int
        L.pz_compress_candidates.argtypes = [vp, sz, ctypes.c_int, ctypes.c_uint, vp, sz, vp, vp]
        L.pz_compress_candidates.restype = ctypes.c_int
        L.pz_compressed_size.argtypes = [vp, sz, ctypes.c_int, ctypes.c_uint, ctypes.c_uint, vp, vp, vp]
        L.pz_compressed_size.restype = ctypes.c_int
        L.pz_test_lookback_timeout.argtypes = [vp, sz, ctypes.c_int, vp, sz, vp, vp]
        L.pz_test_lookback_timeout.restype = ctypes.c_int
        L.pz_swap_work_bytes.argtypes = [sz]
        L.pz_swap_work_bytes.restype = sz
        L.pz_swap_capacity.argtypes = [sz, sz]
        L.pz_swap_capacity.restype = sz
        L.pz_swap_out.argtypes = [vp, sz, ctypes.c_int, sz, vp, sz, vp, sz, ctypes.POINTER(sz), vp]
        L.pz_swap_out.restype = ctypes.c_int
        L.pz_swap_in.argtypes = [vp, sz, vp, sz, vp, sz, vp, vp]
        L.pz_swap_in.restype = ctypes.c_int
        u32 = ctypes.c_uint
        L.pz_pool_bytes.argtypes = [sz, sz]
        L.pz_pool_bytes.restype = sz
        L.pz_pool_init.argtypes = [vp, sz, sz, ctypes.POINTER(vp)]
        L.pz_pool_init.restype = ctypes.c_int
        L.pz_pool_free_slots.argtypes = [vp]
        L.pz_pool_free_slots.restype = sz
        L.pz_pool_swap_out.argtypes = [vp, vp, sz, ctypes.c_int, sz, vp, sz, ctypes.POINTER(u32), ctypes.POINTER(sz),
                                       vp]
        L.pz_pool_swap_out.restype = ctypes.c_int
        L.pz_pool_swap_in.argtypes = [vp, u32, vp, sz, vp, sz, vp, vp]
        L.pz_pool_swap_in.restype = ctypes.c_int
        L.pz_pool_release.argtypes = [vp, u32]
        L.pz_pool_release.restype = ctypes.c_int
        _lib = L
    return _lib


def pz_max_compressed_bytes(nbytes: int) -> int:
    return int(load().pz_max_compressed_bytes(nbytes))


def pz_compress(d_in: int, nbytes: int, elem_width: int, d_out: int, out_capacity: int,
                d_total_bytes: int, stream: int = 0) -> int:
    """Raw C-ABI call with integer device addresses; returns the status code."""
    return int(load().pz_compress(d_in or None, nbytes, elem_width, d_out or None, out_capacity,
                                  d_total_bytes or None, stream or None))


def pz_decompress(d_in: int, comp_bytes: int, elem_width: int, d_out: int, nbytes: int,
                  d_status: int, stream: int = 0) -> int:
    return int(load().pz_decompress(d_in or None, comp_bytes, elem_width, d_out or None, nbytes,
                                    d_status or None, stream or None))


def pz_compress_noalloc(d_in: int, nbytes: int, elem_width: int, d_out: int, out_capacity: int,
                        d_total_bytes: int, stream: int = 0) -> int:
    """Raw C-ABI call of the allocation-free compress (scratch in a static
    device array; out_capacity only needs 2*C + nbytes); returns the status."""
    return int(load().pz_compress_noalloc(d_in or None, nbytes, elem_width, d_out or None, out_capacity,
                                          d_total_bytes or None, stream or None))


def pz_compress_candidates(d_in: int, nbytes: int, elem_width: int, candidates: int, d_out: int,
                           out_capacity: int, d_total_bytes: int, stream: int = 0) -> int:
    return int(load().pz_compress_candidates(d_in or None, nbytes, elem_width, candidates, d_out or None,
                                             out_capacity, d_total_bytes or None, stream or None))


def pz_compressed_size(d_in: int, nbytes: int, elem_width: int, candidates: int, chunk_stride: int,
                       d_sizes: int, d_total: int, stream: int = 0) -> int:
    return int(load().pz_compressed_size(d_in or None, nbytes, elem_width, candidates, chunk_stride,
                                         d_sizes or None, d_total or None, stream or None))


def pz_test_lookback_timeout(d_in: int, nbytes: int, elem_width: int, d_out: int, out_capacity: int,
                             d_total_bytes: int, stream: int = 0) -> int:
    """Test hook: the encoder with chunk 0 never taken (its look-back wait
    runs out); *d_total_bytes ends as UINT64_MAX."""
    return int(load().pz_test_lookback_timeout(d_in or None, nbytes, elem_width, d_out or None, out_capacity,
                                               d_total_bytes or None, stream or None))


def pz_swap_work_bytes(piece_bytes: int) -> int:
    return int(load().pz_swap_work_bytes(piece_bytes))


def pz_swap_capacity(nbytes: int, piece_bytes: int) -> int:
    return int(load().pz_swap_capacity(nbytes, piece_bytes))


def pz_swap_out(d_in: int, nbytes: int, elem_width: int, piece_bytes: int, d_work: int, work_bytes: int,
                h_out: int, h_capacity: int, stream: int = 0) -> tuple[int, int]:
    """Returns (status, container length written at h_out)."""
    total = ctypes.c_size_t(0)
    rc = load().pz_swap_out(d_in or None, nbytes, elem_width, piece_bytes, d_work or None, work_bytes,
                            h_out or None, h_capacity, ctypes.byref(total), stream or None)
    return int(rc), int(total.value)


def pz_swap_in(h_in: int, h_bytes: int, d_work: int, work_bytes: int, d_out: int, nbytes: int, d_status: int,
               stream: int = 0) -> int:
    return int(load().pz_swap_in(h_in or None, h_bytes, d_work or None, work_bytes, d_out or None, nbytes,
                                 d_status or None, stream or None))


def pz_pool_bytes(slot_bytes: int, nslots: int) -> int:
    return int(load().pz_pool_bytes(slot_bytes, nslots))


def pz_pool_init(h_mem: int, nbytes: int, slot_bytes: int) -> tuple[int, int]:
    """Returns (status, pool handle as an integer address)."""
    pool = ctypes.c_void_p(0)
    rc = load().pz_pool_init(h_mem or None, nbytes, slot_bytes, ctypes.byref(pool))
    return int(rc), int(pool.value or 0)


def pz_pool_free_slots(pool: int) -> int:
    return int(load().pz_pool_free_slots(pool or None))


def pz_pool_swap_out(pool: int, d_in: int, nbytes: int, elem_width: int, piece_bytes: int, d_work: int,
                     work_bytes: int, stream: int = 0) -> tuple[int, int, int]:
    """Returns (status, tensor handle, stored container bytes)."""
    tensor, stored = ctypes.c_uint(0), ctypes.c_size_t(0)
    rc = load().pz_pool_swap_out(pool or None, d_in or None, nbytes, elem_width, piece_bytes, d_work or None,
                                 work_bytes, ctypes.byref(tensor), ctypes.byref(stored), stream or None)
    return int(rc), int(tensor.value), int(stored.value)


def pz_pool_swap_in(pool: int, tensor: int, d_work: int, work_bytes: int, d_out: int, nbytes: int, d_status: int,
                    stream: int = 0) -> int:
    return int(load().pz_pool_swap_in(pool or None, tensor, d_work or None, work_bytes, d_out or None, nbytes,
                                      d_status or None, stream or None))


def pz_pool_release(pool: int, tensor: int) -> int:
    return int(load().pz_pool_release(pool or None, tensor))


# ---------------------------------------------------------------- torch glue

def _current_stream_handle(device) -> int:
    import torch

    return int(torch.cuda.current_stream(device).cuda_stream)


def compress_tensor(x, elem_width: int, out=None, total=None, candidates: int = PZ_CAND_ALL):
    """Compress the bytes of a contiguous CUDA tensor.

    Returns ``(out, total)``: ``out`` is a uint8 CUDA tensor of
    ``pz_max_compressed_bytes`` bytes whose first ``total.item()`` bytes are
    the stream; ``total`` is a 1-element int64 CUDA tensor. Asynchronous on
    the current stream."""
    import torch

    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("compress_tensor needs a contiguous CUDA tensor")
    nbytes = x.numel() * x.element_size()
    cap = pz_max_compressed_bytes(nbytes)
    if out is None:
        out = torch.empty(max(cap, 16), dtype=torch.uint8, device=x.device)
    if total is None:
        total = torch.empty(1, dtype=torch.int64, device=x.device)
    rc = pz_compress_candidates(x.data_ptr(), nbytes, elem_width, candidates, out.data_ptr(), out.numel(),
                                total.data_ptr(), _current_stream_handle(x.device))
    if rc != PZ_OK:
        raise PlaneZipError("pz_compress_candidates", rc)
    return out, total


def compressed_size_tensor(x, elem_width: int, chunk_stride: int = 1, candidates: int = PZ_CAND_ALL,
                           with_sizes: bool = True):
    """Sizes only (no stream): returns ``(sizes, total)``. ``sizes`` is a
    uint16-valued int32 CUDA tensor of ceil(C / chunk_stride) entries (None
    when ``with_sizes`` is false); ``total`` is a 1-element int64 CUDA tensor
    with the sum of 2 + L over the visited chunks. Asynchronous."""
    import torch

    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("compressed_size_tensor needs a contiguous CUDA tensor")
    nbytes = x.numel() * x.element_size()
    C = (nbytes + 4095) // 4096
    n = (C + chunk_stride - 1) // chunk_stride
    sizes = torch.zeros(max(n, 1), dtype=torch.int16, device=x.device) if with_sizes else None
    total = torch.empty(1, dtype=torch.int64, device=x.device)
    rc = pz_compressed_size(x.data_ptr(), nbytes, elem_width, candidates, chunk_stride,
                            sizes.data_ptr() if sizes is not None else 0, total.data_ptr(),
                            _current_stream_handle(x.device))
    if rc != PZ_OK:
        raise PlaneZipError("pz_compressed_size", rc)
    if sizes is not None:
        sizes = sizes[:n].to(torch.int32) & 0xFFFF
    return sizes, total


def decompress_tensor(stream_buf, comp_bytes: int, elem_width: int, nbytes: int, out=None, status=None):
    """Decompress ``comp_bytes`` of a uint8 CUDA tensor into ``nbytes``.

    Returns ``(out, status)``; ``status`` is a 1-element int32 CUDA tensor
    holding PZ_OK, PZ_ERR_CORRUPT or PZ_ERR_TIMEOUT once the stream completes."""
    import torch

    if out is None:
        out = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=stream_buf.device)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=stream_buf.device)
    rc = pz_decompress(stream_buf.data_ptr(), comp_bytes, elem_width, out.data_ptr(), nbytes,
                       status.data_ptr(), _current_stream_handle(stream_buf.device))
    if rc != PZ_OK:
        raise PlaneZipError("pz_decompress", rc)
    return out, status


class SwapBuffers:
    """Device staging and a pinned host container for swapping tensors of up
    to ``max_bytes`` bytes in pieces of ``piece_bytes`` (torch allocations;
    the swap itself runs in the library)."""

    def __init__(self, max_bytes: int, piece_bytes: int = 64 << 20, device="cuda"):
        import torch

        self.piece_bytes = piece_bytes
        self.work_bytes = pz_swap_work_bytes(piece_bytes)
        if self.work_bytes == 0:
            raise ValueError("piece_bytes must be a positive multiple of 4096")
        self.work = torch.empty(self.work_bytes, dtype=torch.uint8, device=device)
        self.host = torch.empty(pz_swap_capacity(max_bytes, piece_bytes), dtype=torch.uint8).pin_memory()
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def swap_out(self, x, elem_width: int) -> int:
        """Container length; the container is in ``self.host[:length]``."""
        nbytes = x.numel() * x.element_size()
        rc, total = pz_swap_out(x.data_ptr(), nbytes, elem_width, self.piece_bytes, self.work.data_ptr(),
                                self.work_bytes, self.host.data_ptr(), self.host.numel(),
                                _current_stream_handle(x.device))
        if rc != PZ_OK:
            raise PlaneZipError("pz_swap_out", rc)
        return total

    def swap_in(self, length: int, out):
        """Decode the container back into ``out`` (asynchronous); returns the
        device status tensor."""
        nbytes = out.numel() * out.element_size()
        rc = pz_swap_in(self.host.data_ptr(), length, self.work.data_ptr(), self.work_bytes, out.data_ptr(), nbytes,
                        self.status.data_ptr(), _current_stream_handle(out.device))
        if rc != PZ_OK:
            raise PlaneZipError("pz_swap_in", rc)
        return self.status


class SwapPool:
    """A pool of fixed-size slots in pinned host memory (torch allocation)
    that swapped tensors occupy, and the device staging the swaps need; the
    pool's bookkeeping and the swaps run in the library."""

    def __init__(self, pool_bytes: int, slot_bytes: int = 4 << 20, piece_bytes: int = 64 << 20, device="cuda"):
        import torch

        self.piece_bytes = piece_bytes
        self.work_bytes = pz_swap_work_bytes(piece_bytes)
        if self.work_bytes == 0:
            raise ValueError("piece_bytes must be a positive multiple of 4096")
        self.work = torch.empty(self.work_bytes, dtype=torch.uint8, device=device)
        # a 4096-byte aligned base: the slots (and so the container's pieces,
        # at 128-byte boundaries of the container) start aligned
        self.host = torch.empty(pool_bytes + 4096, dtype=torch.uint8).pin_memory()
        base = (self.host.data_ptr() + 4095) // 4096 * 4096
        rc, self.pool = pz_pool_init(base, pool_bytes, slot_bytes)
        if rc != PZ_OK:
            raise PlaneZipError("pz_pool_init", rc)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def free_slots(self) -> int:
        return pz_pool_free_slots(self.pool)

    def swap_out(self, x, elem_width: int) -> tuple[int, int]:
        """(tensor handle, stored bytes); blocks until the tensor is in the pool."""
        rc, tensor, stored = pz_pool_swap_out(self.pool, x.data_ptr(), x.numel() * x.element_size(), elem_width,
                                              self.piece_bytes, self.work.data_ptr(), self.work_bytes,
                                              _current_stream_handle(x.device))
        if rc != PZ_OK:
            raise PlaneZipError("pz_pool_swap_out", rc)
        return tensor, stored

    def swap_in(self, tensor: int, out):
        """Decode a pooled tensor into ``out`` (asynchronous); returns the
        device status tensor. Release the tensor after the stream is done."""
        rc = pz_pool_swap_in(self.pool, tensor, self.work.data_ptr(), self.work_bytes, out.data_ptr(),
                             out.numel() * out.element_size(), self.status.data_ptr(),
                             _current_stream_handle(out.device))
        if rc != PZ_OK:
            raise PlaneZipError("pz_pool_swap_in", rc)
        return self.status

    def release(self, tensor: int) -> None:
        rc = pz_pool_release(self.pool, tensor)
        if rc != PZ_OK:
            raise PlaneZipError("pz_pool_release", rc)
