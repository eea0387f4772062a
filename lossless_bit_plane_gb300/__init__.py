"""PlaneZip block codec on GB300 (sm_103a).

The codec (arXiv:2610.25033v1, Section III-A) runs in the CUDA library
``libplanezip.so`` behind the C ABI of ``include/planezip.h``; this package
holds that library's sources (``csrc/``), its build step (``build.py``), a
ctypes binding with the same names (``_lib.py``) and the seeded input
generators (``workloads.py``).
"""
from ._lib import (  # noqa: F401
    EXPORTS,
    PZ_ERR_ARG,
    PZ_ERR_CAPACITY,
    PZ_ERR_CORRUPT,
    PZ_ERR_CUDA,
    PZ_ERR_TIMEOUT,
    PZ_OK,
    PlaneZipError,
    compress_tensor,
    decompress_tensor,
    load,
    pz_compress,
    pz_compress_noalloc,
    pz_decompress,
    pz_max_compressed_bytes,
)
