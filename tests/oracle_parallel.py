"""The oracle's stream of a whole tensor, computed chunk-parallel on the host.

Section III-A "Stream format" of the paper codes every 4 KB chunk on its own
and lays the stream out as all chunk sizes, then all payloads. So the input
cut at chunk boundaries, each slice compressed by the unchanged oracle, gives
slice streams whose size tables concatenate into the whole size table and
whose payloads concatenate into the whole payload area (a property pinned on
the CPU by ``tests/test_oracle_pins.py::test_chunk_aligned_split_concatenates``
and ``tests/test_oracle_parallel.py``). The oracle's C calls run without the
GIL, so a thread pool spreads the slices over the host cores.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle


def host_threads() -> int:
    if hasattr(os, "sched_getaffinity"):
        return max(1, len(os.sched_getaffinity(0)))
    return max(1, os.cpu_count() or 1)


def compress(data, elem_width: int, candidates: int = oracle.CAND_ALL, threads: int | None = None,
             slices_per_thread: int = 4) -> bytes:
    """oracle.compress(data, elem_width, candidates), chunk-parallel."""
    raw = np.ascontiguousarray(np.frombuffer(bytes(data), np.uint8) if isinstance(data, (bytes, bytearray))
                               else np.asarray(data).view(np.uint8).reshape(-1))
    n = raw.size
    C = (n + 4095) // 4096
    threads = threads or host_threads()
    k = max(1, min(C, threads * slices_per_thread))
    cuts = [C * i // k for i in range(k + 1)]
    pieces = [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]

    def one(ab):
        a, b = ab
        s = oracle.compress(raw[4096 * a: min(n, 4096 * b)], elem_width, candidates)
        return s[: 2 * (b - a)], s[2 * (b - a):]

    if len(pieces) <= 1:
        return oracle.compress(raw, elem_width, candidates)
    with ThreadPoolExecutor(max_workers=min(threads, len(pieces))) as pool:
        parts = list(pool.map(one, pieces))
    return b"".join(h for h, _ in parts) + b"".join(p for _, p in parts)
