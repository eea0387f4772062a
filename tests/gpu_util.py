"""GPU-side helpers for the parity tests: run the C-ABI codec on host bytes
and explain the first difference from the oracle's stream."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from lossless_bit_plane_gb300 import _lib


def to_device(data) -> torch.Tensor:
    arr = np.frombuffer(bytes(data), dtype=np.uint8).copy() if not isinstance(data, np.ndarray) else data.view(np.uint8).reshape(-1)
    x = torch.empty(arr.size, dtype=torch.uint8, device="cuda")
    if arr.size:
        x.copy_(torch.from_numpy(np.ascontiguousarray(arr)))
    return x


def gpu_compress_dev(x: torch.Tensor, ew: int):
    out, total = _lib.compress_tensor(x, ew)
    torch.cuda.synchronize()
    return out, int(total.item())


def gpu_compress(data, ew: int) -> bytes:
    out, total = gpu_compress_dev(to_device(data), ew)
    return out[:total].cpu().numpy().tobytes()


def gpu_decompress(stream: bytes, nbytes: int, ew: int, comp_bytes: int | None = None):
    s = to_device(stream + bytes(16))  # slack so that comp_bytes < len is expressible
    out, st = _lib.decompress_tensor(s, len(stream) if comp_bytes is None else comp_bytes, ew, nbytes)
    torch.cuda.synchronize()
    return int(st.item()), out[:nbytes].cpu().numpy().tobytes()


def chunk_table(stream: bytes, nbytes: int):
    C = (nbytes + 4095) // 4096
    lens = np.frombuffer(stream[: 2 * C], dtype="<u2").astype(np.int64)
    offs = 2 * C + np.concatenate([[0], np.cumsum(lens)[:-1]]) if C else np.zeros(0, np.int64)
    return lens, offs


def explain_mismatch(data, ew: int, got: bytes, want: bytes) -> str:
    n = len(data)
    if len(got) != len(want):
        msg = f"length {len(got)} != oracle {len(want)}; "
    else:
        msg = ""
    C = (n + 4095) // 4096
    g_l, g_o = chunk_table(got, n)
    w_l, w_o = chunk_table(want, n)
    for c in range(C):
        gl = int(g_l[c]) if c < len(g_l) else -1
        if gl != w_l[c] or got[g_o[c]:g_o[c] + gl] != want[w_o[c]:w_o[c] + w_l[c]]:
            raw = bytes(data)[4096 * c: 4096 * c + 4096]
            tags, bits, _ = oracle.analyze(raw, ew)
            return (msg + f"first differing chunk {c}: L gpu {gl} oracle {int(w_l[c])}; "
                    f"oracle tags {tags.tolist()} bits {bits.tolist()}")
    return msg + "headers and payloads equal"
