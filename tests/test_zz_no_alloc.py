"""pz_compress_noalloc: the allocation-free compress entry point.

It serves callers that cannot allocate device memory when they compress (for
example a swap runtime evicting activations because device memory is full).
Its encoder scratch lives in a static device array of the library rather than
in the caller's output buffer, so the output only has to hold the stream.
This file checks it through the C ABI against the regular pz_compress on the
same inputs: the streams and sizes must be identical (integer work, exact),
over several calls in a row that share the static scratch.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest

from lossless_bit_plane_gb300 import _lib, build
from lossless_bit_plane_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    _lib.load()


def _reference(x: torch.Tensor, ew: int) -> bytes:
    out, total = _lib.compress_tensor(x, ew)
    torch.cuda.synchronize()
    return out[: int(total.item())].cpu().numpy().tobytes()


def _noalloc(x: torch.Tensor, ew: int) -> bytes:
    nbytes = x.numel()
    C = (nbytes + 4095) // 4096
    cap = 2 * C + nbytes                       # the stream alone, no scratch tail
    out = torch.empty(max(cap, 16), dtype=torch.uint8, device=x.device)
    total = torch.empty(1, dtype=torch.int64, device=x.device)
    stream = torch.cuda.current_stream(x.device).cuda_stream
    rc = _lib.pz_compress_noalloc(x.data_ptr(), nbytes, ew, out.data_ptr(), cap, total.data_ptr(), stream)
    assert rc == _lib.PZ_OK, _lib.STATUS_NAMES.get(rc, rc)
    torch.cuda.synchronize()
    return out[: int(total.item())].cpu().numpy().tobytes()


def _dev(arr: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(arr.view(np.uint8)).copy()).cuda()


def test_noalloc_matches_pz_compress_on_calls_in_a_row():
    rng = np.random.default_rng(31)
    big = _dev(W.relu_values(3 * (1 << 20) + 777, rng))                      # 12 MiB FP32, ragged tail
    small = _dev(W.f32_to_bf16_rne(W.gelu_values(5000, rng)))                # 10 KB BF16
    cases = [(big, 4), (small, 2), (big, 4), (_dev(W.edge_blocks_bf16()), 2)]
    for x, ew in cases:
        want = _reference(x, ew)
        got = _noalloc(x, ew)
        assert len(got) == len(want)
        assert got == want


def test_noalloc_at_its_maximum_size():
    # nbytes == PZ_NOALLOC_MAX_BYTES: 65,536 chunks, so the look-back words
    # and the ticket fill the static scratch array to its last word; then a
    # ragged input just below the maximum, and the maximum again (each call
    # finds the previous call's contents in the array).
    rng = np.random.default_rng(37)
    n = _lib.NOALLOC_MAX_BYTES
    full = _dev(W.relu_values(n // 4, rng))
    assert full.numel() == n
    ragged = full[: n - 4096 + 100]
    for x, ew in ((full, 4), (ragged, 2), (full, 4)):
        want = _reference(x, ew)
        got = _noalloc(x, ew)
        assert got == want


def test_noalloc_rejects_sizes_beyond_its_scratch():
    FAKE = 0x100000  # never dereferenced: the size checks come first
    n = _lib.NOALLOC_MAX_BYTES + 1
    C = (n + 4095) // 4096
    assert _lib.pz_compress_noalloc(FAKE, n, 4, FAKE, 2 * C + n, FAKE) == _lib.PZ_ERR_CAPACITY
    n = 8192
    assert _lib.pz_compress_noalloc(FAKE, n, 4, FAKE, 2 * 2 + n - 1, FAKE) == _lib.PZ_ERR_CAPACITY
