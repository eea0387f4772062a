"""The Python usage example given to users of the library (compress,
decompress, sampled sizes, swap out and in), run as written through the C
ABI, so that the documented usage stays correct."""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def test_usage_example():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from lossless_bit_plane_gb300 import _lib, build

    build.build()
    torch.manual_seed(0)
    x = torch.randn(1 << 20, device="cuda").relu()        # FP32 activations
    out, total = _lib.compress_tensor(x, elem_width=4)     # device stream, device length
    n = int(total.item())
    back, status = _lib.decompress_tensor(out, n, 4, x.numel() * 4)
    assert int(status.item()) == 0 and torch.equal(back.view(torch.float32), x)

    sizes, est_total = _lib.compressed_size_tensor(x, 4, chunk_stride=4)   # sampled sizes only
    torch.cuda.synchronize()
    C = (x.numel() * 4 + 4095) // 4096
    assert sizes.numel() == (C + 3) // 4
    headers = out[: 2 * C].cpu().view(torch.int16).to(torch.int32) & 0xFFFF
    assert torch.equal(sizes.cpu(), headers[::4])
    swap = _lib.SwapBuffers(x.numel() * 4)                 # pieces of at most 64 MiB by default
    length = swap.swap_out(x, 4)                           # compressed container in pinned host memory
    back.zero_()
    status = swap.swap_in(length, back)                    # back on the device (asynchronous)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and torch.equal(back.view(torch.float32), x)

    pool = _lib.SwapPool(64 << 20, slot_bytes=1 << 20)     # 64 MiB of pinned host slots
    free = pool.free_slots()
    handle, stored = pool.swap_out(x, 4)                   # the tensor occupies ceil(stored / 1 MiB) slots
    assert free - pool.free_slots() == (stored + (1 << 20) - 1) // (1 << 20)
    back.zero_()
    status = pool.swap_in(handle, back)
    torch.cuda.synchronize()
    pool.release(handle)
    assert int(status.item()) == 0 and torch.equal(back.view(torch.float32), x)
    assert pool.free_slots() == free
