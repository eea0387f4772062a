"""The encoder's bounded waits, exercised without a GPU fault: the test hook
pz_test_lookback_timeout runs the encoder with chunk 0 never taken, so a
look-back waits on a status word that nothing publishes. The wait must give
up after its iteration limit, the launch must end with the timeout report
(*d_total_bytes = UINT64_MAX), and the context must stay usable."""
import time

import numpy as np
import pytest

import oracle
from lossless_bit_plane_gb300 import _lib, build
from lossless_bit_plane_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def test_lookback_wait_gives_up_and_reports_timeout():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    data = W.relu_values(64 * 1024, np.random.default_rng(9)).view(np.uint8)  # 64 chunks
    x = torch.from_numpy(data.copy()).cuda()
    cap = _lib.pz_max_compressed_bytes(x.numel())
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    total = torch.zeros(1, dtype=torch.int64, device="cuda")
    t0 = time.perf_counter()
    rc = _lib.pz_test_lookback_timeout(x.data_ptr(), x.numel(), 4, out.data_ptr(), cap, total.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert rc == _lib.PZ_OK
    assert int(total.item()) == -1  # UINT64_MAX: the timeout report
    assert waited < 60
    # the context is usable: a normal call on the same buffers is exact
    out2, total2 = _lib.compress_tensor(x, 4, out, total)
    torch.cuda.synchronize()
    assert out2[: int(total2.item())].cpu().numpy().tobytes() == oracle.compress(data, 4)
