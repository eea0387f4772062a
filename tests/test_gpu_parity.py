"""GPU parity: the CUDA codec, called through the C ABI, against the CPU
oracle on the same seeded bytes. Streams, chunk sizes and round trips must
be bit-exact (integer work: no tolerance).

Paper: arXiv:2610.25033v1, Section III-A "Codec" and "Stream format".
"""
import numpy as np
import pytest

import oracle
from lossless_bit_plane_gb300 import _lib, build
from lossless_bit_plane_gb300 import workloads as W
from tests import golden_io, oracle_parallel

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    _lib.load()


from tests.gpu_util import (  # noqa: E402
    chunk_table,
    explain_mismatch,
    gpu_compress,
    gpu_compress_dev,
    gpu_decompress,
    to_device,
)


def full_parity(data, ew):
    data = bytes(data)
    got = gpu_compress(data, ew)
    want = oracle.compress(data, ew)
    assert got == want, explain_mismatch(data, ew, got, want)
    st, back = gpu_decompress(got, len(data), ew)
    assert st == _lib.PZ_OK and back == data
    return got


# ------------------------------------------------------------ small cases

@pytest.mark.parametrize("case", golden_io.all_cases(), ids=lambda c: c["name"])
def test_golden_streams(case):
    got = gpu_compress(case["input"], case["elem_width"])
    assert got.hex(" ") == case["stream"].hex(" ")
    st, back = gpu_decompress(case["stream"], len(case["input"]), case["elem_width"])
    assert st == 0 and back == case["input"]


@pytest.mark.parametrize("ew", [4, 2])
@pytest.mark.parametrize("which", ["fp32", "bf16"])
def test_edge_blocks(ew, which):
    data = W.edge_blocks_fp32() if which == "fp32" else W.edge_blocks_bf16()
    full_parity(data, ew)
    # one block per chunk as well (each edge block alone, then padded tails)
    for i in range(0, 64, 7):
        full_parity(data[128 * i: 128 * i + 128], ew)


@pytest.mark.parametrize("ew", [4, 2, 1, 8])
def test_tiny_alphabet_multi_chunk(ew):
    dt = "bf16" if ew == 2 else "fp32"
    full_parity(W.tiny_alphabet_blocks(32 * 70 + 5, dt, seed=ew), ew)


@pytest.mark.parametrize("ew", [4, 2])
def test_tail_sizes(ew):
    rng = np.random.default_rng(21)
    for n in W.TAIL_SIZES + (4096 * 3 + 130, 4096 * 5 - 2):
        for data in (bytes(n), rng.integers(0, 256, n, dtype=np.uint8).tobytes(),
                     W.relu_values(n // 4 + 1, rng).tobytes()[:n],
                     W.f32_to_bf16_rne(W.gelu_values(n // 2 + 1, rng)).tobytes()[:n]):
            if n == 0:
                got = gpu_compress(data, ew)
                assert got == b"" and oracle.compress(data, ew) == b""
                st, back = gpu_decompress(b"", 0, ew)
                assert st == 0
                continue
            full_parity(data, ew)


def test_random_and_zero_chunks():
    rng = np.random.default_rng(22)
    data = np.concatenate([np.zeros(4096 * 3, np.uint8), rng.integers(0, 256, 4096 * 3, dtype=np.uint8),
                           np.zeros(100, np.uint8)])
    for ew in (4, 2):
        s = full_parity(data, ew)
        lens, _ = chunk_table(s, data.size)
        assert list(lens[3:6]) == [4096] * 3


# ------------------------------------------------------ workload configs

def test_config1_relu_fp32_4mib_full():
    t = W.relu_fp32_4mib()
    s = full_parity(t.data, 4)
    assert t.nbytes / len(s) > 1.5


def test_config2_conv_bf16_full():
    t = W.conv_bf16()
    s = full_parity(t.data, 2)
    assert t.nbytes / len(s) > 1.5


def _large_case(t):
    # The whole stream -- every header and every payload byte -- against the
    # oracle's stream of the same bytes, computed chunk-parallel on the host;
    # the GPU stream is the one of the bench's launch configuration (one
    # pz_compress call on the full tensor). Then the full GPU round trip.
    x = to_device(t.data)
    out, total = gpu_compress_dev(x, t.elem_width)
    C = (t.nbytes + 4095) // 4096
    stream = out[:total].cpu().numpy().tobytes()
    want = oracle_parallel.compress(t.data, t.elem_width)
    assert total == len(want)
    assert stream[: 2 * C] == want[: 2 * C], explain_mismatch(t.data, t.elem_width, stream, want)
    assert stream == want, explain_mismatch(t.data, t.elem_width, stream, want)
    back, st = _lib.decompress_tensor(out, total, t.elem_width, t.nbytes)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(back[: t.nbytes], x)
    return total


def test_config3_attention_bf16_full():
    t = W.attention_bf16()
    total = _large_case(t)
    assert t.nbytes / total > 1.5


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_config4_mlp_ln_full(dtype):
    for t in W.mlp_ln(dtype=dtype):
        _large_case(t)


@pytest.mark.parametrize("ew", [4, 2])
@pytest.mark.parametrize("nchunks", [1000, 5000, 6300])
def test_verbatim_runs_of_every_length_on_each_walk(nchunks, ew):
    # 1,000 chunks: the fused walk and decode; 5,000: the cooperative walk;
    # 6,300: the thread walk. Whole stream against the oracle, then the
    # round trip.
    # Blocks whose top k planes are constant and whose low planes are random,
    # k cycling through 0..w: verbatim runs of every length, shorter than,
    # equal to and longer than the flags one walk step tests.
    data = W.verbatim_run_blocks(nchunks, ew, seed=89 + nchunks + ew)
    t = W.Tensor(f"verbatim_runs_{nchunks}_{ew}", "fp32" if ew == 4 else "bf16", data)
    _large_case(t)
    lens = np.frombuffer(oracle_parallel.compress(data, ew)[: 2 * nchunks], dtype=np.uint16)
    assert (lens < 4096).mean() > 0.9  # coded chunks, not raw ones


@pytest.mark.parametrize("seg", list(range(len(W.SWEEP_SEGMENTS))))
def test_config5_sweep_segments_full(seg):
    kind, dt = W.SWEEP_SEGMENTS[seg]
    _large_case(W.sweep_segment(kind, dt))


# ----------------------------------------------------------- decoder only

def test_decodes_oracle_streams():
    t = W.relu_fp32_4mib()
    s = oracle.compress(t.data, 4)
    st, back = gpu_decompress(s, t.nbytes, 4)
    assert st == 0 and back == t.data.tobytes()
    t2 = W.conv_bf16()
    s2 = oracle.compress(t2.data, 2)
    st, back = gpu_decompress(s2, t2.nbytes, 2)
    assert st == 0 and back == t2.data.tobytes()


def test_corrupt_streams_report_status():
    rng = np.random.default_rng(23)
    data = W.relu_values(4 * 1024 + 300, rng).tobytes()
    n = len(data)
    s = bytearray(oracle.compress(data, 4))
    C = (n + 4095) // 4096
    bad = bytearray(s); bad[0:2] = (0).to_bytes(2, "little")
    assert gpu_decompress(bytes(bad), n, 4)[0] == _lib.PZ_ERR_CORRUPT
    bad = bytearray(s); bad[0:2] = (4097).to_bytes(2, "little")
    assert gpu_decompress(bytes(bad), n, 4)[0] == _lib.PZ_ERR_CORRUPT
    assert gpu_decompress(bytes(s), n, 4, comp_bytes=len(s) - 1)[0] == _lib.PZ_ERR_CORRUPT
    bad = bytearray(s); bad[2 * C] = (bad[2 * C] & ~7) | 6          # tag 6
    assert gpu_decompress(bytes(bad), n, 4)[0] == _lib.PZ_ERR_CORRUPT
    for _ in range(200):
        bad = bytearray(s)
        pos = int(rng.integers(16 * 8, len(bad) * 8))
        bad[pos // 8] ^= 1 << (pos % 8)
        st, out = gpu_decompress(bytes(bad), n, 4)
        rc_ref, out_ref = oracle.decompress_status(bytes(bad), n, 4)
        assert st in (_lib.PZ_OK, _lib.PZ_ERR_CORRUPT)
        assert st == rc_ref
        if st == 0:
            assert out == out_ref


@pytest.mark.parametrize("dtype,ew", [("fp32", 4), ("bf16", 2)])
def test_corrupt_attention_streams_on_the_cooperative_walk(dtype, ew):
    # 1,024 / 512 chunks of causal attention (DBX and BX blocks with runs of
    # short codes, parsed several per step by the cooperative warp walk; at
    # this size one resident wave of warps walks and decodes every chunk in a
    # single launch): one random bit flipped per call anywhere past the size
    # table, judged by the oracle on the whole stream.
    t = W.sweep_segment("attention", dtype, seed=41, seg_bytes=(4 if dtype == "fp32" else 2) << 20)
    data = t.data.tobytes()
    n = len(data)
    s = bytearray(oracle.compress(data, ew))
    C = (n + 4095) // 4096
    assert C <= 6144
    st, back = gpu_decompress(bytes(s), n, ew)
    assert st == 0 and back == data
    rng = np.random.default_rng(43)
    for _ in range(64):
        bad = bytearray(s)
        pos = int(rng.integers(16 * C, len(bad) * 8))
        bad[pos // 8] ^= 1 << (pos % 8)
        st, out = gpu_decompress(bytes(bad), n, ew)
        rc_ref, out_ref = oracle.decompress_status(bytes(bad), n, ew)
        assert st == rc_ref, pos
        if st == 0:
            assert out == out_ref


@pytest.mark.parametrize("dtype,seg_mib", [("fp32", 22), ("bf16", 20)])
def test_corrupt_attention_streams_on_the_standalone_cooperative_walk(dtype, seg_mib):
    # 5,120 chunks (whole 1024 x 1024 attention matrices: 20 MiB of FP32 from
    # the 22 MiB asked for, 20 MiB of BF16): more than one resident wave of
    # the fused walk and decode (6 blocks of 4 warps per SM on 152 SMs), so
    # the cooperative walk runs as a launch of its own and the decode kernel
    # follows it. Clean
    # round trip first, then one bit flipped per call in the last chunks,
    # each flip judged by the oracle on the flipped chunk alone.
    t = W.sweep_segment("attention", dtype, seed=47, seg_bytes=seg_mib << 20)
    ew = t.elem_width
    data = t.data
    n = data.size
    s = bytearray(oracle.compress(data, ew))
    lens, offs = chunk_table(bytes(s), n)
    C = lens.size
    assert 3648 < C <= 6144
    st, back = gpu_decompress(bytes(s), n, ew)
    assert st == 0 and back == data.tobytes()
    rng = np.random.default_rng(53)
    for _ in range(32):
        c = int(rng.integers(C - 256, C))
        L = int(lens[c])
        bad = bytearray(s)
        bit = int(rng.integers(0, 8 * L))
        bad[offs[c] + bit // 8] ^= 1 << (bit % 8)
        st, out = gpu_decompress(bytes(bad), n, ew)
        piece = data[4096 * c: 4096 * c + 4096]
        mini = int(L).to_bytes(2, "little") + bytes(bad[offs[c]: offs[c] + L])
        rc_ref, out_ref = oracle.decompress_status(mini, piece.size, ew)
        assert st == rc_ref, (c, bit)
        if st == 0:
            assert out[4096 * c: 4096 * c + piece.size] == out_ref


def test_corrupt_streams_report_status_above_the_cooperative_walk_size():
    # 8,500 chunks: decompress walks chunks one thread each (inputs of up to
    # 6,144 chunks take the cooperative warp walk, covered above). Bits are
    # flipped in the payloads of the last chunks only; since chunks are
    # independent, the oracle judges each flip on that chunk alone.
    rng = np.random.default_rng(29)
    data = W.relu_values(8500 * 1024 - 77, rng).view(np.uint8)
    n = data.size
    s = bytearray(oracle.compress(data, 4))
    lens, offs = chunk_table(bytes(s), n)
    C = lens.size
    st, back = gpu_decompress(bytes(s), n, 4)
    assert st == 0 and back == data.tobytes()
    for _ in range(24):
        c = int(rng.integers(C - 12, C))
        L = int(lens[c])
        bad = bytearray(s)
        bit = int(rng.integers(0, 8 * L))
        bad[offs[c] + bit // 8] ^= 1 << (bit % 8)
        st, out = gpu_decompress(bytes(bad), n, 4)
        piece = data[4096 * c: 4096 * c + 4096]
        mini = int(L).to_bytes(2, "little") + bytes(bad[offs[c]: offs[c] + L])
        rc_ref, out_ref = oracle.decompress_status(mini, piece.size, 4)
        assert st == rc_ref, (c, bit)
        if st == 0:
            assert out[4096 * c: 4096 * c + piece.size] == out_ref


@pytest.mark.parametrize("dtype,seg_mib", [("fp32", 36), ("bf16", 34)])
def test_corrupt_attention_streams_above_the_cooperative_walk_size(dtype, seg_mib):
    # Causal-attention data codes most blocks as DBX or BX with several short
    # (non-verbatim) plane codes per block, which the thread walk parses up to
    # two at a time; 9,216 / 8,704 chunks take that walk. One bit is flipped
    # per call, in the last rows' chunks (the longest code sequences), and the
    # oracle judges the flipped chunk on its own.
    t = W.sweep_segment("attention", dtype, seed=31, seg_bytes=seg_mib << 20)
    ew = t.elem_width
    data = t.data
    n = data.size
    s = bytearray(oracle.compress(data, ew))
    lens, offs = chunk_table(bytes(s), n)
    C = lens.size
    assert C > 6144
    st, back = gpu_decompress(bytes(s), n, ew)
    assert st == 0 and back == data.tobytes()
    rng = np.random.default_rng(37)
    for _ in range(32):
        c = int(rng.integers(C - 256, C))
        L = int(lens[c])
        bad = bytearray(s)
        bit = int(rng.integers(0, 8 * L))
        bad[offs[c] + bit // 8] ^= 1 << (bit % 8)
        st, out = gpu_decompress(bytes(bad), n, ew)
        piece = data[4096 * c: 4096 * c + 4096]
        mini = int(L).to_bytes(2, "little") + bytes(bad[offs[c]: offs[c] + L])
        rc_ref, out_ref = oracle.decompress_status(mini, piece.size, ew)
        assert st == rc_ref, (c, bit)
        if st == 0:
            assert out[4096 * c: 4096 * c + piece.size] == out_ref


def test_calls_queued_back_to_back_on_one_stream():
    # Compress and decompress calls of four sizes, one per decode path (the
    # fused walk and decode alone and after the size sums, the standalone
    # cooperative walk, the thread walk), queued on one stream with no host
    # synchronisation: each call's first kernel follows the previous call's
    # last one, and the kernels inside a call are launched as programmatic
    # dependents. Every stream equals the oracle's and every round trip is
    # exact.
    rng = np.random.default_rng(61)
    items = [(W.relu_values(256 * 1024, rng).view(np.uint8), 4),
             (W.conv_bf16().data.view(np.uint8), 2),
             (W.sweep_segment("attention", "fp32", seed=67, seg_bytes=20 << 20).data.view(np.uint8), 4),
             (W.sweep_segment("attention", "bf16", seed=71, seg_bytes=34 << 20).data.view(np.uint8), 2)]
    assert [(a.size + 4095) // 4096 for a, _ in items] == [256, 3136, 5120, 8704]
    xs = [to_device(a) for a, _ in items]
    torch.cuda.synchronize()
    results = []
    for _ in range(2):
        for x, (a, ew) in zip(xs, items):
            out, total = _lib.compress_tensor(x, ew)
            back, st = _lib.decompress_tensor(out, out.numel(), ew, a.size)
            results.append((x, out, total, back, st, a, ew))
    torch.cuda.synchronize()
    for x, out, total, back, st, a, ew in results:
        n = int(total.item())
        assert int(st.item()) == 0
        assert torch.equal(back[: a.size], x)
        stream = out[:n].cpu().numpy().tobytes()
        assert stream == oracle_parallel.compress(a, ew)


def test_repeated_calls_and_streams_are_deterministic():
    t = W.relu_fp32_4mib()
    x = to_device(t.data)
    ref = None
    s2 = torch.cuda.Stream()
    for i in range(4):
        with torch.cuda.stream(s2 if i % 2 else torch.cuda.current_stream()):
            out, total = _lib.compress_tensor(x, 4)
        torch.cuda.synchronize()
        got = out[: int(total.item())].cpu()
        if ref is None:
            ref = got
        assert torch.equal(got, ref)


def test_fused_walk_and_decode_while_another_stream_holds_sms():
    # 3,000 chunks of causal attention (FP32, 12 MiB) and of ReLU data:
    # decompress takes the fused walk-and-decode path, one launch whose warps
    # overwrite their chunks' output regions while other warps of the same
    # launch may not have started yet. A 256 MiB compress on a second stream
    # keeps SMs busy, so the launch's blocks start in several waves. Chunk
    # offsets come from the header table alone, so every round trip stays
    # exact whatever the order in which the blocks run.
    rng = np.random.default_rng(73)
    att = W.sweep_segment("attention", "fp32", seed=79, seg_bytes=12 << 20).data.view(np.uint8)
    relu = W.relu_values(3000 * 1024 - 5, rng).view(np.uint8)
    busy = to_device(rng.integers(0, 1 << 32, (256 << 20) // 4, dtype=np.uint32).view(np.uint8))
    busy_out = torch.empty(_lib.pz_max_compressed_bytes(busy.numel()), dtype=torch.uint8, device="cuda")
    busy_tot = torch.empty(1, dtype=torch.int64, device="cuda")
    s2 = torch.cuda.Stream()
    for a in (att, relu):
        assert 2048 < (a.size + 4095) // 4096 <= 3072
        x = to_device(a)
        out, total = gpu_compress_dev(x, 4)
        assert out[:total].cpu().numpy().tobytes() == oracle_parallel.compress(a, 4)
        backs = []
        torch.cuda.synchronize()
        for _ in range(6):
            with torch.cuda.stream(s2):
                _lib.compress_tensor(busy, 4, busy_out, busy_tot)
            backs.append(_lib.decompress_tensor(out, total, 4, a.size))
        torch.cuda.synchronize()
        for back, st in backs:
            assert int(st.item()) == 0
            assert torch.equal(back[: a.size], x)
