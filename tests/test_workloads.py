"""The seeded synthetic inputs follow the recipes the benchmark configurations
state (shapes and sizes, value distributions, exact zeros, BF16 rounding),
and the same seed gives the same bytes. CPU only; small instances where the
full configuration would take long to generate."""
from __future__ import annotations

import math
import struct

import numpy as np

from lossless_bit_plane_gb300 import workloads as W


def _f32(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def _bf16_nearest_even(bits: int) -> int:
    """BF16 pattern nearest to the finite FP32 value `bits`, ties to an even
    pattern: the two candidates are the truncation and the next pattern up in
    magnitude, compared by exact distance (both differences are exact in
    double precision)."""
    lo = bits >> 16
    hi = lo + 1
    v = _f32(bits)
    d_lo = abs(v - _f32(lo << 16))
    d_hi = abs(_f32(hi << 16) - v)
    if d_lo < d_hi:
        return lo
    if d_hi < d_lo:
        return hi
    return lo if lo % 2 == 0 else hi


def test_bf16_rounding_is_round_to_nearest_even():
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32)
    exp = (bits >> 23) & 0xFF
    bits = bits[exp < 0xFE]  # finite, and rounding up cannot leave the finite range
    got = W.f32_to_bf16_rne(bits.view(np.float32))
    want = np.array([_bf16_nearest_even(int(b)) for b in bits], dtype=np.uint16)
    assert np.array_equal(got, want)
    # ties: 1 + 2^-8 lies halfway between 0x3F80 and 0x3F81 and goes to the
    # even 0x3F80; 0x3F818000 lies halfway between 0x3F81 and 0x3F82 and goes
    # to 0x3F82; signs, zeros, infinities and NaN
    special = np.array([0x3F800000, 0x3F808000, 0x3F818000, 0x80000000, 0x00000000, 0x7F800000, 0xFF800000,
                        0x7FC00000, 0x7F800001, 0xBF808001], dtype=np.uint32)
    out = W.f32_to_bf16_rne(special.view(np.float32)).tolist()
    assert out[:7] == [0x3F80, 0x3F80, 0x3F82, 0x8000, 0x0000, 0x7F80, 0xFF80]
    assert out[7] == 0x7FC0 and (out[8] & 0x7FC0) == 0x7FC0  # NaN stays a quiet NaN
    assert out[9] == 0xBF81  # just above the tie: away from zero in magnitude


def test_relu_config_recipe():
    t = W.relu_fp32_4mib()
    assert (t.nbytes, t.elem_width) == (4 << 20, 4)
    x = t.data.view(np.float32)
    assert x.size == 1 << 20 and np.all(x >= 0) and not np.signbit(x).any()
    zero = np.mean(x == 0)
    assert abs(zero - 0.5) < 0.005  # 0 with probability 0.5 (sd of the estimate 0.0005)
    # |N(0,1)| has mean sqrt(2 / pi)
    assert abs(float(x[x > 0].mean()) - math.sqrt(2 / math.pi)) < 0.005


def test_conv_config_recipe_on_a_small_shape():
    # the full configuration is [32,64,56,56] BF16 = 12,845,056 bytes
    assert 32 * 64 * 56 * 56 * 2 == 12_845_056
    t = W.conv_bf16(shape=(2, 8, 56, 56))
    assert (t.nbytes, t.elem_width) == (2 * 8 * 56 * 56 * 2, 2)
    h = t.data.view(np.uint16)
    assert not np.any(h & 0x8000)  # after ReLU: no negative values (and no -0)
    zero = np.mean(h == 0)
    assert 0.35 < zero < 0.65  # ReLU of a zero-mean field
    # the Gaussian taps are normalised, and the blur makes neighbours alike:
    # a pixel and its right neighbour are both zero or both non-zero far
    # more often than independent pixels would be
    taps = W._gauss_taps()
    assert taps.size == 13 and abs(taps.sum() - 1.0) < 1e-12 and np.argmax(taps) == 6
    img = (h.reshape(16, 56, 56) != 0)
    same = np.mean(img[:, :, 1:] == img[:, :, :-1])
    assert same > 0.85


def test_attention_config_recipe_on_a_small_shape():
    seq = 64
    t = W.attention_bf16(batch=1, heads=2, seq=seq)
    assert (t.nbytes, t.elem_width) == (2 * seq * seq * 2, 2)
    h = t.data.view(np.uint16).reshape(2, seq, seq)
    upper = np.triu(np.ones((seq, seq), dtype=bool), k=1)
    assert np.all(h[:, upper] == 0)  # exact zeros above the diagonal
    assert np.all(h[:, ~upper] != 0)  # softmax weights are positive
    assert np.all(h[:, 0, 0] == 0x3F80)  # row 0: one weight, exactly 1.0
    vals = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # BF16 rounding changes each positive weight by at most 2^-9 relative,
    # so a row that sums to 1 sums to 1 within 2^-9 (plus FP32 rounding)
    assert np.all(np.abs(vals.sum(axis=2) - 1.0) <= 2.0 ** -9 + 1e-6)
    # the full configuration: [8,12,1024,1024] BF16 = 192 MiB, 49,152 chunks
    assert 8 * 12 * 1024 * 1024 * 2 == 192 << 20 and (192 << 20) // 4096 == 49_152


def test_mlp_config_recipe():
    rng = W._rng(9)
    g = W.gelu_values(1 << 20, rng)
    # GELU's minimum is about -0.16997; E[x Phi(x)] for x ~ N(0,1) is 1 / (2 sqrt(pi))
    assert float(g.min()) >= -0.17 and float(g.min()) < -0.16
    assert abs(float(g.mean()) - 1 / (2 * math.sqrt(math.pi))) < 0.003
    assert np.any(g != 0)
    ln = W.layernorm_values(4096, 768, W._rng(11))
    sd = ln.std(axis=0)
    mu = ln.mean(axis=0)
    assert sd.min() > 0.45 and sd.max() < 1.6  # gamma ~ U(0.5, 1.5) per feature
    assert np.abs(mu).max() < 0.5 and 0.07 < float(mu.std()) < 0.13  # beta ~ N(0, 0.1^2)
    # the full configuration's sizes: FP32 96 + 24 MiB, BF16 48 + 12 MiB
    assert 8 * 1024 * 3072 * 4 == 96 << 20 and 8 * 1024 * 768 * 4 == 24 << 20


def test_sweep_layout_and_random_segment():
    assert len(W.SWEEP_SEGMENTS) == 7 and W.SWEEP_SEGMENTS[-1] == ("random", "u32")
    kinds = {k for k, _ in W.SWEEP_SEGMENTS[:-1]}
    assert kinds == {"relu", "conv", "attention"}
    assert {d for _, d in W.SWEEP_SEGMENTS[:-1]} == {"fp32", "bf16"}
    # 6 x 128 MiB + 256 MiB = 1 GiB; the random segment is twice seg_bytes
    assert 6 * (128 << 20) + (256 << 20) == 1 << 30
    r = W.sweep_segment("random", "u32", seg_bytes=1 << 20)
    assert (r.nbytes, r.elem_width) == (2 << 20, 4)
    words = r.data.view(np.uint32)
    assert abs(float(words.mean()) / 2.0 ** 32 - 0.5) < 0.01
    assert abs(np.unpackbits(r.data).mean() - 0.5) < 0.002


def test_same_seed_same_bytes():
    assert W.sha256(W.relu_fp32_4mib().data) == W.sha256(W.relu_fp32_4mib().data)
    assert W.sha256(W.relu_fp32_4mib(seed=1).data) != W.sha256(W.relu_fp32_4mib().data)
    a = W.sweep_segment("conv", "bf16", seg_bytes=1 << 20)
    b = W.sweep_segment("conv", "bf16", seg_bytes=1 << 20)
    assert a.nbytes == 1 << 20 and np.array_equal(a.data, b.data)
    c = W.attention_bf16(batch=1, heads=1, seq=32)
    d = W.attention_bf16(batch=1, heads=1, seq=32)
    assert np.array_equal(c.data, d.data)


def test_verbatim_run_blocks_give_runs_of_every_length():
    # The recipe's premise, checked with the oracle's per-block analysis:
    # blocks sharing k top bits over random low bits take BX (or DBX) with
    # w - k verbatim planes, so the coded blocks span run lengths on both
    # sides of the walks' flag windows (26 for 32-bit, 10 for 16-bit symbols).
    import oracle

    for ew, bx_ks in ((4, range(2, 11)), (2, range(1, 16))):
        w = 8 * ew
        data = W.verbatim_run_blocks(4, ew, seed=5)
        assert data.size == 4 * 4096
        tags = np.asarray(oracle.analyze(data, ew)[0]).reshape(-1)
        for b, t in enumerate(tags):
            if b % (w + 1) in bx_ks:
                assert int(t) == oracle.TAG_BX, (ew, b)
        sym = data.view("<u4" if ew == 4 else "<u2").reshape(-1, 128 // ew).astype(np.uint64)
        for b in range(tags.size):
            k = b % (w + 1)
            if k:  # the top k bits are the block's own constant
                assert np.unique(sym[b] >> np.uint64(w - k)).size == 1
