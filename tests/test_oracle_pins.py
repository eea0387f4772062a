"""Pins of the CPU oracle against what the paper and arithmetic fix.

Paper: "PlaneZip: Lossless Bit-Plane Compression of Training Activations
Offloaded over PCIe" (arXiv:2610.25033v1), Section III-A "Codec" (block,
symbols, candidates, plane code lengths, 3-bit tag, smallest kept) and
"Stream format" (4 KB chunks, 16-bit sizes, raw fallback, ratios include tags,
headers and padding); Section III-A "Validation" (size model vs bit-exact
encoder). Every expected number below was derived by hand from those
definitions and the readings R1-R14; none was produced by running code.
"""
import numpy as np
import pytest

import oracle
from lossless_bit_plane_gb300 import workloads as W
from tests import golden_io

CASES = golden_io.all_cases()


def u32(vals):
    return np.array(vals, dtype="<u4").tobytes()


def u16(vals):
    return np.array(vals, dtype="<u2").tobytes()


def blocks(buf: bytes):
    return [buf[i:i + 128] for i in range(0, len(buf), 128)]


# ---------------------------------------------------------------- goldens

@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_golden_stream(case):
    stream = oracle.compress(case["input"], case["elem_width"])
    assert stream.hex(" ") == case["stream"].hex(" ")
    assert oracle.decompress(case["stream"], len(case["input"]), case["elem_width"]) == case["input"]


# ------------------------------------------------------- worked examples

# (block, elem_width, {tag: bits}, chosen tag), all derived by hand
WORKED = [
    # 1.0f constant: g = 0x20400000 -> BX 7+5+7+5+7
    (u32([0x3F800000] * 32), 4, {0: 1056, 1: 39, 2: 31, 3: 63, 4: 1024}, 2),
    # BF16 1.0 constant: DBX = 16 + one run of 17 planes (6)
    (u16([0x3F80] * 64), 2, {0: 1088, 1: 22, 2: 28, 3: 92, 4: 1024}, 1),
    # integer ramp: DBX 32 + run32 + all-ones
    (u32(list(range(32))), 4, {0: 1024, 1: 44, 4: 1024}, 1),
    # descending ramp: every delta is -1 = 2^33 - 1: only X32 is non-zero (all ones)
    (u32([31 - k for k in range(32)]), 4, {1: 44}, 1),
    # a single word: ZVC 64; ZBX 111 (1-bit planes go verbatim in 2 bits); BX 167
    (u32([0x12345678] + [0] * 31), 4, {0: 64, 2: 167, 3: 111, 4: 1024}, 0),
    # all-zero FP32: BX is one run code (7); ZVC = N = ZBX = 32 ties by tag order
    (bytes(128), 4, {0: 32, 1: 39, 2: 7, 3: 32, 4: 1024}, 2),
    # all-zero BF16: BX one run code of 16 planes (6); DBX 16 + 6
    (bytes(128), 2, {0: 64, 1: 22, 2: 6, 3: 64, 4: 1024}, 2),
    # BF16 s_0 = 1, rest 0: BX run15 (6) + single one (11) = 17; DBX = base 16
    # + the 17th (borrow) plane, d_1 = -1 mod 2^17, Gray code bit 16 alone:
    # single one q = 0 (11) + run of the 16 planes below (6) = 33; ZBX = mask
    # 64 + run15 (6) + the 1-bit plane, verbatim in 2 bits = 72
    (u16([1] + [0] * 63), 2, {0: 80, 1: 33, 2: 17, 3: 72, 4: 1024}, 2),
    # s_k = rotl(0x0F0F0F0F, (k-3) mod 8): every BX plane verbatim (32 x 33),
    # DBX 32 + 32 + 3 + 31 x 32 (its plane 31 is the only zero plane); RAW wins
    (u32([0xE1E1E1E1, 0xC3C3C3C3, 0x87878787, 0x0F0F0F0F, 0x1E1E1E1E, 0x3C3C3C3C, 0x78787878,
          0xF0F0F0F0] * 4), 4, {0: 1056, 1: 1059, 2: 1056, 3: 1088, 4: 1024}, 4),
]


@pytest.mark.parametrize("i", range(len(WORKED)))
def test_worked_example_sizes(i):
    blk, ew, expect, tag = WORKED[i]
    enc, model, chosen = oracle.block_candidates(blk, ew)
    for t, bits in expect.items():
        assert enc[t] == bits, (oracle.TAG_NAMES[t], enc)
        assert model[t] == bits
    assert chosen == tag


def test_dbx_borrow_bit_pins_unsigned_delta():
    # R5: s_0 = 0x80000000, rest 0. Unsigned: d_1 = 0 - 0x80000000 mod 2^33
    # = 0x1_8000_0000 (bits 32 and 31), g = bits 32 and 30. Top-down codes:
    # X32 single one q=0 (00011 00000), X31 single zero (001), X30 pre-XOR zero
    # (00001; P30 = 0), X29..X0 run 30 (01 00111). With the base: 57 bits:
    # 00 00 00 80 | 18 10 CA 01. (A signed delta would make X32 zero instead.)
    blk = u32([0x80000000] + [0] * 31)
    n, payload = oracle.encode_candidate(blk, 4, oracle.TAG_DBX)
    assert n == 57
    assert payload.hex(" ") == "00 00 00 80 18 10 ca 01"


def test_bf16_symbol_order_pins_little_endian_halves():
    # R2: BF16 symbols are little-endian half-words in memory order. Bytes
    # 01 00 00 00 ... give s_0 = 1 (BX: run15 6 + single one 11 = 17 bits);
    # bytes 00 01 ... give s_0 = 0x0100, g = 0x0180: X15..X9 run 7 (6), X8 single
    # one (11), X7 pre-XOR zero (5), X6..X0 run 7 (6) = 28.
    a = bytes([1, 0]) + bytes(126)
    b = bytes([0, 1]) + bytes(126)
    assert oracle.block_candidates(a, 2)[0][oracle.TAG_BX] == 17
    assert oracle.block_candidates(b, 2)[0][oracle.TAG_BX] == 28


# ----------------------------------------------------------- closed forms

def test_zvc_and_raw_closed_forms():
    rng = np.random.default_rng(11)
    for ew, w, N in ((4, 32, 32), (2, 16, 64)):
        for _ in range(200):
            sym = rng.integers(1, 1 << w, N, dtype=np.uint64)
            sym[rng.random(N) < rng.random()] = 0
            blk = sym.astype("<u4" if w == 32 else "<u2").tobytes()
            n = int(np.count_nonzero(sym))
            enc, model, _ = oracle.block_candidates(blk, ew)
            assert enc[oracle.TAG_ZVC] == N + n * w == model[oracle.TAG_ZVC]
            assert enc[oracle.TAG_RAW] == 1024


def test_zero_chunk_sizes():
    # FP32: 32 blocks x (3 + 7) bits = 320 bits = 40 bytes + 2 header bytes.
    # BF16: 32 blocks x (3 + 6) bits = 288 bits = 36 bytes + 2.
    assert len(oracle.compress(bytes(4096), 4)) == 42
    assert len(oracle.compress(bytes(4096), 2)) == 38


def test_random_chunk_is_raw():
    # random words: ZVC 1056, BX 1056, DBX 1088, ZBX 1088 > RAW 1024, so each
    # block is 1027 bits; 32 * 1027 > 8 * 4096, so the chunk is stored raw.
    rng = np.random.default_rng(5)
    data = rng.integers(0, 256, 4096, dtype=np.uint8).tobytes()
    for ew in (4, 2):
        s = oracle.compress(data, ew)
        assert len(s) == 4098
        assert s[:2] == bytes([0x00, 0x10]) and s[2:] == data
        assert abs(4096 / len(s) - 0.99951) < 1e-5
        enc, _, tag = oracle.block_candidates(data[:128], ew)
        assert tag == oracle.TAG_RAW


def test_chunk_of_raw_blocks_is_raw_chunk():
    rng = np.random.default_rng(6)
    data = rng.integers(0, 256, 3 * 4096 + 700, dtype=np.uint8).tobytes()
    tags, bits, lens = oracle.analyze(data, 4)
    assert list(lens) == [4096, 4096, 4096, 700]
    assert (tags == 255).all()


def test_tail_sizes_round_trip_and_raw_rule():
    rng = np.random.default_rng(8)
    for n in W.TAIL_SIZES:
        for data in (bytes(n), rng.integers(0, 256, n, dtype=np.uint8).tobytes(),
                     W.relu_values(n // 4 + 1, rng).tobytes()[:n]):
            for ew in (4, 2):
                s = oracle.compress(data, ew)
                C = (n + 4095) // 4096
                assert len(s) >= 2 * C
                lens = np.frombuffer(s[:2 * C], dtype="<u2")
                raw_lens = [min(4096, n - 4096 * c) for c in range(C)]
                assert all(1 <= L <= r for L, r in zip(lens, raw_lens))
                assert len(s) == 2 * C + int(lens.sum())
                assert oracle.decompress(s, n, ew) == data


# --------------------------------------------- model vs encoder, selection

def _all_test_blocks():
    out = []
    out += [(b, 4) for b in blocks(W.edge_blocks_fp32().tobytes())]
    out += [(b, 2) for b in blocks(W.edge_blocks_fp32().tobytes())]
    out += [(b, 2) for b in blocks(W.edge_blocks_bf16().tobytes())]
    out += [(b, 4) for b in blocks(W.edge_blocks_bf16().tobytes())]
    out += [(b, 4) for b in blocks(W.tiny_alphabet_blocks(300, "fp32").tobytes())]
    out += [(b, 2) for b in blocks(W.tiny_alphabet_blocks(300, "bf16").tobytes())]
    rng = np.random.default_rng(9)
    out += [(b, 4) for b in blocks(W.relu_values(32 * 64, rng).tobytes())]
    out += [(b, 2) for b in blocks(W.f32_to_bf16_rne(W.relu_values(64 * 64, rng)).tobytes())]
    out += [(b, 4) for b in blocks(W.gelu_values(32 * 64, rng).tobytes())]
    out += [(b, 2) for b in blocks(W.f32_to_bf16_rne(W.gelu_values(64 * 64, rng)).tobytes())]
    return out


def test_size_model_equals_encoder_bits():
    # Section III-A "Validation": the size model and the bit-exact encoder
    # must agree exactly on every candidate of every block.
    for blk, ew in _all_test_blocks():
        enc, model, _ = oracle.block_candidates(blk, ew)
        assert enc == model, (ew, blk.hex(), enc, model)


def test_selected_tag_is_first_minimum():
    for blk, ew in _all_test_blocks():
        enc, _, tag = oracle.block_candidates(blk, ew)
        assert enc[tag] == min(enc)
        assert tag == enc.index(min(enc))


def test_all_zero_block_selects_the_minimum_not_zvc():
    # The paper keeps the smallest candidate. An all-zero block costs ZVC = N,
    # but BX codes all w planes as one zero run: 7 bits (FP32), 6 bits (BF16).
    for ew, bx, N in ((4, 7, 32), (2, 6, 64)):
        enc, _, tag = oracle.block_candidates(bytes(128), ew)
        assert tag == oracle.TAG_BX and enc[oracle.TAG_BX] == bx
        assert enc[oracle.TAG_ZVC] == N == enc[oracle.TAG_ZBX]


# ------------------------------------------------------------- round trip

def test_round_trip_edge_and_tiny_alphabet_blocks():
    for blk, ew in _all_test_blocks():
        s = oracle.compress(blk, ew)
        assert oracle.decompress(s, 128, ew) == blk


def test_round_trip_every_candidate_decodes():
    # force every candidate through the decoder by building one-block streams
    # by hand: tag + candidate payload, byte-padded, and a header L (< 128).
    for blk, ew in _all_test_blocks()[:400]:
        for tag in range(5):
            n, payload = oracle.encode_candidate(blk, ew, tag)
            bits = 3 + n
            L = (bits + 7) // 8
            if L >= 128:
                continue
            body = np.zeros(L + 1, dtype=np.uint8)
            acc = tag | (int.from_bytes(payload, "little") << 3)
            body[:L] = np.frombuffer(acc.to_bytes(L + 1, "little")[:L], dtype=np.uint8)
            stream = bytes([L & 0xFF, L >> 8]) + body[:L].tobytes()
            assert oracle.decompress(stream, 128, ew) == blk, (tag, ew)


def test_round_trip_multi_chunk_tensors():
    rng = np.random.default_rng(10)
    data = np.concatenate([
        W.edge_blocks_fp32(), W.relu_values(3000, rng).view(np.uint8),
        W.f32_to_bf16_rne(W.gelu_values(5000, rng)).view(np.uint8),
        rng.integers(0, 256, 5000, dtype=np.uint8)]).tobytes()
    for ew in (4, 2, 1, 8):
        s = oracle.compress(data, ew)
        assert oracle.decompress(s, len(data), ew) == data


def test_chunk_aligned_split_concatenates():
    # Section III-A "Stream format": every 4 KB chunk is coded on its own, so
    # splitting the input at chunk boundaries and compressing each piece gives
    # the pieces' size tables and payloads, which concatenate (all tables,
    # then all payloads) into the whole input's stream.
    rng = np.random.default_rng(11)
    data = np.concatenate([
        W.relu_values(4096 * 3, rng).view(np.uint8), rng.integers(0, 256, 4096 * 2, dtype=np.uint8),
        np.zeros(4096 * 2, np.uint8), W.f32_to_bf16_rne(W.gelu_values(4096 * 2 + 777, rng)).view(np.uint8)]).tobytes()
    n = len(data)
    C = (n + 4095) // 4096
    for ew in (4, 2):
        whole = oracle.compress(data, ew)
        for cuts in ([0, C], [0, 1, C], [0, 3, 5, 8, C], list(range(C + 1))):
            heads, bodies = [], []
            for a, b in zip(cuts[:-1], cuts[1:]):
                s = oracle.compress(data[4096 * a: min(n, 4096 * b)], ew)
                heads.append(s[:2 * (b - a)])
                bodies.append(s[2 * (b - a):])
            assert b"".join(heads) + b"".join(bodies) == whole, (ew, cuts)


def test_ratio_accounting_includes_tags_headers_and_padding():
    rng = np.random.default_rng(12)
    data = W.relu_values(5 * 1024 + 77, rng).tobytes()
    s = oracle.compress(data, 4)
    C = (len(data) + 4095) // 4096
    lens = np.frombuffer(s[:2 * C], dtype="<u2").astype(int)
    tags, bits, lens2 = oracle.analyze(data, 4)
    assert (lens == lens2).all()
    # per compressed chunk: L = ceil(sum of block bits incl. 3-bit tags / 8)
    for c in range(C):
        raw_len = min(4096, len(data) - 4096 * c)
        b = bits[32 * c: 32 * c + (raw_len + 127) // 128]
        if lens[c] < raw_len:
            assert lens[c] == (int(b.sum()) + 7) // 8
    assert len(s) == 2 * C + lens.sum()
    assert len(data) / len(s) == pytest.approx(len(data) / (2 * C + lens.sum()))


# ---------------------------------------------------------- corrupt input

def test_corrupt_headers_and_tags_are_reported():
    data = W.relu_values(2048, np.random.default_rng(13)).tobytes()  # 2 chunks
    s = bytearray(oracle.compress(data, 4))
    C = 2
    assert oracle.decompress_status(bytes(s), len(data), 4)[0] == oracle.OK
    bad = bytearray(s); bad[0:2] = (0).to_bytes(2, "little")          # L = 0
    assert oracle.decompress_status(bytes(bad), len(data), 4)[0] == oracle.ERR_CORRUPT
    bad = bytearray(s); bad[0:2] = (4097).to_bytes(2, "little")       # L > raw
    assert oracle.decompress_status(bytes(bad), len(data), 4)[0] == oracle.ERR_CORRUPT
    assert oracle.decompress_status(bytes(s[:-1]), len(data), 4)[0] == oracle.ERR_CORRUPT  # truncated
    assert oracle.decompress_status(bytes(s[:2 * C + 1]), len(data), 4)[0] == oracle.ERR_CORRUPT
    assert oracle.decompress_status(bytes(s[:1]), len(data), 4)[0] == oracle.ERR_ARG      # < 2C
    bad = bytearray(s); bad[2 * C] = (bad[2 * C] & ~7) | 5             # tag 5
    assert oracle.decompress_status(bytes(bad), len(data), 4)[0] == oracle.ERR_CORRUPT


def test_random_bit_flips_never_crash():
    rng = np.random.default_rng(14)
    data = W.relu_values(4096, rng).tobytes()
    s = oracle.compress(data, 4)
    for _ in range(300):
        bad = bytearray(s)
        pos = int(rng.integers(0, len(bad) * 8))
        bad[pos // 8] ^= 1 << (pos % 8)
        rc, out = oracle.decompress_status(bytes(bad), len(data), 4)
        assert rc in (oracle.OK, oracle.ERR_CORRUPT)
