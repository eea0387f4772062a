"""Pins of the oracle's restricted block selection (candidate masks).

The paper compares PlaneZip with single encodings applied to every block
(Section V-A, Fig. 3: ZVC, BPC = DBX on every block, the best single
encoding). A candidate mask (bit t = tag t) restricts the per-block choice;
the raw block always stays allowed, and a chunk that would grow is still
stored raw (Section III-A "Stream format"). What pins it, independently of
the restricted encoder itself:
  - the block's size equals 3 + the minimum over the allowed candidates of
    the independent size model's lengths (ties to the lowest tag);
  - closed forms for all-zero chunks and ramps (from the code lengths);
  - the full candidate set reproduces the unrestricted stream byte for byte;
  - every restricted stream round-trips, and none is shorter than the full one.
"""
import numpy as np
import pytest

import oracle
from lossless_bit_plane_gb300 import workloads as W

MASKS = {
    "zvc": 1 << oracle.TAG_ZVC,
    "dbx": 1 << oracle.TAG_DBX,
    "bx": 1 << oracle.TAG_BX,
    "zbx": 1 << oracle.TAG_ZBX,
    "raw": 1 << oracle.TAG_RAW,
    "zvc+zbx": (1 << oracle.TAG_ZVC) | (1 << oracle.TAG_ZBX),
    "dbx+bx": (1 << oracle.TAG_DBX) | (1 << oracle.TAG_BX),
}


def _cases():
    rng = np.random.default_rng(11)
    relu = W.relu_values(8192, rng).view(np.uint8)                       # 32 KB FP32, 8 chunks
    gelu16 = W.f32_to_bf16_rne(W.gelu_values(8192, rng)).view(np.uint8)  # 16 KB BF16
    return [
        ("edge_fp32", W.edge_blocks_fp32(), 4),
        ("edge_fp32_as16", W.edge_blocks_fp32(), 2),
        ("edge_bf16", W.edge_blocks_bf16(), 2),
        ("relu_fp32", relu, 4),
        ("gelu_bf16", gelu16, 2),
        ("tiny_fp32", W.tiny_alphabet_blocks(64, "fp32"), 4),
        ("tiny_bf16", W.tiny_alphabet_blocks(64, "bf16"), 2),
    ]


CASES = _cases()


@pytest.mark.parametrize("name,data,ew", CASES, ids=[c[0] for c in CASES])
def test_all_candidates_is_the_unrestricted_stream(name, data, ew):
    assert oracle.compress(data, ew, oracle.CAND_ALL) == oracle.compress(data, ew)


@pytest.mark.parametrize("mask_name", list(MASKS))
@pytest.mark.parametrize("name,data,ew", CASES, ids=[c[0] for c in CASES])
def test_restricted_choice_is_the_allowed_minimum(name, data, ew, mask_name):
    mask = MASKS[mask_name] | (1 << oracle.TAG_RAW)
    buf = np.ascontiguousarray(data).view(np.uint8).reshape(-1)
    tags, bits, lens = oracle.analyze(buf, ew, mask)
    stream = oracle.compress(buf, ew, mask)
    for b in range(tags.size):
        if tags[b] == 255:  # block of a chunk stored raw
            continue
        assert (mask >> int(tags[b])) & 1, (b, tags[b])
        block = np.zeros(128, dtype=np.uint8)
        chunk = buf[128 * b: 128 * b + 128]
        block[: chunk.size] = chunk
        _, model, _ = oracle.block_candidates(block, ew)
        allowed = [t for t in range(5) if (mask >> t) & 1]
        best = min(allowed, key=lambda t: (model[t], t))
        assert int(tags[b]) == best and int(bits[b]) == 3 + model[best], (b, model)
    # the stream decodes back and is never shorter than the unrestricted one
    assert oracle.decompress(stream, buf.size, ew) == buf.tobytes()
    assert len(stream) >= len(oracle.compress(buf, ew))
    C = (buf.size + 4095) // 4096
    assert len(stream) == 2 * C + int(lens.astype(np.int64).sum())


def test_raw_only_mask_stores_every_chunk_raw():
    buf = W.relu_values(4096, np.random.default_rng(3)).view(np.uint8)  # 16 KB
    stream = oracle.compress(buf, 4, 1 << oracle.TAG_RAW)
    C = buf.size // 4096
    assert len(stream) == 2 * C + buf.size
    assert all(int.from_bytes(stream[2 * c: 2 * c + 2], "little") == 4096 for c in range(C))


@pytest.mark.parametrize("mask_name,ew,L", [
    ("zvc", 4, (32 * (3 + 32) + 7) // 8),   # ZVC = N bits when every symbol is zero
    ("zvc", 2, (32 * (3 + 64) + 7) // 8),
    ("dbx", 4, (32 * (3 + 32 + 7) + 7) // 8),  # base 32 + one zero run over 33 planes (2 + 5)
    ("dbx", 2, (32 * (3 + 16 + 6) + 7) // 8),  # base 16 + one zero run over 17 planes (2 + 4)
    ("bx", 4, 40),                           # the unrestricted choice: 32 x 10 bits
    ("zbx", 4, (32 * (3 + 32) + 7) // 8),    # mask only when n = 0
])
def test_all_zero_chunk_closed_forms(mask_name, ew, L):
    stream = oracle.compress(np.zeros(4096, np.uint8), ew, MASKS[mask_name] | (1 << oracle.TAG_RAW))
    assert len(stream) == 2 + L
    assert int.from_bytes(stream[:2], "little") == L


def test_bpc_on_an_integer_ramp():
    # s_k = k: DBX = base 32 + zero run over planes 32..1 (2 + 5) + all-ones plane 0 (5) = 44 bits,
    # plus the tag: 47 bits per block, with DBX the only allowed coded candidate
    ramp = np.tile(np.arange(32, dtype=np.uint32), 32)
    tags, bits, lens = oracle.analyze(ramp.view(np.uint8), 4, MASKS["dbx"] | (1 << oracle.TAG_RAW))
    assert set(tags.tolist()) == {oracle.TAG_DBX}
    assert set(bits.tolist()) == {47}
    assert lens.tolist() == [(32 * 47 + 7) // 8]
