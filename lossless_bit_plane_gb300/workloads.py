"""Seeded synthetic inputs for the PlaneZip block codec.

This module only MAKES input bytes; it holds none of the codec's arithmetic.
Both the CUDA path's tests and the CPU oracle's tests draw their inputs from
here, so that the two sides see identical bytes.

The paper ("PlaneZip: Lossless Bit-Plane Compression of Training Activations
Offloaded over PCIe", Section IV "Methodology" and Table III) measures
activations captured from five trained models. Those tensors are not
available, so these generators stand in for them with the structure that the
paper names for each producer: ReLU zeros, smooth convolution maps, causally
masked softmax rows, GELU and LayerNorm outputs, and BF16 tensors obtained by
round-to-nearest-even from FP32 (Section IV).

Every generator uses ``numpy.random.Generator(PCG64(seed))`` and is
deterministic across machines.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np

MiB = 1 << 20


# --------------------------------------------------------------------------
# Element conversions (input preparation, not codec arithmetic)
# --------------------------------------------------------------------------

def f32_to_bf16_rne(x) -> np.ndarray:
    """FP32 -> BF16 bit patterns by round-to-nearest-even; NaN -> quiet NaN."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = ((u.astype(np.uint64) + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    if nan.any():
        rounded = np.where(nan, ((u >> 16) | 0x0040).astype(np.uint16), rounded)
    return rounded


def as_dtype_bytes(x_f32: np.ndarray, dtype: str) -> np.ndarray:
    """Flat uint8 view of an FP32 array stored as 'fp32' or 'bf16'."""
    if dtype == "fp32":
        return np.ascontiguousarray(x_f32, dtype=np.float32).reshape(-1).view(np.uint8)
    if dtype == "bf16":
        return f32_to_bf16_rne(x_f32.reshape(-1)).view(np.uint8)
    raise ValueError(dtype)


def elem_width(dtype: str) -> int:
    return {"fp32": 4, "bf16": 2, "u32": 4}[dtype]


def sha256(buf: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(buf).view(np.uint8).tobytes()).hexdigest()


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# --------------------------------------------------------------------------
# Distributions (FP32 values, generated in FP64 where a formula is applied)
# --------------------------------------------------------------------------

def relu_values(n: int, rng: np.random.Generator) -> np.ndarray:
    """Post-ReLU activations: 0 with probability 0.5, else |N(0,1)|."""
    v = np.abs(rng.standard_normal(n)).astype(np.float32)
    v[rng.random(n) < 0.5] = 0.0
    return v


def _gauss_taps(sigma: float = 2.0, radius: int = 6) -> np.ndarray:
    t = np.arange(-radius, radius + 1, dtype=np.float64)
    w = np.exp(-0.5 * (t / sigma) ** 2)
    return w / w.sum()


def conv_fields(nfields: int, h: int, w: int, gains: np.ndarray, rng: np.random.Generator) -> np.ndarray:
    """Smooth post-ReLU conv maps: per field an N(0,1) image blurred separably
    with a Gaussian (sigma 2 px, radius 6, reflect boundary) in FP64, times a
    per-field gain, then ReLU; returned as FP32 [nfields, h, w]."""
    taps = _gauss_taps()
    r = (taps.size - 1) // 2
    out = np.empty((nfields, h, w), dtype=np.float32)
    step = 256
    for f0 in range(0, nfields, step):
        f1 = min(nfields, f0 + step)
        x = rng.standard_normal((f1 - f0, h, w))
        xp = np.pad(x, ((0, 0), (r, r), (0, 0)), mode="reflect")
        y = sum(taps[i] * xp[:, i:i + h, :] for i in range(taps.size))
        yp = np.pad(y, ((0, 0), (0, 0), (r, r)), mode="reflect")
        z = sum(taps[i] * yp[:, :, i:i + w] for i in range(taps.size))
        z *= gains[f0:f1, None, None]
        np.maximum(z, 0.0, out=z)
        out[f0:f1] = z.astype(np.float32)
    return out


def causal_softmax_rows(nmat: int, seq: int, rng: np.random.Generator) -> np.ndarray:
    """Causally masked attention probabilities: row i is the softmax of N(0,1)
    logits over columns j <= i (FP64 -> FP32); columns j > i are exactly 0."""
    out = np.empty((nmat, seq, seq), dtype=np.float32)
    mask = np.tril(np.ones((seq, seq), dtype=bool))
    for m in range(nmat):
        x = rng.standard_normal((seq, seq))
        x = np.where(mask, x, -np.inf)
        x -= x.max(axis=1, keepdims=True)
        e = np.exp(x)
        out[m] = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return out


def gelu_values(n: int, rng: np.random.Generator) -> np.ndarray:
    """Exact GELU x * Phi(x) of N(0,1) inputs, computed in FP64."""
    from scipy.special import erf

    out = np.empty(n, dtype=np.float32)
    step = 1 << 22
    for i in range(0, n, step):
        x = rng.standard_normal(min(step, n - i))
        out[i:i + x.size] = (x * 0.5 * (1.0 + erf(x / np.sqrt(2.0)))).astype(np.float32)
    return out


def layernorm_values(rows: int, features: int, rng: np.random.Generator) -> np.ndarray:
    """LayerNorm outputs N(0,1) * gamma + beta, gamma ~ U(0.5, 1.5) and
    beta ~ N(0, 0.1^2) per feature (0.1 read as the standard deviation)."""
    gamma = rng.uniform(0.5, 1.5, features)
    beta = rng.normal(0.0, 0.1, features)
    out = np.empty((rows, features), dtype=np.float32)
    step = 4096
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        out[r0:r1] = (rng.standard_normal((r1 - r0, features)) * gamma + beta).astype(np.float32)
    return out


# --------------------------------------------------------------------------
# The five workloads
# --------------------------------------------------------------------------

@dataclass
class Tensor:
    name: str
    dtype: str        # 'fp32', 'bf16' or 'u32'
    data: np.ndarray  # flat uint8

    @property
    def elem_width(self) -> int:
        return elem_width(self.dtype)

    @property
    def nbytes(self) -> int:
        return int(self.data.size)


def relu_fp32_4mib(seed: int = 0) -> Tensor:
    """FP32 post-ReLU tensor of 1,048,576 elements (4 MiB, 1024 chunks)."""
    return Tensor("relu_fp32_4MiB", "fp32", as_dtype_bytes(relu_values(1 << 20, _rng(seed)), "fp32"))


def conv_bf16(seed: int = 1, shape=(32, 64, 56, 56)) -> Tensor:
    """BF16 conv feature map NCHW [32,64,56,56]: per-(n,c) blurred N(0,1)
    fields, per-channel gain U(0.1,4) shared across n, ReLU, RNE to BF16."""
    rng = _rng(seed)
    n, c, h, w = shape
    gain_c = rng.uniform(0.1, 4.0, c)
    gains = np.tile(gain_c, n)
    x = conv_fields(n * c, h, w, gains, rng)
    return Tensor("conv_bf16_[32,64,56,56]", "bf16", as_dtype_bytes(x, "bf16"))


def attention_bf16(seed: int = 2, batch: int = 8, heads: int = 12, seq: int = 1024) -> Tensor:
    """BF16 causal attention probabilities [8,12,1024,1024] (192 MiB)."""
    rng = _rng(seed)
    parts = [f32_to_bf16_rne(causal_softmax_rows(1, seq, rng)[0].reshape(-1)) for _ in range(batch * heads)]
    return Tensor("attention_bf16_[8,12,1024,1024]", "bf16", np.concatenate(parts).view(np.uint8))


def mlp_ln(seed: int = 3, dtype: str = "fp32") -> list[Tensor]:
    """GELU output [8,1024,3072] and LayerNorm output [8,1024,768]."""
    rng = _rng(seed)
    g = gelu_values(8 * 1024 * 3072, rng)
    ln = layernorm_values(8 * 1024, 768, rng)
    return [Tensor(f"gelu_{dtype}_[8,1024,3072]", dtype, as_dtype_bytes(g, dtype)),
            Tensor(f"layernorm_{dtype}_[8,1024,768]", dtype, as_dtype_bytes(ln, dtype))]


SWEEP_SEGMENTS = (
    ("relu", "fp32"), ("relu", "bf16"),
    ("conv", "fp32"), ("conv", "bf16"),
    ("attention", "fp32"), ("attention", "bf16"),
    ("random", "u32"),
)


def sweep_segment(kind: str, dtype: str, seed: int = 4, seg_bytes: int = 128 * MiB) -> Tensor:
    """One segment of the 1 GiB sweep: 128 MiB of a config 1-3 distribution in
    FP32 or BF16, or 256 MiB of uniform random u32 (the raw-fallback case)."""
    idx = SWEEP_SEGMENTS.index((kind, dtype))
    rng = _rng(seed * 1000 + idx)
    if kind == "random":
        nbytes = 2 * seg_bytes
        data = rng.integers(0, 1 << 32, nbytes // 4, dtype=np.uint32).view(np.uint8)
        return Tensor("random_u32_256MiB", "u32", data)
    n = seg_bytes // (4 if dtype == "fp32" else 2)
    if kind == "relu":
        x = relu_values(n, rng)
    elif kind == "conv":
        per = 56 * 56
        nf = -(-n // per)
        gains = rng.uniform(0.1, 4.0, 64)
        x = conv_fields(nf, 56, 56, np.resize(gains, nf), rng).reshape(-1)[:n]
    elif kind == "attention":
        seq = 1024
        x = np.concatenate([causal_softmax_rows(1, seq, rng)[0].reshape(-1) for _ in range(n // (seq * seq))])
    else:
        raise ValueError(kind)
    return Tensor(f"{kind}_{dtype}_128MiB", dtype, as_dtype_bytes(x, dtype))


def sweep_1gib(seed: int = 4) -> list[Tensor]:
    """The 1 GiB throughput sweep: 7 segments, compressed one call each."""
    return [sweep_segment(k, d, seed) for k, d in SWEEP_SEGMENTS]


# --------------------------------------------------------------------------
# Edge blocks and small-alphabet blocks
# --------------------------------------------------------------------------

F32 = {
    "one": 0x3F800000, "m2.5": 0xC0200000, "maxf": 0x7F7FFFFF, "qnan": 0x7FC00000,
    "snan": 0x7F800001, "inf": 0x7F800000, "ninf": 0xFF800000, "nzero": 0x80000000,
    "minsub": 0x00000001, "maxsub": 0x007FFFFF, "ones": 0xFFFFFFFF,
}
TINY_ALPHABET_32 = np.array([0, 1, 0x80000000, 0x3F800000, 0x7FC00000, 0xFFFFFFFF], dtype=np.uint32)
TINY_ALPHABET_16 = np.array([0, 1, 0x8000, 0x3F80, 0x7FC0, 0xFFFF], dtype=np.uint16)


def edge_blocks_fp32(seed: int = 0) -> np.ndarray:
    """64 hand-built 128-byte blocks (32 words each), returned as flat uint8.

    All-zero, -0, +-0 mixes, constants, ramps, alternating signs, NaN and Inf
    payloads, subnormals, single and adjacent non-zeros at the start, middle
    and end, all-ones words, random words, zero/value interleaves, and
    constants and sparse words chosen so that every plane code (zero runs of
    many lengths, single zeros, all-ones, pre-XOR-zero, one and two adjacent
    ones, verbatim) appears at top, middle and bottom planes."""
    rng = _rng(seed + 100)
    k = np.arange(32, dtype=np.uint32)
    B = []

    def const(v):
        B.append(np.full(32, v, dtype=np.uint32))

    def sparse(pos, vals):
        b = np.zeros(32, dtype=np.uint32)
        b[list(pos)] = vals
        B.append(b)

    const(0)                                                    # all +0
    const(F32["nzero"])                                          # all -0
    B.append(np.where(k % 2 == 0, 0, F32["nzero"]).astype(np.uint32))  # +-0 alternating
    const(F32["one"]); const(F32["m2.5"]); const(F32["maxf"])    # constants
    B.append(k.copy())                                           # integer ramp
    B.append((k.astype(np.float32) * 0.5).view(np.uint32))       # float ramp k*0.5
    B.append(np.where(k % 2 == 0, 1.5, -1.5).astype(np.float32).view(np.uint32))  # alternating +-x
    const(F32["qnan"])
    B.append((F32["snan"] + k).astype(np.uint32))                # sNaN payloads
    const(F32["inf"]); const(F32["ninf"])
    B.append(np.where(k % 2 == 0, F32["inf"], F32["ninf"]).astype(np.uint32))
    const(F32["minsub"]); const(F32["maxsub"])
    sparse([0], [0x12345678]); sparse([16], [0x12345678]); sparse([31], [0x12345678])
    sparse([7, 8], [0x3F800000, 0x3F800000])                     # two adjacent non-zeros
    const(F32["ones"])
    B.append(rng.integers(0, 1 << 32, 32, dtype=np.uint64).astype(np.uint32))  # random u32
    B.append(np.where(k % 2 == 0, 0, (1.0 + k * 2.0 ** -20)).astype(np.float32).view(np.uint32))
    B.append(np.where(k % 2 == 1, 0, (1.0 + k * 2.0 ** -20)).astype(np.float32).view(np.uint32))
    B.append((31 - k).astype(np.uint32))                         # descending ramp
    B.append(np.resize(np.array([F32["qnan"], F32["inf"], F32["minsub"], 0, F32["nzero"],
                                 F32["maxsub"], F32["ninf"], F32["snan"]], dtype=np.uint32), 32))
    B.append((np.uint32(1) << k).astype(np.uint32))               # one-hot powers of two
    sparse([5], [0x80000000]); sparse([3], [1 << 16]); sparse([9], [1])       # single one: top/mid/bottom
    sparse([4, 5], [0x80000000] * 2); sparse([10, 11], [1 << 15] * 2); sparse([30, 31], [1, 1])  # two adjacent
    B.append(np.where(k % 2 == 0, 0x40000000, 0x60000000).astype(np.uint32))  # pre-XOR-zero planes
    B.append((0x80000000 | (k << 8)).astype(np.uint32))          # all-ones top plane
    for c in (0x00000001, 0x33333333, 0xCCCCCCCC, 0x0F0F0F0F, 0x00FF00FF, 0x0000FFFF,
              0xFFFF0000, 0x7FFFFFFF, 0x55555555, 0xAAAAAAAA, 0x00010000):
        const(c)                                                 # runs of many lengths
    for n in (1, 2, 3, 4, 5, 7, 9):                              # few survivors: tiny ZBX planes
        b = np.zeros(32, dtype=np.uint32)
        pos = rng.choice(32, n, replace=False)
        b[pos] = 0x3F800000 | rng.integers(0, 1 << 10, n, dtype=np.uint64).astype(np.uint32)
        B.append(b)
    while len(B) < 64:                                           # small-alphabet blocks
        B.append(TINY_ALPHABET_32[rng.integers(0, TINY_ALPHABET_32.size, 32)])
    arr = np.stack(B[:64]).astype("<u4")
    return arr.reshape(-1).view(np.uint8)


def edge_blocks_bf16(seed: int = 0) -> np.ndarray:
    """64 BF16 blocks (64 half-words each): the BF16 analogues of the FP32
    edge blocks, returned as flat uint8."""
    rng = _rng(seed + 200)
    k = np.arange(64, dtype=np.uint32)
    B = []

    def const(v):
        B.append(np.full(64, v, dtype=np.uint16))

    def sparse(pos, vals):
        b = np.zeros(64, dtype=np.uint16)
        b[list(pos)] = vals
        B.append(b)

    const(0); const(0x8000)
    B.append(np.where(k % 2 == 0, 0, 0x8000).astype(np.uint16))
    const(0x3F80); const(0xC020); const(0x7F7F)
    B.append(k.astype(np.uint16))
    B.append(f32_to_bf16_rne(k.astype(np.float32) * 0.5))
    B.append(f32_to_bf16_rne(np.where(k % 2 == 0, 1.5, -1.5)))
    const(0x7FC0); B.append((0x7F81 + k).astype(np.uint16)); const(0x7F80); const(0xFF80)
    B.append(np.where(k % 2 == 0, 0x7F80, 0xFF80).astype(np.uint16))
    const(0x0001); const(0x007F)
    sparse([0], [0x1234]); sparse([32], [0x1234]); sparse([63], [0x1234]); sparse([31], [0x1234])
    sparse([31, 32], [0x3F80, 0x3F80])                           # adjacent across the half split
    sparse([7, 8], [0x3F80, 0x3F80])
    const(0xFFFF)
    B.append(rng.integers(0, 1 << 16, 64, dtype=np.uint64).astype(np.uint16))
    B.append(np.where(k % 2 == 0, 0, 0x3F80 + (k % 8)).astype(np.uint16))
    B.append(np.where(k % 2 == 1, 0, 0x3F80 + (k % 8)).astype(np.uint16))
    B.append((63 - k).astype(np.uint16))
    B.append(((np.uint32(1) << (k % 16))).astype(np.uint16))
    sparse([5], [0x8000]); sparse([40], [1 << 8]); sparse([9], [1])
    sparse([4, 5], [0x8000] * 2); sparse([40, 41], [1 << 7] * 2); sparse([62, 63], [1, 1])
    B.append(np.where(k < 32, 0, 0x3F80).astype(np.uint16))      # zeros then survivors
    B.append(np.where(k >= 32, 0, 0x3F80).astype(np.uint16))     # survivors then zeros
    for c in (0x3333, 0xCCCC, 0x0F0F, 0x00FF, 0x7FFF, 0x5555, 0xAAAA, 0x0100):
        const(c)
    for n in (1, 2, 3, 4, 5, 7, 9, 33):
        b = np.zeros(64, dtype=np.uint16)
        pos = rng.choice(64, n, replace=False)
        b[pos] = 0x3F00 | rng.integers(0, 1 << 7, n, dtype=np.uint64).astype(np.uint16)
        B.append(b)
    while len(B) < 64:
        B.append(TINY_ALPHABET_16[rng.integers(0, TINY_ALPHABET_16.size, 64)])
    arr = np.stack(B[:64]).astype("<u2")
    return arr.reshape(-1).view(np.uint8)


def tiny_alphabet_blocks(nblocks: int, dtype: str, seed: int = 7) -> np.ndarray:
    """Random blocks whose symbols come from a six-value alphabet
    ({0, 1, -0, 1.0, qNaN, all-ones} and the BF16 analogues)."""
    rng = _rng(seed)
    if dtype == "bf16":
        return TINY_ALPHABET_16[rng.integers(0, 6, nblocks * 64)].astype("<u2").view(np.uint8)
    return TINY_ALPHABET_32[rng.integers(0, 6, nblocks * 32)].astype("<u4").view(np.uint8)



def verbatim_run_blocks(nchunks: int, elem_width: int, seed: int = 89) -> np.ndarray:
    """Blocks whose symbols share their top k bits (a constant of the block)
    over uniform random low bits, k cycling through 0..w across blocks (w =
    8 x elem_width): the top k planes are constant and the low w - k random,
    so coded blocks carry verbatim-plane runs of every length."""
    rng = _rng(seed)
    w = 8 * elem_width
    nblk = nchunks * 32
    k = (np.arange(nblk, dtype=np.uint64) % np.uint64(w + 1))[:, None]
    lowmask = (np.uint64(1) << (np.uint64(w) - k)) - np.uint64(1)
    low = rng.integers(0, 1 << w, (nblk, 128 // elem_width), dtype=np.uint64)
    top = rng.integers(0, 1 << w, (nblk, 1), dtype=np.uint64)
    vals = (top & ~lowmask) | (low & lowmask)
    return vals.astype("<u4" if elem_width == 4 else "<u2").view(np.uint8).reshape(-1)

TAIL_SIZES = (0, 2, 4, 126, 128, 130, 4094, 4096, 4098)
