// pz_format.cuh — the PlaneZip stream format as this library writes it.
//
// Paper: "PlaneZip: Lossless Bit-Plane Compression of Training Activations
// Offloaded over PCIe" (arXiv:2610.25033v1), Section III-A "Codec" and
// "Stream format"; Section II-B for BPC's delta bit-plane XOR transform.
//
// The paper fixes block (128 B), symbol widths (w = 16, N = 64 for BF16;
// w = 32, N = 32 for every other element type), the candidates, the plane
// code LENGTHS, the 3-bit tag, the 4 KB chunk and the 16-bit size. Where it
// leaves the layout open, this library fixes it as follows:
//   - LSB-first bit order; an m-bit field is written bit 0 first.
//   - Symbols are little-endian unsigned; "zero" means all w bits zero.
//   - Tags: ZVC 0, DBX 1, BX 2, ZBX 3, RAW 4; a block keeps the smallest
//     candidate, ties to the lowest tag; payload follows the tag directly.
//   - ZVC: N-bit non-zero mask (symbol 0 first), then the non-zero symbols.
//   - DBX: base s_0 in w bits, then the w+1 planes of the deltas
//     d_j = (s_j - s_{j-1}) mod 2^(w+1), j = 1..N-1, unsigned (bit w is the
//     borrow); plane width N-1.
//   - BX: the w planes of the symbols, width N.
//   - ZBX: N-bit mask, then BX over the n non-zero symbols in index order,
//     width n; nothing more when n = 0.
//   - RAW: the 128 block bytes.
//   - Planes are XORed with the plane above (X_top = P_top,
//     X_i = P_i ^ P_{i+1}), i.e. the planes of g = v ^ (v >> 1) in P-bit
//     arithmetic, and coded top plane first:
//       zero run of L >= 2 planes   0 1 + (L-2) in K bits
//       single zero plane           0 0 1
//       all-ones plane              0 0 0 0 0
//       pre-XOR plane P_i zero      0 0 0 0 1     (below the top plane only)
//       two adjacent ones q, q+1    0 0 0 1 0 + q in p bits
//       single one at q             0 0 0 1 1 + q in p bits
//       verbatim                    1 + the W plane bits, bit 0 first
//     K = ceil(log2(P-1)) (5 for 32/33 planes, 4 for 16/17), p =
//     ceil(log2 W) (0 for W <= 1). Zero planes always form maximal runs; a
//     non-zero plane takes the shortest applicable code, ties in the order
//     all-ones, pre-XOR-zero, two-adjacent, single-one, verbatim.
//   - Chunk: 32 blocks, bit-contiguous, zero-padded to a byte; a final
//     partial block is zero-padded to 128 B for coding only. L =
//     ceil(bits/8); if L >= raw size the chunk is stored raw with L = raw
//     size.
//   - Stream: C little-endian u16 sizes, then the payloads, unpadded.
#pragma once

#include <cstdint>

namespace pz {

constexpr int kBlockBytes = 128;
constexpr int kChunkBytes = 4096;
constexpr int kBlocksPerChunk = 32;

enum Tag : uint32_t { kTagZVC = 0, kTagDBX = 1, kTagBX = 2, kTagZBX = 3, kTagRAW = 4 };

// status codes shared with include/planezip.h
constexpr int kOk = 0;
constexpr int kErrCorrupt = 3;
constexpr int kErrTimeout = 5;

}  // namespace pz
