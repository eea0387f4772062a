/*
 * PlaneZip block codec: plain, single-threaded CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library. The product path (the CUDA
 * library under lossless_bit_plane_gb300/) never links, loads or calls it,
 * and the two share no code.
 *
 * What it computes follows "PlaneZip: Lossless Bit-Plane Compression of
 * Training Activations Offloaded over PCIe" (arXiv:2610.25033v1):
 *   - Section III-A "Codec": 128-byte blocks read as N symbols of w bits
 *     (w = 16 and N = 64 for BF16, w = 32 and N = 32 otherwise); the four
 *     encodings ZVC, DBX, BX, ZBX plus the raw block; BPC's plane prefix code;
 *     the smallest candidate kept behind a 3-bit tag.
 *   - Section III-A "Stream format": 32 blocks per 4 KB chunk, byte-aligned
 *     chunks, a 16-bit size per chunk, a chunk that would grow stored raw.
 *   - Section II-B "Memory Compression": BPC's Delta-BitPlane-XOR transform.
 * Where the paper leaves a bit layout open the oracle follows the readings
 * R1..R14 written out at the top of pz_oracle.c.
 *
 * Parity status: the code LENGTHS are the paper's; the bit PATTERNS, field
 * orders and tie-breaks are this codec's documented readings, pinned by
 * hand-derived golden streams, closed forms and round trips rather than by a
 * stream printed in the paper (the paper prints none).
 *
 * All pointers are host pointers. Return values are PZO_* status codes.
 */
#ifndef PZ_ORACLE_H
#define PZ_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  PZO_OK = 0,
  PZO_ERR_ARG = 1,
  PZO_ERR_CAPACITY = 2,
  PZO_ERR_CORRUPT = 3
};

enum { PZO_TAG_ZVC = 0, PZO_TAG_DBX = 1, PZO_TAG_BX = 2, PZO_TAG_ZBX = 3, PZO_TAG_RAW = 4 };

/* Candidate masks (bit t = tag t). The raw block is always a candidate. */
#define PZO_CAND_ALL 0x1Fu

/* Largest possible stream for nbytes of input: 2 bytes of header per chunk
 * plus every chunk stored raw. */
size_t pzo_max_stream_bytes(size_t nbytes);

/* Compress nbytes at `in` into `out` (capacity `cap`). On success *total is
 * the stream length 2C + sum(L). elem_width 2 selects 16-bit symbols; any
 * other positive width selects 32-bit symbols. */
int pzo_compress(const uint8_t *in, size_t nbytes, int elem_width,
                 uint8_t *out, size_t cap, size_t *total);

/* The same stream format with block selection restricted to the candidates
 * in `candidates` (bit t = tag t; raw is always allowed): the smallest
 * allowed candidate is kept, ties to the lowest tag. PZO_CAND_ALL gives
 * pzo_compress. This reproduces the paper's single-encoding comparisons
 * (Section V-A "Compression Ratio", Fig. 3: ZVC only, BPC = DBX on every block, ...). */
int pzo_compress_candidates(const uint8_t *in, size_t nbytes, int elem_width, unsigned candidates,
                            uint8_t *out, size_t cap, size_t *total);

/* Decompress a stream of comp_bytes (>= the stream's own length) into
 * nbytes at `out`. Returns PZO_ERR_CORRUPT on any malformed field. */
int pzo_decompress(const uint8_t *in, size_t comp_bytes, int elem_width,
                   uint8_t *out, size_t nbytes);

/* One 128-byte block: the five candidate sizes in bits (tag excluded), in
 * tag order ZVC, DBX, BX, ZBX, RAW, measured by the bit-exact encoders
 * (enc_bits) and by the independent size model (model_bits); *tag is the
 * candidate the block encoder keeps. Either output array may be NULL. */
int pzo_block_candidates(const uint8_t block[128], int elem_width,
                         int enc_bits[5], int model_bits[5], int *tag);

/* Bit-exact encoding of one block as candidate `tag` (without the 3-bit tag)
 * into buf (zeroed by the caller, cap_bytes long); returns the bit count or a
 * negative value if it does not fit. */
int pzo_encode_candidate(const uint8_t block[128], int elem_width, int tag,
                         uint8_t *buf, size_t cap_bytes);

/* Per-block analysis of a whole tensor, chunk by chunk: tags[i] and
 * bits[i] (tag included) for every block i, and per-chunk L in lens[c].
 * Blocks of chunks stored raw get tag 255. Arrays hold ceil(nbytes/128),
 * ceil(nbytes/128) and ceil(nbytes/4096) entries. */
int pzo_analyze(const uint8_t *in, size_t nbytes, int elem_width,
                uint8_t *tags, uint16_t *bits, uint16_t *lens);

/* pzo_analyze with block selection restricted as in pzo_compress_candidates. */
int pzo_analyze_candidates(const uint8_t *in, size_t nbytes, int elem_width, unsigned candidates,
                           uint8_t *tags, uint16_t *bits, uint16_t *lens);

#ifdef __cplusplus
}
#endif

#endif
