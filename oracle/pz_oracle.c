/*
 * PlaneZip block codec: plain, single-threaded CPU oracle. It keeps no state
 * between calls, so separate threads may run it on separate buffers.
 *
 * TEST INFRASTRUCTURE ONLY (see pz_oracle.h). It is written for a reader to
 * check against the paper by eye: every plane is an explicit array of bits,
 * every code is written one bit at a time, and nothing is fused or reordered.
 *
 * Paper: "PlaneZip: Lossless Bit-Plane Compression of Training Activations
 * Offloaded over PCIe", arXiv:2610.25033v1. Section III-A "Codec" defines the
 * block, the symbols, the five candidates and the plane code lengths;
 * Section III-A "Stream format" defines chunks, headers and raw fallback;
 * Section II-B defines BPC's DBX transform.
 *
 * Readings where the paper leaves the layout open (the GPU path follows the
 * same readings bit for bit):
 *  R1  Streams are LSB-first: stream bit b is bit (b mod 8) of byte b/8; an
 *      m-bit field with value v is written v bit 0 first.
 *  R2  Symbols are little-endian unsigned integers of w bits.
 *  R3  A symbol is zero only if all w bits are zero (-0.0 is non-zero).
 *  R4  The DBX base symbol is stored verbatim in w bits.
 *  R5  DBX deltas are (s_j - s_{j-1}) mod 2^(w+1) of the UNSIGNED symbols, so
 *      bit w of a delta is the borrow [s_j < s_{j-1}].
 *  R6  ZBX with no non-zero symbol writes its N-bit mask and no plane codes.
 *  R7  Plane codes are written top plane first, down to plane 0.
 *  R8  The run-length field has k = ceil(log2(P-1)) bits for P planes
 *      (5 for 32/33 planes, 4 for 16/17 planes: "6 or 7" bits per run code).
 *  R9  The position field has p = ceil(log2 W) bits for planes W bits wide
 *      (p = 0 when W <= 1).
 *  R10 Code bit patterns, first stream bit on the left:
 *        zero run (L >= 2 zero planes)  0 1 + (L-2) in k bits
 *        single zero plane              0 0 1
 *        all-ones plane                 0 0 0 0 0
 *        pre-XOR plane zero             0 0 0 0 1
 *        two adjacent ones at q, q+1    0 0 0 1 0 + q in p bits
 *        single one at q                0 0 0 1 1 + q in p bits
 *        verbatim                       1 + the W plane bits, bit 0 first
 *  R11 Zero planes always form maximal runs coded by the first two codes.
 *      A non-zero plane takes the shortest applicable code among all-ones,
 *      pre-XOR-zero, two-adjacent, single-one, verbatim; ties go to the
 *      earlier one in that list. Pre-XOR-zero applies below the top plane.
 *  R12 Tags: ZVC 0, DBX 1, BX 2, ZBX 3, RAW 4 in a 3-bit field; a block keeps
 *      the smallest candidate and ties go to the lowest tag.
 *  R13 A final partial block is zero-padded to 128 bytes for encoding; the
 *      decoder writes only the chunk's real bytes.
 *  R14 The stream is the table of C little-endian 16-bit chunk sizes L
 *      followed by the chunk payloads, byte-aligned and unpadded. A chunk
 *      whose coded size L would reach its raw size is stored raw with
 *      L = raw size, so L == raw size marks a raw chunk.
 */
#include "pz_oracle.h"

#include <stdlib.h>
#include <string.h>

#define BLOCK_BYTES 128
#define CHUNK_BYTES 4096
#define BLOCKS_PER_CHUNK 32
#define MAX_SYMBOLS 64
#define MAX_PLANES 33

/* ------------------------------------------------------------------ */
/* Bit writer / reader (R1: LSB-first).                                */
/* ------------------------------------------------------------------ */

typedef struct {
  uint8_t *buf;
  size_t cap_bits;
  size_t pos;
  int overflow;
} bitwriter;

static void put_bit(bitwriter *w, int bit) {
  if (w->pos >= w->cap_bits) {
    w->overflow = 1;
    w->pos++;
    return;
  }
  uint8_t m = (uint8_t)(1u << (w->pos % 8));
  if (bit)
    w->buf[w->pos / 8] |= m;
  else
    w->buf[w->pos / 8] &= (uint8_t)~m;
  w->pos++;
}

static void put_field(bitwriter *w, uint64_t value, int nbits) {
  for (int i = 0; i < nbits; i++) put_bit(w, (int)((value >> i) & 1u));
}

typedef struct {
  const uint8_t *buf;
  size_t nbits;
  size_t pos;
  int overrun;
} bitreader;

static int get_bit(bitreader *r) {
  if (r->pos >= r->nbits) {
    r->overrun = 1;
    r->pos++;
    return 0;
  }
  int b = (r->buf[r->pos / 8] >> (r->pos % 8)) & 1;
  r->pos++;
  return b;
}

static uint64_t get_field(bitreader *r, int nbits) {
  uint64_t v = 0;
  for (int i = 0; i < nbits; i++) v |= (uint64_t)get_bit(r) << i;
  return v;
}

/* ------------------------------------------------------------------ */
/* Block and symbols (Section III-A "Codec"; R2).                      */
/* ------------------------------------------------------------------ */

typedef struct {
  int w; /* symbol width in bits */
  int N; /* symbols per block */
} geometry;

static geometry geometry_for(int elem_width) {
  geometry g;
  g.w = (elem_width == 2) ? 16 : 32; /* BF16 uses 16-bit symbols; others 32 */
  g.N = (BLOCK_BYTES * 8) / g.w;
  return g;
}

static void block_to_symbols(const uint8_t *block, geometry g, uint32_t *sym) {
  int bytes = g.w / 8;
  for (int k = 0; k < g.N; k++) {
    uint32_t v = 0;
    for (int b = 0; b < bytes; b++) v |= (uint32_t)block[k * bytes + b] << (8 * b);
    sym[k] = v;
  }
}

static void symbols_to_block(const uint32_t *sym, geometry g, uint8_t *block) {
  int bytes = g.w / 8;
  for (int k = 0; k < g.N; k++)
    for (int b = 0; b < bytes; b++) block[k * bytes + b] = (uint8_t)(sym[k] >> (8 * b));
}

static int ceil_log2(int v) {
  int k = 0;
  while ((1 << k) < v) k++;
  return k; /* 0 for v <= 1 */
}

/* ------------------------------------------------------------------ */
/* Bit-planes (Section II-B, Section III-A).                           */
/*   pre[i][j] = bit i of value j            (the planes before XOR)   */
/*   x[top] = pre[top]; x[i] = pre[i] XOR pre[i+1] for i < top.        */
/* ------------------------------------------------------------------ */

typedef struct {
  int P;   /* number of planes */
  int W;   /* plane width in bits */
  uint8_t pre[MAX_PLANES][MAX_SYMBOLS];
  uint8_t x[MAX_PLANES][MAX_SYMBOLS];
} planes;

static void make_planes(planes *pl, const uint64_t *values, int W, int P) {
  pl->P = P;
  pl->W = W;
  for (int i = 0; i < P; i++)
    for (int j = 0; j < W; j++) pl->pre[i][j] = (uint8_t)((values[j] >> i) & 1u);
  for (int i = 0; i < P; i++)
    for (int j = 0; j < W; j++)
      pl->x[i][j] = (i == P - 1) ? pl->pre[i][j] : (uint8_t)(pl->pre[i][j] ^ pl->pre[i + 1][j]);
}

static int count_ones(const uint8_t *bits, int W) {
  int c = 0;
  for (int j = 0; j < W; j++) c += bits[j];
  return c;
}

static int first_one(const uint8_t *bits, int W) {
  for (int j = 0; j < W; j++)
    if (bits[j]) return j;
  return -1;
}

/* Plane code kinds, in the R11 tie order for non-zero planes. */
enum { CODE_ALL_ONES = 0, CODE_PREXOR_ZERO = 1, CODE_TWO_ADJ = 2, CODE_SINGLE = 3, CODE_VERBATIM = 4 };

/* Choose the code for non-zero plane i (R11) and report its length. */
static int choose_plane_code(const planes *pl, int i, int *q_out, int *len_out) {
  int W = pl->W, top = pl->P - 1, p = ceil_log2(W);
  const uint8_t *x = pl->x[i];
  int ones = count_ones(x, W);
  int q = first_one(x, W);
  int applicable[5], length[5];
  applicable[CODE_ALL_ONES] = (ones == W);
  length[CODE_ALL_ONES] = 5;
  applicable[CODE_PREXOR_ZERO] = (i < top) && (count_ones(pl->pre[i], W) == 0);
  length[CODE_PREXOR_ZERO] = 5;
  applicable[CODE_TWO_ADJ] = (ones == 2) && (q + 1 < W) && x[q + 1];
  length[CODE_TWO_ADJ] = 5 + p;
  applicable[CODE_SINGLE] = (ones == 1);
  length[CODE_SINGLE] = 5 + p;
  applicable[CODE_VERBATIM] = 1;
  length[CODE_VERBATIM] = 1 + W;
  int shortest = length[CODE_VERBATIM];
  for (int c = 0; c < 5; c++)
    if (applicable[c] && length[c] < shortest) shortest = length[c];
  int best = CODE_VERBATIM; /* the first applicable code of that length */
  for (int c = 4; c >= 0; c--)
    if (applicable[c] && length[c] == shortest) best = c;
  *q_out = q;
  *len_out = length[best];
  return best;
}

static int plane_is_zero(const planes *pl, int i) { return count_ones(pl->x[i], pl->W) == 0; }

/* Write the P plane codes, top plane first (R7, R10, R11). */
static void write_plane_codes(bitwriter *w, const planes *pl) {
  int k = ceil_log2(pl->P - 1), p = ceil_log2(pl->W);
  int i = pl->P - 1;
  while (i >= 0) {
    if (plane_is_zero(pl, i)) {
      int run = 0;
      while (i - run >= 0 && plane_is_zero(pl, i - run)) run++;
      if (run == 1) {
        put_bit(w, 0); put_bit(w, 0); put_bit(w, 1);
      } else {
        put_bit(w, 0); put_bit(w, 1);
        put_field(w, (uint64_t)(run - 2), k);
      }
      i -= run;
      continue;
    }
    int q, len;
    int code = choose_plane_code(pl, i, &q, &len);
    switch (code) {
      case CODE_ALL_ONES:
        put_bit(w, 0); put_bit(w, 0); put_bit(w, 0); put_bit(w, 0); put_bit(w, 0);
        break;
      case CODE_PREXOR_ZERO:
        put_bit(w, 0); put_bit(w, 0); put_bit(w, 0); put_bit(w, 0); put_bit(w, 1);
        break;
      case CODE_TWO_ADJ:
        put_bit(w, 0); put_bit(w, 0); put_bit(w, 0); put_bit(w, 1); put_bit(w, 0);
        put_field(w, (uint64_t)q, p);
        break;
      case CODE_SINGLE:
        put_bit(w, 0); put_bit(w, 0); put_bit(w, 0); put_bit(w, 1); put_bit(w, 1);
        put_field(w, (uint64_t)q, p);
        break;
      default:
        put_bit(w, 1);
        for (int j = 0; j < pl->W; j++) put_bit(w, pl->x[i][j]);
        break;
    }
    i--;
  }
}

/* Read P plane codes into pl->x / pl->pre (top plane first). */
static int read_plane_codes(bitreader *r, planes *pl, int W, int P) {
  int k = ceil_log2(P - 1), p = ceil_log2(W), top = P - 1;
  pl->P = P;
  pl->W = W;
  int i = top;
  while (i >= 0) {
    int run = 0; /* planes this code sets to zero */
    if (get_bit(r)) { /* 1: verbatim */
      for (int j = 0; j < W; j++) pl->x[i][j] = (uint8_t)get_bit(r);
    } else if (get_bit(r)) { /* 0 1: zero run */
      run = 2 + (int)get_field(r, k);
    } else if (get_bit(r)) { /* 0 0 1: single zero plane */
      run = 1;
    } else {
      int b3 = get_bit(r), b4 = get_bit(r);
      memset(pl->x[i], 0, (size_t)W);
      if (!b3 && !b4) { /* all ones */
        for (int j = 0; j < W; j++) pl->x[i][j] = 1;
      } else if (!b3 && b4) { /* pre-XOR plane zero: x[i] = pre[i+1] */
        if (i == top) return PZO_ERR_CORRUPT;
        for (int j = 0; j < W; j++) pl->x[i][j] = pl->pre[i + 1][j];
      } else {
        int q = (int)get_field(r, p);
        if (b4 == 0) { /* two adjacent ones */
          if (q + 1 >= W) return PZO_ERR_CORRUPT;
          pl->x[i][q] = 1;
          pl->x[i][q + 1] = 1;
        } else { /* single one */
          if (q >= W) return PZO_ERR_CORRUPT;
          pl->x[i][q] = 1;
        }
      }
    }
    if (r->overrun) return PZO_ERR_CORRUPT;
    if (run > 0) {
      if (run > i + 1) return PZO_ERR_CORRUPT;
      for (int t = 0; t < run; t++) {
        memset(pl->x[i], 0, (size_t)W);
        for (int j = 0; j < W; j++) pl->pre[i][j] = (i == top) ? 0 : pl->pre[i + 1][j];
        i--;
      }
      continue;
    }
    for (int j = 0; j < W; j++)
      pl->pre[i][j] = (i == top) ? pl->x[i][j] : (uint8_t)(pl->x[i][j] ^ pl->pre[i + 1][j]);
    i--;
  }
  return PZO_OK;
}

/* value j = sum_i pre[i][j] * 2^i */
static uint64_t plane_value(const planes *pl, int j) {
  uint64_t v = 0;
  for (int i = 0; i < pl->P; i++) v |= (uint64_t)pl->pre[i][j] << i;
  return v;
}

/* ------------------------------------------------------------------ */
/* The candidates (Section III-A "Codec"). Each writes its payload      */
/* (without the tag) and returns the number of bits written.            */
/* ------------------------------------------------------------------ */

/* ZVC: an N-bit mask of non-zero symbols, then the non-zero symbols. */
static void encode_zvc(bitwriter *w, const uint32_t *s, geometry g) {
  for (int k = 0; k < g.N; k++) put_bit(w, s[k] != 0);
  for (int k = 0; k < g.N; k++)
    if (s[k] != 0) put_field(w, s[k], g.w);
}

/* DBX: the base symbol (R4), then the w+1 bit-planes of the N-1 deltas
 * (R5), with adjacent planes XORed. */
static void encode_dbx(bitwriter *w, const uint32_t *s, geometry g) {
  planes pl;
  uint64_t d[MAX_SYMBOLS];
  uint64_t mod_mask = (1ull << (g.w + 1)) - 1;
  put_field(w, s[0], g.w);
  for (int j = 1; j < g.N; j++) d[j - 1] = ((uint64_t)s[j] - (uint64_t)s[j - 1]) & mod_mask;
  make_planes(&pl, d, g.N - 1, g.w + 1);
  write_plane_codes(w, &pl);
}

/* BX: the w bit-planes of the symbols themselves, adjacent planes XORed. */
static void encode_bx(bitwriter *w, const uint32_t *s, geometry g) {
  planes pl;
  uint64_t v[MAX_SYMBOLS];
  for (int j = 0; j < g.N; j++) v[j] = s[j];
  make_planes(&pl, v, g.N, g.w);
  write_plane_codes(w, &pl);
}

/* ZBX: the N-bit zero mask, then BX over the n non-zero symbols compacted
 * to the front, each plane n bits wide (R6 for n = 0). */
static void encode_zbx(bitwriter *w, const uint32_t *s, geometry g) {
  planes pl;
  uint64_t t[MAX_SYMBOLS];
  int n = 0;
  for (int k = 0; k < g.N; k++) put_bit(w, s[k] != 0);
  for (int k = 0; k < g.N; k++)
    if (s[k] != 0) t[n++] = s[k];
  if (n == 0) return;
  make_planes(&pl, t, n, g.w);
  write_plane_codes(w, &pl);
}

/* RAW: the 1024 bits of the block, byte by byte. */
static void encode_raw(bitwriter *w, const uint8_t *block) {
  for (int b = 0; b < BLOCK_BYTES; b++) put_field(w, block[b], 8);
}

static void encode_candidate(bitwriter *w, int tag, const uint8_t *block, const uint32_t *s, geometry g) {
  switch (tag) {
    case PZO_TAG_ZVC: encode_zvc(w, s, g); break;
    case PZO_TAG_DBX: encode_dbx(w, s, g); break;
    case PZO_TAG_BX: encode_bx(w, s, g); break;
    case PZO_TAG_ZBX: encode_zbx(w, s, g); break;
    default: encode_raw(w, block); break;
  }
}

/* Bits each candidate takes, measured by running its encoder. */
static void candidate_bits_by_encoding(const uint8_t *block, geometry g, int out[5]) {
  uint32_t s[MAX_SYMBOLS];
  uint8_t scratch[512];
  block_to_symbols(block, g, s);
  for (int tag = 0; tag < 5; tag++) {
    bitwriter w = {scratch, sizeof(scratch) * 8, 0, 0};
    encode_candidate(&w, tag, block, s, g);
    out[tag] = (int)w.pos;
  }
}

/* ------------------------------------------------------------------ */
/* Size model: the same lengths counted from plane classes, without a  */
/* bit writer (the paper's "vectorized size model" cross-check,        */
/* Section III-A "Validation"). Written independently of the encoder:  */
/* it scans planes bottom-up and adds code lengths arithmetically.     */
/* ------------------------------------------------------------------ */

static int model_plane_codes(const planes *pl) {
  int P = pl->P, W = pl->W, top = P - 1;
  int k = ceil_log2(P - 1), p = ceil_log2(W);
  int total = 0, run = 0;
  for (int i = 0; i <= top; i++) {
    int ones = 0, pre_ones = 0, adjacent_pairs = 0;
    for (int j = 0; j < W; j++) {
      ones += pl->x[i][j];
      pre_ones += pl->pre[i][j];
      if (j + 1 < W && pl->x[i][j] && pl->x[i][j + 1]) adjacent_pairs++;
    }
    if (ones == 0) {
      run++;
      continue;
    }
    if (run) total += (run == 1) ? 3 : 2 + k;
    run = 0;
    int len = 1 + W; /* verbatim always applies */
    if (ones == W && 5 < len) len = 5;
    if (i < top && pre_ones == 0 && 5 < len) len = 5;
    if ((ones == 1 || (ones == 2 && adjacent_pairs == 1)) && 5 + p < len) len = 5 + p;
    total += len;
  }
  if (run) total += (run == 1) ? 3 : 2 + k;
  return total;
}

static void candidate_bits_by_model(const uint8_t *block, geometry g, int out[5]) {
  planes pl;
  uint32_t s[MAX_SYMBOLS];
  uint64_t v[MAX_SYMBOLS] = {0};
  block_to_symbols(block, g, s);
  int n = 0;
  for (int k = 0; k < g.N; k++) n += (s[k] != 0);
  out[PZO_TAG_ZVC] = g.N + n * g.w;
  for (int j = 1; j < g.N; j++)
    v[j - 1] = ((uint64_t)s[j] - (uint64_t)s[j - 1]) & ((1ull << (g.w + 1)) - 1);
  make_planes(&pl, v, g.N - 1, g.w + 1);
  out[PZO_TAG_DBX] = g.w + model_plane_codes(&pl);
  for (int j = 0; j < g.N; j++) v[j] = s[j];
  make_planes(&pl, v, g.N, g.w);
  out[PZO_TAG_BX] = model_plane_codes(&pl);
  int m = 0;
  for (int j = 0; j < g.N; j++)
    if (s[j]) v[m++] = s[j];
  if (m == 0) {
    out[PZO_TAG_ZBX] = g.N;
  } else {
    make_planes(&pl, v, m, g.w);
    out[PZO_TAG_ZBX] = g.N + model_plane_codes(&pl);
  }
  out[PZO_TAG_RAW] = BLOCK_BYTES * 8;
}

/* The block keeps the smallest candidate; ties go to the lowest tag (R12).
 * Only the candidates in the mask `allowed` (bit t = tag t) are considered;
 * the raw block is always allowed, so a choice always exists. */
static int select_tag(const int bits[5], unsigned allowed) {
  allowed |= 1u << PZO_TAG_RAW;
  int best = PZO_TAG_RAW;
  for (int t = 0; t < 5; t++)
    if (((allowed >> t) & 1u) && (bits[t] < bits[best] || (bits[t] == bits[best] && t < best))) best = t;
  return best;
}

/* ------------------------------------------------------------------ */
/* Block decoder (the inverse of each candidate).                      */
/* ------------------------------------------------------------------ */

static int decode_block(bitreader *r, geometry g, uint8_t *block) {
  planes pl;
  uint32_t s[MAX_SYMBOLS];
  int tag = (int)get_field(r, 3);
  if (r->overrun) return PZO_ERR_CORRUPT;
  memset(s, 0, sizeof(s));
  switch (tag) {
    case PZO_TAG_ZVC: {
      int mask[MAX_SYMBOLS];
      for (int k = 0; k < g.N; k++) mask[k] = get_bit(r);
      for (int k = 0; k < g.N; k++)
        if (mask[k]) s[k] = (uint32_t)get_field(r, g.w);
      break;
    }
    case PZO_TAG_DBX: {
      s[0] = (uint32_t)get_field(r, g.w);
      if (r->overrun) return PZO_ERR_CORRUPT;
      int rc = read_plane_codes(r, &pl, g.N - 1, g.w + 1);
      if (rc) return rc;
      uint64_t wmask = (g.w == 32) ? 0xFFFFFFFFull : 0xFFFFull;
      for (int j = 1; j < g.N; j++) s[j] = (uint32_t)(((uint64_t)s[j - 1] + plane_value(&pl, j - 1)) & wmask);
      break;
    }
    case PZO_TAG_BX: {
      int rc = read_plane_codes(r, &pl, g.N, g.w);
      if (rc) return rc;
      for (int j = 0; j < g.N; j++) s[j] = (uint32_t)plane_value(&pl, j);
      break;
    }
    case PZO_TAG_ZBX: {
      int mask[MAX_SYMBOLS], n = 0;
      for (int k = 0; k < g.N; k++) {
        mask[k] = get_bit(r);
        n += mask[k];
      }
      if (r->overrun) return PZO_ERR_CORRUPT;
      if (n > 0) {
        int rc = read_plane_codes(r, &pl, n, g.w);
        if (rc) return rc;
        int t = 0;
        for (int k = 0; k < g.N; k++)
          if (mask[k]) s[k] = (uint32_t)plane_value(&pl, t++);
      }
      break;
    }
    case PZO_TAG_RAW:
      for (int b = 0; b < BLOCK_BYTES; b++) block[b] = (uint8_t)get_field(r, 8);
      return r->overrun ? PZO_ERR_CORRUPT : PZO_OK;
    default:
      return PZO_ERR_CORRUPT;
  }
  if (r->overrun) return PZO_ERR_CORRUPT;
  symbols_to_block(s, g, block);
  return PZO_OK;
}

/* ------------------------------------------------------------------ */
/* Chunks and stream (Section III-A "Stream format"; R13, R14).        */
/* ------------------------------------------------------------------ */

static size_t num_chunks(size_t nbytes) { return (nbytes + CHUNK_BYTES - 1) / CHUNK_BYTES; }

size_t pzo_max_stream_bytes(size_t nbytes) { return 2 * num_chunks(nbytes) + nbytes; }

/* Encode one chunk of raw_len bytes into `payload`; returns its length L
 * and fills per-block tags/bits when asked. */
static size_t encode_chunk(const uint8_t *src, size_t raw_len, geometry g, unsigned allowed, uint8_t *payload,
                           uint8_t *tags, uint16_t *bits) {
  uint8_t coded[CHUNK_BYTES + 64];
  memset(coded, 0, sizeof(coded));
  bitwriter w = {coded, sizeof(coded) * 8, 0, 0};
  size_t nblocks = (raw_len + BLOCK_BYTES - 1) / BLOCK_BYTES;
  for (size_t b = 0; b < nblocks; b++) {
    uint8_t block[BLOCK_BYTES];
    uint32_t s[MAX_SYMBOLS];
    memset(block, 0, sizeof(block));
    size_t take = raw_len - b * BLOCK_BYTES;
    if (take > BLOCK_BYTES) take = BLOCK_BYTES;
    memcpy(block, src + b * BLOCK_BYTES, take);
    int cand[5];
    candidate_bits_by_encoding(block, g, cand);
    int tag = select_tag(cand, allowed);
    size_t start = w.pos;
    put_field(&w, (uint64_t)tag, 3);
    block_to_symbols(block, g, s);
    encode_candidate(&w, tag, block, s, g);
    if (tags) tags[b] = (uint8_t)tag;
    if (bits) bits[b] = (uint16_t)(w.pos - start);
  }
  size_t L = (w.pos + 7) / 8;
  if (L >= raw_len) { /* a chunk that would grow is stored raw */
    memcpy(payload, src, raw_len);
    if (tags)
      for (size_t b = 0; b < nblocks; b++) tags[b] = 255;
    return raw_len;
  }
  memcpy(payload, coded, L);
  return L;
}

int pzo_compress(const uint8_t *in, size_t nbytes, int elem_width, uint8_t *out, size_t cap,
                 size_t *total) {
  return pzo_compress_candidates(in, nbytes, elem_width, PZO_CAND_ALL, out, cap, total);
}

int pzo_compress_candidates(const uint8_t *in, size_t nbytes, int elem_width, unsigned candidates,
                            uint8_t *out, size_t cap, size_t *total) {
  if (elem_width <= 0 || (!in && nbytes) || !total) return PZO_ERR_ARG;
  size_t C = num_chunks(nbytes);
  if (cap < pzo_max_stream_bytes(nbytes)) return PZO_ERR_CAPACITY;
  if (!out && C) return PZO_ERR_ARG;
  geometry g = geometry_for(elem_width);
  size_t pos = 2 * C;
  for (size_t c = 0; c < C; c++) {
    size_t raw_len = nbytes - c * CHUNK_BYTES;
    if (raw_len > CHUNK_BYTES) raw_len = CHUNK_BYTES;
    size_t L = encode_chunk(in + c * CHUNK_BYTES, raw_len, g, candidates, out + pos, NULL, NULL);
    out[2 * c] = (uint8_t)(L & 0xFF);
    out[2 * c + 1] = (uint8_t)(L >> 8);
    pos += L;
  }
  *total = pos;
  return PZO_OK;
}

int pzo_decompress(const uint8_t *in, size_t comp_bytes, int elem_width, uint8_t *out,
                   size_t nbytes) {
  if (elem_width <= 0 || (!out && nbytes)) return PZO_ERR_ARG;
  size_t C = num_chunks(nbytes);
  if (comp_bytes < 2 * C || (!in && C)) return PZO_ERR_ARG;
  geometry g = geometry_for(elem_width);
  size_t pos = 2 * C;
  for (size_t c = 0; c < C; c++) {
    size_t L = (size_t)in[2 * c] | ((size_t)in[2 * c + 1] << 8);
    size_t raw_len = nbytes - c * CHUNK_BYTES;
    if (raw_len > CHUNK_BYTES) raw_len = CHUNK_BYTES;
    if (L == 0 || L > raw_len || pos + L > comp_bytes) return PZO_ERR_CORRUPT;
    uint8_t *dst = out + c * CHUNK_BYTES;
    if (L == raw_len) {
      memcpy(dst, in + pos, raw_len);
    } else {
      bitreader r = {in + pos, 8 * L, 0, 0};
      size_t nblocks = (raw_len + BLOCK_BYTES - 1) / BLOCK_BYTES;
      for (size_t b = 0; b < nblocks; b++) {
        uint8_t block[BLOCK_BYTES];
        int rc = decode_block(&r, g, block);
        if (rc) return rc;
        size_t take = raw_len - b * BLOCK_BYTES;
        if (take > BLOCK_BYTES) take = BLOCK_BYTES;
        memcpy(dst + b * BLOCK_BYTES, block, take);
      }
      /* the chunk is exactly ceil(bits/8) bytes and its padding bits are 0 */
      if (8 * L - r.pos >= 8) return PZO_ERR_CORRUPT;
      while (r.pos < 8 * L)
        if (get_bit(&r)) return PZO_ERR_CORRUPT;
    }
    pos += L;
  }
  return PZO_OK;
}

int pzo_block_candidates(const uint8_t block[128], int elem_width, int enc_bits[5],
                         int model_bits[5], int *tag) {
  if (!block || elem_width <= 0) return PZO_ERR_ARG;
  geometry g = geometry_for(elem_width);
  int e[5];
  candidate_bits_by_encoding(block, g, e);
  if (enc_bits) memcpy(enc_bits, e, sizeof(e));
  if (model_bits) candidate_bits_by_model(block, g, model_bits);
  if (tag) *tag = select_tag(e, PZO_CAND_ALL);
  return PZO_OK;
}

int pzo_encode_candidate(const uint8_t block[128], int elem_width, int tag, uint8_t *buf,
                         size_t cap_bytes) {
  if (!block || !buf || elem_width <= 0 || tag < 0 || tag > 4) return -1;
  geometry g = geometry_for(elem_width);
  uint32_t s[MAX_SYMBOLS];
  block_to_symbols(block, g, s);
  bitwriter w = {buf, cap_bytes * 8, 0, 0};
  encode_candidate(&w, tag, block, s, g);
  return w.overflow ? -1 : (int)w.pos;
}

int pzo_analyze(const uint8_t *in, size_t nbytes, int elem_width, uint8_t *tags, uint16_t *bits,
                uint16_t *lens) {
  return pzo_analyze_candidates(in, nbytes, elem_width, PZO_CAND_ALL, tags, bits, lens);
}

int pzo_analyze_candidates(const uint8_t *in, size_t nbytes, int elem_width, unsigned candidates,
                           uint8_t *tags, uint16_t *bits, uint16_t *lens) {
  if (elem_width <= 0 || (!in && nbytes)) return PZO_ERR_ARG;
  geometry g = geometry_for(elem_width);
  size_t C = num_chunks(nbytes);
  uint8_t payload[CHUNK_BYTES];
  for (size_t c = 0; c < C; c++) {
    size_t raw_len = nbytes - c * CHUNK_BYTES;
    if (raw_len > CHUNK_BYTES) raw_len = CHUNK_BYTES;
    size_t L = encode_chunk(in + c * CHUNK_BYTES, raw_len, g, candidates, payload,
                            tags ? tags + c * BLOCKS_PER_CHUNK : NULL,
                            bits ? bits + c * BLOCKS_PER_CHUNK : NULL);
    if (lens) lens[c] = (uint16_t)L;
  }
  return PZO_OK;
}
