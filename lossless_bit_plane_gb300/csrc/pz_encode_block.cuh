// pz_encode_block.cuh — the per-block work of the PlaneZip encoder: one lane
// codes one 128-byte block. Classification (the five candidate sizes from
// bit-sliced plane classes), selection, and emission of the kept candidate
// through a lane's bit writer. Included by encode.cu; the kernel around it
// (loads, chunk close, look-back, copy-out) lives there.
//
// Paper: "PlaneZip: Lossless Bit-Plane Compression of Training Activations
// Offloaded over PCIe" (arXiv:2610.25033v1), Section III-A "Codec" (ZVC,
// DBX, BX, ZBX and raw per 128-byte block; BPC's plane prefix code; the
// smallest candidate behind a 3-bit tag) and Section II-B (BPC's
// Delta-BitPlane-XOR transform).
//
// Stage layout: a lane's block is one 128-byte row of the warp's 4 KB stage,
// 16-byte units swizzled as a 128-byte-swizzled TMA tile leaves them (unit u
// of row r at unit u ^ (r & 7)). Shared memory is addressed by 32-bit
// shared-window addresses.
#pragma once

#include <cstdint>

#include "pz_device.cuh"
#include "pz_format.cuh"

namespace pz {

// ------------------------------------------------------------ cost helpers

// Zero planes (bits of Z, only the first P bits may be set) form maximal
// runs: a run of one costs 3 bits, a longer run 2 + K bits.
__device__ __forceinline__ int run_cost(uint64_t Z, int K) {
  uint64_t start = Z & ~(Z << 1);
  uint64_t single = start & ~(Z >> 1);
  int R = __popcll(start), S = __popcll(single);
  return 3 * S + (2 + K) * (R - S);
}

// Class of every plane of one candidate (bit i = plane i): non-zero, and the
// code each non-zero plane takes: verbatim, a 5-bit code (all-ones or, if
// not all-ones, pre-XOR-zero), or a 5+p-bit position code (single one or,
// if not, two adjacent ones). FP32 DBX has a 33rd plane, whose six class
// bits are packed in `top`.
struct Plan {
  uint32_t nz, v, f5, fa, m, ms;
  uint32_t top;
};

// Shortest applicable code per non-zero plane of width W (position field
// p), ties in the order all-ones, pre-XOR-zero, two-adjacent, single-one,
// verbatim: 5-bit codes unless verbatim (1+W) is shorter, position codes
// unless verbatim is shorter.
__device__ __forceinline__ Plan make_plan(uint32_t NZ, uint32_t A, uint32_t PX, uint32_t S1, uint32_t T2, int W,
                                          int p) {
  const int lv = 1 + W, lm = 5 + p;
  uint32_t f5 = (A | PX) & NZ;
  uint32_t m = (S1 | T2) & NZ & ~f5;
  if (5 > lv) f5 = 0;
  if (lm > lv) m = 0;
  Plan pl;
  pl.nz = NZ;
  pl.f5 = f5;
  pl.fa = A & f5;
  pl.m = m;
  pl.ms = S1 & m;
  pl.v = NZ & ~f5 & ~m;
  pl.top = 0;
  return pl;
}

__device__ __forceinline__ int plan_cost(const Plan &pl, int W, int p) {
  return 5 * __popc(pl.f5) + (5 + p) * __popc(pl.m) + (1 + W) * __popc(pl.v);
}

struct Sizes {
  int s[5];
  uint32_t m0, m1;  // non-zero symbol masks: symbols 0..31 and (BF16) 32..63
  uint32_t tag, bits;  // the kept candidate and its size (tag excluded)
  Plan win;            // its plan (plane candidates only)
  uint64_t bp;         // DBX's borrow plane (bit q = borrow of delta q+1)
};

// Pick the smallest allowed candidate (bit t of cand = tag t; the raw block
// is always allowed), ties to the lowest tag, and keep its plan.
__device__ __forceinline__ void keep_smallest(Sizes &z, const Plan &bx, const Plan &zbx, const Plan &dbx,
                                              uint32_t cand) {
  uint32_t tag = kTagRAW;
  int best = z.s[kTagRAW];
#pragma unroll
  for (int t = 3; t >= 0; --t)
    if (((cand >> t) & 1u) && z.s[t] <= best) {
      best = z.s[t];
      tag = (uint32_t)t;
    }
  z.tag = tag;
  z.bits = (uint32_t)best;
  z.win = (tag == kTagZBX) ? zbx : (tag == kTagDBX) ? dbx : bx;
}

// The lane's block in its 128-byte row of the stage, as the TMA left it
// (16-byte units swizzled by row): unit u holds words 4u .. 4u+3.
// Row addresses: a lane's 128-byte row of the stage starts on a 128-byte
// boundary (the stage is 1024-aligned), so a byte offset below 128, however
// swizzled, can be XORed into the row's address instead of added; the
// lane-dependent part of the swizzle (row_swz) is then common to every
// access and the per-access cost is one shift and one XOR.
__device__ __forceinline__ uint32_t row_swz(uint32_t rowbase, uint32_t r) { return rowbase ^ ((r & 7u) << 4); }
__device__ __forceinline__ uint4 stage_unit(uint32_t rowbase, uint32_t r, uint32_t u) {  // u < 8
  return lds128(row_swz(rowbase, r) ^ (u << 4));
}
// The lane's row of DBX words: 32 words in a 128-byte-aligned row, 16-byte
// units swizzled like a stage row (unit u at u ^ (lane & 7)). The classifier
// leaves there, as it streams the block, the Gray-coded deltas that DBX codes
// (word 0: zero, the base is coded verbatim), so that emission takes them as
// they are instead of deriving them again.
__device__ __forceinline__ uint32_t drow_unit(uint32_t drow, uint32_t lane, uint32_t u) {  // u < 8
  return row_swz(drow, lane) ^ (u << 4);
}

// ------------------------------------------------------------ FP32 classify
// The five candidate sizes (tag excluded) of the lane's block of 32 symbols
// and the kept candidate's plan. The words are streamed from the stage row four at a time, so that only the
// accumulators stay in registers; DBX's Gray-coded deltas go to the lane's
// DBX row (drow) unit by unit.
__device__ __forceinline__ Sizes classify32(uint32_t rowbase, uint32_t lane, uint32_t cand, uint32_t drow) {
  uint32_t a = 0, b = 0, c = 0, adj = 0, andx = ~0u, ors = 0, gprev = 0;  // BX
  uint32_t nz = 0, zn = 0, adjz = 0, last = 0;                            // ZBX / ZVC
  uint32_t ad = 0, bd = 0, cd = 0, adjd = 0, andd = ~0u, ord = 0, Bw = 0, gdprev = 0;  // DBX
  uint32_t xprev = 0;
  // word k of the block; the loop runs over 16-byte units (4 words each) so
  // that the kernel's code stays small
  auto step = [&](uint32_t x, uint32_t k) -> uint32_t {
    const uint32_t g = x ^ (x >> 1);
    ors |= x;
    c |= b & g;
    b |= a & g;
    a |= g;
    if (k) adj |= gprev & g;
    andx &= g;
    gprev = g;
    const uint32_t m = x ? 0xFFFFFFFFu : 0u;
    nz = __funnelshift_r(nz, m, 1);  // word k's flag enters at bit 31; after 32 words it sits at bit k
    zn |= ~g & m;  // some survivor has a 0 in the plane
    adjz |= last & g;
    last = x ? g : last;
    uint32_t gdk = 0;
    if (k) {
      const uint64_t d = (uint64_t)x - (uint64_t)xprev;
      const uint32_t lo = (uint32_t)d, hi = (uint32_t)(d >> 32);  // hi: borrow mask
      const uint32_t gd = lo ^ __funnelshift_r(lo, hi, 1);
      ord |= lo;
      Bw = __funnelshift_r(Bw, hi, 1);  // borrow of delta k ends at bit k (bit 0 stays 0)
      cd |= bd & gd;
      bd |= ad & gd;
      ad |= gd;
      if (k > 1) adjd |= gdprev & gd;
      andd &= gd;
      gdprev = gd;
      gdk = gd;
    }
    xprev = x;
    return gdk;
  };
  {
    const uint4 q = stage_unit(rowbase, lane, 0);
    step(q.x, 0);
    const uint32_t d1 = step(q.y, 1), d2 = step(q.z, 2), d3 = step(q.w, 3);
    sts128(drow_unit(drow, lane, 0), 0u, d1, d2, d3);
  }
#pragma unroll 1
  for (uint32_t u = 1; u < 8; ++u) {
    const uint4 q = stage_unit(rowbase, lane, u);
    const uint32_t d0 = step(q.x, 4 * u), d1 = step(q.y, 4 * u + 1), d2 = step(q.z, 4 * u + 2),
                   d3 = step(q.w, 4 * u + 3);
    sts128(drow_unit(drow, lane, u), d0, d1, d2, d3);
  }
  Bw >>= 1;  // borrow of delta k at bit k-1
  Sizes z;
  z.m0 = nz;
  z.m1 = 0;
  int n = __popc(nz);
  z.s[kTagZVC] = 32 + 32 * n;
  z.s[kTagRAW] = 1024;
  // BX: 32 planes of width 32, top plane 31
  const uint32_t PX = (~ors & a) & 0x7FFFFFFFu;
  const Plan bx = make_plan(a, andx, PX, a & ~b, b & ~c & adj, 32, 5);
  z.s[kTagBX] = run_cost((uint32_t)~a, 5) + plan_cost(bx, 32, 5);
  // ZBX: mask + 32 planes of width n over the survivors
  Plan zbx;
  if (n == 0) {
    zbx = make_plan(0, 0, 0, 0, 0, 1, 0);
    z.s[kTagZBX] = 32;
  } else {
    const int pn = (int)ceil_log2_u32((uint32_t)n);
    zbx = make_plan(a, ~zn & a, PX, a & ~b, b & ~c & adjz, n, pn);
    z.s[kTagZBX] = 32 + run_cost((uint32_t)~a, 5) + plan_cost(zbx, n, pn);
  }
  // DBX: base + 33 planes of width 31 (plane 32 = borrow plane, the top)
  Plan dbx = make_plan(ad, andd, ~ord & ad, ad & ~bd, bd & ~cd & adjd, 31, 5);
  {
    const int ones = __popc(Bw);
    const Plan tp = make_plan(Bw != 0, Bw == 0x7FFFFFFFu, 0, ones == 1, ones == 2 && (Bw & (Bw >> 1)), 31, 5);
    dbx.top = tp.nz | (tp.v << 1) | (tp.f5 << 2) | (tp.fa << 3) | (tp.m << 4) | (tp.ms << 5);
    const uint64_t Z = (uint64_t)(uint32_t)~ad | ((uint64_t)(Bw == 0) << 32);
    z.s[kTagDBX] = 32 + run_cost(Z, 5) + plan_cost(dbx, 31, 5) + plan_cost(tp, 31, 5);
  }
  z.bp = Bw;
  keep_smallest(z, bx, zbx, dbx, cand);
  return z;
}

// ------------------------------------------------------------ BF16 classify
// As classify32 for a block of 64 BF16 symbols, on split-packed words.
// Split-packed words (word j = symbol j | symbol j+32 << 16) are built while
// streaming the stage row: word j needs raw words j/2 and 16 + j/2. DBX's
// Gray-coded deltas, split-packed the same way, go to the lane's DBX row.
__device__ __forceinline__ Sizes classify16(uint32_t rowbase, uint32_t lane, uint32_t cand, uint32_t drow) {
  uint32_t a = 0, b = 0, c = 0, adj = 0, andx = ~0u, ors = 0, gprev = 0, g0 = 0;
  uint32_t mlo = 0, mhi = 0, zn = 0, adjz = 0, last = 0;
  uint32_t ad = 0, bd = 0, cd = 0, adjd = 0, andd = ~0u, ord = 0, Blo = 0, Bhi = 0, gdprev = 0,
           gd0 = 0, d32b = 0;
  const uint32_t s31lo = stage_unit(rowbase, lane, 3).w & 0xFFFF0000u;  // symbol 31 in the high half
  uint32_t xprev = 0;
  // split-packed word j >= 1 (symbols j and j+32); the loop below runs over
  // half 16-byte units (4 words each) so that the kernel's code stays small
  auto step = [&](uint32_t x, uint32_t j) -> uint32_t {
    const uint32_t g = x ^ ((x >> 1) & 0x7FFF7FFFu);
    ors |= x;
    c |= b & g;
    b |= a & g;
    a |= g;
    adj |= gprev & g;
    andx &= g;
    gprev = g;
    const uint32_t m = halfmask_nonzero(x);
    mlo = __funnelshift_r(mlo, m, 1);  // symbol j's flag enters at bit 31, ends at bit j
    mhi = __funnelshift_l(m, mhi, 1);  // symbol j+32's flag enters at bit 0 (reversed below)
    zn |= ~g & m;
    adjz |= last & g;
    last = (g & m) | (last & ~m);
    // DBX: lo half d_j = s_j - s_{j-1}, hi half d_{j+32} = s_{j+32} - s_{j+31}
    uint32_t bo;
    const uint32_t d = sub16x2(x, xprev, bo);
    const uint32_t gd = d ^ (((d >> 1) & 0x7FFF7FFFu) | bo);
    ord |= d;
    cd |= bd & gd;
    bd |= ad & gd;
    ad |= gd;
    andd &= gd;
    adjd |= gdprev & gd;
    gdprev = gd;
    Blo = __funnelshift_r(Blo, bo >> 15, 1);  // d_j's borrow ends at bit j (shifted to j-1 below)
    Bhi = __funnelshift_l(bo, Bhi, 1);        // d_{j+32}'s borrow enters at bit 0 (reversed below)
    xprev = x;
    return gd;
  };
  {
    const uint4 qa = stage_unit(rowbase, lane, 0), qb = stage_unit(rowbase, lane, 4);
    // word 0: no delta for symbol 0 (the DBX base); d_32 = s_32 - s_31
    const uint32_t x = prmt(qa.x, qb.x, 0x5410u);
    const uint32_t g = x ^ ((x >> 1) & 0x7FFF7FFFu);
    ors = x;
    a = g;
    g0 = g;
    andx = g;
    gprev = g;
    const uint32_t m = halfmask_nonzero(x);
    mlo = m << 31;
    mhi = m >> 31;
    zn = ~g & m;
    last = g & m;
    uint32_t bo;
    uint32_t d = sub16x2(x, s31lo, bo);
    d &= 0xFFFF0000u;
    bo &= 0x80000000u;
    const uint32_t gd = d ^ (((d >> 1) & 0x7FFF7FFFu) | bo);
    ord = d;
    ad = gd;
    andd = gd | 0x0000FFFFu;
    gd0 = gd;
    gdprev = gd;
    Blo = 0;  // d_32's borrow (bo bit 31) goes to plane position 31 after the loop
    d32b = bo;
    xprev = x;
    const uint32_t d1 = step(prmt(qa.x, qb.x, 0x7632u), 1);
    const uint32_t d2 = step(prmt(qa.y, qb.y, 0x5410u), 2);
    const uint32_t d3 = step(prmt(qa.y, qb.y, 0x7632u), 3);
    sts128(drow_unit(drow, lane, 0), gd, d1, d2, d3);
  }
#pragma unroll 1
  for (uint32_t h = 1; h < 8; ++h) {
    const uint4 qa = stage_unit(rowbase, lane, h >> 1), qb = stage_unit(rowbase, lane, 4u + (h >> 1));
    const bool hi = (h & 1u) != 0;
    const uint32_t a0 = hi ? qa.z : qa.x, a1 = hi ? qa.w : qa.y, b0 = hi ? qb.z : qb.x, b1 = hi ? qb.w : qb.y;
    const uint32_t d0 = step(prmt(a0, b0, 0x5410u), 4u * h);
    const uint32_t d1 = step(prmt(a0, b0, 0x7632u), 4u * h + 1u);
    const uint32_t d2 = step(prmt(a1, b1, 0x5410u), 4u * h + 2u);
    const uint32_t d3 = step(prmt(a1, b1, 0x7632u), 4u * h + 3u);
    sts128(drow_unit(drow, lane, h), d0, d1, d2, d3);
  }
  // the accumulations above left word j's bits at j (low halves) or 31 - j
  // (high halves); bring them to the plane positions the masks use
  mhi = __brev(mhi);
  Blo = (Blo >> 1) | d32b;
  Bhi = __brev(Bhi) >> 1;
  // combine the two halves (symbols 0..31 and 32..63) into 16-plane masks
  auto lo = [](uint32_t v) { return v & 0xFFFFu; };
  auto hi = [](uint32_t v) { return v >> 16; };
  Sizes z;
  z.m0 = mlo;
  z.m1 = mhi;
  int n = __popc(mlo) + __popc(mhi);
  z.s[kTagZVC] = 64 + 16 * n;
  z.s[kTagRAW] = 1024;
  uint32_t a16 = lo(a) | hi(a);
  uint32_t b16 = lo(b) | hi(b) | (lo(a) & hi(a));
  uint32_t c16 = lo(c) | hi(c) | (lo(a) & hi(b)) | (lo(b) & hi(a));
  uint32_t ors16 = lo(ors) | hi(ors);
  uint32_t Z16 = ~a16 & 0xFFFFu;
  uint32_t PX16 = (~ors16 & a16) & 0x7FFFu;
  Plan bx, zbx, dbx;
  // BX: 16 planes of width 64; adjacency across the half split is (31, 32)
  {
    const uint32_t adj16 = lo(adj) | hi(adj) | (lo(gprev) & hi(g0));
    const uint32_t and16 = lo(andx) & hi(andx);
    bx = make_plan(a16, and16, PX16, a16 & ~b16, b16 & ~c16 & adj16, 64, 6);
    z.s[kTagBX] = run_cost(Z16, 4) + plan_cost(bx, 64, 6);
  }
  if (n == 0) {
    zbx = make_plan(0, 0, 0, 0, 0, 1, 0);
    z.s[kTagZBX] = 64;
  } else {
    // the pair across the split: the last survivor among symbols 0..31 and
    // the first among 32..63 (its Gray code read back from the stage row)
    uint32_t gfirst = 0;
    if (mhi) {
      const uint32_t v = lds16(row_swz(rowbase, lane) ^ ((32u + (uint32_t)(__ffs(mhi) - 1)) << 1));
      gfirst = v ^ (v >> 1);
    }
    const uint32_t adjz16 = lo(adjz) | hi(adjz) | (lo(last) & gfirst);
    const uint32_t A = ~(lo(zn) | hi(zn)) & a16;
    const int pn = (int)ceil_log2_u32((uint32_t)n);
    zbx = make_plan(a16, A, PX16, a16 & ~b16, b16 & ~c16 & adjz16, n, pn);
    z.s[kTagZBX] = 64 + run_cost(Z16, 4) + plan_cost(zbx, n, pn);
  }
  // DBX: base + 17 planes of width 63 (plane 16 = borrow plane, the top)
  {
    const uint32_t ad16 = lo(ad) | hi(ad);
    const uint32_t bd16 = lo(bd) | hi(bd) | (lo(ad) & hi(ad));
    const uint32_t cd16 = lo(cd) | hi(cd) | (lo(ad) & hi(bd)) | (lo(bd) & hi(ad));
    const uint32_t adjd16 = lo(adjd) | hi(adjd) | (lo(gdprev) & hi(gd0));
    const uint32_t andd16 = lo(andd) & hi(andd);
    const uint32_t ord16 = lo(ord) | hi(ord);
    const uint64_t Bp = (uint64_t)Blo | ((uint64_t)Bhi << 32);
    z.bp = Bp;
    const int bones = __popcll(Bp);
    const uint32_t tnz = (Bp != 0), tA = (Bp == (1ull << 63) - 1), tS = (bones == 1),
                   tT = (bones == 2) && ((Bp & (Bp >> 1)) != 0);
    dbx = make_plan(ad16 | (tnz << 16), andd16 | (tA << 16), ~ord16 & ad16, (ad16 & ~bd16) | (tS << 16),
                    (bd16 & ~cd16 & adjd16) | (tT << 16), 63, 6);
    const uint32_t Z = ~dbx.nz & 0x1FFFFu;
    z.s[kTagDBX] = 16 + run_cost(Z, 4) + plan_cost(dbx, 63, 6);
  }
  keep_smallest(z, bx, zbx, dbx, cand);
  return z;
}

// ------------------------------------------------------------------ emit
// Emission works out of the lane's own 128-byte row of the stage: first the
// block's words as the TMA left them (128-byte swizzle), later the lane's 32
// transposed plane rows.

__device__ __forceinline__ uint32_t stage_word(uint32_t rowbase, uint32_t r, uint32_t k) {  // k < 32
  return row_swz(rowbase, r) ^ (k << 2);
}
__device__ __forceinline__ uint32_t stage_half(uint32_t rowbase, uint32_t r, uint32_t h) {  // h < 64
  return row_swz(rowbase, r) ^ (h << 1);
}
// Plane rows after the transpose: a lane's 32 rows fill its own 128-byte
// stage row as eight 16-byte units, unit g (rows 4g .. 4g+3) at position
// (g ^ lane) & 7, so that eight consecutive lanes reading their unit g read
// eight different units (all 32 banks) and one 16-byte load brings four
// planes.
__device__ __forceinline__ uint32_t plane_unit(uint32_t rowbase, uint32_t lane, uint32_t g) {  // g < 8
  return rowbase + (((g ^ lane) & 7u) << 4);
}
__device__ __forceinline__ void store_planes(uint32_t rowbase, uint32_t lane, const uint32_t (&T)[32]) {
#pragma unroll
  for (uint32_t g = 0; g < 8; ++g) sts128(plane_unit(rowbase, lane, g), T[4 * g], T[4 * g + 1], T[4 * g + 2], T[4 * g + 3]);
}

// LSB-first writer of one lane's bits into a zeroed shared-memory word
// buffer: each field is ORed in at its bit position, with one shared
// reduction per word it touches (so neighbouring lanes may share words), and
// the position advances. A coded chunk is shorter than its raw size, so every
// word touched lies inside the chunk's buffer (1024 words and slack).
struct PosWriter {
  uint32_t buf;  // shared address of word 0
  uint32_t pos;  // bit position of the next field
  __device__ __forceinline__ void init(uint32_t b, uint32_t bitpos) {
    buf = b;
    pos = bitpos;
  }
  __device__ __forceinline__ uint32_t word_addr() const { return buf + ((pos >> 5) << 2); }
  // len <= 32 bits of v (v < 2^len)
  __device__ __forceinline__ void put(uint32_t v, uint32_t len) {
    const uint32_t sh = pos & 31u, a = word_addr();
    ors32(a, v << sh);
    if (sh + len > 32u) ors32(a + 4, __funnelshift_l(v, 0u, sh));
    pos += len;
  }
  // len <= 64 bits: lo = bits 0..31, hi = bits 32..len-1 (zero when len <=
  // 32; the second reduction then ORs in only what spills past the word)
  __device__ __forceinline__ void put_wide(uint32_t lo, uint32_t hi, uint32_t len) {
    const uint32_t sh = pos & 31u, a = word_addr();
    ors32(a, lo << sh);
    ors32(a + 4, __funnelshift_l(lo, hi, sh));
    if (sh + len > 64u) ors32(a + 8, __funnelshift_l(hi, 0u, sh));
    pos += len;
  }
  // a 1 then the W plane bits of X (the verbatim code; X < 2^W): W <= 32
  // (FP32 planes) or W <= 64 (BF16 planes), one code path each
  template <bool W16>
  __device__ __forceinline__ void put_verbatim(uint32_t xl, uint32_t xh, uint32_t W) {
    const uint32_t v0 = (xl << 1) | 1u, v1 = __funnelshift_l(xl, xh, 1);  // code bits 0..31, 32..63
    const uint32_t sh = pos & 31u, a = word_addr(), end = sh + W + 1u;
    ors32(a, v0 << sh);
    if (end > 32u) ors32(a + 4, __funnelshift_l(v0, v1, sh));
    if (W16 && end > 64u) ors32(a + 8, __funnelshift_l(v1, xh >> 31, sh));
    if (W16 && end > 96u) ors32(a + 12, __funnelshift_l(xh >> 31, 0u, sh));
    pos += W + 1u;
  }
  // the verbatim codes of four planes of 32 bits, X3 (the highest) first:
  // 132 bits, five words before the shift to the position
  __device__ __forceinline__ void put_verbatim32x4(uint32_t X3, uint32_t X2, uint32_t X1, uint32_t X0) {
    const uint32_t c0 = (X3 << 1) | 1u;
    const uint32_t c1 = (X3 >> 31) | 2u | (X2 << 2);
    const uint32_t c2 = (X2 >> 30) | 4u | (X1 << 3);
    const uint32_t c3 = (X1 >> 29) | 8u | (X0 << 4);
    const uint32_t c4 = X0 >> 28;
    const uint32_t sh = pos & 31u, a = word_addr();
    ors32(a, c0 << sh);
    ors32(a + 4, __funnelshift_l(c0, c1, sh));
    ors32(a + 8, __funnelshift_l(c1, c2, sh));
    ors32(a + 12, __funnelshift_l(c2, c3, sh));
    ors32(a + 16, __funnelshift_l(c3, c4, sh));
    if (sh > 28u) ors32(a + 20, __funnelshift_l(c4, 0u, sh));
    pos += 132;
  }
  // N whole words (len bits, the last word possibly partial), B[0] first
  template <int N>
  __device__ __forceinline__ void put_words(const uint32_t (&B)[N], uint32_t len) {
    const uint32_t sh = pos & 31u, a = word_addr();
    ors32(a, B[0] << sh);
#pragma unroll
    for (int k = 1; k < N; ++k) ors32(a + 4u * (uint32_t)k, __funnelshift_l(B[k - 1], B[k], sh));
    if (sh + len > 32u * (uint32_t)N) ors32(a + 4u * (uint32_t)N, __funnelshift_l(B[N - 1], 0u, sh));
    pos += len;
  }
  // the verbatim codes of four BF16 planes of 64 bits (X = hi:lo), X3 first:
  // 4 x 65 bits, nine words before the shift to the position
  __device__ __forceinline__ void put_verbatim64x4(uint32_t l3, uint32_t h3, uint32_t l2, uint32_t h2, uint32_t l1,
                                                   uint32_t h1, uint32_t l0, uint32_t h0) {
    // code k = 1 | X << 1 as three words e0, e1, e2 (e2 one bit)
    auto e0 = [](uint32_t l) { return (l << 1) | 1u; };
    auto e1 = [](uint32_t l, uint32_t h) { return __funnelshift_l(l, h, 1); };
    const uint32_t B[9] = {e0(l3),
                           e1(l3, h3),
                           (h3 >> 31) | (e0(l2) << 1),
                           __funnelshift_l(e0(l2), e1(l2, h2), 1),
                           __funnelshift_l(e1(l2, h2), h2 >> 31, 1) | (e0(l1) << 2),
                           __funnelshift_l(e0(l1), e1(l1, h1), 2),
                           __funnelshift_l(e1(l1, h1), h1 >> 31, 2) | (e0(l0) << 3),
                           __funnelshift_l(e0(l0), e1(l0, h0), 3),
                           __funnelshift_l(e1(l0, h0), h0 >> 31, 3)};
    put_words<9>(B, 260u);
  }
  // the verbatim codes of four planes of W <= 31 bits (FP32 DBX, ZBX), each
  // 1 + W bits given as its code word c = 1 | X << 1: two pairs of codes, each
  // pair at most 64 bits
  __device__ __forceinline__ void put_verbatim_pairs(uint32_t c3, uint32_t c2, uint32_t c1, uint32_t c0, uint32_t W) {
    const uint32_t s = W + 1u;
    const uint64_t A = (uint64_t)c3 | ((uint64_t)c2 << s), B = (uint64_t)c1 | ((uint64_t)c0 << s);
    put_wide((uint32_t)A, (uint32_t)(A >> 32), 2u * s);
    put_wide((uint32_t)B, (uint32_t)(B >> 32), 2u * s);
  }
};

// The code of zero planes i .. hb+1 (a run of r = i - hb planes): 0 0 1 for
// one plane, 0 1 + (r - 2) in K bits for more.
__device__ __forceinline__ void run_code(int r, int K, uint32_t &code, uint32_t &len) {
  code = (r == 1) ? 4u : 2u | ((uint32_t)(r - 2) << 2);
  len = (r == 1) ? 3u : 2u + (uint32_t)K;
}

// The code of a plane that is not verbatim, at most 11 bits (a zero run at
// its top plane i, down to the highest non-zero plane below; 0 0 0 0 0 all
// ones; 0 0 0 0 1 pre-XOR plane zero; 0 0 0 1 1 + q single one at q; 0 0 0 1
// 0 + q two adjacent ones at q, q+1), picked by selects.
__device__ __forceinline__ void put_short(PosWriter &wr, int i, uint32_t below_nz, bool zero, bool f5, bool fa,
                                          bool ms, uint32_t xl, uint32_t xh, uint32_t lm, int K) {
  const int hb = below_nz ? 31 - __clz((int)below_nz) : -1;
  uint32_t rcode, rlen;
  run_code(i - hb, K, rcode, rlen);
  const uint32_t q = xl ? (uint32_t)(__ffs((int)xl) - 1) : 32u + (uint32_t)(__ffs((int)xh) - 1);
  const uint32_t mcode = (ms ? 24u : 8u) | (q << 5);
  const uint32_t code = zero ? rcode : f5 ? (fa ? 0u : 16u) : mcode;
  const uint32_t len = zero ? rlen : f5 ? 5u : lm;
  wr.put(code, len);
}

// Plane codes, top plane first, driven by the candidate's plan (bit i of each
// mask = plane i). For FP32 DBX the 33rd plane (the borrow plane, class bits
// in pl.top) and for BF16 DBX the 17th (bit 16 of the masks) is coded first
// from its value topv; a zero top plane starts a run down to the highest
// non-zero plane below. Then planes 31..0 (FP32) or 15..0 (BF16) in groups of
// four, the group's rows brought by one 16-byte load (BF16: two, the low and
// the high 32 symbols), every lane of the warp at the same group. For DBX a
// row's bit j is delta j, so plane bit q = delta q+1 is the row shifted by
// one. A verbatim plane takes the first branch -- four at once where the
// block's whole group is verbatim (FP32 BX: five words of codes; FP32 DBX
// and ZBX, at most 31 bits a plane: two pairs of codes; BF16 BX: nine words;
// BF16 DBX: eight; BF16 ZBX: four codes of at most 64 bits), as the low
// planes of activations are in whole warps -- and every other code (a zero run at its
// top plane, a 5-bit code, a position code) the second; zero planes below a
// run's top plane emit nothing. Each path exists once in the code (rolled
// loops), which keeps the kernel's instructions within the instruction
// cache.
template <bool W16>
__device__ __forceinline__ void emit_plane_codes(PosWriter &wr, uint32_t rowbase, uint32_t lane, int W, int p,
                                                 bool dbx, uint64_t topv, const Plan &pl) {
  constexpr int K = W16 ? 4 : 5;
  constexpr int kTop = W16 ? 16 : 32;  // the DBX borrow plane
  const uint32_t lowmask = W16 ? 0xFFFFu : 0xFFFFFFFFu;
  const uint32_t NZ = pl.nz & lowmask, V = pl.v & lowmask, F5 = pl.f5, FA = pl.fa, MS = pl.ms;
  const uint32_t lm = 5u + (uint32_t)p;
  int first = W16 ? 15 : 31;  // the lane's highest plane not yet coded
  if (dbx) {
    // class bits of the top plane: nz, verbatim, 5-bit, all-ones, position, single-one
    const uint32_t tb = W16 ? (((pl.nz >> 16) & 1u) | (((pl.v >> 16) & 1u) << 1) | (((pl.f5 >> 16) & 1u) << 2) |
                               (((pl.fa >> 16) & 1u) << 3) | (((pl.m >> 16) & 1u) << 4) | (((pl.ms >> 16) & 1u) << 5))
                            : pl.top;
    const uint32_t tl = (uint32_t)topv, th = (uint32_t)(topv >> 32);
    if (!(tb & 1u)) {  // zero: a run down to the highest non-zero plane below
      const int hb = NZ ? 31 - __clz((int)NZ) : -1;
      uint32_t code, len;
      run_code(kTop - hb, K, code, len);
      wr.put(code, len);
      first = hb;
    } else if (tb & 2u) {
      wr.put_verbatim<W16>(tl, th, (uint32_t)W);
    } else {
      put_short(wr, kTop, 0u, false, (tb & 4u) != 0, (tb & 8u) != 0, (tb & 32u) != 0, tl, th, lm, K);
    }
  }
  const uint32_t live = (first < 0) ? 0u : ((2u << first) - 1u);  // planes not yet coded
  const uint32_t Zm = ~NZ & live;
  const uint32_t RSm = Zm & ~(Zm >> 1);  // zero planes that start a run
  const uint32_t SH = RSm | (NZ & ~V);    // planes with a short code
#pragma unroll 1
  for (int g = W16 ? 3 : 7; g >= 0; --g) {
    uint32_t gv = (V >> (4 * g)) & 15u, gs = (SH >> (4 * g)) & 15u;
    if (!(gv | gs)) continue;
    uint4 qa = lds128(plane_unit(rowbase, lane, (uint32_t)g));
    uint4 qb = make_uint4(0, 0, 0, 0);
    if (W16) qb = lds128(plane_unit(rowbase, lane, (uint32_t)g + 4u));
    if (W16 && gv == 15u) {  // four verbatim BF16 planes
      if (dbx) {  // 63 bits: a row pair is X << 1, so each code is the pair | 1, 64 bits
        const uint32_t B[8] = {qa.w | 1u, qb.w, qa.z | 1u, qb.z, qa.y | 1u, qb.y, qa.x | 1u, qb.x};
        wr.put_words<8>(B, 256u);
      } else if (W == 64) {
        wr.put_verbatim64x4(qa.w, qb.w, qa.z, qb.z, qa.y, qb.y, qa.x, qb.x);
      } else {  // ZBX, at most 63 bits: one code of at most 64 bits each
        const uint32_t s = (uint32_t)W + 1u;
        wr.put_wide((qa.w << 1) | 1u, __funnelshift_l(qa.w, qb.w, 1), s);
        wr.put_wide((qa.z << 1) | 1u, __funnelshift_l(qa.z, qb.z, 1), s);
        wr.put_wide((qa.y << 1) | 1u, __funnelshift_l(qa.y, qb.y, 1), s);
        wr.put_wide((qa.x << 1) | 1u, __funnelshift_l(qa.x, qb.x, 1), s);
      }
      continue;
    }
    if (!W16 && gv == 15u) {  // four verbatim planes: 32 bits (BX) or at most 31 (DBX, ZBX)
      if (W == 32) {
        wr.put_verbatim32x4(qa.w, qa.z, qa.y, qa.x);
      } else {  // a DBX row is X << 1 already
        const uint32_t sh1 = dbx ? 0u : 1u;
        wr.put_verbatim_pairs((qa.w << sh1) | 1u, (qa.z << sh1) | 1u, (qa.y << sh1) | 1u, (qa.x << sh1) | 1u,
                              (uint32_t)W);
      }
      continue;
    }
    // planes 4g+3 .. 4g: the rows move down one place per step (the top row in .w)
#pragma unroll 1
    for (int i = 4 * g + 3; i >= 4 * g; --i) {
      const uint32_t lo = qa.w, hi = qb.w;
      qa = make_uint4(0, qa.x, qa.y, qa.z);
      if (W16) qb = make_uint4(0, qb.x, qb.y, qb.z);
      // the plane X: FP32 the row (DBX: shifted); BF16 low row | high row << 32 (DBX: shifted by one)
      const uint32_t xl = dbx ? (W16 ? __funnelshift_r(lo, hi, 1) : lo >> 1) : lo;
      const uint32_t xh = W16 ? (dbx ? hi >> 1 : hi) : 0u;
      const uint32_t bit = 1u << i;
      if (V & bit) {
        wr.put_verbatim<W16>(xl, xh, (uint32_t)W);
      } else if (SH & bit) {
        put_short(wr, i, NZ & (bit - 1u), !(NZ & bit), (F5 & bit) != 0, (FA & bit) != 0, (MS & bit) != 0, xl, xh, lm,
                  K);
      }
    }
  }
}

// Planes of the kept candidate, before anything is written to the output
// buffer (the DBX rows lie in it): the candidate's words -- DBX's
// Gray-coded deltas from the lane's DBX row, the block's words (BX) from the
// stage row, or its survivors (ZBX), stored in order at their ranks into the
// lane's DBX row, which ZBX does not need (read from the stage row instead
// where they are the block's first W symbols already), Gray-coded here --
// go through one 32x32 bit transpose into the stage row as plane rows
// (store_planes). Every lane runs the same loads, from a row picked by its
// candidate. Returns the plane width W (0: no plane codes) and, for DBX,
// the base symbol, read before the stage row is overwritten.
struct Prep {
  uint32_t W;
  uint32_t base;
};

__device__ __forceinline__ Prep prep32(uint32_t tag, uint32_t nz, uint32_t rowbase, uint32_t lane, uint32_t drow) {
  Prep pr{0u, 0u};
  if (tag == kTagRAW || tag == kTagZVC || (tag == kTagZBX && nz == 0)) return pr;
  const bool dbx = (tag == kTagDBX);
  pr.base = lds32(stage_word(rowbase, lane, 0));
  pr.W = dbx ? 31u : 32u;
  // survivors that are the block's first W symbols (a causal mask's rows)
  // are in place already: the planes come from the stage row as for BX
  const bool moved = (tag == kTagZBX) && (nz & (nz + 1u)) != 0u;
  if (moved) {  // the survivors, in order, to the lane's DBX row (which ZBX does not use)
    const uint32_t dx = row_swz(drow, lane);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint4 q = stage_unit(rowbase, lane, (uint32_t)u);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = 4 * u + k;
        if (nz & (1u << j)) sts32(dx ^ ((uint32_t)__popc(nz & ((1u << j) - 1u)) << 2), w[k]);
      }
    }
  }
  if (tag == kTagZBX) pr.W = (uint32_t)__popc(nz);
  // DBX rows are Gray-coded already (row bit j = delta j, bit 0 zero)
  const uint32_t src = (dbx || moved) ? drow : rowbase, gmask = dbx ? 0u : 0xFFFFFFFFu;
  uint32_t T[32];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint4 q = lds128(row_swz(src, lane) ^ ((uint32_t)u << 4));
    T[4 * u] = q.x;
    T[4 * u + 1] = q.y;
    T[4 * u + 2] = q.z;
    T[4 * u + 3] = q.w;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) T[j] ^= (T[j] >> 1) & gmask;
  transpose32(T);
  if (pr.W < 32u && !dbx) {  // ZBX: plane bits past the survivors come from stale words
    const uint32_t keep = (1u << pr.W) - 1u;
#pragma unroll
    for (int i = 0; i < 32; ++i) T[i] &= keep;
  }
  store_planes(rowbase, lane, T);
  return pr;
}

// FP32 emit of the chosen candidate after prep32. nz: non-zero symbol mask.
__device__ __forceinline__ void emit32(PosWriter &wr, uint32_t tag, uint32_t nz, uint32_t rowbase, uint32_t lane,
                                      const Plan &pl, uint64_t bp, const Prep &pr) {
  if (tag == kTagRAW) {
#pragma unroll 4
    for (uint32_t k = 0; k < 32; ++k) wr.put(lds32(stage_word(rowbase, lane, k)), 32);
    return;
  }
  if (tag == kTagZVC || tag == kTagZBX) wr.put(nz, 32);
  if (tag == kTagZVC) {
    for (uint32_t m = nz; m; m &= m - 1) wr.put(lds32(stage_word(rowbase, lane, __ffs(m) - 1)), 32);
    return;
  }
  if (pr.W == 0) return;  // ZBX without survivors: the mask alone
  const bool dbx = (tag == kTagDBX);
  if (dbx) wr.put(pr.base, 32);
  emit_plane_codes<false>(wr, rowbase, lane, (int)pr.W, (int)ceil_log2_u32(pr.W), dbx, dbx ? bp : 0ull, pl);
}

// BF16 planes of the kept candidate (as prep32, but ZBX's survivors are
// compacted in place in the stage row): split-packed words (word j = symbol
// j | symbol j+32 << 16) -- DBX's from its row as they are, the others built
// from the raw or compacted row.
__device__ __forceinline__ Prep prep16(uint32_t tag, uint32_t mlo, uint32_t mhi, uint32_t rowbase, uint32_t lane,
                                      uint32_t drow) {
  Prep pr{0u, 0u};
  if (tag == kTagRAW || tag == kTagZVC || (tag == kTagZBX && (mlo | mhi) == 0)) return pr;
  const bool dbx = (tag == kTagDBX);
  pr.base = lds16(stage_half(rowbase, lane, 0));
  pr.W = dbx ? 63u : 64u;
  if (tag == kTagZBX) {
    // the survivors' half-words compacted in place (cnt <= h); for 64
    // half-words this loop over the survivors measured as fast as storing
    // every half-word at its rank. Survivors that are the block's first W
    // symbols (a causal mask's rows) are in place already.
    const bool prefix = (mhi == 0u) ? (mlo & (mlo + 1u)) == 0u : (mlo == ~0u && (mhi & (mhi + 1u)) == 0u);
    if (!prefix) {
      uint32_t cnt = 0;
      for (uint32_t m = mlo; m; m &= m - 1, ++cnt)
        sts16(stage_half(rowbase, lane, cnt), lds16(stage_half(rowbase, lane, __ffs(m) - 1)));
      for (uint32_t m = mhi; m; m &= m - 1, ++cnt)
        sts16(stage_half(rowbase, lane, cnt), lds16(stage_half(rowbase, lane, 31 + __ffs(m))));
    }
    pr.W = (uint32_t)(__popc(mlo) + __popc(mhi));
  }
  const uint32_t src = dbx ? drow : rowbase, gmask = dbx ? 0u : 0x7FFF7FFFu;
  uint32_t R[32], T[32];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint4 q = lds128(row_swz(src, lane) ^ ((uint32_t)u << 4));
    R[4 * u] = q.x;
    R[4 * u + 1] = q.y;
    R[4 * u + 2] = q.z;
    R[4 * u + 3] = q.w;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const uint32_t t = dbx ? R[j] : split_word(R, j);
    T[j] = t ^ ((t >> 1) & gmask);
  }
  transpose32(T);  // T[i] = plane i of symbols 0..31, T[16 + i] = plane i of symbols 32..63
  if (pr.W < 64u && !dbx) {  // ZBX: plane bits past the survivors come from stale half-words
    const uint32_t keep_lo = (pr.W >= 32u) ? 0xFFFFFFFFu : ((1u << pr.W) - 1u);
    const uint32_t keep_hi = (pr.W <= 32u) ? 0u : ((1u << (pr.W - 32u)) - 1u);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      T[i] &= keep_lo;
      T[16 + i] &= keep_hi;
    }
  }
  store_planes(rowbase, lane, T);
  return pr;
}

// BF16 emit of the chosen candidate after prep16. mlo/mhi: non-zero masks of
// symbols 0..31 / 32..63.
__device__ __forceinline__ void emit16(PosWriter &wr, uint32_t tag, uint32_t mlo, uint32_t mhi, uint32_t rowbase,
                                      uint32_t lane, const Plan &pl, uint64_t bp, const Prep &pr) {
  if (tag == kTagRAW) {
#pragma unroll 4
    for (uint32_t k = 0; k < 32; ++k) wr.put(lds32(stage_word(rowbase, lane, k)), 32);
    return;
  }
  if (tag == kTagZVC || tag == kTagZBX) {
    wr.put(mlo, 32);
    wr.put(mhi, 32);
  }
  if (tag == kTagZVC) {
    for (uint32_t m = mlo; m; m &= m - 1) wr.put(lds16(stage_half(rowbase, lane, __ffs(m) - 1)), 16);
    for (uint32_t m = mhi; m; m &= m - 1) wr.put(lds16(stage_half(rowbase, lane, 31 + __ffs(m))), 16);
    return;
  }
  if (pr.W == 0) return;  // ZBX without survivors: the masks alone
  const bool dbx = (tag == kTagDBX);
  if (dbx) wr.put(pr.base, 16);
  emit_plane_codes<true>(wr, rowbase, lane, (int)pr.W, (int)ceil_log2_u32(pr.W), dbx, dbx ? bp : 0ull, pl);
}

}  // namespace pz
