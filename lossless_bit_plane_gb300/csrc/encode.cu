// encode.cu — PlaneZip block encoder for sm_103a.
//
// Paper: "PlaneZip: Lossless Bit-Plane Compression of Training Activations
// Offloaded over PCIe" (arXiv:2610.25033v1), Section III-A "Codec" (per
// 128-byte block: ZVC, DBX, BX, ZBX and raw; the smallest is kept behind a
// 3-bit tag; BPC's plane prefix code) and "Stream format" (32 blocks per
// byte-aligned 4 KB chunk with a 16-bit size; a chunk that would grow is
// stored raw); Section II-B (BPC's Delta-BitPlane-XOR).
//
// GPU design (one kernel does load, classify, select, emit, scan, scatter):
//  - Persistent warps take chunks in ticket order (atomic counter), the next
//    ticket only once the current chunk is done. The launch is the
//    programmatic dependent of the small kernel that zeroes the look-back
//    words, the ticket and the total, so that its launch overlaps that
//    kernel; each warp waits for it before its first ticket. A warp owns a
//    4 KB chunk; LANE b OWNS BLOCK b and works on it alone, so the per-block
//    work is SIMD over 32 blocks rather than cooperative.
//  - The chunk arrives by a 2D TMA tile load (32 rows x 128 B, 128-byte
//    swizzle) into the warp's shared stage; the other warps of the SM cover
//    its latency, and each warp prefetches into L2 the chunk one wave of
//    tickets ahead. The swizzle makes each lane's row read (8 x 16 B)
//    bank-conflict free.
//  - Candidate sizes come from plane CLASSES, computed bit-sliced over the
//    32 words a lane holds: the XOR of adjacent planes is the Gray code
//    g = v ^ (v >> 1) of each symbol, and per-plane "any one", "two or more",
//    "three or more", "all ones", "adjacent pair" and "pre-XOR plane zero"
//    flags are plain OR/AND accumulations across words. BF16 runs the same
//    word loop on two 16-bit symbols per word (symbols j and j+32).
//  - Only the winning candidate is materialised: its planes come from one
//    32x32 bit transpose in registers, and its codes go into a shared chunk
//    buffer through an LSB-first writer at the block's bit offset (a warp
//    prefix sum over the lanes' block sizes), plane by plane with every lane
//    of the warp at the same plane.
//  - Chunk offsets come from a single-pass decoupled look-back over 8-byte
//    status words (flag | value) in the scratch tail of the output buffer,
//    with a bounded spin; the warp then copies its chunk to its final byte
//    offset with aligned 16-byte stores and byte stores at the two edges.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "pz_device.cuh"
#include "pz_format.cuh"
#include "pz_kernels.h"

namespace pz {

constexpr uint64_t kFlagAgg = 1ull << 62;
constexpr uint64_t kFlagInc = 2ull << 62;
constexpr uint64_t kValueMask = (1ull << 62) - 1;
constexpr uint32_t kLookbackSpinLimit = 1u << 21;
constexpr uint32_t kMbarPollLimit = 1u << 24;

// ------------------------------------------------------------ cost helpers

// Zero planes (bits of Z, only the first P bits may be set) form maximal
// runs: a run of one costs 3 bits, a longer run 2 + K bits.
__device__ __forceinline__ int run_cost(uint64_t Z, int K) {
  uint64_t start = Z & ~(Z << 1);
  uint64_t single = start & ~(Z >> 1);
  int R = __popcll(start), S = __popcll(single);
  return 3 * S + (2 + K) * (R - S);
}

// Cost of the non-zero planes NZ of width W (position field p): planes that
// are all ones or whose pre-XOR plane is zero (c5) take the 5-bit code, or
// verbatim if shorter; planes with one or two adjacent ones take 5 + p (or
// verbatim); the rest are verbatim, 1 + W.
__device__ __forceinline__ int nonzero_cost(uint64_t NZ, uint64_t A, uint64_t PX, uint64_t ST,
                                            int W, int p) {
  uint64_t c5 = (A | PX) & NZ;
  uint64_t cm = ST & NZ & ~c5;
  uint64_t cv = NZ & ~(c5 | cm);
  int lv = 1 + W;
  int l5 = min(5, lv), lm = min(5 + p, lv);
  return l5 * __popcll(c5) + lm * __popcll(cm) + lv * __popcll(cv);
}

// Class of a single plane given as a word: 0 zero, else its code length.
template <typename T>
__device__ __forceinline__ int single_plane_len(T X, T full, int W, int p) {
  if (X == 0) return 0;
  int ones = (sizeof(T) == 8) ? __popcll((uint64_t)X) : __popc((uint32_t)X);
  int lv = 1 + W;
  if (X == full) return min(5, lv);
  bool adj2 = (ones == 2) && ((X & (X >> 1)) != 0);
  if (ones == 1 || adj2) return min(5 + p, lv);
  return lv;
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
  uint4 q;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(q.x), "=r"(q.y), "=r"(q.z), "=r"(q.w)
               : "r"(row_swz(rowbase, r) ^ (u << 4))
               : "memory");
  return q;
}
__device__ __forceinline__ uint32_t unit_word(const uint4 &q, int k) {
  return (k == 0) ? q.x : (k == 1) ? q.y : (k == 2) ? q.z : q.w;
}
// The block's 32 words into registers (FP32), or its split-packed words
// (BF16: word j = symbol j | symbol j+32 << 16).
template <bool W16>
__device__ __forceinline__ void load_block(uint32_t rowbase, uint32_t lane, uint32_t (&s)[32]) {
  uint32_t raw[32];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint4 q = stage_unit(rowbase, lane, u);
    raw[4 * u] = q.x;
    raw[4 * u + 1] = q.y;
    raw[4 * u + 2] = q.z;
    raw[4 * u + 3] = q.w;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) s[j] = W16 ? split_word(raw, j) : raw[j];
}

// ------------------------------------------------------------ FP32 classify
// s: the block's 32 symbols. Returns the five candidate sizes (tag excluded).
// The words are streamed from the stage row four at a time, so that only the
// accumulators stay in registers.
__device__ __forceinline__ Sizes classify32(uint32_t rowbase, uint32_t lane, uint32_t cand) {
  uint32_t a = 0, b = 0, c = 0, adj = 0, andx = ~0u, ors = 0, gprev = 0;  // BX
  uint32_t nz = 0, zn = 0, adjz = 0, last = 0;                            // ZBX / ZVC
  uint32_t ad = 0, bd = 0, cd = 0, adjd = 0, andd = ~0u, ord = 0, Bw = 0, gdprev = 0;  // DBX
  uint32_t xprev = 0;
  // word k of the block; the loop runs over 16-byte units (4 words each) so
  // that the kernel's code stays small
  auto step = [&](uint32_t x, uint32_t k) {
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
    }
    xprev = x;
  };
  {
    const uint4 q = stage_unit(rowbase, lane, 0);
    step(q.x, 0);
    step(q.y, 1);
    step(q.z, 2);
    step(q.w, 3);
  }
#pragma unroll 1
  for (uint32_t u = 1; u < 8; ++u) {
    const uint4 q = stage_unit(rowbase, lane, u);
    step(q.x, 4 * u);
    step(q.y, 4 * u + 1);
    step(q.z, 4 * u + 2);
    step(q.w, 4 * u + 3);
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
// sp: split-packed block (word j = symbol j | symbol j+32 << 16).
// Split-packed words (word j = symbol j | symbol j+32 << 16) are built while
// streaming the stage row: word j needs raw words j/2 and 16 + j/2.
__device__ __forceinline__ Sizes classify16(uint32_t rowbase, uint32_t lane, uint32_t cand) {
  uint32_t a = 0, b = 0, c = 0, adj = 0, andx = ~0u, ors = 0, gprev = 0, g0 = 0;
  uint32_t mlo = 0, mhi = 0, zn = 0, adjz = 0, last = 0, fst = 0, seen = 0;
  uint32_t ad = 0, bd = 0, cd = 0, adjd = 0, andd = ~0u, ord = 0, Blo = 0, Bhi = 0, gdprev = 0,
           gd0 = 0, d32b = 0;
  const uint32_t s31lo = stage_unit(rowbase, lane, 3).w & 0xFFFF0000u;  // symbol 31 in the high half
  uint32_t xprev = 0;
  // split-packed word j >= 1 (symbols j and j+32); the loop below runs over
  // half 16-byte units (4 words each) so that the kernel's code stays small
  auto step = [&](uint32_t x, uint32_t j) {
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
    fst |= g & ~seen;
    seen |= m;
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
    fst = g;
    seen = m;
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
    step(prmt(qa.x, qb.x, 0x7632u), 1);
    step(prmt(qa.y, qb.y, 0x5410u), 2);
    step(prmt(qa.y, qb.y, 0x7632u), 3);
  }
#pragma unroll 1
  for (uint32_t h = 1; h < 8; ++h) {
    const uint4 qa = stage_unit(rowbase, lane, h >> 1), qb = stage_unit(rowbase, lane, 4u + (h >> 1));
    const bool hi = (h & 1u) != 0;
    const uint32_t a0 = hi ? qa.z : qa.x, a1 = hi ? qa.w : qa.y, b0 = hi ? qb.z : qb.x, b1 = hi ? qb.w : qb.y;
    step(prmt(a0, b0, 0x5410u), 4u * h);
    step(prmt(a0, b0, 0x7632u), 4u * h + 1u);
    step(prmt(a1, b1, 0x5410u), 4u * h + 2u);
    step(prmt(a1, b1, 0x7632u), 4u * h + 3u);
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
    const uint32_t adjz16 = lo(adjz) | hi(adjz) | (lo(last) & hi(fst));
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
// transposed plane rows (XOR-swizzled by lane). Per-plane work runs as short
// runtime loops over that row so that the kernel's code stays small.

__device__ __forceinline__ uint32_t stage_word(uint32_t rowbase, uint32_t r, uint32_t k) {  // k < 32
  return row_swz(rowbase, r) ^ (k << 2);
}
__device__ __forceinline__ uint32_t stage_half(uint32_t rowbase, uint32_t r, uint32_t h) {  // h < 64
  return row_swz(rowbase, r) ^ (h << 1);
}
__device__ __forceinline__ uint32_t plane_row(uint32_t rowbase, uint32_t lane, uint32_t i) {  // i, lane < 32
  return (rowbase ^ (lane << 2)) ^ (i << 2);
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts16(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"((unsigned short)v) : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void emit_run(BitWriter &bw, int run, int K) {
  if (run == 1)
    bw.put(4u, 3);  // 0 0 1
  else
    bw.put(2u | ((uint32_t)(run - 2) << 2), 2 + K);  // 0 1 + (run-2)
}

// One non-zero plane X (T = uint32_t for planes up to 32 bits, uint64_t up to
// 64): the shortest applicable code, ties in the order all-ones,
// pre-XOR-zero, two-adjacent, single-one, verbatim.
template <typename T>
__device__ __forceinline__ void emit_plane(BitWriter &bw, T X, bool prexor_zero, int W, int p, T full) {
  const int ones = (sizeof(T) == 8) ? __popcll((uint64_t)X) : __popc((uint32_t)X);
  const int q = (sizeof(T) == 8) ? (__ffsll((long long)X) - 1) : (__ffs((int)(uint32_t)X) - 1);
  const bool A = (X == full);
  const bool T2 = (ones == 2) && ((X >> q) == (T)3);
  const bool S1 = (ones == 1);
  int len = 1 + W;
  uint32_t val = 0;
  bool verbatim = true;
  if (S1 && 5 + p <= len) { len = 5 + p; val = 24u | ((uint32_t)q << 5); verbatim = false; }  // 0 0 0 1 1 + q
  if (T2 && 5 + p <= len) { len = 5 + p; val = 8u | ((uint32_t)q << 5); verbatim = false; }   // 0 0 0 1 0 + q
  if (prexor_zero && 5 <= len) { len = 5; val = 16u; verbatim = false; }                        // 0 0 0 0 1
  if (A && 5 <= len) { len = 5; val = 0u; verbatim = false; }                                    // 0 0 0 0 0
  if (!verbatim) {
    bw.put(val, (uint32_t)len);
  } else if (sizeof(T) == 4 || W <= 32) {
    bw.put_wide(((uint64_t)X << 1) | 1u, (uint32_t)W + 1);  // 1 + the plane
  } else {
    bw.put_wide(((uint64_t)(uint32_t)X << 1) | 1u, 33);
    bw.put_wide((uint64_t)X >> 32, (uint32_t)W - 32);
  }
}

// Plane codes, top plane first, driven by the candidate's plan: a zero
// plane starts a run that extends to the next non-zero plane (found with a
// leading-zero count), a 5-bit code needs no plane data, and only verbatim
// and position codes read the plane. Plane i < 32 (FP32) or < 16 (BF16, low
// and high 32 symbols in rows i and 16+i) comes from the transposed rows; for
// DBX the rows hold deltas at bit j = delta index j, so plane bit q = delta
// q+1 needs a shift. FP32 DBX has a 33rd plane, the borrow plane, on top: it
// is coded first from its class bits in pl.top and its value topv, so that
// the loop works on 32-bit masks.
//
// The loop is plane-major: every lane of the warp stands at the same plane in
// the same iteration (planes 31..0 for FP32, 16..0 for BF16, where a block
// without a borrow plane has nothing at 16), so the lanes' branches agree
// wherever their blocks' planes take the same code, as the low, verbatim
// planes of activations do. A zero plane emits its run's code at the run's
// top plane only (RSm); planes above the lane's first uncoded plane were
// coded already (FP32 DBX) or do not exist.
template <bool W16>
__device__ __forceinline__ void emit_plane_codes(BitWriter &bw, uint32_t rowbase, uint32_t lane, int top,
                                                 int W, int p, bool dbx, uint64_t topv, const Plan &pl) {
  constexpr int K = W16 ? 4 : 5;
  const uint32_t NZ = pl.nz, V = pl.v, F5 = pl.f5, FA = pl.fa, MS = pl.ms;
  const uint32_t lm = 5u + (uint32_t)p;
  int first = top;  // the lane's highest plane not yet coded
  if (!W16 && dbx) {  // FP32 DBX: plane 32 first
    if (!(pl.top & 1u)) {  // zero: a run down to the highest non-zero plane below
      const int hb = NZ ? 31 - __clz((int)NZ) : -1;
      emit_run(bw, 32 - hb, K);
      first = hb;
    } else {
      if (pl.top & 4u) {
        bw.put((pl.top & 8u) ? 0u : 16u, 5);  // all ones / pre-XOR plane zero
      } else if (pl.top & 2u) {
        bw.put_wide((topv << 1) | 1u, (uint32_t)W + 1);
      } else {
        const uint32_t q = (uint32_t)(__ffsll((long long)topv) - 1);
        bw.put(((pl.top & 32u) ? 24u : 8u) | (q << 5), lm);
      }
      first = 31;
    }
  }
  const uint32_t Zm = (first < 0) ? 0u : (~NZ & ((2u << first) - 1u));
  const uint32_t RSm = Zm & ~(Zm >> 1);
#pragma unroll 1
  for (int i = W16 ? 16 : 31; i >= 0; --i) {
    const uint32_t bit = 1u << i;
    if (!(NZ & bit)) {  // zero planes i .. hb+1
      if (RSm & bit) {
        const uint32_t below = NZ & (bit - 1u);
        const int hb = below ? 31 - __clz((int)below) : -1;
        emit_run(bw, i - hb, K);
      }
      continue;
    }
    if (F5 & bit) {
      bw.put((FA & bit) ? 0u : 16u, 5);  // 0 0 0 0 0 all ones / 0 0 0 0 1 pre-XOR plane zero
    } else {
      uint64_t X;
      if (W16 && dbx && i == 16) {
        X = topv;
      } else {
        const uint32_t lo = lds32(plane_row(rowbase, lane, (uint32_t)i));
        if (W16) {
          const uint32_t hi = lds32(plane_row(rowbase, lane, (uint32_t)i + 16));
          X = dbx ? ((uint64_t)(lo >> 1) | ((uint64_t)hi << 31)) : ((uint64_t)lo | ((uint64_t)hi << 32));
        } else {
          X = dbx ? (uint64_t)(lo >> 1) : (uint64_t)lo;
        }
      }
      if (V & bit) {  // 1 + the plane
        if (W <= 32) {
          bw.put_wide((X << 1) | 1u, (uint32_t)W + 1);
        } else {
          bw.put_wide(((X & 0xFFFFFFFFull) << 1) | 1u, 33);
          bw.put_wide(X >> 32, (uint32_t)W - 32);
        }
      } else {  // 0 0 0 1 1 + q single one / 0 0 0 1 0 + q two adjacent ones
        const uint32_t q = (uint32_t)(__ffsll((long long)X) - 1);
        bw.put(((MS & bit) ? 24u : 8u) | (q << 5), lm);
      }
    }
  }
}

// FP32 emit of the chosen candidate. s: the block's symbols; nz: non-zero mask.
__device__ __forceinline__ void emit32(BitWriter &bw, uint32_t tag, uint32_t nz, uint32_t rowbase, uint32_t lane,
                                      const Plan &pl, uint64_t bp) {
  if (tag == kTagRAW) {
#pragma unroll 4
    for (uint32_t k = 0; k < 32; ++k) bw.put(lds32(stage_word(rowbase, lane, k)), 32);
    return;
  }
  if (tag == kTagZVC || tag == kTagZBX) bw.put(nz, 32);
  if (tag == kTagZVC) {
    for (uint32_t m = nz; m; m &= m - 1) bw.put(lds32(stage_word(rowbase, lane, __ffs(m) - 1)), 32);
    return;
  }
  uint32_t T[32];
  uint64_t topv = 0;
  int top = 31, W = 32;
  if (tag == kTagZBX) {
    if (nz == 0) return;
    uint32_t cnt = 0;  // compact the survivors in place (cnt <= k)
    for (uint32_t m = nz; m; m &= m - 1, ++cnt)
      sts32(stage_word(rowbase, lane, cnt), lds32(stage_word(rowbase, lane, __ffs(m) - 1)));
    W = (int)cnt;
  }
  {
    load_block<false>(rowbase, lane, T);  // BX, DBX and the compacted ZBX row
    if (tag == kTagDBX) {  // deltas (33 bits: bit 32 is the borrow), Gray-coded; the borrow plane came from classify
      bw.put(T[0], 32);
      uint32_t prev = T[0];
      T[0] = 0;
#pragma unroll
      for (int j = 1; j < 32; ++j) {
        const uint32_t cur = T[j];
        const uint64_t d = (uint64_t)cur - (uint64_t)prev;
        const uint32_t lo = (uint32_t)d, hi = (uint32_t)(d >> 32);
        T[j] = lo ^ __funnelshift_r(lo, hi, 1);
        prev = cur;
      }
      topv = bp;
      top = 32;
      W = 31;
    } else {  // BX, or ZBX over its first W (compacted) words
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t t = (j < W) ? T[j] : 0u;
        T[j] = t ^ (t >> 1);
      }
    }
  }
  transpose32(T);
#pragma unroll
  for (int i = 0; i < 32; ++i) sts32(plane_row(rowbase, lane, i), T[i]);
  emit_plane_codes<false>(bw, rowbase, lane, top, W, (int)ceil_log2_u32((uint32_t)W), tag == kTagDBX, topv, pl);
}

// BF16 emit of the chosen candidate. sp: split-packed symbols (word j =
// symbol j | symbol j+32 << 16); mlo/mhi: non-zero masks of 0..31 / 32..63.
__device__ __forceinline__ void emit16(BitWriter &bw, uint32_t tag, uint32_t mlo, uint32_t mhi, uint32_t rowbase,
                                      uint32_t lane, const Plan &pl, uint64_t bp) {
  if (tag == kTagRAW) {
#pragma unroll 4
    for (uint32_t k = 0; k < 32; ++k) bw.put(lds32(stage_word(rowbase, lane, k)), 32);
    return;
  }
  if (tag == kTagZVC || tag == kTagZBX) {
    bw.put(mlo, 32);
    bw.put(mhi, 32);
  }
  if (tag == kTagZVC) {
    for (uint32_t m = mlo; m; m &= m - 1) bw.put(lds16(stage_half(rowbase, lane, __ffs(m) - 1)), 16);
    for (uint32_t m = mhi; m; m &= m - 1) bw.put(lds16(stage_half(rowbase, lane, 31 + __ffs(m))), 16);
    return;
  }
  uint32_t T[32];
  uint64_t topv = 0;
  int top = 15, W = 64;
  if (tag == kTagZBX) {
    uint32_t cnt = 0;  // compact the survivors' half-words in place (cnt <= h)
    for (uint32_t m = mlo; m; m &= m - 1, ++cnt)
      sts16(stage_half(rowbase, lane, cnt), lds16(stage_half(rowbase, lane, __ffs(m) - 1)));
    for (uint32_t m = mhi; m; m &= m - 1, ++cnt)
      sts16(stage_half(rowbase, lane, cnt), lds16(stage_half(rowbase, lane, 31 + __ffs(m))));
    if (cnt == 0) return;
    W = (int)cnt;
  }
  {
    load_block<true>(rowbase, lane, T);  // BX, DBX and the compacted ZBX row
    if (tag == kTagDBX) {  // deltas (17 bits: bit 16 is the borrow), Gray-coded; the borrow plane came from classify
      bw.put(T[0] & 0xFFFFu, 16);
      uint32_t prev = T[31] << 16;  // word 0: no delta for s_0 (the base); d_32 = s_32 - s_31
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t cur = T[j];
        uint32_t bo;
        uint32_t d = sub16x2(cur, prev, bo);
        if (j == 0) {
          d &= 0xFFFF0000u;
          bo &= 0x80000000u;
        }
        T[j] = d ^ (((d >> 1) & 0x7FFF7FFFu) | bo);
        prev = cur;
      }
      topv = bp;
      top = 16;
      W = 63;
    } else {  // BX, or ZBX over its first W (compacted) half-words
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t keep = ((j < W) ? 0x0000FFFFu : 0u) | ((j + 32 < W) ? 0xFFFF0000u : 0u);
        const uint32_t t = T[j] & keep;
        T[j] = t ^ ((t >> 1) & 0x7FFF7FFFu);
      }
    }
  }
  transpose32(T);
#pragma unroll
  for (int i = 0; i < 32; ++i) sts32(plane_row(rowbase, lane, i), T[i]);
  emit_plane_codes<true>(bw, rowbase, lane, top, W, (int)ceil_log2_u32((uint32_t)W), tag == kTagDBX, topv, pl);
}

// --------------------------------------------------------------- look-back

// Exclusive prefix of the chunk sizes before chunk t. Each chunk publishes
// (AGG | L) as soon as its size is known and (INC | prefix + L) once its own
// prefix is known; a warp sums the predecessors' values, 32 at a time,
// back to the nearest inclusive one.
__device__ __forceinline__ uint64_t lookback(unsigned long long *status, uint32_t t,
                                             uint32_t lane, bool &timed_out) {
  uint64_t excl = 0;
  int64_t base = (int64_t)t - 1;
  uint32_t spins = 0;
  while (base >= 0) {
    int64_t idx = base - (int64_t)lane;
    uint64_t v = (idx >= 0) ? ld_relaxed_u64(status + idx) : kFlagInc;
    uint32_t flag = (uint32_t)(v >> 62);
    uint32_t pm = __ballot_sync(0xFFFFFFFFu, flag == 2);
    uint32_t zm = __ballot_sync(0xFFFFFFFFu, flag == 0);
    uint32_t firstP = pm ? (uint32_t)(__ffs(pm) - 1) : 32u;
    uint32_t window = (firstP < 31) ? ((2u << firstP) - 1u) : 0xFFFFFFFFu;
    if (zm & window) {
      if (++spins > kLookbackSpinLimit) {
        timed_out = true;
        break;
      }
      __nanosleep(64);
      continue;
    }
    // the words before the first inclusive one are chunk sizes (at most 4096
    // each), so their sum fits one 32-bit warp reduction; the inclusive
    // word's value comes from its lane
    const uint32_t sizes = (lane < firstP) ? (uint32_t)(v & kValueMask) : 0u;
    const uint64_t inc = (firstP < 32) ? (__shfl_sync(0xFFFFFFFFu, v, firstP) & kValueMask) : 0ull;
    excl += (uint64_t)__reduce_add_sync(0xFFFFFFFFu, sizes) + inc;
    if (firstP < 32) break;
    base -= 32;
  }
  return excl;
}

// ------------------------------------------------------------- copy out
// Copy L bytes from the shared word buffer to global byte address dst
// (any alignment): aligned 16-byte stores inside, byte stores at the edges.
__device__ __forceinline__ void copy_out(const uint32_t *buf, uint32_t L, uint8_t *dst,
                                         uint32_t lane) {
  if (L == 0) return;
  const uint64_t a0 = reinterpret_cast<uint64_t>(dst);
  const uint64_t v0 = a0 & ~15ull;
  const uint32_t nvec = (uint32_t)(((a0 + L - 1) & ~15ull) - v0) / 16 + 1;
  const int nwords = (int)((L + 3) >> 2);
  for (uint32_t i = lane; i < nvec; i += 32) {
    const uint64_t A = v0 + 16ull * i;
    const int o = (int)((int64_t)A - (int64_t)a0);  // source byte of A, may be < 0
    const int wi = o >> 2;                          // floor
    const uint32_t sh = (uint32_t)(o & 3) * 8;
    uint32_t w5[5];
#pragma unroll
    for (int k = 0; k < 5; ++k) {
      int idx = wi + k;
      w5[k] = (idx >= 0 && idx < nwords) ? buf[idx] : 0u;
    }
    uint32_t v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = __funnelshift_r(w5[k], w5[k + 1], sh);
    if (o >= 0 && o + 16 <= (int)L) {
      *reinterpret_cast<uint4 *>(A) = make_uint4(v[0], v[1], v[2], v[3]);
    } else {
#pragma unroll
      for (int byte = 0; byte < 16; ++byte) {
        int so = o + byte;
        if (so >= 0 && so < (int)L)
          reinterpret_cast<uint8_t *>(A)[byte] = (uint8_t)(v[byte >> 2] >> ((byte & 3) * 8));
      }
    }
  }
}

// ------------------------------------------------------------------ kernel

constexpr int kEncWarps = 8;
constexpr int kOutWords = 1024 + 4;

// Shared memory per warp: one 4 KB stage buffer (1024-aligned, the TMA
// destination), the chunk's output word buffer, an mbarrier (16 bytes
// reserved). One stage at three CTAs per SM (24 warps): the next chunk is
// loaded after this one is done, and the other warps cover that load's
// latency. (A second stage, with the next chunk's load in flight, needs more
// shared memory than three CTAs allow.)
template <bool W16>
struct EncCfg {
  static constexpr int kMinCtas = 3;
  static constexpr size_t kStageBytes = 4096;
  static constexpr size_t kOutBytes = kOutWords * 4;
  static constexpr size_t kBytes = 1024 + kEncWarps * kStageBytes + kEncWarps * kOutBytes + kEncWarps * 16;
};

// Byte address of 16-byte unit u of row r in a 128-byte-swizzled stage.
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t u) {
  return r * 128u + ((u ^ (r & 7u)) << 4);
}

// The encoder is launched as the programmatic dependent of the kernel that
// zeroes its scratch words, and may start before that kernel ends.
__global__ void zero_scratch_kernel(unsigned long long *scratch, uint32_t nwords, unsigned long long *total) {
  griddep_launch_dependents();
  const uint32_t i0 = blockIdx.x * blockDim.x + threadIdx.x;
  for (uint32_t i = i0; i < nwords; i += gridDim.x * blockDim.x) scratch[i] = 0;
  if (i0 == 0) *total = 0;
}

// kSizeOnly: the sizes-only launch (no stream). It classifies chunks 0,
// stride, 2*stride, ... (warps take them in a fixed round-robin, no ticket),
// and reports each L and the sum of 2 + L, without emitting, locating or
// writing any payload.
template <bool W16, bool kSizeOnly>
__global__ void __launch_bounds__(kEncWarps * 32, EncCfg<W16>::kMinCtas)
    encode_kernel(const __grid_constant__ CUtensorMap tmap, EncodeArgs p) {
  using Cfg = EncCfg<W16>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t lane = lane_id();
  const uint32_t warp = threadIdx.x >> 5;
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *st = base + warp * Cfg::kStageBytes;
  uint32_t *outbuf = reinterpret_cast<uint32_t *>(base + kEncWarps * Cfg::kStageBytes + warp * Cfg::kOutBytes);
  uint64_t *mbar = reinterpret_cast<uint64_t *>(base + kEncWarps * Cfg::kStageBytes + kEncWarps * Cfg::kOutBytes) +
                   2 * warp;
  const uint32_t mb = smem_u32(mbar);
  if (lane == 0) {
    mbar_init(mb, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const uint32_t C = p.num_chunks;
  const uint64_t nbytes = p.nbytes;
  uint32_t parity = 0;
  bool failed = false;

  // a chunk is loaded by TMA if its first row lies inside the tensor map
  auto uses_tma = [&](uint32_t t) { return (uint64_t)t * 32u < p.tma_rows; };
  auto issue = [&](uint32_t t) {
    if (lane == 0 && uses_tma(t)) {
      mbar_arrive_expect_tx(mb, 4096);
      tma_load_2d(smem_u32(st), &tmap, 0, (int)(t * 32u), mb);
    }
  };
  // plain loads for bytes that the tensor map does not cover
  auto patch = [&](uint32_t t) {
    const uint64_t c0 = (uint64_t)t * 4096u;
    const uint32_t raw_len = (uint32_t)umin64(4096u, nbytes - c0);
    uint32_t from = 0;
    if (uses_tma(t)) {
      from = (uint32_t)(umin64((uint64_t)p.tma_rows * 128u, c0 + 4096u) - c0);
      if (from >= raw_len) return;
    } else {
      for (uint32_t u = lane; u < 256; u += 32)
        *reinterpret_cast<uint4 *>(st + swz(u >> 3, u & 7)) = make_uint4(0, 0, 0, 0);
      __syncwarp();
    }
    for (uint32_t i = from + lane; i < raw_len; i += 32)
      st[swz(i >> 7, (i >> 4) & 7) + (i & 15)] = p.in[c0 + i];
    __syncwarp();
  };

  // work units: chunk t itself, or (sizes only) chunk t * stride
  const uint32_t U = kSizeOnly ? (C + p.stride - 1) / p.stride : C;
  const uint32_t warp_id = blockIdx.x * kEncWarps + warp, nwarps = gridDim.x * kEncWarps;
  auto next_unit = [&](uint32_t u) -> uint32_t {
    if (kSizeOnly) return u + nwarps;
    uint32_t v = 0;
    if (lane == 0) v = atomicAdd(p.ticket, 1u);
    return p.unit0 + __shfl_sync(0xFFFFFFFFu, v, 0);
  };
  auto chunk_of = [&](uint32_t u) -> uint32_t { return kSizeOnly ? u * p.stride : u; };
  unsigned long long size_sum = 0;  // sizes only: this warp's sum of 2 + L

  // the ticket counter is zeroed by the preceding kernel: wait for it before
  // the first ticket (the sizes-only launch waits before its first store)
  bool scratch_ready = false;
  if (!kSizeOnly) {
    griddep_wait();
    scratch_ready = true;
  }
  uint32_t u = kSizeOnly ? warp_id : next_unit(0);
  if (u < U) issue(chunk_of(u));

  while (u < U) {
    const uint32_t t = chunk_of(u);
    if (uses_tma(t)) {
      if (!mbar_wait(mb, parity, kMbarPollLimit)) failed = true;
      parity ^= 1u;
    }
    patch(t);

    const uint64_t c0 = (uint64_t)t * 4096u;
    const uint32_t raw_len = (uint32_t)umin64(4096u, nbytes - c0);
    const uint32_t nblk = (raw_len + 127u) >> 7;
    const bool active = lane < nblk;

    const uint32_t rowbase = smem_u32(st) + lane * 128u;
    Sizes z = W16 ? classify16(rowbase, lane, p.candidates) : classify32(rowbase, lane, p.candidates);
    const uint32_t tag = z.tag;
    uint32_t bits = z.bits;
    bits = active ? bits + 3 : 0;

    // block bit offsets: warp prefix sum
    uint32_t incl = bits;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= (uint32_t)o) incl += v;
    }
    const uint32_t total_bits = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const uint32_t off = incl - bits;
    uint32_t L = (total_bits + 7) >> 3;
    const bool raw_chunk = L >= raw_len;
    if (raw_chunk) L = raw_len;
    if (!scratch_ready) {  // sizes only: before the first store to the sizes or the total
      griddep_wait();
      scratch_ready = true;
    }
    if (kSizeOnly) {
      if (lane == 0) {
        if (p.sizes) p.sizes[u] = (uint16_t)L;
        size_sum += 2u + L;
      }
      __syncwarp();
      fence_proxy_async_smem();  // generic-proxy use of the stage before the next TMA write
      u = next_unit(u);
      if (u < U) issue(chunk_of(u));
      continue;
    }
    if (lane == 0) st_relaxed_u64(p.status + t, (t == 0 ? kFlagInc : kFlagAgg) | L);

    if (!raw_chunk) {
      const uint32_t nw = (L + 3) / 4 + 1;
      for (uint32_t i = lane; i < nw; i += 32) outbuf[i] = 0;
      __syncwarp();
      if (active) {
        BitWriter bw;
        bw.init(outbuf, off, kOutWords);
        bw.put(tag, 3);
        const Plan &pl = z.win;
        if (W16)
          emit16(bw, tag, z.m0, z.m1, rowbase, lane, pl, z.bp);
        else
          emit32(bw, tag, z.m0, rowbase, lane, pl, z.bp);
        bw.flush();
      }
    } else {
      for (uint32_t u = lane; u < 256; u += 32)
        reinterpret_cast<uint4 *>(outbuf)[u] = *reinterpret_cast<const uint4 *>(st + swz(u >> 3, u & 7));
    }
    __syncwarp();

    bool to = false;
    const uint64_t excl = (t == 0) ? 0 : lookback(p.status, t, lane, to);
    if (to) failed = true;
    if (lane == 0) {
      if (t) st_relaxed_u64(p.status + t, kFlagInc | (excl + L));
      p.out[2ull * t] = (uint8_t)(L & 0xFF);
      p.out[2ull * t + 1] = (uint8_t)(L >> 8);
      if (t == C - 1) atomicMax(p.total, 2ull * C + excl + L);
    }
    copy_out(outbuf, L, p.out + 2ull * C + excl, lane);

    __syncwarp();
    fence_proxy_async_smem();  // generic-proxy use of the stage before the next TMA write
    // The next ticket is taken only now: a warp that holds a ticket is always
    // working toward that chunk's size, so no look-back waits on a chunk whose
    // warp is still busy with its previous one.
    u = next_unit(u);
    if (u < U) issue(chunk_of(u));  // one stage: load the next chunk now that this one is done
    // The chunk one wave of tickets ahead (every warp of the grid takes one
    // ticket per wave) is brought into L2, so that its warp's TMA load finds
    // it there; each chunk is prefetched once, by the warp one wave before.
    if (lane == 0 && (uint64_t)(u + nwarps + 1) * 32u <= p.tma_rows)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.in + (uint64_t)(u + nwarps) * 4096u),
                   "r"(4096u)
                   : "memory");
  }
  if (kSizeOnly && lane == 0 && size_sum) atomicAdd(p.total, size_sum);
  if (failed && lane == 0) atomicMax(p.total, ~0ull);
}

template __global__ void encode_kernel<false, false>(const __grid_constant__ CUtensorMap, EncodeArgs);
template __global__ void encode_kernel<true, false>(const __grid_constant__ CUtensorMap, EncodeArgs);
template __global__ void encode_kernel<false, true>(const __grid_constant__ CUtensorMap, EncodeArgs);
template __global__ void encode_kernel<true, true>(const __grid_constant__ CUtensorMap, EncodeArgs);

size_t encode_smem_bytes(bool w16) { return w16 ? EncCfg<true>::kBytes : EncCfg<false>::kBytes; }
int encode_threads() { return kEncWarps * 32; }
int encode_warps() { return kEncWarps; }

const void *zero_scratch_kernel_ptr() { return reinterpret_cast<const void *>(&zero_scratch_kernel); }
const void *encode_kernel_ptr(bool w16, bool size_only) {
  if (size_only)
    return w16 ? reinterpret_cast<const void *>(&encode_kernel<true, true>)
               : reinterpret_cast<const void *>(&encode_kernel<false, true>);
  return w16 ? reinterpret_cast<const void *>(&encode_kernel<true, false>)
             : reinterpret_cast<const void *>(&encode_kernel<false, false>);
}

}  // namespace pz
