// decode.cu — PlaneZip block decoder for sm_103a.
//
// Paper: "PlaneZip: Lossless Bit-Plane Compression of Training Activations
// Offloaded over PCIe" (arXiv:2610.25033v1), Section III-A "Stream format":
// the decompressor locates every chunk with a prefix sum over the 16-bit
// chunk sizes and decodes chunks in parallel; each block is the inverse of
// its tagged candidate (Section III-A "Codec").
//
// GPU design:
//  - The format stores no per-block offsets: block b of a chunk starts where
//    block b-1 ends, so a chunk's blocks must be parsed in order. Parallelism
//    therefore comes from chunks: LANE = CHUNK. A warp decodes 32 chunks at
//    once, each lane walking its own chunk's 32 blocks in sequence, so the
//    serial prefix-code parse runs SIMD across 32 chunks.
//  - Chunk offsets: each CTA sums all headers before its first chunk
//    (16-byte vector loads, L2-resident, reduced in shared memory) and scans
//    its own 128 headers; no scratch memory and no inter-CTA waiting.
//  - Raw chunks (L == raw size) are copied by the whole warp with coalesced
//    16-byte stores; compressed chunks are parsed by their lane through an
//    LSB-first bit reader over read-only cached 32-bit loads with one word
//    of look-ahead.
//  - Planes are rebuilt top-down in registers (pre-XOR plane P_i = X_i ^
//    P_{i+1}), turned back into symbols by one 32x32 bit transpose, then the
//    delta is undone (prefix sum) or the survivors are scattered back (ZBX)
//    through a lane-private shared-memory scratch.
//  - Every field is validated; a malformed chunk sets PZ_ERR_CORRUPT in the
//    status word and stops; no write leaves the chunk's output range and no
//    read leaves the input.
#include <cuda_runtime.h>

#include <cstdint>

#include "pz_device.cuh"
#include "pz_format.cuh"
#include "pz_kernels.h"

namespace pz {

constexpr int kDecWarps = 8;
constexpr uint32_t kStageWords = (4096 + 16) / 4 + 4;  // 257 16-byte units + slack for 64-bit peeks

__device__ __forceinline__ uint32_t lds32d(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds16d(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void sts32d(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts16d(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"((unsigned short)v) : "memory");
}
// Lane-private 32-word row, XOR-swizzled by lane (conflict-free across lanes).
__device__ __forceinline__ uint32_t prow(uint32_t row, uint32_t lane, uint32_t word) {
  return row + (((word ^ lane) & 31u) << 2);
}
__device__ __forceinline__ uint32_t prow_half(uint32_t row, uint32_t lane, uint32_t h) {
  return prow(row, lane, h >> 1) + ((h & 1u) << 1);
}

// A chunk's payload staged in shared memory: word k holds stream bytes
// [a0 + 4k, a0 + 4k + 4), where a0 is the payload's first byte rounded down
// to 16; bit q counts from a0. The buffer has slack words past the data.
struct StageBits {
  uint32_t base;  // shared address of word 0
  // word address of bit q, clamped so that a malformed stream cannot read
  // outside the buffer (valid streams never reach the clamp)
  __device__ __forceinline__ uint32_t addr(uint32_t q) const { return base + (min(q >> 5, kStageWords - 3u) << 2); }
  __device__ __forceinline__ uint32_t peek32(uint32_t q) const {
    const uint32_t a = addr(q);
    return __funnelshift_r(lds32d(a), lds32d(a + 4), q & 31u);
  }
  // bits [q, q + 64) and bit q + 64
  __device__ __forceinline__ uint64_t peek64(uint32_t q, uint32_t &bit64) const {
    const uint32_t a = addr(q), sh = q & 31u;
    const uint32_t w0 = lds32d(a), w1 = lds32d(a + 4), w2 = lds32d(a + 8);
    bit64 = (w2 >> sh) & 1u;
    return (uint64_t)__funnelshift_r(w0, w1, sh) | ((uint64_t)__funnelshift_r(w1, w2, sh) << 32);
  }
};

// Decode the block whose tag is at stage bit q into o[32] (the block's 32
// words in memory order); q advances past the block. Plane codes are parsed
// by a per-plane loop that is the same instruction stream for every lane
// (the code class picks values by selects, not branches): each plane is
// X_i, rebuilt to the pre-XOR plane P_i = X_i ^ P_{i+1} and stored in the
// lane's row (FP32 plane i < 32 in word i; BF16 plane i < 16 in words i and
// 16+i; DBX rows pre-shifted so row bit j is delta j). One 32x32 bit
// transpose then turns rows into symbols. Returns false on a malformed code.
template <bool W16>
__device__ __forceinline__ bool decode_block(const StageBits &sb, uint32_t &q, uint32_t (&o)[32], uint32_t row,
                                             uint32_t lane) {
  constexpr int K = W16 ? 4 : 5;
  const uint32_t tag = sb.peek32(q) & 7u;
  q += 3;
  if (tag > kTagRAW) return false;
  if (tag == kTagRAW) {
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = sb.peek32(q + 32u * k);
    q += 1024;
    return true;
  }
  if (tag == kTagZVC) {
    if (W16) {
      const uint32_t mlo = sb.peek32(q), mhi = sb.peek32(q + 32);
      q += 64;
#pragma unroll 1
      for (uint32_t h = 0; h < 64; ++h) {
        const uint32_t bit = ((h < 32) ? (mlo >> h) : (mhi >> (h - 32))) & 1u;
        sts16d(prow_half(row, lane, h), bit ? (sb.peek32(q) & 0xFFFFu) : 0u);
        q += bit * 16u;
      }
    } else {
      const uint32_t mask = sb.peek32(q);
      q += 32;
#pragma unroll 1
      for (uint32_t k = 0; k < 32; ++k) {
        const uint32_t bit = (mask >> k) & 1u;
        sts32d(prow(row, lane, k), bit ? sb.peek32(q) : 0u);
        q += bit * 32u;
      }
    }
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = lds32d(prow(row, lane, k));
    return true;
  }
  uint32_t basesym = 0, mlo = 0, mhi = 0;
  int top = W16 ? 15 : 31, W = W16 ? 64 : 32;
  if (tag == kTagDBX) {
    basesym = sb.peek32(q) & (W16 ? 0xFFFFu : 0xFFFFFFFFu);
    q += W16 ? 16 : 32;
    ++top;
    --W;
  } else if (tag == kTagZBX) {
    mlo = sb.peek32(q);
    q += 32;
    if (W16) {
      mhi = sb.peek32(q);
      q += 32;
    }
    W = __popc(mlo) + __popc(mhi);
    if (W == 0) {
#pragma unroll
      for (int k = 0; k < 32; ++k) o[k] = 0;
      return true;
    }
  }
  const bool dbx = (tag == kTagDBX);
  const uint32_t p = (uint32_t)ceil_log2_int(W);
  const uint32_t pmask = (1u << p) - 1u;
  // code length by class (leading zero bits, capped at 4), 7 bits each
  const uint32_t lens = (1u + (uint32_t)W) | ((2u + K) << 7) | (3u << 14) | ((5u + p) << 21);
  // The walk kernel has already checked run lengths and the pre-XOR-zero
  // code's plane; the position field's range is checked here.
  bool bad = false;
  int run = 0;
  if (!W16) {
    const uint32_t full = (W >= 32) ? ~0u : ((1u << W) - 1u);
    uint32_t Pup = 0;
#pragma unroll 1
    for (int i = top; i >= 0; --i) {
      uint32_t X = 0;
      if (run > 0) {
        --run;
      } else {
        const uint32_t a = sb.addr(q), sh = q & 31u;
        const uint32_t w0 = lds32d(a), w1 = lds32d(a + 4), w2 = lds32d(a + 8);
        const uint32_t lo = __funnelshift_r(w0, w1, sh), hi = __funnelshift_r(w1, w2, sh);
        const uint32_t tz = (uint32_t)__ffs(lo | 16u) - 1u;
        const uint32_t qf = (lo >> 5) & pmask;
        const bool hi4 = (lo & 16u) != 0;
        const uint32_t xv = __funnelshift_r(lo, hi, 1) & full;
        const uint32_t xp = (hi4 ? 1u : 3u) << qf;
        const uint32_t x5 = hi4 ? Pup : full;
        X = (tz == 0u) ? xv : (tz == 3u) ? xp : (tz == 4u) ? x5 : 0u;
        q += (tz == 4u) ? 5u : ((lens >> (7u * tz)) & 127u);
        if (tz == 1u) run = 1 + (int)((lo >> 2) & ((1u << K) - 1u));
        bad |= (tz == 3u) && (qf + (hi4 ? 0u : 1u) >= (uint32_t)W);
      }
      const uint32_t Pi = (i == top) ? X : (X ^ Pup);
      Pup = Pi;
      if (i < 32) sts32d(prow(row, lane, (uint32_t)i), dbx ? (Pi << 1) : Pi);
    }
  } else {
    const uint64_t full = (W >= 64) ? ~0ull : ((1ull << W) - 1);
    uint64_t Pup = 0;
#pragma unroll 1
    for (int i = top; i >= 0; --i) {
      uint64_t X = 0;
      if (run > 0) {
        --run;
      } else {
        uint32_t b64;
        const uint64_t win = sb.peek64(q, b64);
        const uint32_t lo = (uint32_t)win;
        const uint32_t tz = (uint32_t)__ffs(lo | 16u) - 1u;
        const uint32_t qf = (lo >> 5) & pmask;
        const bool hi4 = (lo & 16u) != 0;
        const uint64_t xv = (W >= 64) ? ((win >> 1) | ((uint64_t)b64 << 63)) : ((win >> 1) & full);
        const uint64_t xp = (hi4 ? 1ull : 3ull) << qf;
        const uint64_t x5 = hi4 ? Pup : full;
        X = (tz == 0u) ? xv : (tz == 3u) ? xp : (tz == 4u) ? x5 : 0ull;
        q += (tz == 4u) ? 5u : ((lens >> (7u * tz)) & 127u);
        if (tz == 1u) run = 1 + (int)((lo >> 2) & ((1u << K) - 1u));
        bad |= (tz == 3u) && (qf + (hi4 ? 0u : 1u) >= (uint32_t)W);
      }
      const uint64_t Pi = (i == top) ? X : (X ^ Pup);
      Pup = Pi;
      if (i < 16) {
        sts32d(prow(row, lane, (uint32_t)i), dbx ? (uint32_t)(Pi << 1) : (uint32_t)Pi);
        sts32d(prow(row, lane, (uint32_t)i + 16), dbx ? (uint32_t)(Pi >> 31) : (uint32_t)(Pi >> 32));
      }
    }
  }
  const bool ok = !bad;
#pragma unroll
  for (int j = 0; j < 32; ++j) o[j] = lds32d(prow(row, lane, j));
  transpose32(o);  // FP32: o[j] = symbol j (or delta j); BF16: split words
  if (!W16) {
    if (dbx) {
      o[0] = basesym;
#pragma unroll
      for (int j = 1; j < 32; ++j) o[j] += o[j - 1];
    } else if (tag == kTagZBX) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < W) sts32d(prow(row, lane, j), o[j]);
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const uint32_t rank = __popc(mlo & ((1u << k) - 1u));
        o[k] = ((mlo >> k) & 1u) ? lds32d(prow(row, lane, rank)) : 0u;
      }
    }
    return ok;
  }
  // BF16: o holds split words (word j = symbol j | symbol j+32 << 16)
  if (dbx) {
    uint32_t prev = basesym;  // s_0
    o[0] = (o[0] & 0xFFFF0000u) | prev;
#pragma unroll
    for (int j = 1; j < 32; ++j) {  // s_j = s_{j-1} + d_j
      prev = (prev + o[j]) & 0xFFFFu;
      o[j] = (o[j] & 0xFFFF0000u) | prev;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {  // s_{j+32} = s_{j+31} + d_{j+32}
      prev = (prev + (o[j] >> 16)) & 0xFFFFu;
      o[j] = (o[j] & 0xFFFFu) | (prev << 16);
    }
  } else if (tag == kTagZBX) {
    // survivors t_0..t_{W-1}: t_j in o[j] low, t_{j+32} in o[j] high; store
    // them as half-words in index order, then gather each symbol by rank
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < W) sts16d(prow_half(row, lane, j), o[j] & 0xFFFFu);
      if (j + 32 < W) sts16d(prow_half(row, lane, j + 32), o[j] >> 16);
    }
    const uint32_t clo = __popc(mlo);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const uint32_t rl = __popc(mlo & ((1u << j) - 1u));
      const uint32_t rh = clo + __popc(mhi & ((1u << j) - 1u));
      const uint32_t vl = ((mlo >> j) & 1u) ? lds16d(prow_half(row, lane, rl)) : 0u;
      const uint32_t vh = ((mhi >> j) & 1u) ? lds16d(prow_half(row, lane, rh)) : 0u;
      o[j] = vl | (vh << 16);
    }
  }
  uint32_t sp[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) sp[j] = o[j];
#pragma unroll
  for (int r = 0; r < 32; ++r) o[r] = raw_word_from_split(sp, r);
  return ok;
}

// ------------------------------------------------------ block boundaries
// The format stores no per-block offsets, so a chunk's block starts come from
// a walk that only measures code lengths (tags, masks, plane-code prefixes).

// 32 stream bits starting at an absolute bit position (reads clamped to the
// input, so a malformed length never reads outside it).
struct Window {
  const uint32_t *w;
  uint64_t nw;
  __device__ __forceinline__ uint32_t ld(uint64_t i) const { return i < nw ? __ldg(w + i) : 0u; }
  __device__ __forceinline__ uint32_t peek32(uint64_t pos) const {
    const uint64_t wi = pos >> 5;
    return __funnelshift_r(ld(wi), ld(wi + 1), (uint32_t)(pos & 31));
  }
};

// Reader over one chunk's bits at chunk-relative positions.
struct WindowReader {  // straight from global memory (clamped to the input)
  Window win;
  uint64_t base;
  __device__ __forceinline__ uint32_t peek(uint32_t pos) const { return win.peek32(base + pos); }
};

// Lane-private 512-byte ring in shared memory, filled ahead of the read
// position with 16-byte cp.async copies (one commit group per copy), so a
// lane streams its chunk without scattered global loads.
constexpr uint32_t kRingUnits = 32;  // 16-byte units per ring
constexpr uint32_t kRingAhead = 24;  // units kept in flight past the read unit

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_ahead() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kRingAhead) : "memory");
}

struct RingReader {
  uint32_t ring;       // shared address of the lane's ring
  const uint8_t *g0;   // 16-byte aligned global address of unit 0
  uint32_t nunits;     // units that hold chunk bytes
  uint32_t fetched;    // units issued so far
  uint32_t bit0;       // bit of unit 0 where the chunk starts
  uint32_t limit;      // a peek at any q = bit0 + pos below this is resident

  __device__ __forceinline__ void init(uint32_t ring_addr, const uint8_t *in, uint64_t off, uint32_t L) {
    const uint64_t a0 = off & ~15ull;
    ring = ring_addr;
    g0 = in + a0;
    bit0 = (uint32_t)(off - a0) * 8u;
    nunits = (uint32_t)((off + L + 15 - a0) >> 4);
    fetched = 0;
    limit = 0;
  }
  __device__ __forceinline__ void refill(uint32_t q) {
    const uint32_t need = ((q + 63) >> 7) + 1;  // units under a 64-bit window at q
    const uint32_t lim = min(need + kRingAhead, nunits);
    while (fetched < lim) {
      cp_async16(ring + (fetched % kRingUnits) * 16u, g0 + 16ull * fetched);
      ++fetched;
    }
    if (fetched == nunits) {
      cp_async_wait_all();
      limit = 0xFFFFFFFFu;
    } else {
      cp_async_wait_ahead();
      limit = (fetched - kRingAhead) * 128u - 63u;  // q + 63 < resident units * 128
    }
  }
  // 32 bits at chunk bit pos; the caller has ensured residency
  __device__ __forceinline__ uint32_t peek_resident(uint32_t pos) const {
    const uint32_t q = bit0 + pos;
    const uint32_t w = q >> 5;
    uint32_t lo, hi;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(lo) : "r"(ring + ((w & (kRingUnits * 4 - 1)) << 2)) : "memory");
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(hi) : "r"(ring + (((w + 1) & (kRingUnits * 4 - 1)) << 2)) : "memory");
    return __funnelshift_r(lo, hi, q & 31u);
  }
  // the single bit at chunk bit pos (resident)
  __device__ __forceinline__ uint32_t bit_resident(uint32_t pos) const {
    const uint32_t q = bit0 + pos;
    uint32_t w;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(ring + (((q >> 5) & (kRingUnits * 4 - 1)) << 2)) : "memory");
    return (w >> (q & 31u)) & 1u;
  }
  // make every peek at or below pos resident
  __device__ __forceinline__ void ensure(uint32_t pos) {
    const uint32_t q = bit0 + pos;
    if (q >= limit) refill(q);
  }
  __device__ __forceinline__ uint32_t peek(uint32_t pos) {
    ensure(pos);
    return peek_resident(pos);
  }
};

struct WindowPeeker {  // adapts WindowReader to the ensure / peek_resident interface
  WindowReader r;
  __device__ __forceinline__ void ensure(uint32_t) const {}
  __device__ __forceinline__ uint32_t peek_resident(uint32_t pos) const { return r.peek(pos); }
  __device__ __forceinline__ uint32_t bit_resident(uint32_t pos) const { return r.peek(pos) & 1u; }
  __device__ __forceinline__ uint32_t peek(uint32_t pos) const { return r.peek(pos); }
};

// Advance pos over the plane codes of planes top..0 of width W. Each step
// tests the flag bits of the next eight codes under the assumption that they
// are verbatim (a verbatim code is 1 + W bits): a run of m leading verbatim
// codes advances m planes at once; otherwise the code at pos is classified
// by its leading zero bits (stream order, capped at 4): 01 run (2+K bits,
// 2+field planes), 001 single zero (3), 0001x position code (5+p), 0000x
// all-ones / pre-XOR-zero (5).
template <typename Reader>
__device__ __forceinline__ bool walk_planes(Reader &rd, uint32_t &pos, int top, int W, int K) {
  constexpr int kSkip = 8;
  const uint32_t p = (uint32_t)ceil_log2_int(W);
  const uint32_t S = 1u + (uint32_t)W;
  const uint32_t kmask = (1u << K) - 1u;
  int i = top;
  bool ok = true;
#pragma unroll 1
  while (i >= 0) {
    rd.ensure(pos + (kSkip - 1) * S);
    uint32_t f = 0;
#pragma unroll
    for (int k = 0; k < kSkip; ++k) f |= rd.bit_resident(pos + (uint32_t)k * S) << k;
    int m = __ffs(~f) - 1;  // leading verbatim codes, 0..kSkip
    if (m > i + 1) m = i + 1;
    if (m > 0) {
      pos += (uint32_t)m * S;
      i -= m;
      continue;
    }
    const uint32_t v0 = rd.peek_resident(pos);
    const uint32_t tz = (uint32_t)__ffs(v0 | 16u) - 1u;  // 1..4
    const uint32_t len = (tz == 1u) ? 2u + K : (tz == 2u) ? 3u : (tz == 3u) ? 5u + p : 5u;
    const int run = (tz == 1u) ? 2 + (int)((v0 >> 2) & kmask) : 1;
    ok = ok && !(run > i + 1) && !(tz == 4u && (v0 & 16u) && i == top);
    pos += len;
    i -= run;
  }
  return ok;
}

// Record each block's start bit (relative to the chunk) and check that the
// chunk is exactly ceil(bits/8) bytes with zero padding.
template <bool W16, typename Reader>
__device__ __forceinline__ bool walk_chunk(Reader &rd, uint32_t L, uint32_t nblk, uint16_t *starts) {
  constexpr int w = W16 ? 16 : 32;
  constexpr int N = W16 ? 64 : 32;
  constexpr int K = W16 ? 4 : 5;
  const uint32_t cap = 8u * L;
  uint32_t pos = 0;
#pragma unroll 1
  for (uint32_t b = 0; b < nblk; ++b) {
    starts[b] = (uint16_t)pos;
    const uint32_t tag = rd.peek(pos) & 7u;
    pos += 3;
    if (tag > kTagRAW) return false;
    if (tag == kTagRAW) {
      pos += 1024;
    } else if (tag == kTagZVC || tag == kTagZBX) {
      uint32_t n = __popc(rd.peek(pos));
      pos += 32;
      if (W16) {
        n += __popc(rd.peek(pos));
        pos += 32;
      }
      if (tag == kTagZVC)
        pos += n * w;
      else if (n && !walk_planes(rd, pos, w - 1, (int)n, K))
        return false;
    } else {
      int top = w - 1, W = N;
      if (tag == kTagDBX) {
        pos += w;
        top = w;
        W = N - 1;
      }
      if (!walk_planes(rd, pos, top, W, K)) return false;
    }
    if (pos > cap) return false;
  }
  if (cap - pos >= 8) return false;
  if (cap > pos && (rd.peek(pos) & ((1u << (cap - pos)) - 1u))) return false;
  return true;
}

// ---------------------------------------------------------------- kernels
//
// Two launches. The walk kernel runs one thread per chunk: it finds the
// chunk's payload offset (sum of all earlier sizes) and, for a coded chunk,
// every block's start bit, and leaves them in the first bytes of that
// chunk's own output region: the offset (8 bytes) then the start bits of
// blocks 1..n-1 (2 bytes each). The decode kernel runs one warp per chunk,
// lane = block: each lane reads its start, the warp synchronises, and only
// then are those bytes overwritten with decoded data. A final chunk too
// short to hold that record (under 72 bytes) is located and walked by its
// decode warp instead.

constexpr int kWalkThreads = 64;
constexpr int kRecordBytes = 72;  // 8-byte offset + 31 x 2-byte start bits + padding

// Sum of the 16-bit sizes of chunks [0, first) by all threads of the block;
// first must be a multiple of 8.
__device__ __forceinline__ unsigned long long sum_sizes_before(const uint8_t *in, uint32_t first) {
  unsigned long long part = 0;
  const uint4 *h4 = reinterpret_cast<const uint4 *>(in);
  for (uint32_t i = threadIdx.x; i < first / 8; i += blockDim.x) {
    const uint4 v = __ldg(h4 + i);
    part += (v.x & 0xFFFFu) + (v.x >> 16) + (v.y & 0xFFFFu) + (v.y >> 16) + (v.z & 0xFFFFu) + (v.z >> 16) +
            (v.w & 0xFFFFu) + (v.w >> 16);
  }
  return part;
}

template <bool W16>
__global__ void __launch_bounds__(kWalkThreads)
    walk_kernel(DecodeArgs p) {
  __shared__ __align__(16) uint8_t rings[kWalkThreads][kRingUnits * 16];
  __shared__ unsigned long long red[kWalkThreads / 32];
  __shared__ uint32_t wsum[kWalkThreads / 32];
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t C = p.num_chunks;
  const uint32_t first = blockIdx.x * kWalkThreads;
  unsigned long long part = warp_sum_u64(sum_sizes_before(p.in, first));
  const uint32_t c = first + threadIdx.x;
  const bool valid = c < C;
  const uint32_t L = valid ? __ldg(reinterpret_cast<const uint16_t *>(p.in) + c) : 0u;
  uint32_t incl = L;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= (uint32_t)o) incl += v;
  }
  if (lane == 0) red[warp] = part;
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (!valid) return;
  unsigned long long base = 0;
  for (int w = 0; w < kWalkThreads / 32; ++w) base += red[w];
  for (uint32_t w = 0; w < warp; ++w) base += wsum[w];
  const uint64_t off = 2ull * C + base + (incl - L);
  const uint32_t raw_len = (uint32_t)umin64(4096u, p.nbytes - (uint64_t)c * 4096u);
  if (L == 0 || L > raw_len || off + L > p.comp_bytes) {
    atomicMax(p.status, kErrCorrupt);
    return;
  }
  if (raw_len < (uint32_t)kRecordBytes) return;  // the decode warp handles it
  uint8_t *rec = p.out + (uint64_t)c * 4096u;
  *reinterpret_cast<unsigned long long *>(rec) = off;
  if (L == raw_len) return;  // raw chunk: the offset is all the decoder needs
  uint16_t starts[32];
  RingReader rd;
  rd.init(smem_u32(rings[threadIdx.x]), p.in, off, L);
  const uint32_t nblk = (raw_len + 127u) >> 7;
  const bool ok = walk_chunk<W16>(rd, L, nblk, starts);
  cp_async_wait_all();  // no copy may be in flight when the thread exits
  if (!ok) {
    atomicMax(p.status, kErrCorrupt);
    return;
  }
  uint16_t *rs = reinterpret_cast<uint16_t *>(rec + 8);
#pragma unroll 1
  for (uint32_t b = 1; b < nblk; ++b) rs[b - 1] = starts[b];
}

// Byte offset of 16-byte unit u of row r in a 128-byte-swizzled 4 KB tile.
__device__ __forceinline__ uint32_t tile_swz(uint32_t r, uint32_t u) { return r * 128u + ((u ^ (r & 7u)) << 4); }

template <bool W16>
__global__ void __launch_bounds__(kDecWarps * 32, 3)
    decode_kernel(DecodeArgs p) {
  __shared__ __align__(16) uint32_t tile[kDecWarps][32 * 32];  // per warp: 32 lane rows of 128 B
  __shared__ __align__(16) uint32_t stage[kDecWarps][kStageWords];  // per warp: the chunk's payload
  __shared__ uint16_t tail_starts[kDecWarps][32];
  const uint32_t lane = lane_id();
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t C = p.num_chunks;
  const uint32_t c = blockIdx.x * kDecWarps + warp;
  if (c >= C) return;
  const uint32_t L = __ldg(reinterpret_cast<const uint16_t *>(p.in) + c);
  const uint32_t raw_len = (uint32_t)umin64(4096u, p.nbytes - (uint64_t)c * 4096u);
  const uint64_t hdr_bytes = 2ull * C;
  if (L == 0 || L > raw_len) return;  // reported by the walk kernel
  uint8_t *dst = p.out + (uint64_t)c * 4096u;
  const uint32_t nblk = (raw_len + 127u) >> 7;
  const Window win{reinterpret_cast<const uint32_t *>(p.in), (p.comp_bytes + 3) / 4};

  // payload offset and this lane's block start bit
  uint64_t off;
  uint32_t s0 = 0, s1 = 0;
  bool ok = true;
  if (raw_len >= (uint32_t)kRecordBytes) {
    off = *reinterpret_cast<const unsigned long long *>(dst);
    if (L < raw_len) {
      const uint16_t *rs = reinterpret_cast<const uint16_t *>(dst + 8);
      s0 = (lane >= 1 && lane < nblk) ? rs[lane - 1] : 0u;
      s1 = (lane + 1 < nblk) ? rs[lane] : 0u;
    }
  } else {  // short final chunk: locate and walk it here
    unsigned long long part = 0;
    for (uint32_t i = lane; i < c; i += 32) part += __ldg(reinterpret_cast<const uint16_t *>(p.in) + i);
    off = hdr_bytes + warp_sum_u64(part);
    if (off + L > p.comp_bytes) return;  // reported by the walk kernel
    if (L < raw_len) {
      if (lane == 0) {
        WindowPeeker rd{WindowReader{win, 8ull * off}};
        ok = walk_chunk<W16>(rd, L, nblk, tail_starts[warp]);
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      if (!ok) {
        if (lane == 0) atomicMax(p.status, kErrCorrupt);
        return;
      }
      __syncwarp();
      s0 = (lane < nblk) ? tail_starts[warp][lane] : 0u;
      s1 = (lane + 1 < nblk) ? tail_starts[warp][lane + 1] : 0u;
    }
  }
  if (off + L > p.comp_bytes) return;  // reported by the walk kernel
  __syncwarp();  // every lane has read the record before any output is written

  if (L == raw_len) {  // raw chunk: the warp copies it (source at any byte offset)
    const uint32_t *w = reinterpret_cast<const uint32_t *>(p.in);
    const uint64_t nw = (p.comp_bytes + 3) / 4;
    const uint32_t sh = (uint32_t)(off & 3) * 8;
    for (uint32_t v = lane; v * 16 < raw_len; v += 32) {
      const uint64_t wi = (off + 16ull * v) >> 2;
      uint32_t w5[5];
#pragma unroll
      for (int k = 0; k < 5; ++k) w5[k] = (wi + k < nw) ? __ldg(w + wi + k) : 0u;
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k] = __funnelshift_r(w5[k], w5[k + 1], sh);
      if (v * 16 + 16 <= raw_len) {
        *reinterpret_cast<uint4 *>(dst + 16ull * v) = make_uint4(o[0], o[1], o[2], o[3]);
      } else {
        for (uint32_t b = 0; v * 16 + b < raw_len; ++b) dst[16ull * v + b] = (uint8_t)(o[b >> 2] >> ((b & 3) * 8));
      }
    }
    return;
  }

  // stage the payload: 16-byte units from a0 = off rounded down to 16
  const uint64_t a0 = off & ~15ull;
  const uint32_t nunits = (uint32_t)((off + L + 15 - a0) >> 4);
  const uint32_t sbase = smem_u32(stage[warp]);
  for (uint32_t u = lane; u < nunits; u += 32) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.in + a0) + u);
    *reinterpret_cast<uint4 *>(&stage[warp][4 * u]) = v;
  }
  __syncwarp();
  const StageBits sb{sbase};
  const uint32_t bit0 = (uint32_t)(off - a0) * 8u;

  uint32_t *tw = tile[warp];
  const uint32_t row = smem_u32(tw) + lane * 128u;
  if (lane < nblk) {
    uint32_t q = bit0 + s0;
    uint32_t o[32];
    ok = decode_block<W16>(sb, q, o, row, lane);
    const uint32_t used = q - bit0 - s0;
    if (lane + 1 < nblk && used != s1 - s0) ok = false;
    if (lane + 1 == nblk && s0 + used > 8u * L) ok = false;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(tw) + tile_swz(lane, u)) =
          make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
  }
  if (!ok) atomicMax(p.status, kErrCorrupt);
  __syncwarp();
  // coalesced write-out of the chunk
#pragma unroll
  for (uint32_t i = 0; i < 8; ++i) {
    const uint32_t v = lane + 32u * i;
    if (16u * v >= raw_len) break;
    const uint4 q = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint8_t *>(tw) + tile_swz(v >> 3, v & 7));
    if (16u * v + 16u <= raw_len) {
      *reinterpret_cast<uint4 *>(dst + 16u * v) = q;
    } else {
      const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
      for (uint32_t b = 0; 16u * v + b < raw_len; ++b) dst[16u * v + b] = (uint8_t)(qq[b >> 2] >> ((b & 3) * 8));
    }
  }
}

template __global__ void walk_kernel<false>(DecodeArgs);
template __global__ void walk_kernel<true>(DecodeArgs);
template __global__ void decode_kernel<false>(DecodeArgs);
template __global__ void decode_kernel<true>(DecodeArgs);

int walk_threads() { return kWalkThreads; }
int decode_threads() { return kDecWarps * 32; }
int decode_chunks_per_cta() { return kDecWarps; }
const void *walk_kernel_ptr(bool w16) {
  return w16 ? reinterpret_cast<const void *>(&walk_kernel<true>)
             : reinterpret_cast<const void *>(&walk_kernel<false>);
}
const void *decode_kernel_ptr(bool w16) {
  return w16 ? reinterpret_cast<const void *>(&decode_kernel<true>)
             : reinterpret_cast<const void *>(&decode_kernel<false>);
}

}  // namespace pz
