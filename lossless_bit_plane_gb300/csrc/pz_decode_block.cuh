// pz_decode_block.cuh — the per-block work of the PlaneZip decoder: one lane
// decodes one 128-byte block of a chunk staged in shared memory, given the
// bit where the block starts. Included by decode.cu; the kernels around it
// (chunk location, walks, staging, write-out) live there.
//
// Paper: "PlaneZip: Lossless Bit-Plane Compression of Training Activations
// Offloaded over PCIe" (arXiv:2610.25033v1), Section III-A "Codec" (each
// block is the inverse of its tagged candidate: ZVC, DBX, BX, ZBX or raw)
// and Section II-B (BPC's Delta-BitPlane-XOR transform).
#pragma once

#include <cstdint>

#include "pz_device.cuh"
#include "pz_format.cuh"

namespace pz {

// A staged payload: 16-byte units from the payload's first byte rounded down
// to 16 (at most 257 units), plus slack words for three-word peeks.
constexpr uint32_t kStageWords = (4096 + 16) / 4 + 4;

// Lane-private 32-word row (the lane's 128-byte row of a 128-aligned tile).
// Word access XOR-swizzled by lane (conflict-free across lanes): the row
// starts on a 128-byte boundary, so the swizzled word offset can be XORed
// into the row's address, and the lane-dependent part is common to every
// access of the lane.
__device__ __forceinline__ uint32_t prow(uint32_t row, uint32_t lane, uint32_t word) {  // word, lane < 32
  return (row ^ (lane << 2)) ^ (word << 2);
}
__device__ __forceinline__ uint32_t prow_half(uint32_t row, uint32_t lane, uint32_t h) {  // h < 64
  return (row ^ (lane << 2)) ^ (h << 1);
}
// A chunk's payload staged in shared memory: word k holds stream bytes
// [a0 + 4k, a0 + 4k + 4), where a0 is the payload's first byte rounded down
// to 16; bit q counts from a0.
struct StageBits {
  uint32_t base;  // shared address of word 0
  // word address of bit q, clamped so that a malformed stream cannot read
  // outside the buffer (valid streams never reach the clamp)
  __device__ __forceinline__ uint32_t addr(uint32_t q) const { return base + (min(q >> 5, kStageWords - 3u) << 2); }
  __device__ __forceinline__ uint32_t peek32(uint32_t q) const {
    const uint32_t a = addr(q);
    return __funnelshift_r(lds32(a), lds32(a + 4), q & 31u);
  }
};

// Decode the block whose tag is at stage bit q into o[32] (the block's 32
// words in memory order); q advances past the block. Plane codes are parsed
// top plane first by a per-plane loop: a verbatim code takes a short branch
// of its own (the low planes of activations are verbatim in nearly every
// block, so whole warps skip the classification there), the other codes pick
// their values by selects rather than branches. Each plane is X_i,
// rebuilt to the pre-XOR plane P_i = X_i ^ P_{i+1} and stored in the lane's
// row (FP32 plane i < 32 in row i; BF16 plane i < 16 in rows i and 16+i; a
// DBX row's bit j is delta j+1). One 32x32 bit transpose then turns rows
// into symbols (or deltas, summed afterwards). Returns false on a malformed
// code.
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
    // the non-zero symbols follow the mask back to back, w bits each: the
    // symbol k is read straight from its rank's position (no serial walk)
    if (W16) {
      const uint32_t mlo = sb.peek32(q), mhi = sb.peek32(q + 32);
      q += 64;
      const uint32_t clo = __popc(mlo);
#pragma unroll
      for (int r = 0; r < 32; ++r) {  // raw word r: symbols 2r and 2r + 1
        const uint32_t m = (r < 16) ? mlo : mhi;
        const int k = (2 * r) & 31;
        const uint32_t r0 = ((r < 16) ? 0u : clo) + __popc(m & ((1u << k) - 1u));
        const uint32_t b0 = (m >> k) & 1u, b1 = (m >> (k + 1)) & 1u;
        const uint32_t v0 = b0 ? (sb.peek32(q + 16u * r0) & 0xFFFFu) : 0u;
        const uint32_t v1 = b1 ? (sb.peek32(q + 16u * (r0 + b0)) & 0xFFFFu) : 0u;
        o[r] = v0 | (v1 << 16);
      }
      q += 16u * (clo + __popc(mhi));
    } else {
      const uint32_t mask = sb.peek32(q);
      q += 32;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const uint32_t rk = __popc(mask & ((1u << k) - 1u));
        o[k] = ((mask >> k) & 1u) ? sb.peek32(q + 32u * rk) : 0u;
      }
      q += 32u * __popc(mask);
    }
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
  const uint32_t p = ceil_log2_u32((uint32_t)W);
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
        // a code spans at most 33 bits (1 + W, W <= 32), so the two words
        // under q hold it: bit q + 32 is bit sh of w1
        const uint32_t a = sb.addr(q), sh = q & 31u;
        const uint32_t w0 = lds32(a), w1 = lds32(a + 4);
        const uint32_t lo = __funnelshift_r(w0, w1, sh);
        if (lo & 1u) {  // verbatim: 1 + the plane
          X = __funnelshift_r(lo, w1 >> sh, 1) & full;
          q += 1u + (uint32_t)W;
        } else {
          const uint32_t tz = (uint32_t)__ffs(lo | 16u) - 1u;  // 1..4
          const uint32_t qf = (lo >> 5) & pmask;
          const bool hi4 = (lo & 16u) != 0;
          const uint32_t xp = (hi4 ? 1u : 3u) << qf;
          const uint32_t x5 = hi4 ? Pup : full;
          X = (tz == 3u) ? xp : (tz == 4u) ? x5 : 0u;
          q += (tz == 4u) ? 5u : ((lens >> (7u * tz)) & 127u);
          if (tz == 1u) run = 1 + (int)((lo >> 2) & ((1u << K) - 1u));
          bad |= (tz == 3u) && (qf + (hi4 ? 0u : 1u) >= (uint32_t)W);
        }
      }
      const uint32_t Pi = X ^ Pup;  // Pup is 0 above the top plane
      Pup = Pi;
      if (i < 32) sts32(row + ((((uint32_t)i ^ lane) & 31u) << 2), Pi);  // prow(row, lane, i), added (faster here)
    }
  } else {
    const uint64_t full = (W >= 64) ? ~0ull : ((1ull << W) - 1);
    const uint32_t full_lo = (uint32_t)full, full_hi = (uint32_t)(full >> 32);
    uint64_t Pup = 0;
#pragma unroll 1
    for (int i = top; i >= 0; --i) {
      uint64_t X = 0;
      if (run > 0) {
        --run;
      } else {
        const uint32_t a = sb.addr(q), sh = q & 31u;
        const uint32_t w0 = lds32(a), w1 = lds32(a + 4), w2 = lds32(a + 8);
        const uint32_t lo = __funnelshift_r(w0, w1, sh), hi = __funnelshift_r(w1, w2, sh);
        if (lo & 1u) {  // verbatim: 1 + the plane (bits 1..64 after the flag)
          const uint32_t xl = __funnelshift_r(lo, hi, 1) & full_lo, xh = __funnelshift_r(hi, w2 >> sh, 1) & full_hi;
          X = (uint64_t)xl | ((uint64_t)xh << 32);
          q += 1u + (uint32_t)W;
        } else {
          const uint32_t tz = (uint32_t)__ffs(lo | 16u) - 1u;  // 1..4
          const uint32_t qf = (lo >> 5) & pmask;
          const bool hi4 = (lo & 16u) != 0;
          const uint64_t xp = (hi4 ? 1ull : 3ull) << qf;
          const uint64_t x5 = hi4 ? Pup : full;
          X = (tz == 3u) ? xp : (tz == 4u) ? x5 : 0ull;
          q += (tz == 4u) ? 5u : ((lens >> (7u * tz)) & 127u);
          if (tz == 1u) run = 1 + (int)((lo >> 2) & ((1u << K) - 1u));
          bad |= (tz == 3u) && (qf + (hi4 ? 0u : 1u) >= (uint32_t)W);
        }
      }
      const uint64_t Pi = X ^ Pup;  // Pup is 0 above the top plane
      Pup = Pi;
      if (i < 16) {
        sts32(prow(row, lane, (uint32_t)i), (uint32_t)Pi);
        sts32(prow(row, lane, (uint32_t)i + 16), (uint32_t)(Pi >> 32));
      }
    }
  }
  const bool ok = !bad;
#pragma unroll
  for (int j = 0; j < 32; ++j) o[j] = lds32(prow(row, lane, j));
  transpose32(o);  // FP32: o[j] = symbol j (or delta j+1); BF16: split words
  if (!W16) {
    if (dbx) {  // s_0 = base, s_j = s_{j-1} + delta j
      uint32_t prev = basesym;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t d = o[j];
        o[j] = prev;
        prev += d;
      }
    } else if (tag == kTagZBX && (mlo & (mlo + 1u)) != 0u) {
      // (survivors that are the block's first W symbols -- a causal mask's
      // rows -- are in place already, and the planes' bits from W on are 0)
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < W) sts32(prow(row, lane, j), o[j]);
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const uint32_t rank = __popc(mlo & ((1u << k) - 1u));
        o[k] = ((mlo >> k) & 1u) ? lds32(prow(row, lane, rank)) : 0u;
      }
    }
    return ok;
  }
  // BF16: o holds split words (word j = symbol j | symbol j+32 << 16); for
  // DBX, word j holds delta j+1 low and delta j+33 high
  if (dbx) {
    uint32_t prev = basesym;  // s_0
#pragma unroll
    for (int j = 0; j < 32; ++j) {  // s_j, then s_{j+1} = s_j + delta j+1
      const uint32_t d = o[j] & 0xFFFFu;
      o[j] = (o[j] & 0xFFFF0000u) | prev;
      prev = (prev + d) & 0xFFFFu;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {  // s_{j+32}, then s_{j+33} = s_{j+32} + delta j+33
      const uint32_t d = o[j] >> 16;
      o[j] = (o[j] & 0xFFFFu) | (prev << 16);
      prev = (prev + d) & 0xFFFFu;
    }
  } else if (tag == kTagZBX && !((mhi == 0u) ? (mlo & (mlo + 1u)) == 0u : (mlo == ~0u && (mhi & (mhi + 1u)) == 0u))) {
    // (survivors that are the block's first W symbols are in place already,
    // zeros after them: the split words become raw words below, as for BX)
    // survivors t_0..t_{W-1}: t_j in o[j] low, t_{j+32} in o[j] high. They
    // go to the lane's row as half-words in index order (word m = t_2m |
    // t_2m+1 << 16, the same pairing as a raw word), and each raw word of
    // the block is gathered from there by its two symbols' ranks.
#pragma unroll
    for (int m = 0; m < 32; ++m) sts32(prow(row, lane, (uint32_t)m), raw_word_from_split(o, m));
    const uint32_t clo = __popc(mlo);
#pragma unroll
    for (int r = 0; r < 32; ++r) {  // symbols 2r and 2r + 1
      const uint32_t m = (r < 16) ? mlo : mhi;
      const int k = (2 * r) & 31;
      const uint32_t r0 = ((r < 16) ? 0u : clo) + __popc(m & ((1u << k) - 1u));
      const uint32_t b0 = (m >> k) & 1u, b1 = (m >> (k + 1)) & 1u;
      const uint32_t v0 = b0 ? lds16(prow_half(row, lane, r0)) : 0u;
      const uint32_t v1 = b1 ? lds16(prow_half(row, lane, r0 + b0)) : 0u;
      o[r] = v0 | (v1 << 16);
    }
    return ok;
  }
  uint32_t sp[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) sp[j] = o[j];
#pragma unroll
  for (int r = 0; r < 32; ++r) o[r] = raw_word_from_split(sp, r);
  return ok;
}


}  // namespace pz
