// decode.cu — PlaneZip block decoder for sm_103a.
//
// Paper: "PlaneZip: Lossless Bit-Plane Compression of Training Activations
// Offloaded over PCIe" (arXiv:2610.25033v1), Section III-A "Stream format":
// the decompressor locates every chunk with a prefix sum over the 16-bit
// chunk sizes and decodes chunks in parallel; each block is the inverse of
// its tagged candidate (Section III-A "Codec").
//
// GPU design (up to three launches per call):
//  - The format stores no per-block offsets: block b of a chunk starts where
//    block b-1 ends, so a chunk's blocks must be measured in order before
//    they can be decoded in parallel. A walk finds every block's start bit;
//    a decode kernel then decodes the blocks, LANE = BLOCK.
//  - Chunk offsets: a small kernel sums the 16-bit sizes of each group of
//    2048 chunks; a walk warp adds the group sums before its group and the
//    sizes of its own group's earlier chunks.
//  - Walk, above 6144 chunks: LANE = CHUNK, one warp per CTA. Each lane
//    measures its chunk's codes through a window in shared memory, refilled
//    warp-wide by bulk copies; a step takes a block header and up to two
//    non-verbatim codes and skips a run of verbatim codes by testing their
//    flag bits. Up to 6144 chunks: WARP = CHUNK, the 32 lanes testing 32
//    flags at once (shorter chains for small inputs). Where every chunk has
//    a resident warp, that warp also decodes its chunk in the same launch.
//  - Records: a chunk's payload offset and its blocks' start bits go into
//    the first 72 bytes of the chunk's own output region; the decode warp
//    reads them before it overwrites those bytes.
//  - Decode: WARP = CHUNK, LANE = BLOCK. The payload is staged in shared
//    memory; each lane rebuilds its planes top-down (pre-XOR plane P_i =
//    X_i ^ P_{i+1}) into a lane-private row, one 32x32 bit transpose turns
//    them into symbols, then the delta is undone (prefix sum) or the
//    survivors are scattered back by rank (ZBX); ZVC symbols are read by
//    rank. Raw chunks are copied by the whole warp with 16-byte stores.
//  - Every field is validated; a malformed chunk sets PZ_ERR_CORRUPT in the
//    status word; no write leaves the chunk's output range and no read
//    leaves the 16-byte granules of the input.
#include <cuda_runtime.h>

#include <cstdint>

#include "pz_decode_block.cuh"
#include "pz_device.cuh"
#include "pz_format.cuh"
#include "pz_kernels.h"

namespace pz {

constexpr int kDecWarps = 8;
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

struct WindowPeeker {  // adapts WindowReader to the ensure / peek_resident interface
  WindowReader r;
  __device__ __forceinline__ void ensure(uint32_t) const {}
  __device__ __forceinline__ uint32_t peek_resident(uint32_t pos) const { return r.peek(pos); }
  __device__ __forceinline__ uint32_t bit_resident(uint32_t pos) const { return r.peek(pos) & 1u; }
  __device__ __forceinline__ void window_resident(uint32_t pos, uint32_t &v0, uint32_t &v1, uint32_t &v2) const {
    v0 = r.peek(pos);
    v1 = r.peek(pos + 32u);
    v2 = r.peek(pos + 64u);
  }
  __device__ __forceinline__ uint32_t peek(uint32_t pos) const { return r.peek(pos); }
};

// Walk one chunk by one thread: record each block's start bit (relative to
// the chunk) through put_start(b, pos) and check that the chunk is exactly
// ceil(bits/8) bytes with zero padding. The decode kernel uses it for a final
// chunk too short (under 72 bytes) to hold a walk record.
//
// An iteration either reads a
// block header (tag; the mask of ZVC / ZBX; the base of DBX) and skips what
// needs no parsing, or advances over plane codes: it tests the flag bits of
// the next eight codes under the assumption that they are verbatim (1 + W
// bits each) and skips the m leading verbatim ones, or, when the first code
// is not verbatim, classifies it by its leading zero bits (stream order,
// capped at 4): 01 run (2+K bits, 2+field planes), 001 single zero (3),
// 0001x position code (5+p), 0000x all-ones / pre-XOR-zero (5).
template <bool W16, typename Reader, typename Sink>
__device__ __forceinline__ bool walk_chunk(Reader &rd, uint32_t L, uint32_t nblk, Sink put_start) {
  constexpr uint32_t w = W16 ? 16u : 32u;   // bits per symbol = BX planes
  constexpr uint32_t N = W16 ? 64u : 32u;   // symbols per block
  constexpr uint32_t K = W16 ? 4u : 5u;     // run field
  constexpr uint32_t kSkip = 8;
  const uint32_t cap = 8u * L;
  uint32_t pos = 0, b = 0;
  int i = -1, top = 0;          // plane still to be walked (-1: next is a header)
  uint32_t S = 2u, p = 0u;      // verbatim code length 1 + W, position field
  bool ok = true;
#pragma unroll 1
  while (ok && (i >= 0 || b < nblk)) {
    const bool hdr = i < 0;
    rd.ensure(pos + (kSkip - 1) * S + 35u);
    uint32_t f = 0;
#pragma unroll
    for (uint32_t k = 1; k < kSkip; ++k) f |= rd.bit_resident(pos + k * S) << k;
    uint32_t v0, v1, v2;
    rd.window_resident(pos, v0, v1, v2);
    f |= v0 & 1u;
    // header
    const uint32_t tag = v0 & 7u;
    const uint32_t n = __popc(__funnelshift_r(v0, v1, 3)) + (W16 ? __popc(__funnelshift_r(v1, v2, 3)) : 0u);
    const bool masked = (tag == kTagZVC) || (tag == kTagZBX);
    uint32_t hadv = 3u;
    hadv += masked ? (W16 ? 64u : 32u) : 0u;
    hadv += (tag == kTagZVC) ? n * w : 0u;
    hadv += (tag == kTagDBX) ? w : 0u;
    hadv += (tag == kTagRAW) ? 1024u : 0u;
    const bool planes = (tag == kTagBX) || (tag == kTagDBX) || (tag == kTagZBX && n != 0);
    const int htop = (tag == kTagDBX) ? (int)w : (int)w - 1;
    const uint32_t hW = (tag == kTagDBX) ? N - 1u : (tag == kTagZBX) ? n : N;
    // plane codes
    int m = __ffs(~f) - 1;  // leading verbatim codes, 0..kSkip
    m = min(m, i + 1);
    const uint32_t tz = (uint32_t)__ffs(v0 | 16u) - 1u;  // 1..4 when not verbatim
    const uint32_t len = (tz == 1u) ? 2u + K : (tz == 2u) ? 3u : (tz == 3u) ? 5u + p : 5u;
    const int run = (tz == 1u) ? 2 + (int)((v0 >> 2) & ((1u << K) - 1u)) : 1;
    const bool pbad = (m == 0) && ((run > i + 1) || (tz == 4u && (v0 & 16u) && i == top));
    if (hdr) {
      put_start(b, pos);
      ok = (tag <= kTagRAW) && pos <= cap;
      pos += hadv;
      i = planes ? htop : -1;
      top = htop;
      S = 1u + hW;
      p = ceil_log2_u32(hW);
      ++b;
    } else {
      ok = !pbad;
      pos += (m > 0) ? (uint32_t)m * S : len;
      i -= (m > 0) ? m : run;
    }
  }
  if (!ok || pos > cap) return false;
  if (cap - pos >= 8) return false;
  if (cap > pos && (rd.peek(pos) & ((1u << (cap - pos)) - 1u))) return false;
  return true;
}

// ---------------------------------------------------------------- kernels
//
// Up to three launches. The walk kernel runs one warp per 32 consecutive
// chunks, lane = chunk: it finds each chunk's payload offset (2C plus the
// sum of all earlier sizes) and, for a coded chunk, every block's start
// bit, and leaves them in the first bytes of that chunk's own output region:
// the offset (8 bytes) then the start bits of blocks 1..n-1 (2 bytes each).
// The decode kernel runs one warp per chunk, lane = block: each lane reads
// its start, the warp synchronises, and only then are those bytes
// overwritten with decoded data. A final chunk too short to hold that record
// (under 72 bytes) is located and walked by its decode warp instead.
//
// For the offsets, a first small kernel sums the sizes of each group of 2048
// chunks (all groups but the last) and leaves the sum at byte 72 of the
// group's first chunk region (a full 4 KB chunk, past its record); a walk
// warp then adds at most one group sum per earlier group and the sizes of
// at most 2047 chunks of its own group.

constexpr uint32_t kRecordBytes = 72;  // 8-byte offset + 31 x 2-byte start bits + padding
constexpr uint32_t kGroupChunks = 2048;
constexpr uint32_t kGroupSumAt = 72;   // byte of the group's first chunk region
constexpr uint32_t kMbarPolls = 1u << 24;

__device__ __forceinline__ unsigned long long sum8_sizes(const uint4 v) {
  return (unsigned long long)((v.x & 0xFFFFu) + (v.x >> 16) + (v.y & 0xFFFFu) + (v.y >> 16) + (v.z & 0xFFFFu) +
                              (v.z >> 16) + (v.w & 0xFFFFu) + (v.w >> 16));
}

__global__ void __launch_bounds__(256) size_sum_kernel(DecodeArgs p) {
  __shared__ unsigned long long red[8];
  griddep_launch_dependents();  // the walk's blocks may be scheduled now; they wait for this kernel's end
  const uint32_t g = blockIdx.x;  // every chunk of the group exists
  const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.in) + (uint64_t)g * (kGroupChunks / 8) + threadIdx.x);
  const unsigned long long s = warp_sum_u64(sum8_sizes(v));
  if (lane_id() == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t = 0;
    for (int w = 0; w < 8; ++w) t += red[w];
    *reinterpret_cast<unsigned long long *>(p.out + (uint64_t)g * kGroupChunks * 4096u + kGroupSumAt) = t;
  }
}

// Sum of the sizes of chunks [0, first) (first a multiple of 32), by a warp.
__device__ __forceinline__ unsigned long long sizes_before(const DecodeArgs &p, uint32_t first, uint32_t lane) {
  const uint32_t g0 = first / kGroupChunks;
  unsigned long long part = 0;
  for (uint32_t g = lane; g < g0; g += 32)
    part += *reinterpret_cast<const unsigned long long *>(p.out + (uint64_t)g * kGroupChunks * 4096u + kGroupSumAt);
  const uint4 *h4 = reinterpret_cast<const uint4 *>(p.in);
  for (uint32_t i = g0 * (kGroupChunks / 8) + lane; i < first / 8; i += 32) part += sum8_sizes(__ldg(h4 + i));
  return warp_sum_u64(part);
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(mbar)
               : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(mbar) : "memory");
}

// Walk kernel shape: warps of 32 chunks (lane = chunk); each lane reads its
// chunk through a window of kWinUnits 16-byte units in shared memory. One
// warp per CTA spreads the warps evenly over the SMs (6 or 7 per SM for a
// 128 MiB input rather than 3 or 4 CTAs of two), and the kernel lasts as long
// as its slowest warp.
constexpr uint32_t kWalkWarps = 1;
constexpr uint32_t kWinUnits = 48;
constexpr uint32_t kWinWords = kWinUnits * 4;
// windows are laid out kWinStride words apart (4 words more than a window,
// a 16-byte multiple for the bulk copies) so that lanes reading the same
// window offset -- as they all do right after a refill -- hit different banks
constexpr uint32_t kWinStride = kWinWords + 4;
constexpr uint32_t kWalkSmem = kWalkWarps * 32 * kWinStride * 4 + kWalkWarps * 8;

// The warp's walk: lane = chunk. It is one loop that every lane runs until
// the last lane is done (lanes that are done, or have nothing to walk, sit
// out both steps). An iteration takes up to two steps per lane:
//  - a header step, when the lane stands at a block: the tag, the mask of
//    ZVC / ZBX or the base of DBX; what needs no parsing (ZVC symbols, a
//    raw block) is skipped, and a block with plane codes goes on to
//  - a plane step in the same iteration: up to two codes that are not
//    verbatim, each classified by its leading zero bits (stream order,
//    capped at 4): 01 run (2+K bits, 2+field planes), 001 single zero (3),
//    0001x position code (5+p), 0000x all-ones / pre-XOR-zero (5); then the
//    flag bits of the next kSkip codes are tested under the assumption that
//    they are verbatim (1 + W bits each) and the m leading verbatim ones are
//    skipped. The header fields and the first two codes are read from the
//    same five words loaded at the position.
// A lane's window holds the units from the one under its position on; when
// any lane's next iteration could read past its window, every walking lane
// re-bases its window at its position with one bulk copy, and the warp waits
// once for all of them. Records: the start bit of block b >= 1 goes to
// rs[b - 1]. Returns false where the chunk is malformed.
template <bool W16>
__device__ __forceinline__ bool walk_warp(const DecodeArgs &p, bool walk, uint64_t off, uint32_t L, uint32_t nblk,
                                          uint16_t *rs, const uint32_t *win, uint32_t mb, bool &timed_out) {
  constexpr uint32_t w = W16 ? 16u : 32u;   // bits per symbol = BX planes
  constexpr uint32_t N = W16 ? 64u : 32u;   // symbols per block
  constexpr uint32_t K = W16 ? 4u : 5u;     // run field
  // flags tested per plane step. FP32: 26, so that a block's trailing run of
  // verbatim planes (the mantissa's, after its last short codes) takes one
  // step; with 14 to 25 flags it takes two, and more than 26 add loads that
  // no run repays. BF16: 10 (12 was no faster), fewer mean more iterations.
  constexpr uint32_t kSkip = W16 ? 10u : 26u;
  // bits an iteration may read past its position: five words at the
  // position, or a plane block's header fields (tag and mask, or tag and
  // base), two codes of at most 11 bits each and kSkip flags N + 1 apart
  constexpr uint32_t kPlaneReach = 3u + N + 22u + (kSkip - 1u) * (N + 1u) + 64u;
  constexpr uint32_t kAhead = (kPlaneReach > 160u ? kPlaneReach : 160u) + 32u;
  const uint32_t lane = lane_id();
  const uint64_t a0 = off & ~15ull;
  const uint8_t *g0 = p.in + a0;
  const uint32_t bit0 = (uint32_t)(off - a0) * 8u;
  const uint32_t nunits = (uint32_t)((off + L + 15 - a0) >> 4);
  const uint32_t cap = 8u * L;
  const uint32_t winaddr = smem_u32(win);
  uint32_t lim = 0;    // absolute bit at which the window ends
  uint32_t wbase = 0;  // absolute bit where the window starts
  uint32_t parity = 0;
  uint32_t pos = 0, b = 0, S = 2u, pf = 0u;
  int i = -1, top = 0;
  bool ok = true;
  bool run = walk;
#pragma unroll 1
  while (true) {
    const uint32_t qa = bit0 + min(pos, cap);
    const bool need = run && qa + kAhead >= lim;
    if (!__any_sync(0xFFFFFFFFu, run)) break;
    if (__any_sync(0xFFFFFFFFu, need)) {
      fence_proxy_async_smem();  // this lane's reads of its window before the bulk write
      if (run) {
        const uint32_t u = qa >> 7;  // <= nunits
        const uint32_t bytes = min(kWinUnits, nunits - u) * 16u;
        if (bytes) {
          mbar_expect_tx(mb, bytes);
          bulk_load(winaddr, g0 + 16ull * u, bytes, mb);
        }
        wbase = u * 128u;
        lim = wbase + kWinUnits * 128u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(mb);
      const bool got = mbar_wait(mb, parity, kMbarPolls);
      if (!__all_sync(0xFFFFFFFFu, got)) {
        mbar_wait(mb, parity, kMbarPolls);  // leave no copy in flight
        timed_out = true;
        return false;
      }
      parity ^= 1u;
    }
    // bit in the window; the clamp only binds for lanes that are done (a
    // walking lane re-based its window above), and keeps every read inside
    const uint32_t ql = min(qa - wbase, kWinUnits * 128u - kAhead);
    // one set of loads serves both steps: the header's fields and the first
    // two plane codes after them lie within the 128 bits at the position
    const uint32_t wi = ql >> 5, sh = ql & 31u;
    const uint32_t x0 = win[wi], x1 = win[wi + 1], x2 = win[wi + 2], x3 = win[wi + 3], x4 = win[wi + 4];
    const uint32_t v0 = __funnelshift_r(x0, x1, sh), v1 = __funnelshift_r(x1, x2, sh),
                   v2 = __funnelshift_r(x2, x3, sh), v3 = __funnelshift_r(x3, x4, sh);
    // the 32 bits at ql + o, o < 96
    auto bits_at = [&](uint32_t o) -> uint32_t {
      const uint32_t wq = o >> 5;
      const uint32_t a = (wq == 0u) ? v0 : (wq == 1u) ? v1 : v2, c = (wq == 0u) ? v1 : (wq == 1u) ? v2 : v3;
      return __funnelshift_r(a, c, o & 31u);
    };
    uint32_t offb = 0;  // bits from ql to the first plane code of this iteration
    if (run && i < 0) {  // header step
      const uint32_t tag = v0 & 7u;
      uint32_t n = __popc(__funnelshift_r(v0, v1, 3));
      if (W16) n += __popc(__funnelshift_r(v1, v2, 3));
      const bool masked = (tag == kTagZVC) || (tag == kTagZBX);
      uint32_t hadv = 3u;
      hadv += masked ? N : 0u;
      hadv += (tag == kTagZVC) ? n * w : 0u;
      hadv += (tag == kTagDBX) ? w : 0u;
      hadv += (tag == kTagRAW) ? 1024u : 0u;
      const bool planes = (tag == kTagBX) || (tag == kTagDBX) || (tag == kTagZBX && n != 0);
      const uint32_t hW = (tag == kTagDBX) ? N - 1u : (tag == kTagZBX) ? n : N;
      if (b > 0) rs[b - 1] = (uint16_t)pos;
      ok = (tag <= kTagRAW) && pos <= cap;
      pos += hadv;
      offb = hadv;  // 3, 3 + w or 3 + N for a block with plane codes
      top = (tag == kTagDBX) ? (int)w : (int)w - 1;
      i = (ok && planes) ? top : -1;
      S = 1u + hW;
      pf = ceil_log2_u32(hW);
      ++b;
    }
    if (run && i >= 0) {  // plane step
      // up to two codes that are not verbatim, each classified by its leading
      // zeros; the second is parsed only after a first and while planes remain
      const uint32_t c1 = bits_at(offb);
      const bool nv1 = (c1 & 1u) == 0u;
      const uint32_t tz1 = (uint32_t)__ffs(c1 | 16u) - 1u;  // 1..4 when not verbatim
      const uint32_t len1 = (tz1 == 1u) ? 2u + K : (tz1 == 2u) ? 3u : (tz1 == 3u) ? 5u + pf : 5u;
      const int rl1 = (tz1 == 1u) ? 2 + (int)((c1 >> 2) & ((1u << K) - 1u)) : 1;
      bool bad = nv1 && ((rl1 > i + 1) || (tz1 == 4u && (c1 & 16u) && i == top));
      const uint32_t o2 = offb + (nv1 ? len1 : 0u);
      i -= nv1 ? rl1 : 0;
      const uint32_t c2 = bits_at(o2);
      const bool nv2 = nv1 && (c2 & 1u) == 0u && i >= 0;  // below the top plane: no pre-XOR-zero check
      const uint32_t tz2 = (uint32_t)__ffs(c2 | 16u) - 1u;
      const uint32_t len2 = (tz2 == 1u) ? 2u + K : (tz2 == 2u) ? 3u : (tz2 == 3u) ? 5u + pf : 5u;
      const int rl2 = (tz2 == 1u) ? 2 + (int)((c2 >> 2) & ((1u << K) - 1u)) : 1;
      bad = bad || (nv2 && rl2 > i + 1);
      const uint32_t o3 = o2 + (nv2 ? len2 : 0u);
      i -= nv2 ? rl2 : 0;
      ok = !bad;
      // flag k: bit t_k of the window, rotated to position k (the rotations
      // are independent, and an OR tree joins them)
      const uint32_t base = ql + o3;
      uint32_t y[kSkip];
#pragma unroll
      for (uint32_t k = 0; k < kSkip; ++k) {
        const uint32_t t = base + k * S;
        y[k] = __funnelshift_r(win[t >> 5], win[t >> 5], t - k) & (1u << k);
      }
      uint32_t f = 0;
#pragma unroll
      for (uint32_t k = 0; k < kSkip; k += 2) f |= y[k] | y[k + 1];
      const int m = min(__ffs(~f) - 1, i + 1);  // leading verbatim codes, 0..kSkip
      pos += (o3 - offb) + (uint32_t)max(m, 0) * S;
      i -= max(m, 0);
    }
    run = run && ok && (i >= 0 || b < nblk);
  }
  if (!walk) return true;
  if (!ok || pos > cap || cap - pos >= 8) return false;
  if (cap > pos) {  // the padding bits must be zero
    const Window gw{reinterpret_cast<const uint32_t *>(p.in), (p.comp_bytes + 3) / 4};
    if (gw.peek32(8ull * off + pos) & ((1u << (cap - pos)) - 1u)) return false;
  }
  return true;
}

template <bool W16>
__global__ void __launch_bounds__(kWalkWarps * 32)
    walk_kernel(DecodeArgs p) {
  extern __shared__ __align__(128) uint8_t walk_smem[];
  griddep_launch_dependents();  // the decode's blocks may be scheduled now
  griddep_wait();               // the group sums are complete
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t *win = reinterpret_cast<const uint32_t *>(walk_smem) + (warp * 32u + lane) * kWinStride;
  const uint32_t mb = smem_u32(walk_smem + kWalkWarps * 32 * kWinStride * 4) + warp * 8u;
  const uint32_t C = p.num_chunks;
  const uint32_t first = (blockIdx.x * kWalkWarps + warp) * 32u;
  if (first >= C) return;
  const uint32_t c = first + lane;
  const bool valid = c < C;
  const unsigned long long before = sizes_before(p, first, lane);
  const uint32_t L = valid ? __ldg(reinterpret_cast<const uint16_t *>(p.in) + c) : 0u;
  uint32_t incl = L;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= (uint32_t)o) incl += v;
  }
  const uint64_t off = 2ull * C + before + (incl - L);
  const uint32_t raw_len = valid ? (uint32_t)umin64(4096u, p.nbytes - (uint64_t)c * 4096u) : 0u;
  const bool bad = valid && (L == 0 || L > raw_len || off + L > p.comp_bytes);
  if (bad) atomicMax(p.status, kErrCorrupt);
  uint8_t *rec = p.out + (uint64_t)c * 4096u;
  const bool has_rec = valid && !bad && raw_len >= kRecordBytes;
  if (has_rec) *reinterpret_cast<unsigned long long *>(rec) = off;
  const bool walk = has_rec && L < raw_len;  // a raw chunk needs only its offset
  if (!__any_sync(0xFFFFFFFFu, walk)) return;
  if (lane == 0) {
    mbar_init(mb, 1);
    fence_mbar_init();
  }
  __syncwarp();
  bool timed_out = false;
  const bool ok = walk_warp<W16>(p, walk, off, L, (raw_len + 127u) >> 7, reinterpret_cast<uint16_t *>(rec + 8), win,
                                 mb, timed_out);
  if (timed_out) {
    if (lane == 0) atomicMax(p.status, kErrTimeout);
  } else if (!ok) {
    atomicMax(p.status, kErrCorrupt);
  }
}

// ------------------------------------------------ cooperative walk (small)
//
// For inputs of up to kCoopMaxChunks chunks the walk kernel above is bound
// by one thread's chain through a whole chunk, whatever the input's size.
// Here a warp walks one chunk instead: the chunk's payload is staged in
// shared memory by one bulk copy, the warp steps through the blocks with
// every value warp-uniform. In a step lane k loads the 64 bits at the k-th
// code ahead under the assumption that the codes are verbatim (1 + W bits
// each), so one ballot of their flag bits skips up to 32 verbatim planes;
// the lane that stands at the first code that is not verbatim hands its 64
// bits to the warp, which parses up to four such codes in a row from them in
// the same step.
// It writes the same record as the walk kernel (offset and block starts at
// the chunk's output region).

constexpr uint32_t kCoopWarps = 8;
constexpr uint32_t kCoopStageBytes = kStageWords * 4;  // a payload from its 16-byte unit, plus slack
constexpr uint32_t kCoopStageWords = kCoopStageBytes / 4;
constexpr uint32_t kCoopSmem = kCoopWarps * kCoopStageBytes + kCoopWarps * 8;
constexpr uint32_t kCoopMaxChunks = 6144;

// Sum of the sizes of chunks [0, c) for any c, by a warp (group sums of
// whole groups, then 16-byte units of headers, then the last few headers).
__device__ __forceinline__ unsigned long long sizes_before_chunk(const DecodeArgs &p, uint32_t c, uint32_t lane) {
  const uint32_t g0 = c / kGroupChunks;
  unsigned long long part = 0;
  for (uint32_t g = lane; g < g0; g += 32)
    part += *reinterpret_cast<const unsigned long long *>(p.out + (uint64_t)g * kGroupChunks * 4096u + kGroupSumAt);
  const uint4 *h4 = reinterpret_cast<const uint4 *>(p.in);
  const uint32_t u1 = c / 8;
  for (uint32_t i = g0 * (kGroupChunks / 8) + lane; i < u1; i += 32) part += sum8_sizes(__ldg(h4 + i));
  if (lane < (c & 7u)) part += __ldg(reinterpret_cast<const uint16_t *>(p.in) + 8u * u1 + lane);
  return warp_sum_u64(part);
}

// The warp's walk of one staged chunk (WARP = CHUNK, every value
// warp-uniform): stage word k holds payload bytes from 4k on, the payload
// starting at stage bit bit0; rec(b, pos) is called with the start bit of
// each block b >= 1 (relative to bit0). Returns false where the chunk is
// malformed.
template <bool W16, typename Rec>
__device__ __forceinline__ bool coop_walk(const uint32_t *stage, uint32_t bit0, uint32_t L, uint32_t nblk,
                                          uint32_t lane, Rec rec) {
  constexpr uint32_t w = W16 ? 16u : 32u;   // bits per symbol = BX planes
  constexpr uint32_t N = W16 ? 64u : 32u;   // symbols per block
  constexpr uint32_t K = W16 ? 4u : 5u;     // run field
  // word indices are clamped to the stage: a malformed stream cannot read
  // outside it (valid streams never reach the clamp)
  auto word = [&](uint32_t i) { return stage[min(i, kCoopStageWords - 1u)]; };
  auto peek = [&](uint32_t pos) {
    const uint32_t q = bit0 + pos, i = q >> 5;
    return __funnelshift_r(word(i), word(i + 1), q & 31u);
  };
  const uint32_t cap = 8u * L;
  uint32_t pos = 0;
  bool ok = true;
#pragma unroll 1
  for (uint32_t b = 0; b < nblk && ok; ++b) {
    if (b) rec(b, pos);
    const uint32_t tag = peek(pos) & 7u;
    if (tag > kTagRAW) {
      ok = false;
      break;
    }
    const uint32_t n = __popc(peek(pos + 3u)) + (W16 ? __popc(peek(pos + 35u)) : 0u);
    const bool masked = (tag == kTagZVC) || (tag == kTagZBX);
    pos += 3u + (masked ? (W16 ? 64u : 32u) : 0u) + ((tag == kTagZVC) ? n * w : 0u) + ((tag == kTagDBX) ? w : 0u) +
           ((tag == kTagRAW) ? 1024u : 0u);
    const bool planes = (tag == kTagBX) || (tag == kTagDBX) || (tag == kTagZBX && n != 0);
    const int top = (tag == kTagDBX) ? (int)w : (int)w - 1;
    const uint32_t W = (tag == kTagDBX) ? N - 1u : (tag == kTagZBX) ? n : N;
    const uint32_t S = 1u + W, pf = ceil_log2_u32(W);
    int i = planes ? top : -1;
#pragma unroll 1
    while (i >= 0) {
      // lane k holds the 64 bits at the k-th code ahead, were the codes
      // before it verbatim; its lowest bit is that code's flag
      // one clamp for the three words (a malformed stream cannot read past
      // the stage; a valid one never reaches the clamp)
      const uint32_t q = bit0 + pos + lane * S, qi = min(q >> 5, kCoopStageWords - 3u);
      const uint32_t x0 = stage[qi], x1 = stage[qi + 1], x2 = stage[qi + 2];
      const uint32_t lo = __funnelshift_r(x0, x1, q & 31u), hi = __funnelshift_r(x1, x2, q & 31u);
      const uint32_t f = __ballot_sync(0xFFFFFFFFu, lo & 1u);
      const int m = (f == 0xFFFFFFFFu) ? 32 : __ffs(~f) - 1;  // leading verbatim codes
      if (m > i) {  // the block's remaining planes are all verbatim
        pos += (uint32_t)(i + 1) * S;
        break;
      }
      pos += (uint32_t)m * S;
      i -= m;
      if (m == 32) continue;  // FP32 DBX: a 33rd plane remains
      // the code after the m verbatim ones is not verbatim: lane m holds the
      // 64 bits at it, from which up to four such codes in a row are parsed
      // (each is at most 11 bits); only a first code with m = 0 can stand at
      // the top plane
      uint64_t v = (uint64_t)__shfl_sync(0xFFFFFFFFu, lo, m) | ((uint64_t)__shfl_sync(0xFFFFFFFFu, hi, m) << 32);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t cw = (uint32_t)v;
        if (k > 0 && (i < 0 || (cw & 1u))) break;  // a verbatim code, or no planes left
        const uint32_t tz = (uint32_t)__ffs(cw | 16u) - 1u;  // 1..4
        const uint32_t len = (tz == 1u) ? 2u + K : (tz == 2u) ? 3u : (tz == 3u) ? 5u + pf : 5u;
        const int rl = (tz == 1u) ? 2 + (int)((cw >> 2) & ((1u << K) - 1u)) : 1;
        if (rl > i + 1 || (tz == 4u && (cw & 16u) && i == top)) {
          ok = false;
          break;
        }
        pos += len;
        i -= rl;
        v >>= len;
      }
      if (!ok) break;
    }
    if (pos > cap) ok = false;
  }
  if (ok && cap - pos >= 8) ok = false;
  if (ok && cap > pos && (peek(pos) & ((1u << (cap - pos)) - 1u))) ok = false;
  return ok;
}

template <bool W16>
__global__ void __launch_bounds__(kCoopWarps * 32)
    walk_coop_kernel(DecodeArgs p) {
  extern __shared__ __align__(128) uint8_t coop_smem[];
  griddep_launch_dependents();  // the decode's blocks may be scheduled now
  griddep_wait();               // the group sums are complete
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t C = p.num_chunks;
  const uint32_t c = blockIdx.x * kCoopWarps + warp;
  if (c >= C) return;
  const uint32_t *stage = reinterpret_cast<const uint32_t *>(coop_smem + warp * kCoopStageBytes);
  const uint32_t mb = smem_u32(coop_smem + kCoopWarps * kCoopStageBytes) + warp * 8u;
  const uint64_t off = 2ull * C + sizes_before_chunk(p, c, lane);
  const uint32_t L = __ldg(reinterpret_cast<const uint16_t *>(p.in) + c);
  const uint32_t raw_len = (uint32_t)umin64(4096u, p.nbytes - (uint64_t)c * 4096u);
  if (L == 0 || L > raw_len || off + L > p.comp_bytes) {
    if (lane == 0) atomicMax(p.status, kErrCorrupt);
    return;
  }
  if (raw_len < kRecordBytes) return;  // the decode warp handles it
  uint8_t *rec = p.out + (uint64_t)c * 4096u;
  if (lane == 0) *reinterpret_cast<unsigned long long *>(rec) = off;
  if (L == raw_len) return;  // raw chunk: the offset is all the decoder needs

  const uint64_t a0 = off & ~15ull;
  const uint32_t bytes = (uint32_t)(((off + L + 15) & ~15ull) - a0);  // <= 4112
  if (lane == 0) {
    mbar_init(mb, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (lane == 0) {
    mbar_arrive_expect_tx(mb, bytes);
    bulk_load(smem_u32(stage), p.in + a0, bytes, mb);
  }
  if (!__all_sync(0xFFFFFFFFu, mbar_wait(mb, 0, kMbarPolls))) {
    mbar_wait(mb, 0, kMbarPolls);  // leave no copy in flight
    if (lane == 0) atomicMax(p.status, kErrTimeout);
    return;
  }
  const uint32_t bit0 = (uint32_t)(off - a0) * 8u;
  uint16_t *rs = reinterpret_cast<uint16_t *>(rec + 8);  // start of block b at rs[b - 1]
  const bool ok = coop_walk<W16>(stage, bit0, L, (raw_len + 127u) >> 7, lane, [rs, lane](uint32_t b, uint32_t pos) {
    if (lane == 0) rs[b - 1] = (uint16_t)pos;
  });
  if (!ok && lane == 0) atomicMax(p.status, kErrCorrupt);
}

// Byte offset of 16-byte unit u of row r in a 128-byte-swizzled 4 KB tile.
__device__ __forceinline__ uint32_t tile_swz(uint32_t r, uint32_t u) { return r * 128u + ((u ^ (r & 7u)) << 4); }

// A raw chunk: the warp copies raw_len bytes from stream byte off (any
// alignment) to dst.
__device__ __forceinline__ void copy_raw_chunk(const uint8_t *in, uint64_t off, uint32_t raw_len, uint8_t *dst,
                                               uint32_t lane) {
  // output unit v comes from aligned source units v and v+1 (16-byte
  // loads), realigned by the chunk's byte offset within a unit, which is
  // the same for the whole warp
  const uint64_t a0 = off & ~15ull;
  const uint32_t s = (uint32_t)(off - a0);
  const uint32_t nunits = (uint32_t)((((off + raw_len + 15) & ~15ull) - a0) >> 4);
  const uint4 *src = reinterpret_cast<const uint4 *>(in + a0);
  const uint32_t ws = s >> 2, bs = (s & 3u) * 8u;
  // a lane's loads are issued four units at a time (eight 16-byte loads in
  // flight), so that enough bytes are in flight to cover the memory latency
  constexpr int kR = 4;
#pragma unroll 1
  for (uint32_t v0 = lane; v0 * 16 < raw_len; v0 += 32u * kR) {
    uint4 As[kR], Bs[kR];
#pragma unroll
    for (int i = 0; i < kR; ++i) {
      const uint32_t v = v0 + 32u * i;
      As[i] = (v < nunits) ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
      Bs[i] = (v + 1 < nunits) ? __ldg(src + v + 1) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kR; ++i) {
      const uint32_t v = v0 + 32u * i;
      if (v * 16 >= raw_len) break;
      const uint4 A = As[i], B = Bs[i];
      const uint32_t a[8] = {A.x, A.y, A.z, A.w, B.x, B.y, B.z, B.w};
      uint32_t o[4];
      switch (ws) {  // the same for every lane
        case 0:
#pragma unroll
          for (int k = 0; k < 4; ++k) o[k] = __funnelshift_r(a[k], a[k + 1], bs);
          break;
        case 1:
#pragma unroll
          for (int k = 0; k < 4; ++k) o[k] = __funnelshift_r(a[k + 1], a[k + 2], bs);
          break;
        case 2:
#pragma unroll
          for (int k = 0; k < 4; ++k) o[k] = __funnelshift_r(a[k + 2], a[k + 3], bs);
          break;
        default:
#pragma unroll
          for (int k = 0; k < 4; ++k) o[k] = __funnelshift_r(a[k + 3], a[k + 4], bs);
          break;
      }
      if (v * 16 + 16 <= raw_len) {
        *reinterpret_cast<uint4 *>(dst + 16ull * v) = make_uint4(o[0], o[1], o[2], o[3]);
      } else {
        for (uint32_t b = 0; v * 16 + b < raw_len; ++b) dst[16ull * v + b] = (uint8_t)(o[b >> 2] >> ((b & 3) * 8));
      }
    }
  }
}

// Decode a staged chunk: lane b < nblk decodes block b, whose code starts at
// stage bit bit0 + s0 (the next block's at bit0 + s1), into its row of the
// warp's tile; the warp then writes the chunk's raw_len bytes to dst with
// coalesced 16-byte stores. Returns false in a lane whose block is malformed.
template <bool W16>
__device__ __forceinline__ bool decode_staged(uint32_t sbase, uint32_t bit0, uint32_t s0, uint32_t s1, uint32_t nblk,
                                              uint32_t L, uint32_t raw_len, uint32_t *tw, uint8_t *dst,
                                              uint32_t lane) {
  const StageBits sb{sbase};
  bool ok = true;
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
  return ok;
}

template <bool W16>
__global__ void __launch_bounds__(kDecWarps * 32, 3)
    decode_kernel(DecodeArgs p) {
  __shared__ __align__(128) uint32_t tile[kDecWarps][32 * 32];  // per warp: 32 lane rows of 128 B
  __shared__ __align__(16) uint32_t stage[kDecWarps][kStageWords];  // per warp: the chunk's payload
  __shared__ uint16_t tail_starts[kDecWarps][32];
  griddep_wait();  // the walk's records are complete
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
        uint16_t *ts = tail_starts[warp];
        ok = walk_chunk<W16>(rd, L, nblk, [ts](uint32_t b, uint32_t pos) { ts[b] = (uint16_t)pos; });
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
    copy_raw_chunk(p.in, off, raw_len, dst, lane);
    return;
  }

  // stage the payload: 16-byte units from a0 = off rounded down to 16
  const uint64_t a0 = off & ~15ull;
  const uint32_t nunits = (uint32_t)((off + L + 15 - a0) >> 4);
  const uint32_t sbase = smem_u32(stage[warp]);
  {  // loads four units at a time before their stores (more bytes in flight)
    const uint4 *src = reinterpret_cast<const uint4 *>(p.in + a0);
#pragma unroll 1
    for (uint32_t u0 = lane; u0 < nunits; u0 += 128) {
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = (u0 + 32u * i < nunits) ? __ldg(src + u0 + 32u * i) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (u0 + 32u * i < nunits) *reinterpret_cast<uint4 *>(&stage[warp][4 * (u0 + 32u * i)]) = v[i];
    }
  }
  __syncwarp();
  const uint32_t bit0 = (uint32_t)(off - a0) * 8u;
  if (!decode_staged<W16>(sbase, bit0, s0, s1, nblk, L, raw_len, tile[warp], dst, lane)) atomicMax(p.status, kErrCorrupt);
}

// ------------------------------------------- fused walk and decode (small)
//
// For inputs whose chunks all fit in one resident wave of warps, a warp walks
// its chunk as the cooperative walk does and decodes it right away: the block
// starts stay in shared memory, the staged payload serves both steps, and
// neither the records nor a third launch are needed. While one warp decodes,
// the other warps of its SM are still walking, so the decode hides under the
// walks' latency.
//
// Chunk offsets come from the header table alone. Every warp of this launch
// overwrites its chunk's output region with decoded bytes, and nothing
// orders a warp that has finished against a warp of the same launch that has
// not started (another stream may hold SMs, so the wave need not be resident
// at once): no value may be read back from the output region here.
constexpr uint32_t kFusedWarps = 4;
constexpr uint32_t kFusedMaxChunks = 65536;  // header sums below fit 32 bits (65536 x 4096 < 2^32)
static_assert(kStageWords == kCoopStageWords, "the walk and the decode read the same staged payload");

// Sum of the sizes of chunks [0, c), c <= kFusedMaxChunks, from the header
// table: 16-byte units of eight sizes, then the last few sizes, by a warp.
__device__ __forceinline__ uint32_t header_sum_before(const DecodeArgs &p, uint32_t c, uint32_t lane) {
  const uint4 *h4 = reinterpret_cast<const uint4 *>(p.in);
  const uint32_t u1 = c / 8;
  uint32_t part = 0;
  for (uint32_t i = lane; i < u1; i += 32) part += (uint32_t)sum8_sizes(__ldg(h4 + i));
  if (lane < (c & 7u)) part += __ldg(reinterpret_cast<const uint16_t *>(p.in) + 8u * u1 + lane);
  return __reduce_add_sync(0xFFFFFFFFu, part);
}

template <bool W16>
__global__ void __launch_bounds__(kFusedWarps * 32, 6)
    walk_decode_kernel(DecodeArgs p) {
  __shared__ __align__(128) uint32_t tile[kFusedWarps][32 * 32];  // per warp: 32 lane rows of 128 B
  __shared__ __align__(16) uint32_t stage[kFusedWarps][kStageWords];  // per warp: the chunk's payload
  __shared__ uint16_t starts[kFusedWarps][32];  // start bit of block b >= 1
  __shared__ __align__(8) unsigned long long mbar[kFusedWarps];
  griddep_wait();  // a previous kernel of the stream is complete
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t C = p.num_chunks;
  const uint32_t c = blockIdx.x * kFusedWarps + warp;
  if (c >= C) return;
  const uint64_t off = 2ull * C + header_sum_before(p, c, lane);
  const uint32_t L = __ldg(reinterpret_cast<const uint16_t *>(p.in) + c);
  const uint32_t raw_len = (uint32_t)umin64(4096u, p.nbytes - (uint64_t)c * 4096u);
  if (L == 0 || L > raw_len || off + L > p.comp_bytes) {
    if (lane == 0) atomicMax(p.status, kErrCorrupt);
    return;
  }
  uint8_t *dst = p.out + (uint64_t)c * 4096u;
  if (L == raw_len) {
    copy_raw_chunk(p.in, off, raw_len, dst, lane);
    return;
  }
  const uint64_t a0 = off & ~15ull;
  const uint32_t bytes = (uint32_t)(((off + L + 15) & ~15ull) - a0);  // <= 4112
  const uint32_t mb = smem_u32(&mbar[warp]);
  const uint32_t sbase = smem_u32(stage[warp]);
  if (lane == 0) {
    mbar_init(mb, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (lane == 0) {
    mbar_arrive_expect_tx(mb, bytes);
    bulk_load(sbase, p.in + a0, bytes, mb);
  }
  if (!__all_sync(0xFFFFFFFFu, mbar_wait(mb, 0, kMbarPolls))) {
    mbar_wait(mb, 0, kMbarPolls);  // leave no copy in flight
    if (lane == 0) atomicMax(p.status, kErrTimeout);
    return;
  }
  const uint32_t bit0 = (uint32_t)(off - a0) * 8u;
  const uint32_t nblk = (raw_len + 127u) >> 7;
  uint16_t *ts = starts[warp];
  const bool ok = coop_walk<W16>(stage[warp], bit0, L, nblk, lane, [ts, lane](uint32_t b, uint32_t pos) {
    if (lane == 0) ts[b] = (uint16_t)pos;
  });
  if (!ok) {  // warp-uniform
    if (lane == 0) atomicMax(p.status, kErrCorrupt);
    return;
  }
  __syncwarp();
  const uint32_t s0 = (lane >= 1 && lane < nblk) ? ts[lane] : 0u;
  const uint32_t s1 = (lane + 1 < nblk) ? ts[lane + 1] : 0u;
  if (!decode_staged<W16>(sbase, bit0, s0, s1, nblk, L, raw_len, tile[warp], dst, lane))
    atomicMax(p.status, kErrCorrupt);
}

template __global__ void walk_kernel<false>(DecodeArgs);
template __global__ void walk_decode_kernel<false>(DecodeArgs);
template __global__ void walk_decode_kernel<true>(DecodeArgs);
template __global__ void walk_coop_kernel<false>(DecodeArgs);
template __global__ void walk_coop_kernel<true>(DecodeArgs);
template __global__ void walk_kernel<true>(DecodeArgs);
template __global__ void decode_kernel<false>(DecodeArgs);
template __global__ void decode_kernel<true>(DecodeArgs);

int walk_threads() { return kWalkWarps * 32; }
uint32_t coop_max_chunks() { return kCoopMaxChunks; }
int coop_warps() { return kCoopWarps; }
size_t coop_smem_bytes() { return kCoopSmem; }
int fused_warps() { return kFusedWarps; }
uint32_t fused_max_chunks() { return kFusedMaxChunks; }
const void *walk_decode_kernel_ptr(bool w16) {
  return w16 ? reinterpret_cast<const void *>(&walk_decode_kernel<true>)
             : reinterpret_cast<const void *>(&walk_decode_kernel<false>);
}
const void *walk_coop_kernel_ptr(bool w16) {
  return w16 ? reinterpret_cast<const void *>(&walk_coop_kernel<true>)
             : reinterpret_cast<const void *>(&walk_coop_kernel<false>);
}
size_t walk_smem_bytes() { return kWalkSmem; }
uint32_t group_chunks() { return kGroupChunks; }
const void *size_sum_kernel_ptr() { return reinterpret_cast<const void *>(&size_sum_kernel); }
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
