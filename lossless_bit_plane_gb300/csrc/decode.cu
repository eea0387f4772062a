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

constexpr int kDecWarps = 4;
constexpr int kDecChunksPerCta = 32 * kDecWarps;

// LSB-first reader over the stream's 32-bit words with one word prefetched.
struct BitReader {
  const uint32_t *words;
  uint64_t nwords;  // words that hold at least one stream byte
  uint64_t wpos;    // index of the word held in nxt
  uint64_t buf;
  uint32_t nbuf;
  uint32_t nxt;
  uint64_t consumed;

  __device__ __forceinline__ uint32_t load(uint64_t i) const { return i < nwords ? __ldg(words + i) : 0u; }
  __device__ __forceinline__ void init(const uint32_t *w, uint64_t nw, uint64_t bitpos) {
    words = w;
    nwords = nw;
    uint64_t wi = bitpos >> 5;
    uint32_t sh = (uint32_t)(bitpos & 31);
    buf = (uint64_t)load(wi) >> sh;
    nbuf = 32 - sh;
    wpos = wi + 1;
    nxt = load(wpos);
    consumed = 0;
  }
  __device__ __forceinline__ void ensure(uint32_t n) {  // n <= 32
    if (nbuf < n) {
      buf |= (uint64_t)nxt << nbuf;
      nbuf += 32;
      nxt = load(++wpos);
    }
  }
  __device__ __forceinline__ uint32_t peek(uint32_t n) const {  // after ensure(n), n <= 32
    return (uint32_t)buf & (uint32_t)((1ull << n) - 1);
  }
  __device__ __forceinline__ void skip(uint32_t n) {
    buf >>= n;
    nbuf -= n;
    consumed += n;
  }
  __device__ __forceinline__ uint32_t get(uint32_t n) {  // n <= 32
    ensure(n);
    uint32_t v = peek(n);
    skip(n);
    return v;
  }
  __device__ __forceinline__ uint64_t get64(uint32_t n) {  // n <= 64
    if (n > 32) {
      uint64_t lo = get(32);
      return lo | ((uint64_t)get(n - 32) << 32);
    }
    return get(n);
  }
};

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

// Parse the P = top+1 plane codes of one block, top plane first, rebuilding
// the pre-XOR planes P_i = X_i ^ P_{i+1}, and store them in the lane's row:
// FP32 plane i < 32 in word i; BF16 plane i < 16 in words i (symbols 0..31)
// and 16+i (symbols 32..63). For DBX the rows are pre-shifted so that row
// bit j holds delta j (plane bit q is delta q+1); the top DBX plane (the
// borrow plane) is not stored. Returns false on a malformed code.
template <bool W16>
__device__ __forceinline__ bool parse_plane_rows(BitReader &br, uint32_t row, uint32_t lane, int top, int W,
                                                 int p, bool dbx) {
  const int K = W16 ? 4 : 5;
  const uint64_t full = (W >= 64) ? ~0ull : ((1ull << W) - 1);
  uint64_t Pup = 0;
  int run = 0;
#pragma unroll 1
  for (int i = top; i >= 0; --i) {
    uint64_t X = 0;
    if (run > 0) {
      --run;
    } else {
      br.ensure(16);
      const uint32_t v = br.peek(16);
      if (v & 1u) {  // 1 + plane
        br.skip(1);
        X = br.get64((uint32_t)W);
      } else if ((v & 3u) == 2u) {  // 0 1 + (run - 2)
        const int L = 2 + (int)((v >> 2) & ((1u << K) - 1));
        br.skip(2 + K);
        if (L > i + 1) return false;
        run = L - 1;
      } else if ((v & 7u) == 4u) {  // 0 0 1
        br.skip(3);
      } else {
        const uint32_t code = v & 31u;
        br.skip(5);
        if (code == 0) {  // 0 0 0 0 0: all ones
          X = full;
        } else if (code == 16) {  // 0 0 0 0 1: pre-XOR plane zero
          if (i == top) return false;
          X = Pup;
        } else {  // 0 0 0 1 0 / 0 0 0 1 1 + q
          const int q = (int)br.get((uint32_t)p);
          if (code == 8) {
            if (q + 1 >= W) return false;
            X = 3ull << q;
          } else {
            if (q >= W) return false;
            X = 1ull << q;
          }
        }
      }
    }
    const uint64_t Pi = (i == top) ? X : (X ^ Pup);
    Pup = Pi;
    if (W16) {
      if (i < 16) {
        sts32d(prow(row, lane, (uint32_t)i), dbx ? (uint32_t)(Pi << 1) : (uint32_t)Pi);
        sts32d(prow(row, lane, (uint32_t)i + 16), dbx ? (uint32_t)(Pi >> 31) : (uint32_t)(Pi >> 32));
      }
    } else {
      if (i < 32) sts32d(prow(row, lane, (uint32_t)i), dbx ? (uint32_t)(Pi << 1) : (uint32_t)Pi);
    }
  }
  return true;
}

// Decode one block into o[32], the block's 32 words in memory order.
template <bool W16>
__device__ __forceinline__ bool decode_block(BitReader &br, uint32_t (&o)[32], uint32_t row, uint32_t lane) {
  const uint32_t tag = br.get(3);
  if (tag > kTagRAW) return false;
  if (tag == kTagRAW) {
#pragma unroll 4
    for (uint32_t k = 0; k < 32; ++k) sts32d(prow(row, lane, k), br.get(32));
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = lds32d(prow(row, lane, k));
    return true;
  }
  if (tag == kTagZVC) {
    if (W16) {
      const uint32_t mlo = br.get(32), mhi = br.get(32);
#pragma unroll 1
      for (uint32_t h = 0; h < 64; ++h) {
        const uint32_t bit = (h < 32) ? (mlo >> h) : (mhi >> (h - 32));
        sts16d(prow_half(row, lane, h), (bit & 1u) ? br.get(16) : 0u);
      }
    } else {
      const uint32_t mask = br.get(32);
#pragma unroll 1
      for (uint32_t k = 0; k < 32; ++k) sts32d(prow(row, lane, k), ((mask >> k) & 1u) ? br.get(32) : 0u);
    }
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = lds32d(prow(row, lane, k));
    return true;
  }
  uint32_t basesym = 0, mlo = 0, mhi = 0;
  int top = W16 ? 15 : 31, W = W16 ? 64 : 32;
  if (tag == kTagDBX) {
    basesym = br.get(W16 ? 16 : 32);
    ++top;
    --W;
  } else if (tag == kTagZBX) {
    mlo = br.get(32);
    if (W16) mhi = br.get(32);
    W = __popc(mlo) + __popc(mhi);
    if (W == 0) {
#pragma unroll
      for (int k = 0; k < 32; ++k) o[k] = 0;
      return true;
    }
  }
  if (!parse_plane_rows<W16>(br, row, lane, top, W, ceil_log2_int(W), tag == kTagDBX)) return false;
#pragma unroll
  for (int j = 0; j < 32; ++j) o[j] = lds32d(prow(row, lane, j));
  transpose32(o);  // FP32: o[j] = symbol j (or delta j); BF16: split words
  if (!W16) {
    if (tag == kTagDBX) {
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
    return true;
  }
  // BF16: o holds split words (word j = symbol j | symbol j+32 << 16)
  if (tag == kTagDBX) {
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
  return true;
}

// ---------------------------------------------------------------- kernel

template <bool W16>
__global__ void __launch_bounds__(kDecWarps * 32)
    decode_kernel(DecodeArgs p) {
  __shared__ unsigned long long red[kDecWarps];
  __shared__ uint32_t wsum[kDecWarps];
  __shared__ __align__(16) uint32_t scratch[kDecWarps][32 * 32];
  const uint32_t lane = lane_id();
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t C = p.num_chunks;
  const uint32_t first = blockIdx.x * kDecChunksPerCta;
  const uint16_t *hdr = reinterpret_cast<const uint16_t *>(p.in);

  // sum of all chunk sizes before this CTA's first chunk
  unsigned long long part = 0;
  {
    const uint4 *h4 = reinterpret_cast<const uint4 *>(p.in);  // first is a multiple of 8
    for (uint32_t i = threadIdx.x; i < first / 8; i += blockDim.x) {
      uint4 v = __ldg(h4 + i);
      part += (v.x & 0xFFFFu) + (v.x >> 16) + (v.y & 0xFFFFu) + (v.y >> 16) + (v.z & 0xFFFFu) +
              (v.z >> 16) + (v.w & 0xFFFFu) + (v.w >> 16);
    }
  }
  part = warp_sum_u64(part);
  // this CTA's own headers
  const uint32_t c = first + warp * 32 + lane;
  const bool valid = c < C;
  const uint32_t L = valid ? __ldg(hdr + c) : 0u;
  uint32_t incl = L;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= (uint32_t)o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  if (lane == 0) red[warp] = part;
  __syncthreads();
  unsigned long long base = 0;
  for (int w = 0; w < kDecWarps; ++w) base += red[w];
  for (uint32_t w = 0; w < warp; ++w) base += wsum[w];
  const uint64_t off = base + (incl - L);  // payload offset after the header table

  const uint64_t hdr_bytes = 2ull * C;
  const uint64_t c0 = (uint64_t)c * 4096u;
  const uint32_t raw_len = valid ? (uint32_t)umin64(4096u, p.nbytes - c0) : 0u;
  bool bad = valid && (L == 0 || L > raw_len || hdr_bytes + off + L > p.comp_bytes);
  if (bad) atomicMax(p.status, kErrCorrupt);
  const bool is_raw = valid && !bad && L == raw_len;
  const bool is_coded = valid && !bad && L < raw_len;

  // raw chunks: the whole warp copies each one (unaligned source)
  uint32_t rm = __ballot_sync(0xFFFFFFFFu, is_raw);
  while (rm) {
    const uint32_t src_lane = __ffs(rm) - 1;
    rm &= rm - 1;
    const uint64_t soff = __shfl_sync(0xFFFFFFFFu, hdr_bytes + off, src_lane);
    const uint32_t rl = __shfl_sync(0xFFFFFFFFu, raw_len, src_lane);
    const uint32_t cc = __shfl_sync(0xFFFFFFFFu, c, src_lane);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(p.in);
    const uint64_t nw = (p.comp_bytes + 3) / 4;
    uint8_t *dst = p.out + (uint64_t)cc * 4096u;
    const uint32_t sh = (uint32_t)(soff & 3) * 8;
    for (uint32_t v = lane; v * 16 < rl; v += 32) {
      const uint64_t wi = (soff + 16ull * v) >> 2;
      uint32_t w5[5];
#pragma unroll
      for (int k = 0; k < 5; ++k) w5[k] = (wi + k < nw) ? __ldg(w + wi + k) : 0u;
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k] = __funnelshift_r(w5[k], w5[k + 1], sh);
      if (v * 16 + 16 <= rl) {
        *reinterpret_cast<uint4 *>(dst + 16ull * v) = make_uint4(o[0], o[1], o[2], o[3]);
      } else {
        for (uint32_t b = 0; v * 16 + b < rl; ++b) dst[16ull * v + b] = (uint8_t)(o[b >> 2] >> ((b & 3) * 8));
      }
    }
  }

  // coded chunks: each lane walks its own chunk
  if (is_coded) {
    BitReader br;
    br.init(reinterpret_cast<const uint32_t *>(p.in), (p.comp_bytes + 3) / 4, 8ull * (hdr_bytes + off));
    const uint32_t nblk = (raw_len + 127u) >> 7;
    const uint32_t row = smem_u32(&scratch[warp][lane * 32]);
    uint8_t *dst = p.out + c0;
    bool ok = true;
    for (uint32_t b = 0; b < nblk && ok; ++b) {
      uint32_t s[32];
      ok = decode_block<W16>(br, s, row, lane);
      if (br.consumed > 8ull * L) ok = false;
      if (!ok) break;
      uint8_t *bd = dst + 128u * b;
      const uint32_t take = min(128u, raw_len - 128u * b);
      if (take == 128u) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
          reinterpret_cast<uint4 *>(bd)[u] = make_uint4(s[4 * u], s[4 * u + 1], s[4 * u + 2], s[4 * u + 3]);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if ((uint32_t)(4 * k + e) < take) bd[4 * k + e] = (uint8_t)(s[k] >> (8 * e));
      }
    }
    if (ok) {
      // exactly ceil(bits/8) bytes, zero padding
      const uint64_t cap = 8ull * L;
      if (cap - br.consumed >= 8) ok = false;
      else {
        const uint32_t pad = (uint32_t)(cap - br.consumed);
        if (pad && br.get(pad) != 0) ok = false;
      }
    }
    if (!ok) atomicMax(p.status, kErrCorrupt);
  }
}

template __global__ void decode_kernel<false>(DecodeArgs);
template __global__ void decode_kernel<true>(DecodeArgs);

int decode_threads() { return kDecWarps * 32; }
int decode_chunks_per_cta() { return kDecChunksPerCta; }
const void *decode_kernel_ptr(bool w16) {
  return w16 ? reinterpret_cast<const void *>(&decode_kernel<true>)
             : reinterpret_cast<const void *>(&decode_kernel<false>);
}

}  // namespace pz
