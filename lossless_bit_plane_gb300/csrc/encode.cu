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
//    32x32 bit transpose in registers (DBX's deltas as the classifier left
//    them in the lane's row of the output region), and its codes go into a
//    shared chunk buffer through an LSB-first writer at the block's bit
//    offset (a warp prefix sum over the lanes' block sizes), four planes at a
//    time with every lane of the warp at the same four planes: four
//    verbatim planes in one step, the others one by one.
//  - Chunk offsets come from a single-pass decoupled look-back over 8-byte
//    status words (flag | value) in the scratch tail of the output buffer,
//    with a bounded spin; the warp then copies its chunk to its final byte
//    offset with aligned 16-byte stores and byte stores at the two edges.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "pz_device.cuh"
#include "pz_encode_block.cuh"
#include "pz_format.cuh"
#include "pz_kernels.h"

namespace pz {

constexpr uint64_t kFlagAgg = 1ull << 62;
constexpr uint64_t kFlagInc = 2ull << 62;
constexpr uint64_t kValueMask = (1ull << 62) - 1;
constexpr uint32_t kLookbackSpinLimit = 1u << 21;
constexpr uint32_t kMbarPollLimit = 1u << 24;

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
// Copy L bytes from the shared word buffer to global byte address dst (any
// alignment): aligned 16-byte stores inside, byte stores at the two edges.
// The buffer must be readable from word -4 to word (L - 1) / 4 + 4: a source
// word outside [0, L) only feeds output bytes that are not stored, so no
// bounds test is needed per word. The source's offset within its word is the
// same for every vector (dst's offset within 16 bytes decides it).
__device__ __forceinline__ void copy_out(const uint32_t *buf, uint32_t L, uint8_t *dst, uint32_t lane) {
  const uint64_t a0 = reinterpret_cast<uint64_t>(dst);
  const int head = (int)(a0 & 15u);  // bytes of the first vector before dst
  const uint32_t nvec = ((uint32_t)head + L + 15u) >> 4;
  const uint32_t sh = (uint32_t)(-head & 3) * 8u;
  uint8_t *const v0 = dst - head;
#pragma unroll 1
  for (uint32_t i = lane; i < nvec; i += 32) {
    const int o = 16 * (int)i - head;  // source byte of the vector's first byte, >= -15
    const uint32_t *w = buf + (o >> 2);
    const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3], w4 = w[4];
    const uint32_t x0 = __funnelshift_r(w0, w1, sh), x1 = __funnelshift_r(w1, w2, sh),
                   x2 = __funnelshift_r(w2, w3, sh), x3 = __funnelshift_r(w3, w4, sh);
    uint8_t *A = v0 + 16ull * i;
    if (o >= 0 && o + 16 <= (int)L) {
      *reinterpret_cast<uint4 *>(A) = make_uint4(x0, x1, x2, x3);
    } else {
      const uint32_t x[4] = {x0, x1, x2, x3};
#pragma unroll
      for (int byte = 0; byte < 16; ++byte) {
        const int so = o + byte;
        if (so >= 0 && so < (int)L) A[byte] = (uint8_t)(x[byte >> 2] >> ((byte & 3) * 8));
      }
    }
  }
}

// ------------------------------------------------------------------ kernel

constexpr int kEncWarps = 8;
constexpr int kOutWords = 1024 + 4;
constexpr int kOutPad = 4;  // readable words before a warp's output buffer (copy_out reads from word -4)

// Shared memory per warp: one 4 KB stage buffer (1024-aligned, the TMA
// destination), the chunk's output region, an mbarrier (16 bytes reserved).
// The output region is 128-byte aligned: before emission it holds the
// lanes' DBX rows (lane l's at byte 128 l), then the output word buffer
// from byte 16 (word 0) on. One stage at three CTAs per SM (24 warps): the
// next chunk is loaded after this one is done, and the other warps cover
// that load's latency. (A second stage, with the next chunk's load in
// flight, needs more shared memory than three CTAs allow.)
template <bool W16>
struct EncCfg {
  static constexpr int kMinCtas = 3;
  static constexpr size_t kStageBytes = 4096;
  static constexpr size_t kOutBytes = ((kOutPad + kOutWords) * 4 + 127) / 128 * 128;
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
  uint8_t *outreg = base + kEncWarps * Cfg::kStageBytes + warp * Cfg::kOutBytes;  // 128-byte aligned
  uint32_t *outbuf = reinterpret_cast<uint32_t *>(outreg) + kOutPad;
  const uint32_t drow = smem_u32(outreg) + lane * 128u;  // this lane's DBX row (until emission)
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
    Sizes z = W16 ? classify16(rowbase, lane, p.candidates, drow) : classify32(rowbase, lane, p.candidates, drow);
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
      // planes first (the DBX rows lie in the output buffer), then the
      // buffer is cleared and the codes go in
      Prep pr{0u, 0u};
      if (active) pr = W16 ? prep16(tag, z.m0, z.m1, rowbase, lane, drow) : prep32(tag, z.m0, rowbase, lane, drow);
      __syncwarp();
      const uint32_t nu = ((L + 3) / 4 + 4) / 4;  // 16-byte units covering the stream's words and one more
      for (uint32_t i = lane; i < nu; i += 32) reinterpret_cast<uint4 *>(outbuf)[i] = make_uint4(0, 0, 0, 0);
      __syncwarp();
      if (active) {
        PosWriter wr;
        wr.init(smem_u32(outbuf), off);
        wr.put(tag, 3);
        const Plan &pl = z.win;
        if (W16)
          emit16(wr, tag, z.m0, z.m1, rowbase, lane, pl, z.bp, pr);
        else
          emit32(wr, tag, z.m0, rowbase, lane, pl, z.bp, pr);
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
