// pz_device.cuh — device helpers shared by the encoder and decoder kernels:
// inline-PTX wrappers (mbarrier, TMA tile load, relaxed global loads/stores,
// shared memory by 32-bit address, byte permute), SWAR helpers for two
// 16-bit symbols per 32-bit word and a 32x32 bit-matrix transpose.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace pz {

// ---------------------------------------------------------------- basics

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }
__device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }
// ceil(log2(v)) for v >= 1 (0 for v <= 1), without a loop
__device__ __forceinline__ uint32_t ceil_log2_u32(uint32_t v) { return v <= 1u ? 0u : 32u - (uint32_t)__clz(v - 1u); }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// 0xFFFF in each 16-bit half of x that is non-zero, 0 in each half that is 0.
__device__ __forceinline__ uint32_t halfmask_nonzero(uint32_t x) {
  uint32_t t = ((x & 0x7FFF7FFFu) + 0x7FFF7FFFu) | x;  // bit 15 / 31: half != 0
  uint32_t r;
  // byte selectors 9 and B with bit 3 set replicate the sign of bytes 1 / 3
  asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(r) : "r"(t));
  return r;
}

// Two independent 16-bit subtractions d = x - y (mod 2^16 per half); bo gets
// each half's borrow (x_half < y_half) in bit 15 / bit 31.
__device__ __forceinline__ uint32_t sub16x2(uint32_t x, uint32_t y, uint32_t &bo) {
  uint32_t t = (x | 0x80008000u) - (y & 0x7FFF7FFFu);
  uint32_t d = t ^ (~(x ^ y) & 0x80008000u);
  bo = ((~x & y) | (~(x ^ y) & d)) & 0x80008000u;
  return d;
}

// Split packing of a BF16 block: word j holds symbol j (low half) and symbol
// j+32 (high half). raw[r] holds symbols 2r, 2r+1 in memory order.
__device__ __forceinline__ uint32_t split_word(const uint32_t *raw, int j) {
  return prmt(raw[j >> 1], raw[16 + (j >> 1)], (j & 1) ? 0x7632u : 0x5410u);
}
__device__ __forceinline__ uint32_t raw_word_from_split(const uint32_t *sp, int r) {
  return (r < 16) ? prmt(sp[2 * r], sp[2 * r + 1], 0x5410u)
                  : prmt(sp[2 * (r - 16)], sp[2 * (r - 16) + 1], 0x7632u);
}

// 32x32 bit-matrix transpose in registers: afterwards bit j of a[i] equals
// bit i of the original a[j].
__device__ __forceinline__ void transpose32(uint32_t (&a)[32]) {
#pragma unroll
  for (int k = 0; k < 16; ++k) {  // swap 16x16 blocks
    uint32_t x = a[k], y = a[k + 16];
    a[k] = prmt(x, y, 0x5410u);
    a[k + 16] = prmt(x, y, 0x7632u);
  }
#pragma unroll
  for (int g = 0; g < 32; g += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k) {  // swap 8x8 blocks
      uint32_t x = a[g + k], y = a[g + k + 8];
      a[g + k] = prmt(x, y, 0x6240u);
      a[g + k + 8] = prmt(x, y, 0x7351u);
    }
#pragma unroll
  for (int g = 0; g < 32; g += 8)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t t = ((a[g + k] >> 4) ^ a[g + k + 4]) & 0x0F0F0F0Fu;
      a[g + k + 4] ^= t;
      a[g + k] ^= t << 4;
    }
#pragma unroll
  for (int g = 0; g < 32; g += 4)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      uint32_t t = ((a[g + k] >> 2) ^ a[g + k + 2]) & 0x33333333u;
      a[g + k + 2] ^= t;
      a[g + k] ^= t << 2;
    }
#pragma unroll
  for (int g = 0; g < 32; g += 2) {
    uint32_t t = ((a[g] >> 1) ^ a[g + 1]) & 0x55555555u;
    a[g + 1] ^= t;
    a[g] ^= t << 1;
  }
}

// --------------------------------------- shared memory by 32-bit address
// Accesses by a shared-window address (smem_u32 of a pointer), so that row
// and swizzle arithmetic stays in 32-bit registers.
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
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 q;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(q.x), "=r"(q.y), "=r"(q.z), "=r"(q.w)
               : "r"(addr)
               : "memory");
  return q;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void sts16(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"((unsigned short)v) : "memory");
}
// *addr |= v as one shared-memory reduction (no value returned)
__device__ __forceinline__ void ors32(uint32_t addr, uint32_t v) {
  asm volatile("red.shared.or.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// --------------------------------------------- programmatic dependent launch
// A kernel launched with the programmatic-serialization attribute right after
// another kernel of the same stream may start before that kernel ends:
// griddepcontrol.wait returns once the predecessor has ended and its stores
// are visible (at once when the launch had no such predecessor), and a
// predecessor's griddepcontrol.launch_dependents lets the dependent's blocks
// be scheduled before it ends.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------ global memory, relaxed
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ------------------------------------------------------ mbarrier + TMA
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t addr, uint32_t bytes) {
  asm volatile(
      "{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(addr),
      "r"(bytes)
      : "memory");
}
// Bounded wait for the phase with the given parity; false after `limit` polls.
__device__ __forceinline__ bool mbar_wait(uint32_t addr, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}
// 2D tiled TMA load of one box into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar)
      : "memory");
}

// --------------------------------------------------------- warp helpers
__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

}  // namespace pz
