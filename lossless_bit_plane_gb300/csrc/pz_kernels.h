// pz_kernels.h — launch-side declarations of the encoder and decoder kernels
// (argument blocks and launch-shape queries), shared by api.cu and the .cu
// files that define the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include "planezip.h"

namespace pz {

struct EncodeArgs {
  const uint8_t *in;             // input tensor (16-byte aligned)
  uint8_t *out;                  // stream: headers then payloads
  unsigned long long *status;    // look-back words, one per chunk, zeroed
  unsigned int *ticket;          // chunk ticket counter, zeroed
  unsigned long long *total;     // stream length (atomicMax target), zeroed
  // ticket k stands for chunk unit0 + k (nonzero only to leave the first
  // chunks unprocessed)
  uint32_t unit0;
  uint64_t nbytes;
  uint64_t tma_rows;             // 128-byte rows covered by the tensor map (0: none)
  uint32_t num_chunks;
  uint32_t candidates;           // allowed block candidates (bit t = tag t; raw always)
  // size-only launches: chunks 0, stride, 2*stride, ... ; sizes[k] = L of
  // chunk k*stride (when not null); *total += sum of 2 + L
  uint32_t stride;
  uint16_t *sizes;
};

struct DecodeArgs {
  const uint8_t *in;
  uint64_t comp_bytes;
  uint8_t *out;
  uint64_t nbytes;
  int *status;                   // zeroed; atomicMax of error codes
  uint32_t num_chunks;
};

size_t encode_smem_bytes(bool w16);
int encode_threads();
int encode_warps();
const void *encode_kernel_ptr(bool w16, bool size_only);
// zero_scratch_kernel(scratch, nwords, total): zeroes nwords 8-byte words
// and *total, and lets its programmatic dependent (the encoder) start at once
const void *zero_scratch_kernel_ptr();

int walk_threads();
size_t walk_smem_bytes();
const void *walk_kernel_ptr(bool w16);
uint32_t group_chunks();              // chunks per size-sum group
uint32_t coop_max_chunks();           // inputs up to this many chunks use the cooperative walk
int coop_warps();                     // chunks per cooperative-walk block (one warp each)
size_t coop_smem_bytes();
const void *walk_coop_kernel_ptr(bool w16);
int fused_warps();                    // chunks per fused walk-and-decode block (one warp each)
uint32_t fused_max_chunks();          // the fused kernel's limit on C (its header sums are 32-bit)
const void *walk_decode_kernel_ptr(bool w16);  // small inputs: walk and decode in one launch
const void *size_sum_kernel_ptr();    // 256 threads, one block per group but the last
int decode_threads();
int decode_chunks_per_cta();
const void *decode_kernel_ptr(bool w16);

// pz_decompress's body; reset_status false leaves *d_status as it is, so
// that several calls accumulate their errors (atomicMax) in one word.
pz_status decompress_launch(const void *d_in, size_t comp_bytes, int elem_width, void *d_out, size_t nbytes,
                            int *d_status, pz_stream_t stream, bool reset_status);

}  // namespace pz
