// api.cu — the C ABI of include/planezip.h: argument checks, the encoder's
// scratch layout in the output buffer's tail, the TMA tensor map of the
// input, launch shapes, and the launches. No device memory is allocated.
//
// Paper: "PlaneZip: Lossless Bit-Plane Compression of Training Activations
// Offloaded over PCIe" (arXiv:2610.25033v1), Section III-A "Codec" and
// "Stream format" (what the two launched kernels compute).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/planezip.h"
#include "../../include/planezip_testing.h"
#include "pz_kernels.h"

namespace {

constexpr size_t kChunk = 4096;
constexpr int kMaxDevices = 64;

size_t num_chunks(size_t nbytes) { return (nbytes + kChunk - 1) / kChunk; }
size_t align16(size_t v) { return (v + 15) & ~size_t(15); }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int enc_ctas_per_sm[4] = {0, 0, 0, 0};  // [2 * size_only + w16]
  size_t fused_max_chunks[2] = {0, 0};   // [w16]: one resident wave of the fused walk and decode
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;

// Per-device launch facts, computed once with the device current.
cudaError_t device_info(DeviceInfo &out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo &d = g_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    for (int w = 0; w < 2; ++w) {
      const size_t smem = pz::encode_smem_bytes(w == 1);
      for (int so = 0; so < 2; ++so) {
        const void *k = pz::encode_kernel_ptr(w == 1, so == 1);
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
          return e;
        int n = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, pz::encode_threads(), smem)) != cudaSuccess)
          return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        d.enc_ctas_per_sm[2 * so + w] = n;
      }
    }
    for (int w = 0; w < 2; ++w)
      if ((e = cudaFuncSetAttribute(pz::walk_kernel_ptr(w == 1), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)pz::walk_smem_bytes())) != cudaSuccess)
        return e;
    for (int w = 0; w < 2; ++w) {
      int n = 0;
      if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, pz::walk_decode_kernel_ptr(w == 1),
                                                             32 * pz::fused_warps(), 0)) != cudaSuccess)
        return e;
      d.fused_max_chunks[w] = (size_t)n * (size_t)d.sms * (size_t)pz::fused_warps();
      if (d.fused_max_chunks[w] > pz::fused_max_chunks()) d.fused_max_chunks[w] = pz::fused_max_chunks();
    }
    if (!g_encode_tiled) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
      g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.ready = true;
  }
  out = d;
  return cudaSuccess;
}

// One kernel launch; with `dependent` it is the programmatic dependent of
// the kernel launched just before it on the stream (the kernel waits for
// that one with griddepcontrol.wait before it touches its results).
cudaError_t launch(const void *fn, size_t grid, size_t threads, size_t smem, void **args, bool dependent,
                   cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// The 2D tensor map over the input (rows of 128 bytes; 32 x u32 each) and
// the encoder launch. `units` is the number of chunks the launch visits
// (every chunk, or every stride-th for sizes only); a.in, a.nbytes and
// a.num_chunks are set by the caller. The encoder's look-back words and
// ticket (scratch_words 8-byte words at a.status) and *a.total are zeroed by
// a small kernel launched first; the encoder is launched as its programmatic
// dependent, so that its launch overlaps the zeroing (its warps wait for the
// zeroing to end before their first ticket or store).
pz_status launch_encoder(pz::EncodeArgs &a, bool w16, bool size_only, size_t units, size_t scratch_words,
                         const DeviceInfo &info, cudaStream_t s) {
  a.tma_rows = a.nbytes / 128;
  alignas(64) CUtensorMap tmap;
  std::memset(&tmap, 0, sizeof(tmap));
  if (a.tma_rows > 0) {
    cuuint64_t dims[2] = {32, (cuuint64_t)a.tma_rows};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode_tiled(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t *>(a.in), dims, strides,
                                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return PZ_ERR_CUDA;
  }
  // a failure above leaves the stream untouched: the launches start here
  {
    unsigned long long *zp = a.status;
    uint32_t zn = (uint32_t)scratch_words;
    unsigned long long *zt = a.total;
    void *zargs[3] = {&zp, &zn, &zt};
    size_t zb = (scratch_words + 255) / 256;
    if (zb < 1) zb = 1;
    if (zb > (size_t)info.sms * 4) zb = (size_t)info.sms * 4;
    if (cudaLaunchKernel(pz::zero_scratch_kernel_ptr(), dim3((unsigned)zb), dim3(256), zargs, 0, s) != cudaSuccess)
      return PZ_ERR_CUDA;
  }
  const int warps = pz::encode_warps();
  size_t grid = (size_t)info.enc_ctas_per_sm[2 * (size_only ? 1 : 0) + (w16 ? 1 : 0)] * info.sms;
  const size_t need = (units + warps - 1) / warps;
  if (grid > need) grid = need;
  void *args[2] = {&tmap, &a};
  if (launch(pz::encode_kernel_ptr(w16, size_only), grid, (size_t)pz::encode_threads(), pz::encode_smem_bytes(w16),
             args, true, s) != cudaSuccess)
    return PZ_ERR_CUDA;
  return PZ_OK;
}

}  // namespace

extern "C" {

size_t pz_max_compressed_bytes(size_t nbytes) {
  const size_t C = num_chunks(nbytes);
  return align16(2 * C + nbytes) + 8 * C + 64;
}

pz_status pz_compress(const void *d_in, size_t nbytes, int elem_width, void *d_out, size_t out_capacity,
                      unsigned long long *d_total_bytes, pz_stream_t stream) {
  return pz_compress_candidates(d_in, nbytes, elem_width, PZ_CAND_ALL, d_out, out_capacity, d_total_bytes, stream);
}

pz_status pz_compress_candidates(const void *d_in, size_t nbytes, int elem_width, unsigned int candidates,
                                 void *d_out, size_t out_capacity, unsigned long long *d_total_bytes,
                                 pz_stream_t stream) {
  if (elem_width <= 0 || !d_total_bytes || (candidates & ~PZ_CAND_ALL)) return PZ_ERR_ARG;
  const size_t C = num_chunks(nbytes);
  if (nbytes && (!d_in || !d_out)) return PZ_ERR_ARG;
  if (nbytes && (!aligned16(d_in) || !aligned16(d_out))) return PZ_ERR_ARG;
  if (C > 0x7FFFFFFFu || nbytes / 128 > 0xFFFFFFFFull) return PZ_ERR_ARG;
  if (out_capacity < pz_max_compressed_bytes(nbytes)) return PZ_ERR_CAPACITY;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (nbytes == 0)
    return cudaMemsetAsync(d_total_bytes, 0, sizeof(unsigned long long), s) == cudaSuccess ? PZ_OK : PZ_ERR_CUDA;

  DeviceInfo info;
  if (device_info(info) != cudaSuccess) return PZ_ERR_CUDA;

  uint8_t *out = static_cast<uint8_t *>(d_out);
  uint8_t *scratch = out + align16(2 * C + nbytes);

  pz::EncodeArgs a{};
  a.in = static_cast<const uint8_t *>(d_in);
  a.out = out;
  a.status = reinterpret_cast<unsigned long long *>(scratch);
  a.ticket = reinterpret_cast<unsigned int *>(scratch + 8 * C);
  a.total = d_total_bytes;
  a.nbytes = nbytes;
  a.num_chunks = (uint32_t)C;
  a.candidates = candidates | PZ_CAND_RAW;
  a.stride = 1;
  return launch_encoder(a, elem_width == 2, false, C, C + 8, info, s);
}

pz_status pz_test_lookback_timeout(const void *d_in, size_t nbytes, int elem_width, void *d_out, size_t out_capacity,
                                   unsigned long long *d_total_bytes, pz_stream_t stream) {
  if (elem_width <= 0 || !d_total_bytes || !d_in || !d_out) return PZ_ERR_ARG;
  const size_t C = num_chunks(nbytes);
  if (C < 2 || C > 4096) return PZ_ERR_ARG;
  if (!aligned16(d_in) || !aligned16(d_out)) return PZ_ERR_ARG;
  if (out_capacity < pz_max_compressed_bytes(nbytes)) return PZ_ERR_CAPACITY;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceInfo info;
  if (device_info(info) != cudaSuccess) return PZ_ERR_CUDA;
  uint8_t *out = static_cast<uint8_t *>(d_out);
  uint8_t *scratch = out + align16(2 * C + nbytes);
  pz::EncodeArgs a{};
  // chunks are numbered from 1: chunk 0 is never taken, so its status word
  // is never published
  a.unit0 = 1;
  a.in = static_cast<const uint8_t *>(d_in);
  a.out = out;
  a.status = reinterpret_cast<unsigned long long *>(scratch);
  a.ticket = reinterpret_cast<unsigned int *>(scratch + 8 * C);
  a.total = d_total_bytes;
  a.nbytes = nbytes;
  a.num_chunks = (uint32_t)C;
  a.candidates = PZ_CAND_ALL;
  a.stride = 1;
  return launch_encoder(a, elem_width == 2, false, C, C + 8, info, s);
}

pz_status pz_compressed_size(const void *d_in, size_t nbytes, int elem_width, unsigned int candidates,
                             unsigned int chunk_stride, unsigned short *d_sizes, unsigned long long *d_total,
                             pz_stream_t stream) {
  if (elem_width <= 0 || !d_total || chunk_stride == 0 || (candidates & ~PZ_CAND_ALL)) return PZ_ERR_ARG;
  const size_t C = num_chunks(nbytes);
  if (nbytes && !d_in) return PZ_ERR_ARG;
  if (nbytes && !aligned16(d_in)) return PZ_ERR_ARG;
  if (C > 0x7FFFFFFFu || nbytes / 128 > 0xFFFFFFFFull) return PZ_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (nbytes == 0) return cudaMemsetAsync(d_total, 0, sizeof(unsigned long long), s) == cudaSuccess ? PZ_OK : PZ_ERR_CUDA;
  DeviceInfo info;
  if (device_info(info) != cudaSuccess) return PZ_ERR_CUDA;
  pz::EncodeArgs a{};
  a.in = static_cast<const uint8_t *>(d_in);
  a.total = d_total;
  a.nbytes = nbytes;
  a.num_chunks = (uint32_t)C;
  a.candidates = candidates | PZ_CAND_RAW;
  a.stride = chunk_stride;
  a.sizes = d_sizes;
  return launch_encoder(a, elem_width == 2, true, (C + chunk_stride - 1) / chunk_stride, 0, info, s);
}

pz_status pz_decompress(const void *d_in, size_t comp_bytes, int elem_width, void *d_out, size_t nbytes,
                        int *d_status, pz_stream_t stream) {
  return pz::decompress_launch(d_in, comp_bytes, elem_width, d_out, nbytes, d_status, stream, true);
}

}  // extern "C"

// pz_decompress's checks and launches; with reset_status false the device
// status word is not cleared first, so that several streams (the pieces of
// a swapped tensor) accumulate their errors into one word.
pz_status pz::decompress_launch(const void *d_in, size_t comp_bytes, int elem_width, void *d_out, size_t nbytes,
                                int *d_status, pz_stream_t stream, bool reset_status) {
  if (elem_width <= 0 || !d_status) return PZ_ERR_ARG;
  const size_t C = num_chunks(nbytes);
  if (nbytes && (!d_in || !d_out)) return PZ_ERR_ARG;
  if (nbytes && (!aligned16(d_in) || !aligned16(d_out))) return PZ_ERR_ARG;
  if (C > 0x7FFFFFFFu) return PZ_ERR_ARG;
  if (comp_bytes < 2 * C) return PZ_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (reset_status && cudaMemsetAsync(d_status, 0, sizeof(int), s) != cudaSuccess) return PZ_ERR_CUDA;
  if (C == 0) return PZ_OK;

  pz::DecodeArgs a;
  a.in = static_cast<const uint8_t *>(d_in);
  a.comp_bytes = comp_bytes;
  a.out = static_cast<uint8_t *>(d_out);
  a.nbytes = nbytes;
  a.status = d_status;
  a.num_chunks = (uint32_t)C;
  const bool w16 = (elem_width == 2);
  DeviceInfo info;
  if (device_info(info) != cudaSuccess) return PZ_ERR_CUDA;
  void *args[1] = {&a};
  if (C <= info.fused_max_chunks[w16 ? 1 : 0]) {
    // one resident wave: a warp walks and decodes each chunk, in one launch
    // that reads its chunk offsets from the header table alone
    const size_t fw = (size_t)pz::fused_warps();
    if (launch(pz::walk_decode_kernel_ptr(w16), (C + fw - 1) / fw, 32 * fw, 0, args, false, s) != cudaSuccess)
      return PZ_ERR_CUDA;
    return PZ_OK;
  }
  const size_t G = pz::group_chunks();
  const size_t groups = (C + G - 1) / G;
  // Each launch after the first kernel is its predecessor's programmatic
  // dependent: its blocks are scheduled while the predecessor runs and wait
  // for its end (griddepcontrol.wait) before they start, which hides the
  // launch gap. The first kernel follows the status memset and is launched
  // plainly.
  if (groups > 1 && cudaLaunchKernel(pz::size_sum_kernel_ptr(), dim3((unsigned)(groups - 1)), dim3(256), args, 0,
                                     s) != cudaSuccess)
    return PZ_ERR_CUDA;
  const bool after_kernel = groups > 1;
  if (C <= pz::coop_max_chunks()) {  // small input: a warp walks each chunk
    const size_t cw = (size_t)pz::coop_warps();
    if (launch(pz::walk_coop_kernel_ptr(w16), (C + cw - 1) / cw, 32 * cw, pz::coop_smem_bytes(), args, after_kernel,
               s) != cudaSuccess)
      return PZ_ERR_CUDA;
  } else {  // a thread walks each chunk
    const size_t wt = (size_t)pz::walk_threads();
    if (launch(pz::walk_kernel_ptr(w16), (C + wt - 1) / wt, wt, pz::walk_smem_bytes(), args, after_kernel, s) !=
        cudaSuccess)
      return PZ_ERR_CUDA;
  }
  const size_t per = (size_t)pz::decode_chunks_per_cta();
  if (launch(pz::decode_kernel_ptr(w16), (C + per - 1) / per, (size_t)pz::decode_threads(), 0, args, true, s) !=
      cudaSuccess)
    return PZ_ERR_CUDA;
  return PZ_OK;
}


// ---------------------------------------------------------------------------
// Allocation-free compress: the same encoder launch as pz_compress, with the
// look-back words and ticket counter in a file-scope device array instead of
// the tail of the caller's output buffer. For callers that cannot allocate
// when they compress (a swap runtime evicting activations because device
// memory is full cannot grow its buffers); the declaration in planezip.h
// states the limits and the sharing rules.
namespace {

constexpr size_t kNoAllocMaxChunks = PZ_NOALLOC_MAX_BYTES / kChunk;
constexpr size_t kNoAllocScratchWords = kNoAllocMaxChunks + 8;  // status words + ticket
static __device__ __align__(256) unsigned long long g_noalloc_scratch[kNoAllocScratchWords];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once
// per device with that device current.
cudaError_t noalloc_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" pz_status pz_compress_noalloc(const void *d_in, size_t nbytes, int elem_width, void *d_out,
                                         size_t out_capacity, unsigned long long *d_total_bytes,
                                         pz_stream_t stream) {
  if (elem_width <= 0 || !d_total_bytes) return PZ_ERR_ARG;
  const size_t C = num_chunks(nbytes);
  if (nbytes && (!d_in || !d_out)) return PZ_ERR_ARG;
  if (nbytes && (!aligned16(d_in) || !aligned16(d_out))) return PZ_ERR_ARG;
  if (nbytes > PZ_NOALLOC_MAX_BYTES) return PZ_ERR_CAPACITY;
  if (out_capacity < 2 * C + nbytes) return PZ_ERR_CAPACITY;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (nbytes == 0)
    return cudaMemsetAsync(d_total_bytes, 0, sizeof(unsigned long long), s) == cudaSuccess ? PZ_OK : PZ_ERR_CUDA;

  DeviceInfo info;
  if (device_info(info) != cudaSuccess) return PZ_ERR_CUDA;
  void *scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return PZ_ERR_CUDA;
  // the previous call's look-back words and ticket must not leak into this
  // one: the encoder launch zeroes them first

  pz::EncodeArgs a{};
  a.in = static_cast<const uint8_t *>(d_in);
  a.out = static_cast<uint8_t *>(d_out);
  a.status = static_cast<unsigned long long *>(scratch);
  a.ticket = reinterpret_cast<unsigned int *>(static_cast<uint8_t *>(scratch) + 8 * C);
  a.total = d_total_bytes;
  a.nbytes = nbytes;
  a.num_chunks = (uint32_t)C;
  a.candidates = PZ_CAND_ALL;
  a.stride = 1;
  return launch_encoder(a, elem_width == 2, false, C, C + 8, info, s);
}
