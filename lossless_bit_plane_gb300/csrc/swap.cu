// swap.cu — the compressed swap path: a tensor leaves device memory as
// PlaneZip streams in pinned host memory and comes back from them.
//
// Paper: "PlaneZip: Lossless Bit-Plane Compression of Training Activations
// Offloaded over PCIe" (arXiv:2610.25033v1), Section III-A (the engine
// compresses device-to-host swap copies and decompresses host-to-device
// ones; the compressed size of a swap is the sum of its chunk headers) and
// Section III-C, Equation 2 (a transfer is limited by the link or by the
// engine: the codec and the link work concurrently). Here the "engine" is
// the codec's kernels on the compute stream and the link is a copy stream:
// the tensor is cut into pieces, and while piece k+1 is being compressed
// (decompressed), piece k is on the link. Host code only; every byte is
// coded by the library's kernels and moved by cudaMemcpyAsync.
//
// Swap container in host memory (all fields little-endian):
//   bytes 0..31   u32 magic "PZSW", u32 piece count n, u64 nbytes,
//                 u64 piece_bytes, u32 elem_width, u32 zero
//   bytes 32..    u64 stream length of each piece (n entries)
//   then          the n piece streams, each a complete pz_compress stream of
//                 its piece's bytes, each starting at a 16-byte boundary.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "planezip.h"
#include "pz_kernels.h"

namespace {

constexpr uint32_t kMagic = 0x57535A50u;  // "PZSW"
constexpr size_t kHead = 32;

size_t align16(size_t v) { return (v + 15) & ~size_t(15); }
size_t pieces_of(size_t nbytes, size_t piece) { return nbytes ? (nbytes + piece - 1) / piece : 0; }
size_t table_end(size_t n) { return align16(kHead + 8 * n); }
bool piece_ok(size_t piece) { return piece >= 4096 && piece % 4096 == 0; }

// Two device staging buffers (each one piece's largest stream plus the
// encoder's scratch), then two stream-length words and one status word.
size_t stage_bytes(size_t piece) { return align16(pz_max_compressed_bytes(piece)); }

// The copy stream and events of the swap calls, created once per device and
// kept; a mutex per device serialises swap calls on that device (each call
// blocks the host until its copies are done, so they would not overlap).
struct Pipe {
  cudaStream_t copy = nullptr;
  cudaEvent_t coded[2] = {nullptr, nullptr};  // compute stream: piece coded (and its length copied)
  cudaEvent_t moved[2] = {nullptr, nullptr};  // copy stream: piece on the link done
  bool ok = false;
};
constexpr int kMaxDevices = 64;
std::mutex g_pipe_mu[kMaxDevices];
Pipe g_pipe[kMaxDevices];

// The current device's pipe, with its mutex held by `lk`; null on failure.
Pipe *device_pipe(std::unique_lock<std::mutex> &lk) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  lk = std::unique_lock<std::mutex>(g_pipe_mu[dev]);
  Pipe &p = g_pipe[dev];
  if (!p.ok) {
    bool ok = cudaStreamCreateWithFlags(&p.copy, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; i < 2 && ok; ++i)
      ok = cudaEventCreateWithFlags(&p.coded[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.moved[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return nullptr;
    p.ok = true;
  }
  return &p;
}

// Waits for the copy stream on every exit path of a call, so that no copy
// of the call is still in flight when it returns.
struct CopyDrain {
  cudaStream_t s;
  ~CopyDrain() { cudaStreamSynchronize(s); }
};

}  // namespace

extern "C" {

size_t pz_swap_work_bytes(size_t piece_bytes) {
  if (!piece_ok(piece_bytes)) return 0;
  return 2 * stage_bytes(piece_bytes) + 32;
}

size_t pz_swap_capacity(size_t nbytes, size_t piece_bytes) {
  if (!piece_ok(piece_bytes)) return 0;
  const size_t n = pieces_of(nbytes, piece_bytes);
  size_t cap = table_end(n);
  for (size_t k = 0; k < n; ++k) {
    const size_t raw = (k + 1 < n) ? piece_bytes : nbytes - k * piece_bytes;
    cap += align16(2 * ((raw + 4095) / 4096) + raw);
  }
  return cap;
}

pz_status pz_swap_out(const void *d_in, size_t nbytes, int elem_width, size_t piece_bytes, void *d_work,
                      size_t work_bytes, void *h_out, size_t h_capacity, size_t *h_total, pz_stream_t stream) {
  if (elem_width <= 0 || !h_out || !h_total || !piece_ok(piece_bytes)) return PZ_ERR_ARG;
  if (nbytes && (!d_in || !d_work)) return PZ_ERR_ARG;
  if (nbytes && ((reinterpret_cast<uintptr_t>(d_in) | reinterpret_cast<uintptr_t>(d_work)) & 15u)) return PZ_ERR_ARG;
  if (nbytes && work_bytes < pz_swap_work_bytes(piece_bytes)) return PZ_ERR_CAPACITY;
  if (h_capacity < pz_swap_capacity(nbytes, piece_bytes)) return PZ_ERR_CAPACITY;
  const size_t n = pieces_of(nbytes, piece_bytes);
  uint8_t *h = static_cast<uint8_t *>(h_out);
  std::memset(h, 0, table_end(n));
  const uint32_t head32[2] = {kMagic, (uint32_t)n};
  const uint64_t head64[2] = {nbytes, piece_bytes};
  const uint32_t tail32[2] = {(uint32_t)elem_width, 0u};
  std::memcpy(h, head32, 8);
  std::memcpy(h + 8, head64, 16);
  std::memcpy(h + 24, tail32, 8);
  *h_total = table_end(n);
  if (n == 0) return PZ_OK;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::unique_lock<std::mutex> lk;
  Pipe *pipe = device_pipe(lk);
  if (!pipe) return PZ_ERR_CUDA;
  Pipe &pp = *pipe;
  CopyDrain drain{pp.copy};
  uint8_t *work = static_cast<uint8_t *>(d_work);
  const size_t sb = stage_bytes(piece_bytes);
  uint8_t *stage[2] = {work, work + sb};
  unsigned long long *dlen = reinterpret_cast<unsigned long long *>(work + 2 * sb);
  uint64_t *table = reinterpret_cast<uint64_t *>(h + kHead);  // filled by device-to-host copies

  // code piece k into stage k%2: wait until the link has taken piece k-2
  // out of that stage, compress, and copy the stream length to the table
  auto code = [&](size_t k) -> pz_status {
    const int b = (int)(k & 1);
    if (k >= 2 && cudaStreamWaitEvent(s, pp.moved[b], 0) != cudaSuccess) return PZ_ERR_CUDA;
    const size_t raw = (k + 1 < n) ? piece_bytes : nbytes - k * piece_bytes;
    const pz_status st = pz_compress(static_cast<const uint8_t *>(d_in) + k * piece_bytes, raw, elem_width, stage[b],
                                     sb, dlen + b, stream);
    if (st != PZ_OK) return st;
    if (cudaMemcpyAsync(table + k, dlen + b, 8, cudaMemcpyDeviceToHost, s) != cudaSuccess) return PZ_ERR_CUDA;
    if (cudaEventRecord(pp.coded[b], s) != cudaSuccess) return PZ_ERR_CUDA;
    return PZ_OK;
  };

  pz_status st = code(0);
  if (st != PZ_OK) return st;
  size_t off = table_end(n);
  for (size_t k = 0; k < n; ++k) {
    if (k + 1 < n && (st = code(k + 1)) != PZ_OK) return st;  // the next piece codes while this one moves
    const int b = (int)(k & 1);
    if (cudaEventSynchronize(pp.coded[b]) != cudaSuccess) return PZ_ERR_CUDA;
    const uint64_t len = table[k];
    if (len == ~0ull) return PZ_ERR_TIMEOUT;
    if (off + len > h_capacity) return PZ_ERR_CAPACITY;  // cannot happen: len <= 2C + raw
    if (cudaMemcpyAsync(h + off, stage[b], len, cudaMemcpyDeviceToHost, pp.copy) != cudaSuccess) return PZ_ERR_CUDA;
    if (cudaEventRecord(pp.moved[b], pp.copy) != cudaSuccess) return PZ_ERR_CUDA;
    off += align16(len);
  }
  if (cudaStreamSynchronize(pp.copy) != cudaSuccess) return PZ_ERR_CUDA;
  *h_total = off;
  return PZ_OK;
}

pz_status pz_swap_in(const void *h_in, size_t h_bytes, void *d_work, size_t work_bytes, void *d_out, size_t nbytes,
                     int *d_status, pz_stream_t stream) {
  if (!h_in || !d_status || h_bytes < kHead) return PZ_ERR_ARG;
  const uint8_t *h = static_cast<const uint8_t *>(h_in);
  uint32_t head32[2], tail32[2];
  uint64_t head64[2];
  std::memcpy(head32, h, 8);
  std::memcpy(head64, h + 8, 16);
  std::memcpy(tail32, h + 24, 8);
  const size_t n = head32[1], piece = head64[1];
  const int elem_width = (int)tail32[0];
  if (head32[0] != kMagic || head64[0] != nbytes || !piece_ok(piece) || elem_width <= 0 ||
      n != pieces_of(nbytes, piece) || h_bytes < table_end(n))
    return PZ_ERR_ARG;
  if (nbytes && (!d_out || !d_work)) return PZ_ERR_ARG;
  if (nbytes && ((reinterpret_cast<uintptr_t>(d_out) | reinterpret_cast<uintptr_t>(d_work)) & 15u)) return PZ_ERR_ARG;
  if (nbytes && work_bytes < pz_swap_work_bytes(piece)) return PZ_ERR_CAPACITY;
  // piece offsets, checked against the container before anything is copied
  const uint64_t *table = reinterpret_cast<const uint64_t *>(h + kHead);
  const size_t sb = stage_bytes(piece);
  size_t off = table_end(n);
  for (size_t k = 0; k < n; ++k) {
    uint64_t len;
    std::memcpy(&len, table + k, 8);
    const size_t raw = (k + 1 < n) ? piece : nbytes - k * piece;
    if (len > sb || len < 2 * ((raw + 4095) / 4096) || off + len > h_bytes) return PZ_ERR_ARG;
    off += align16(len);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(d_status, 0, sizeof(int), s) != cudaSuccess) return PZ_ERR_CUDA;
  if (n == 0) return PZ_OK;

  std::unique_lock<std::mutex> lk;
  Pipe *pipe = device_pipe(lk);
  if (!pipe) return PZ_ERR_CUDA;
  Pipe &pp = *pipe;
  CopyDrain drain{pp.copy};
  uint8_t *work = static_cast<uint8_t *>(d_work);
  uint8_t *stage[2] = {work, work + sb};
  // the link may start as soon as the caller's earlier work is done
  if (cudaEventRecord(pp.coded[0], s) != cudaSuccess || cudaStreamWaitEvent(pp.copy, pp.coded[0], 0) != cudaSuccess)
    return PZ_ERR_CUDA;
  off = table_end(n);
  size_t offs[2] = {0, 0}, lens[2] = {0, 0};
  // move piece k into stage k%2 once piece k-2 has been decoded out of it
  auto move = [&](size_t k, size_t at) -> pz_status {
    const int b = (int)(k & 1);
    uint64_t len;
    std::memcpy(&len, table + k, 8);
    if (k >= 2 && cudaStreamWaitEvent(pp.copy, pp.coded[b], 0) != cudaSuccess) return PZ_ERR_CUDA;
    if (cudaMemcpyAsync(stage[b], h + at, len, cudaMemcpyHostToDevice, pp.copy) != cudaSuccess) return PZ_ERR_CUDA;
    if (cudaEventRecord(pp.moved[b], pp.copy) != cudaSuccess) return PZ_ERR_CUDA;
    offs[b] = at;
    lens[b] = len;
    return PZ_OK;
  };
  pz_status st = move(0, off);
  if (st != PZ_OK) return st;
  for (size_t k = 0; k < n; ++k) {
    const int b = (int)(k & 1);
    const size_t next = offs[b] + align16(lens[b]);
    if (k + 1 < n && (st = move(k + 1, next)) != PZ_OK) return st;  // the next piece moves while this one decodes
    if (cudaStreamWaitEvent(s, pp.moved[b], 0) != cudaSuccess) return PZ_ERR_CUDA;
    const size_t raw = (k + 1 < n) ? piece : nbytes - k * piece;
    st = pz::decompress_launch(stage[b], lens[b], elem_width, static_cast<uint8_t *>(d_out) + k * piece, raw,
                               d_status, stream, false);
    if (st != PZ_OK) return st;
    if (cudaEventRecord(pp.coded[b], s) != cudaSuccess) return PZ_ERR_CUDA;
  }
  // the copy stream's last copies have been waited for by the decodes; the
  // caller's stream orders everything that follows
  return PZ_OK;
}

}  // extern "C"
