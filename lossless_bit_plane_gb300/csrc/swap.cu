// swap.cu — the compressed swap path: a tensor leaves device memory as
// PlaneZip streams in pinned host memory and comes back from them, either
// into one caller buffer or into a pool of fixed-size host slots.
//
// Paper: "PlaneZip: Lossless Bit-Plane Compression of Training Activations
// Offloaded over PCIe" (arXiv:2610.25033v1), Section III-A (the engine
// compresses device-to-host swap copies and decompresses host-to-device
// ones; on the host, compressed tensors occupy fixed-size chunks of a pinned
// pool, so that their variable sizes do not fragment the allocator) and
// Section III-C, Equation 2 (a transfer is limited by the link or by the
// engine, and the runtime bypasses the engine when compression would not
// shorten the transfer). Here the "engine" is the codec's kernels on the
// caller's stream and the link is a copy stream: the tensor is cut into
// pieces, and while piece k+1 is being compressed (decompressed), piece k is
// on the link. Every byte is coded by the library's kernels and moved by
// cudaMemcpyAsync; the only device code here is a one-thread kernel that
// hands each piece's stream length to the host.
//
// Pieces: a first piece of half the largest piece P, then pieces of P, so
// that the first piece's coding (swap-out) or transfer (swap-in), which
// nothing overlaps, is shorter. Every piece is one codec call with a fixed
// latency of its own, so pieces stay large: a ramp of small pieces at both
// ends left the link idle behind latency-bound codec calls and was slower.
//
// Bypass: a piece whose stream would not be shorter than its raw bytes is
// moved raw (Equation 2 with a ratio c <= 1). On the device the codec is far
// faster than the host link (B_CE > gamma), so every other piece is coded.
//
// Swap container (all fields little-endian):
//   bytes 0..31     u32 magic "PZS3", u32 piece count n, u64 nbytes,
//                   u64 largest piece P, u32 elem_width, u32 zero
//   bytes 32..      n entries of 16 bytes: u64 raw bytes of the piece, u64
//                   stored bytes | (1 << 63 if the piece is stored raw)
//   then            the n pieces, each starting at a 128-byte boundary: the
//                   pz_compress stream of the piece's bytes, or the bytes.
// In a pool the container is laid over a chain of slots: byte x of the
// container is byte x % S of the (x / S)-th slot of the chain (S = slot
// size), so a piece may continue in the next slot.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "planezip.h"
#include "pz_kernels.h"

struct PoolHead;

namespace {

constexpr uint32_t kMagic = 0x33535A50u;  // "PZS3"
constexpr size_t kHead = 32;
constexpr size_t kEntry = 16;
constexpr uint64_t kRawFlag = 1ull << 63;

size_t align16(size_t v) { return (v + 15) & ~size_t(15); }
// Pieces start at 128-byte boundaries of the container: a host-to-device
// copy from a host address that is not 128-byte aligned measured 182 GB/s on
// NVLink-C2C against 210 GB/s aligned (device-to-host copies do not care).
constexpr size_t kPieceAlign = 128;
size_t align_piece(size_t v) { return (v + kPieceAlign - 1) & ~(kPieceAlign - 1); }
size_t table_end(size_t n) { return align_piece(kHead + kEntry * n); }
bool piece_ok(size_t piece) { return piece >= 4096 && piece % 4096 == 0; }

// Piece sizes of a swap of nbytes with largest piece P: a first piece of
// half of P (rounded down to 4096, at least 4096), then pieces of P, the
// last one possibly shorter.
std::vector<size_t> piece_sizes(size_t nbytes, size_t P) {
  std::vector<size_t> out;
  size_t rem = nbytes;
  for (size_t s = std::max<size_t>(4096, (P / 2) & ~size_t(4095)); rem; s = P) {
    const size_t a = std::min(s, rem);
    out.push_back(a);
    rem -= a;
  }
  return out;
}

// Two device staging buffers (each the largest piece's largest stream plus
// the encoder's scratch), then two stream-length words.
size_t stage_bytes(size_t piece) { return align16(pz_max_compressed_bytes(piece)); }

// The copy stream and events of the swap calls, created once per device and
// kept; a mutex per device serialises swap calls on that device.
struct Pipe {
  cudaStream_t copy = nullptr;
  cudaStream_t dec2 = nullptr;  // swap-in: the decodes out of stage 1 (stage 0's run on the caller's stream)
  cudaEvent_t coded[2] = {nullptr, nullptr};  // piece coded / decoded out of stage b
  cudaEvent_t moved[2] = {nullptr, nullptr};  // copy stream: stage b (or the raw piece) moved
  cudaEvent_t joined = nullptr;               // swap-in: the second decode stream's end
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
    bool ok = cudaStreamCreateWithFlags(&p.copy, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.dec2, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.joined, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < 2 && ok; ++i)
      ok = cudaEventCreateWithFlags(&p.coded[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.moved[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return nullptr;
    p.ok = true;
  }
  return &p;
}

// On an error return, waits for the copy stream so that no copy of the call
// is still in flight.
struct CopyDrain {
  cudaStream_t s;
  bool armed = true;
  ~CopyDrain() {
    if (armed) cudaStreamSynchronize(s);
  }
};

// A piece's stream length, from the encoder's total word into the
// container's table in pinned host memory mapped for the device: stored by
// the GPU, so that it does not queue on the copy engine behind the previous
// piece's copy to the host (an 8-byte cudaMemcpyAsync would, and the host
// needs the length before it can issue the piece's own copy).
__global__ void store_length_kernel(const unsigned long long *src, unsigned long long *dst) { *dst = *src; }

// The device address of host memory h if it is pinned and mapped, else null
// (pageable memory gets its lengths by cudaMemcpyAsync).
void *mapped_address(void *h) {
  cudaPointerAttributes at;
  void *d = nullptr;
  if (cudaPointerGetAttributes(&at, h) != cudaSuccess || at.type != cudaMemoryTypeHost ||
      cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess)
    d = nullptr;
  (void)cudaGetLastError();  // pageable memory is not an error of the call
  return d;
}

// ------------------------------------------------------------ host layout

// The container's host bytes: one caller buffer, or a chain of pool slots.
struct HostSpan {
  uint8_t *base = nullptr;  // one buffer of cap bytes
  size_t cap = 0;
  struct PoolHead *pool = nullptr;  // or a pool's slot chain
  std::vector<uint32_t> chain;

  // Host address of container byte x and the bytes that follow it in the
  // same buffer or slot.
  uint8_t *at(size_t x, size_t &run) const;
  // Make container bytes [0, end) addressable (pool: take slots).
  pz_status reserve(size_t end);
  // Zero container bytes [x, x + len) on the host (the padding after a
  // piece, so that a container's bytes depend on the tensor alone).
  void zero(size_t x, size_t len) const {
    while (len) {
      size_t run = 0;
      uint8_t *h = at(x, run);
      const size_t m = std::min(run, len);
      std::memset(h, 0, m);
      x += m;
      len -= m;
    }
  }
  // One copy per contiguous run between container bytes [x, x + len) and a
  // device buffer.
  pz_status copy(size_t x, void *dev, size_t len, cudaMemcpyKind kind, cudaStream_t s) const {
    while (len) {
      size_t run = 0;
      uint8_t *h = at(x, run);
      const size_t m = std::min(run, len);
      const cudaError_t e = (kind == cudaMemcpyDeviceToHost) ? cudaMemcpyAsync(h, dev, m, kind, s)
                                                              : cudaMemcpyAsync(dev, h, m, kind, s);
      if (e != cudaSuccess) return PZ_ERR_CUDA;
      x += m;
      len -= m;
      dev = static_cast<uint8_t *>(dev) + m;
    }
    return PZ_OK;
  }
};

}  // namespace

// ------------------------------------------------------------------ pool

// A pool laid out in caller-provided host memory: this head, the slots'
// next links (u32, kNone ends a chain), then the slots, 4096-aligned. Free
// slots form one chain from free_head.
struct PoolHead {
  uint64_t magic;
  uint64_t slot_bytes;
  uint64_t nslots;
  uint64_t data_off;  // slot 0, from the head
  uint32_t free_head;
  uint32_t nfree;
  std::mutex mu;
  uint32_t *next() { return reinterpret_cast<uint32_t *>(this + 1); }
  uint8_t *slot(uint32_t i) { return reinterpret_cast<uint8_t *>(this) + data_off + (uint64_t)i * slot_bytes; }
};
struct pz_pool_s : PoolHead {};

namespace {

constexpr uint64_t kPoolMagic = 0x31304C4F4F505A50ull;  // "PZPOOL01"
constexpr uint32_t kNone = 0xFFFFFFFFu;

size_t pool_data_off(size_t nslots) { return (sizeof(PoolHead) + 4 * nslots + 4095) & ~size_t(4095); }

uint8_t *HostSpan::at(size_t x, size_t &run) const {
  if (base) {
    run = cap - x;
    return base + x;
  }
  const size_t S = pool->slot_bytes;
  run = S - x % S;
  return pool->slot(chain[x / S]) + x % S;
}

pz_status HostSpan::reserve(size_t end) {
  if (base) return end <= cap ? PZ_OK : PZ_ERR_CAPACITY;
  const size_t need = (end + pool->slot_bytes - 1) / pool->slot_bytes;
  if (need <= chain.size()) return PZ_OK;
  std::lock_guard<std::mutex> lk(pool->mu);
  if (need - chain.size() > pool->nfree) return PZ_ERR_CAPACITY;
  uint32_t *nx = pool->next();
  while (chain.size() < need) {
    const uint32_t s = pool->free_head;
    pool->free_head = nx[s];
    --pool->nfree;
    nx[s] = kNone;
    if (!chain.empty()) nx[chain.back()] = s;
    chain.push_back(s);
  }
  return PZ_OK;
}

void pool_release_chain(PoolHead *pool, uint32_t first) {
  std::lock_guard<std::mutex> lk(pool->mu);
  uint32_t *nx = pool->next();
  for (uint32_t s = first; s != kNone;) {
    const uint32_t n = nx[s];
    nx[s] = pool->free_head;
    pool->free_head = s;
    ++pool->nfree;
    s = n;
  }
}

// ------------------------------------------------------------- swap out

// Compress nbytes at d_in piece by piece into the container `span` (head,
// table, pieces). Blocks until the container is complete: each piece's
// stored length is needed on the host before its copy can be issued.
pz_status swap_out_core(HostSpan &span, const void *d_in, size_t nbytes, int elem_width, size_t P, void *d_work,
                        size_t *h_total, cudaStream_t s) {
  const std::vector<size_t> sizes = piece_sizes(nbytes, P);
  const size_t n = sizes.size();
  pz_status st = span.reserve(table_end(n));
  if (st != PZ_OK) return st;
  size_t run = 0;
  uint8_t *h = span.at(0, run);
  if (run < table_end(n)) return PZ_ERR_CAPACITY;  // the head and table lie in the first buffer or slot
  std::memset(h, 0, table_end(n));
  const uint32_t head32[2] = {kMagic, (uint32_t)n};
  const uint64_t head64[2] = {nbytes, P};
  const uint32_t tail32[2] = {(uint32_t)elem_width, 0u};
  std::memcpy(h, head32, 8);
  std::memcpy(h + 8, head64, 16);
  std::memcpy(h + 24, tail32, 8);
  uint64_t *table = reinterpret_cast<uint64_t *>(h + kHead);  // entry k: table[2k] raw, table[2k+1] stored
  for (size_t k = 0; k < n; ++k) table[2 * k] = sizes[k];
  *h_total = table_end(n);
  if (n == 0) return PZ_OK;
  unsigned long long *table_dev = static_cast<unsigned long long *>(mapped_address(table));

  std::unique_lock<std::mutex> lk;
  Pipe *pipe = device_pipe(lk);
  if (!pipe) return PZ_ERR_CUDA;
  Pipe &pp = *pipe;
  CopyDrain drain{pp.copy};
  uint8_t *work = static_cast<uint8_t *>(d_work);
  const size_t sb = stage_bytes(P);
  uint8_t *stage[2] = {work, work + sb};
  unsigned long long *dlen = reinterpret_cast<unsigned long long *>(work + 2 * sb);
  const uint8_t *in = static_cast<const uint8_t *>(d_in);

  // code piece k into stage k%2: wait until the link has taken piece k-2
  // out of that stage, compress, and copy the stream length to the table
  auto code = [&](size_t k, size_t at) -> pz_status {
    const int b = (int)(k & 1);
    if (k >= 2 && cudaStreamWaitEvent(s, pp.moved[b], 0) != cudaSuccess) return PZ_ERR_CUDA;
    const pz_status cs = pz_compress(in + at, sizes[k], elem_width, stage[b], sb, dlen + b, s);
    if (cs != PZ_OK) return cs;
    if (table_dev) {
      const unsigned long long *src = dlen + b;
      unsigned long long *dst = table_dev + 2 * k + 1;
      void *args[2] = {&src, &dst};
      if (cudaLaunchKernel(reinterpret_cast<const void *>(&store_length_kernel), dim3(1), dim3(1), args, 0, s) !=
          cudaSuccess)
        return PZ_ERR_CUDA;
    } else if (cudaMemcpyAsync(table + 2 * k + 1, dlen + b, 8, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
      return PZ_ERR_CUDA;
    }
    if (cudaEventRecord(pp.coded[b], s) != cudaSuccess) return PZ_ERR_CUDA;
    return PZ_OK;
  };

  if ((st = code(0, 0)) != PZ_OK) return st;
  size_t off = table_end(n), src = 0;
  for (size_t k = 0; k < n; ++k) {
    if (k + 1 < n && (st = code(k + 1, src + sizes[k])) != PZ_OK) return st;  // the next piece codes while this one moves
    const int b = (int)(k & 1);
    if (cudaEventSynchronize(pp.coded[b]) != cudaSuccess) return PZ_ERR_CUDA;
    const uint64_t len = table[2 * k + 1];
    if (len == ~0ull) return PZ_ERR_TIMEOUT;
    const bool raw = len >= sizes[k];  // compression would not shorten it: move the bytes
    const size_t stored = raw ? sizes[k] : (size_t)len;
    table[2 * k + 1] = stored | (raw ? kRawFlag : 0ull);
    if ((st = span.reserve(off + stored)) != PZ_OK) return st;
    // a raw piece is moved from d_in: its stage is free at once
    if (raw && cudaEventRecord(pp.moved[b], pp.copy) != cudaSuccess) return PZ_ERR_CUDA;
    if ((st = span.copy(off, raw ? const_cast<uint8_t *>(in + src) : stage[b], stored, cudaMemcpyDeviceToHost,
                        pp.copy)) != PZ_OK)
      return st;
    if (!raw && cudaEventRecord(pp.moved[b], pp.copy) != cudaSuccess) return PZ_ERR_CUDA;
    const size_t pad = align_piece(stored) - stored;  // outside the bytes the copy writes
    if (pad) {
      if ((st = span.reserve(off + stored + pad)) != PZ_OK) return st;
      span.zero(off + stored, pad);
    }
    off += align_piece(stored);
    src += sizes[k];
  }
  if (cudaStreamSynchronize(pp.copy) != cudaSuccess) return PZ_ERR_CUDA;
  drain.armed = false;
  *h_total = off;
  return PZ_OK;
}

// -------------------------------------------------------------- swap in

// Check the container's head and table against nbytes and its bytes; fills
// the piece sizes and stored lengths. PZ_ERR_ARG if anything disagrees.
pz_status read_table(const HostSpan &span, size_t h_bytes, size_t nbytes, int &elem_width, size_t &P,
                     std::vector<uint64_t> &raw, std::vector<uint64_t> &stored) {
  if (h_bytes < kHead) return PZ_ERR_ARG;
  size_t run = 0;
  const uint8_t *h = span.at(0, run);
  if (run < kHead) return PZ_ERR_ARG;
  uint32_t head32[2], tail32[2];
  uint64_t head64[2];
  std::memcpy(head32, h, 8);
  std::memcpy(head64, h + 8, 16);
  std::memcpy(tail32, h + 24, 8);
  const size_t n = head32[1];
  P = head64[1];
  elem_width = (int)tail32[0];
  if (head32[0] != kMagic || head64[0] != nbytes || !piece_ok(P) || elem_width <= 0 || tail32[1] != 0 ||
      table_end(n) > std::min(run, h_bytes))
    return PZ_ERR_ARG;
  raw.resize(n);
  stored.resize(n);
  size_t off = table_end(n), sum = 0;
  for (size_t k = 0; k < n; ++k) {
    uint64_t e[2];
    std::memcpy(e, h + kHead + kEntry * k, 16);
    const uint64_t len = e[1] & ~kRawFlag;
    const bool is_raw = (e[1] & kRawFlag) != 0;
    const uint64_t C = (e[0] + 4095) / 4096;
    if (e[0] == 0 || e[0] > P || (is_raw ? len != e[0] : (len >= e[0] || len < 2 * C)) || off + len > h_bytes)
      return PZ_ERR_ARG;
    raw[k] = e[0];
    stored[k] = e[1];
    sum += e[0];
    off += align_piece(len);
  }
  return sum == nbytes ? PZ_OK : PZ_ERR_ARG;
}

// Move the pieces back and decode them into d_out. Returns once everything is
// enqueued: the caller's stream completes the call (the host bytes must stay
// unchanged until it has).
pz_status swap_in_core(const HostSpan &span, size_t h_bytes, void *d_work, size_t work_bytes, void *d_out,
                       size_t nbytes, int *d_status, cudaStream_t s) {
  int elem_width = 0;
  size_t P = 0;
  std::vector<uint64_t> raw, stored;
  pz_status st = read_table(span, h_bytes, nbytes, elem_width, P, raw, stored);
  if (st != PZ_OK) return st;
  const size_t n = raw.size();
  if (nbytes && (!d_out || !d_work)) return PZ_ERR_ARG;
  if (nbytes && ((reinterpret_cast<uintptr_t>(d_out) | reinterpret_cast<uintptr_t>(d_work)) & 15u)) return PZ_ERR_ARG;
  if (nbytes && work_bytes < pz_swap_work_bytes(P)) return PZ_ERR_CAPACITY;
  if (cudaMemsetAsync(d_status, 0, sizeof(int), s) != cudaSuccess) return PZ_ERR_CUDA;
  if (n == 0) return PZ_OK;

  std::unique_lock<std::mutex> lk;
  Pipe *pipe = device_pipe(lk);
  if (!pipe) return PZ_ERR_CUDA;
  Pipe &pp = *pipe;
  CopyDrain drain{pp.copy};
  uint8_t *work = static_cast<uint8_t *>(d_work);
  const size_t sb = stage_bytes(P);
  uint8_t *stage[2] = {work, work + sb};
  uint8_t *out = static_cast<uint8_t *>(d_out);
  // the link and the second decode stream may start as soon as the
  // caller's earlier work is done
  if (cudaEventRecord(pp.coded[0], s) != cudaSuccess || cudaStreamWaitEvent(pp.copy, pp.coded[0], 0) != cudaSuccess ||
      cudaStreamWaitEvent(pp.dec2, pp.coded[0], 0) != cudaSuccess)
    return PZ_ERR_CUDA;
  CopyDrain drain2{pp.dec2};
  std::vector<size_t> at(n + 1), dst(n + 1);
  at[0] = table_end(n);
  dst[0] = 0;
  for (size_t k = 0; k < n; ++k) {
    at[k + 1] = at[k] + align_piece(stored[k] & ~kRawFlag);
    dst[k + 1] = dst[k] + raw[k];
  }
  // The coded pieces alternate between the two stages (the j-th coded piece
  // in stage j%2), and the decodes out of stage 1 run on a second stream, so
  // that one piece's walk may overlap the previous piece's decode. A coded
  // piece is moved into its stage once the coded piece two before it has
  // been decoded out of that stage; a raw piece is moved straight to its
  // place in d_out and waits for nothing.
  std::vector<int> sidx(n, -1);
  for (size_t k = 0, j = 0; k < n; ++k)
    if (!(stored[k] & kRawFlag)) sidx[k] = (int)(j++);
  // A run of raw pieces lies back to back in the container (a raw piece is
  // a multiple of 4096 bytes, the last one excepted) and in d_out: the first
  // piece of the run moves the whole run with one copy, the others nothing.
  // (Measured as fast as one copy per piece; kept for the fewer calls.)
  std::vector<size_t> run_bytes(n, 0);
  for (size_t k = n; k-- > 0;)
    if (stored[k] & kRawFlag)
      run_bytes[k] = raw[k] + ((k + 1 < n && (stored[k + 1] & kRawFlag) && at[k + 1] == at[k] + raw[k])
                                   ? run_bytes[k + 1]
                                   : 0);
  auto move = [&](size_t k) -> pz_status {
    if (stored[k] & kRawFlag) {
      const bool continues = k > 0 && (stored[k - 1] & kRawFlag) && at[k] == at[k - 1] + raw[k - 1];
      return continues ? PZ_OK : span.copy(at[k], out + dst[k], run_bytes[k], cudaMemcpyHostToDevice, pp.copy);
    }
    const int j = sidx[k], b = j & 1;
    if (j >= 2 && cudaStreamWaitEvent(pp.copy, pp.coded[b], 0) != cudaSuccess) return PZ_ERR_CUDA;
    const pz_status cs = span.copy(at[k], stage[b], stored[k], cudaMemcpyHostToDevice, pp.copy);
    if (cs != PZ_OK) return cs;
    if (cudaEventRecord(pp.moved[b], pp.copy) != cudaSuccess) return PZ_ERR_CUDA;
    return PZ_OK;
  };
  if ((st = move(0)) != PZ_OK) return st;
  for (size_t k = 0; k < n; ++k) {
    if (k + 1 < n && (st = move(k + 1)) != PZ_OK) return st;  // the next piece moves while this one decodes
    if (stored[k] & kRawFlag) continue;
    const int b = sidx[k] & 1;
    const cudaStream_t ds = b ? pp.dec2 : s;
    if (cudaStreamWaitEvent(ds, pp.moved[b], 0) != cudaSuccess) return PZ_ERR_CUDA;
    st = pz::decompress_launch(stage[b], stored[k], elem_width, out + dst[k], raw[k], d_status, ds, false);
    if (st != PZ_OK) return st;
    if (cudaEventRecord(pp.coded[b], ds) != cudaSuccess) return PZ_ERR_CUDA;
  }
  // the caller's stream waits for the second decode stream
  if (cudaEventRecord(pp.joined, pp.dec2) != cudaSuccess || cudaStreamWaitEvent(s, pp.joined, 0) != cudaSuccess)
    return PZ_ERR_CUDA;
  // the caller's stream waits for the last copies (the raw pieces' too)
  if (cudaEventRecord(pp.moved[0], pp.copy) != cudaSuccess || cudaStreamWaitEvent(s, pp.moved[0], 0) != cudaSuccess)
    return PZ_ERR_CUDA;
  drain.armed = false;
  drain2.armed = false;
  return PZ_OK;
}

bool out_args_ok(const void *d_in, size_t nbytes, int elem_width, size_t piece_bytes, const void *d_work) {
  if (elem_width <= 0 || !piece_ok(piece_bytes)) return false;
  if (nbytes && (!d_in || !d_work)) return false;
  if (nbytes && ((reinterpret_cast<uintptr_t>(d_in) | reinterpret_cast<uintptr_t>(d_work)) & 15u)) return false;
  return true;
}

}  // namespace

extern "C" {

size_t pz_swap_work_bytes(size_t piece_bytes) {
  if (!piece_ok(piece_bytes)) return 0;
  return 2 * stage_bytes(piece_bytes) + 32;
}

size_t pz_swap_capacity(size_t nbytes, size_t piece_bytes) {
  if (!piece_ok(piece_bytes)) return 0;
  const std::vector<size_t> sizes = piece_sizes(nbytes, piece_bytes);
  size_t cap = table_end(sizes.size());
  for (size_t r : sizes) cap += align_piece(r);  // a piece never stores more than its raw bytes
  return cap;
}

pz_status pz_swap_out(const void *d_in, size_t nbytes, int elem_width, size_t piece_bytes, void *d_work,
                      size_t work_bytes, void *h_out, size_t h_capacity, size_t *h_total, pz_stream_t stream) {
  if (!h_out || !h_total || !out_args_ok(d_in, nbytes, elem_width, piece_bytes, d_work)) return PZ_ERR_ARG;
  if (nbytes && work_bytes < pz_swap_work_bytes(piece_bytes)) return PZ_ERR_CAPACITY;
  if (h_capacity < pz_swap_capacity(nbytes, piece_bytes)) return PZ_ERR_CAPACITY;
  HostSpan span;
  span.base = static_cast<uint8_t *>(h_out);
  span.cap = h_capacity;
  return swap_out_core(span, d_in, nbytes, elem_width, piece_bytes, d_work, h_total,
                       reinterpret_cast<cudaStream_t>(stream));
}

pz_status pz_swap_in(const void *h_in, size_t h_bytes, void *d_work, size_t work_bytes, void *d_out, size_t nbytes,
                     int *d_status, pz_stream_t stream) {
  if (!h_in || !d_status) return PZ_ERR_ARG;
  HostSpan span;
  span.base = const_cast<uint8_t *>(static_cast<const uint8_t *>(h_in));
  span.cap = h_bytes;
  return swap_in_core(span, h_bytes, d_work, work_bytes, d_out, nbytes, d_status,
                      reinterpret_cast<cudaStream_t>(stream));
}

size_t pz_pool_bytes(size_t slot_bytes, size_t nslots) {
  if (!piece_ok(slot_bytes) || nslots == 0 || nslots >= kNone) return 0;
  return pool_data_off(nslots) + nslots * slot_bytes;
}

pz_status pz_pool_init(void *h_mem, size_t bytes, size_t slot_bytes, pz_pool **pool) {
  if (!h_mem || !pool || !piece_ok(slot_bytes) || (reinterpret_cast<uintptr_t>(h_mem) & 63u)) return PZ_ERR_ARG;
  // the largest slot count whose layout fits in `bytes`
  size_t nslots = bytes / slot_bytes;
  while (nslots && pz_pool_bytes(slot_bytes, nslots) > bytes) --nslots;
  if (nslots == 0 || nslots >= kNone) return PZ_ERR_CAPACITY;
  PoolHead *p = new (h_mem) pz_pool_s();
  p->magic = kPoolMagic;
  p->slot_bytes = slot_bytes;
  p->nslots = nslots;
  p->data_off = pool_data_off(nslots);
  uint32_t *nx = p->next();
  for (size_t i = 0; i < nslots; ++i) nx[i] = (i + 1 < nslots) ? (uint32_t)(i + 1) : kNone;
  p->free_head = 0;
  p->nfree = (uint32_t)nslots;
  *pool = static_cast<pz_pool *>(p);
  return PZ_OK;
}

size_t pz_pool_free_slots(pz_pool *pool) {
  if (!pool || pool->magic != kPoolMagic) return 0;
  std::lock_guard<std::mutex> lk(pool->mu);
  return pool->nfree;
}

pz_status pz_pool_swap_out(pz_pool *pool, const void *d_in, size_t nbytes, int elem_width, size_t piece_bytes,
                           void *d_work, size_t work_bytes, unsigned int *tensor, size_t *stored_bytes,
                           pz_stream_t stream) {
  if (!pool || pool->magic != kPoolMagic || !tensor || !out_args_ok(d_in, nbytes, elem_width, piece_bytes, d_work))
    return PZ_ERR_ARG;
  if (nbytes && work_bytes < pz_swap_work_bytes(piece_bytes)) return PZ_ERR_CAPACITY;
  if (table_end(piece_sizes(nbytes, piece_bytes).size()) > pool->slot_bytes) return PZ_ERR_ARG;
  HostSpan span;
  span.pool = pool;
  size_t total = 0;
  const pz_status st = swap_out_core(span, d_in, nbytes, elem_width, piece_bytes, d_work, &total,
                                     reinterpret_cast<cudaStream_t>(stream));
  if (st != PZ_OK) {
    if (!span.chain.empty()) pool_release_chain(pool, span.chain.front());
    return st;
  }
  *tensor = span.chain.front();
  if (stored_bytes) *stored_bytes = total;
  return PZ_OK;
}

pz_status pz_pool_swap_in(pz_pool *pool, unsigned int tensor, void *d_work, size_t work_bytes, void *d_out,
                          size_t nbytes, int *d_status, pz_stream_t stream) {
  if (!pool || pool->magic != kPoolMagic || !d_status || tensor >= pool->nslots) return PZ_ERR_ARG;
  HostSpan span;
  span.pool = pool;
  {  // the tensor's slot chain (a chain longer than the pool is not one)
    std::lock_guard<std::mutex> lk(pool->mu);
    const uint32_t *nx = pool->next();
    for (uint32_t s = tensor; s != kNone; s = nx[s]) {
      if (s >= pool->nslots || span.chain.size() >= pool->nslots) return PZ_ERR_ARG;
      span.chain.push_back(s);
    }
  }
  return swap_in_core(span, span.chain.size() * pool->slot_bytes, d_work, work_bytes, d_out, nbytes, d_status,
                      reinterpret_cast<cudaStream_t>(stream));
}

pz_status pz_pool_release(pz_pool *pool, unsigned int tensor) {
  if (!pool || pool->magic != kPoolMagic || tensor >= pool->nslots) return PZ_ERR_ARG;
  {  // a tensor's first slot starts with its container's head; clearing it
     // makes a second release of the same handle an error
    std::lock_guard<std::mutex> lk(pool->mu);
    uint32_t magic = 0;
    std::memcpy(&magic, pool->slot(tensor), 4);
    if (magic != kMagic) return PZ_ERR_ARG;
    std::memset(pool->slot(tensor), 0, 4);
  }
  pool_release_chain(pool, tensor);
  return PZ_OK;
}

}  // extern "C"
