/*
 * planezip.h — C ABI of the PlaneZip block codec on GB300 (sm_103a).
 *
 * The codec is the one of "PlaneZip: Lossless Bit-Plane Compression of
 * Training Activations Offloaded over PCIe" (arXiv:2610.25033v1),
 * Section III-A "Codec" and "Stream format": a tensor is cut into 128-byte
 * blocks, each block is coded as the smallest of ZVC, DBX, BX, ZBX and the
 * raw block behind a 3-bit tag, and 32 blocks form a 4 KB chunk that is
 * byte-aligned, carries a 16-bit size, and is stored raw if coding would
 * grow it.
 *
 * Stream layout produced and consumed here (for nbytes of input, C chunks):
 *   bytes [0, 2C)            C little-endian uint16 chunk sizes L_c
 *   bytes [2C, 2C + sum L)   chunk payloads, concatenated, byte-aligned
 * A chunk with L_c equal to its raw size (4096, or the tail size for the
 * last chunk) is stored verbatim. The bit-level format (field orders, code
 * patterns, tie-breaks) is written out in
 * lossless_bit_plane_gb300/csrc/pz_format.cuh.
 *
 * Conventions for every call:
 *   - "d_" pointers are DEVICE pointers of the current CUDA device; the
 *     caller owns every buffer. The calls allocate nothing.
 *   - Work is enqueued on `stream` and the call returns without waiting;
 *     device-side results are valid after the stream is synchronized.
 *   - A non-PZ_OK return means nothing was enqueued (argument errors) or a
 *     launch failed (PZ_ERR_CUDA, with the CUDA error left to the caller's
 *     next cudaGetLastError()).
 *   - Thread-safe and stateless apart from per-device caches of device
 *     attributes and of the driver's tensor-map encoder.
 */
#ifndef PLANEZIP_H
#define PLANEZIP_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *pz_stream_t; /* == cudaStream_t; NULL = legacy default stream */

typedef enum {
  PZ_OK = 0,
  PZ_ERR_ARG = 1,      /* null pointer, bad width, misaligned pointer, stream too short */
  PZ_ERR_CAPACITY = 2, /* out_capacity below pz_max_compressed_bytes(nbytes) */
  PZ_ERR_CORRUPT = 3,  /* (device status) malformed compressed stream */
  PZ_ERR_CUDA = 4,     /* a CUDA launch or memset failed */
  PZ_ERR_TIMEOUT = 5   /* (device status) an inter-chunk wait hit its iteration limit */
} pz_status;

/* Bytes the caller must allocate for pz_compress's output buffer when
 * compressing nbytes: the largest stream, 2*C + nbytes (every chunk raw),
 * rounded up to 16, plus the encoder's scratch area (8 bytes per chunk + 64)
 * that lives in the tail of the same buffer. Host-only, pure function.
 * Source: Section III-A "Stream format" (16-bit size per chunk; a chunk that
 * would grow is stored raw, so the stream never exceeds 2*C + nbytes). */
size_t pz_max_compressed_bytes(size_t nbytes);

/* Compress nbytes at d_in into d_out.
 * Source: Section III-A "Codec" (block split, symbol width from the element
 * type, the five candidates, smallest kept with a 3-bit tag) and "Stream
 * format" (chunks, headers, raw fallback, prefix-sum location).
 *   d_in          device, >= nbytes readable; 16-byte aligned.
 *   nbytes        input size in bytes; any value (0 gives an empty stream).
 *   elem_width    element size in bytes: 2 selects 16-bit symbols (BF16,
 *                 64 per block); any other positive value selects 32-bit
 *                 symbols (FP32 and all other types, 32 per block).
 *   d_out         device, out_capacity bytes; 16-byte aligned. Receives the
 *                 stream in [0, *d_total_bytes); bytes past the stream are
 *                 scratch and are left unspecified.
 *   out_capacity  must be >= pz_max_compressed_bytes(nbytes).
 *   d_total_bytes device uint64: set to the stream length 2*C + sum(L)
 *                 (the compressed size the paper's engine reports, Section
 *                 III-B), or to UINT64_MAX if a device-side wait timed out.
 *   stream        CUDA stream.
 * Errors: PZ_ERR_ARG (null/misaligned pointer, elem_width <= 0),
 * PZ_ERR_CAPACITY, PZ_ERR_CUDA. Calls that overlap on the GPU must use
 * distinct d_out buffers. */
pz_status pz_compress(const void *d_in, size_t nbytes, int elem_width,
                      void *d_out, size_t out_capacity,
                      unsigned long long *d_total_bytes, pz_stream_t stream);

/* Decompress a stream produced by pz_compress (or the identical CPU
 * oracle) back into nbytes at d_out.
 * Source: Section III-A "Stream format" (chunks located by a prefix sum
 * over the headers and decoded in parallel) and the inverse of each
 * candidate of Section III-A "Codec".
 *   d_in        device, 16-byte aligned; readable up to comp_bytes rounded
 *               up to a multiple of 16 (the decoder copies whole 16-byte
 *               units into shared memory; an allocation of comp_bytes from
 *               cudaMalloc or PyTorch always covers that).
 *   comp_bytes  bytes available at d_in: >= 2*C, and the stream's own
 *               length 2*C + sum(L) must not exceed it (trailing bytes are
 *               ignored).
 *   elem_width  the width given to pz_compress.
 *   d_out       device, nbytes writable; 16-byte aligned. Only [0, nbytes)
 *               is written.
 *   nbytes      the original size.
 *   d_status    device int: set to PZ_OK, or PZ_ERR_CORRUPT if any field of
 *               the stream is malformed (bad size, tag, code, position,
 *               overrun, non-zero padding), or PZ_ERR_TIMEOUT if a
 *               device-side wait for a copy into shared memory hit its
 *               iteration limit (the larger code wins). The output is then
 *               unspecified but no byte outside [0, nbytes) is written, and
 *               reads stay inside the 16-byte-aligned granules that
 *               [0, comp_bytes) touches.
 * Errors: PZ_ERR_ARG (null/misaligned pointer, elem_width <= 0,
 * comp_bytes < 2*C), PZ_ERR_CUDA. */
pz_status pz_decompress(const void *d_in, size_t comp_bytes, int elem_width,
                        void *d_out, size_t nbytes, int *d_status,
                        pz_stream_t stream);

/* Candidate masks for block selection: bit t allows the encoding with tag t
 * (Section III-A "Codec": ZVC 0, DBX 1, BX 2, ZBX 3, raw 4). The raw block is
 * always allowed, so every mask gives a valid stream in the same format. */
#define PZ_CAND_ZVC 0x01u
#define PZ_CAND_DBX 0x02u
#define PZ_CAND_BX 0x04u
#define PZ_CAND_ZBX 0x08u
#define PZ_CAND_RAW 0x10u
#define PZ_CAND_ALL 0x1Fu

/* pz_compress with block selection restricted to `candidates` (a mask of
 * PZ_CAND_* bits; PZ_CAND_RAW is implied): each block keeps the smallest
 * ALLOWED candidate, ties to the lowest tag; chunks that would grow are
 * still stored raw. PZ_CAND_ALL is pz_compress. The stream decodes with
 * pz_decompress like any other.
 * Source: Section V-A "Compression Ratio" and Fig. 3, which compare PlaneZip
 * with single encodings applied to every block (ZVC as in cDMA; BPC = DBX on
 * every block; the best single encoding) -- PZ_CAND_ZVC, PZ_CAND_DBX, ...
 * reproduce those columns on the same data. Arguments, buffers, capacity and
 * errors as pz_compress; a mask with bits outside PZ_CAND_ALL gives
 * PZ_ERR_ARG. */
pz_status pz_compress_candidates(const void *d_in, size_t nbytes, int elem_width,
                                 unsigned int candidates, void *d_out,
                                 size_t out_capacity,
                                 unsigned long long *d_total_bytes,
                                 pz_stream_t stream);

/* Compressed sizes only: no stream is written and no scratch is used.
 * Visits chunks 0, s, 2s, ... (s = chunk_stride >= 1) and reports
 *   d_sizes[k]  (device, u16, ceil(C/s) entries; may be NULL): the size L of
 *               chunk k*s, exactly the header pz_compress_candidates writes
 *               for it with the same candidates;
 *   *d_total    (device u64): the sum over the visited chunks of 2 + L, i.e.
 *               the full stream length 2*C + sum(L) when s = 1 (the total
 *               pz_compress reports), or UINT64_MAX if a device-side wait
 *               timed out.
 * With s > 1 the ratio estimate is (raw bytes of the visited chunks) /
 * *d_total; the host knows the former: s = 4 on tensors above 32 MB is the
 * paper's sampling.
 * Source: Section III-B "Compressibility Predictor" (the engine reports a
 * tensor's compressed size as the sum of its chunk headers; tensors that are
 * not swapped are measured in a profiling iteration that compresses into a
 * scratch buffer and discards the output -- this computes the same sizes
 * without the output) and Section IV "Methodology", "Tensor capture"
 * (tensors above 32 MB are compressed on every fourth 4 KB chunk).
 *   d_in, nbytes, elem_width, candidates: as pz_compress_candidates.
 * Errors: PZ_ERR_ARG (null/misaligned d_in with nbytes > 0, null d_total,
 * elem_width <= 0, chunk_stride == 0, bad mask), PZ_ERR_CUDA. */
pz_status pz_compressed_size(const void *d_in, size_t nbytes, int elem_width,
                             unsigned int candidates, unsigned int chunk_stride,
                             unsigned short *d_sizes,
                             unsigned long long *d_total, pz_stream_t stream);

/* ------------------------------------------------------------------------
 * The compressed swap path. A tensor is swapped out to host memory as
 * PlaneZip streams and swapped back in from them; the codec and the host
 * link work at the same time (Section III-A: the engine compresses
 * device-to-host swaps and decompresses host-to-device ones; Section III-C,
 * Equation 2: a transfer is limited by the link or by the engine, whichever
 * is slower, and the runtime bypasses the engine when compression would not
 * shorten the transfer). The tensor is cut into pieces of at most
 * piece_bytes (a multiple of 4096): a first piece of half that size (so
 * that the first step, which nothing overlaps, is shorter), then pieces of
 * piece_bytes. Piece k+1 is coded on `stream` while piece k is on the link
 * (an internal copy stream). A piece whose stream would not be shorter than its bytes is
 * moved raw. Host memory should be pinned for the copies to overlap
 * (pageable memory works, serialised).
 *
 * Container (little-endian): a 32-byte head (u32 "PZS3", u32 pieces n, u64
 * nbytes, u64 piece_bytes, u32 elem_width, u32 0), n entries of 16 bytes
 * (u64 raw bytes of the piece; u64 stored bytes, bit 63 set when the piece
 * is stored raw), then each piece -- its pz_compress stream, or its bytes --
 * at a 128-byte boundary of the container, the bytes between pieces zero (a
 * copy to the device from a host address that is not 128-byte aligned is
 * slower; give h_out, or the pool's memory, a 128-byte aligned start).
 *
 * Swap-out blocks the host until the container is complete (each piece's
 * stored length is needed on the host to copy it). Swap-in only enqueues:
 * the host bytes must stay unchanged until `stream` has completed the call.
 * Calls that share d_work must be ordered on the same stream.
 * ---------------------------------------------------------------------- */

/* Device staging bytes both calls need for piece_bytes (0 if piece_bytes is
 * not a positive multiple of 4096): two pieces' largest streams plus the
 * encoder's scratch. Host-only, pure. */
size_t pz_swap_work_bytes(size_t piece_bytes);

/* Host bytes pz_swap_out may write for nbytes in pieces of at most
 * piece_bytes (0 for an invalid piece size): the head and table plus every
 * piece's raw bytes, each rounded up to 128. Host-only, pure. */
size_t pz_swap_capacity(size_t nbytes, size_t piece_bytes);

/* Swap out nbytes at d_in (device, 16-byte aligned) into the container at
 * h_out (host, h_capacity >= pz_swap_capacity). d_work: device, 16-byte
 * aligned, work_bytes >= pz_swap_work_bytes(piece_bytes). Returns when the
 * container is complete; *h_total (host) = its length.
 * Errors: PZ_ERR_ARG (bad pointer, width, piece size), PZ_ERR_CAPACITY,
 * PZ_ERR_TIMEOUT (a device-side wait of the encoder timed out), PZ_ERR_CUDA. */
pz_status pz_swap_out(const void *d_in, size_t nbytes, int elem_width,
                      size_t piece_bytes, void *d_work, size_t work_bytes,
                      void *h_out, size_t h_capacity, size_t *h_total,
                      pz_stream_t stream);

/* Swap in: decode the container of h_bytes at h_in (host) back into nbytes
 * at d_out (device, 16-byte aligned). The container's head must match
 * nbytes and its table must be consistent with h_bytes (else PZ_ERR_ARG,
 * nothing enqueued). d_work as for pz_swap_out with the container's piece
 * size. Returns once the copies and decodes are enqueued on `stream`;
 * *d_status (device int) becomes PZ_OK or PZ_ERR_CORRUPT when the stream
 * completes. */
pz_status pz_swap_in(const void *h_in, size_t h_bytes, void *d_work,
                     size_t work_bytes, void *d_out, size_t nbytes,
                     int *d_status, pz_stream_t stream);

/* A pool of fixed-size host slots for swapped tensors (Section III-A: on the
 * host, compressed tensors occupy fixed-size chunks of a pinned pool, so
 * that their variable sizes do not fragment the allocator). A swapped
 * tensor's container is laid over a chain of slots (container byte x in the
 * (x / slot_bytes)-th slot of the chain); its handle is the index of its
 * first slot. The pool lives in host memory the caller provides (pinned for
 * the copies to overlap) and keeps all its state there; calls on one pool
 * are thread-safe. */
typedef struct pz_pool_s pz_pool;

/* Host bytes of a pool of nslots slots of slot_bytes (a multiple of 4096):
 * the pool's head and slot links, then the slots, 4096-aligned. 0 for an
 * invalid size. Host-only, pure. */
size_t pz_pool_bytes(size_t slot_bytes, size_t nslots);

/* Lay a pool out in h_mem (host, 64-byte aligned, `bytes` long; as many
 * slots as fit). The slots lie at 4096-byte offsets from h_mem: with h_mem
 * 4096-byte aligned (pinned allocations are), every piece of a pooled
 * container starts 128-byte aligned in host memory, which copies to the
 * device need for the link's full rate. *pool points into h_mem; the pool
 * needs no teardown beyond freeing h_mem once no call uses it. Errors:
 * PZ_ERR_ARG, PZ_ERR_CAPACITY (not one slot fits). */
pz_status pz_pool_init(void *h_mem, size_t bytes, size_t slot_bytes,
                       pz_pool **pool);

/* Slots not held by a swapped tensor. */
size_t pz_pool_free_slots(pz_pool *pool);

/* pz_swap_out into slots of the pool: *tensor (host) = the handle, and
 * *stored_bytes (host, may be NULL) = the container's length. The head and
 * piece table must fit in one slot (PZ_ERR_ARG otherwise). PZ_ERR_CAPACITY
 * when the pool runs out of slots (the slots taken are given back).
 * Other arguments and errors as pz_swap_out. */
pz_status pz_pool_swap_out(pz_pool *pool, const void *d_in, size_t nbytes,
                           int elem_width, size_t piece_bytes, void *d_work,
                           size_t work_bytes, unsigned int *tensor,
                           size_t *stored_bytes, pz_stream_t stream);

/* pz_swap_in of a tensor of the pool; the tensor keeps its slots (release
 * them once `stream` has completed the call). Arguments and errors as
 * pz_swap_in. */
pz_status pz_pool_swap_in(pz_pool *pool, unsigned int tensor, void *d_work,
                          size_t work_bytes, void *d_out, size_t nbytes,
                          int *d_status, pz_stream_t stream);

/* Give a tensor's slots back to the pool (after every call that uses them
 * has completed on its stream). PZ_ERR_ARG for a handle that is not a
 * swapped tensor's, including one already released. */
pz_status pz_pool_release(pz_pool *pool, unsigned int tensor);

/* Largest input pz_compress_noalloc accepts: 256 MiB (65,536 chunks). */
#define PZ_NOALLOC_MAX_BYTES ((size_t)256 << 20)

/* pz_compress without a scratch area in the caller's buffer. The paper has
 * no counterpart: this entry point exists for callers that cannot allocate
 * device memory when they compress. The typical one is a swap runtime that
 * compresses activations precisely because device memory has run out: it
 * cannot enlarge its output buffer by the scratch tail that pz_compress
 * needs, and a code path that runs out of memory must not ask for more.
 *
 * It computes exactly what pz_compress computes (same kernel, same stream,
 * same *d_total_bytes) but keeps the encoder's scratch (one 8-byte look-back
 * word per chunk and a ticket counter) in a file-scope device array of the
 * library, sized for PZ_NOALLOC_MAX_BYTES of input (about 512 KB); every GPU
 * that loads the library holds that array until the process exits.
 *   Arguments as for pz_compress, except:
 *   out_capacity  must be >= 2*C + nbytes (the stream alone; C =
 *                 ceil(nbytes / 4096)), else PZ_ERR_CAPACITY.
 *   nbytes        must be <= PZ_NOALLOC_MAX_BYTES, else PZ_ERR_CAPACITY
 *                 (nothing is enqueued).
 * The call allocates nothing (no cudaMalloc, no allocating library call);
 * it clears the scratch it needs with a kernel of its own on `stream`,
 * launched just before the encoder.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. All calls in the process share the one array
 * per device, which keeps the last call's contents: calls that may overlap
 * on the GPU (different streams, or concurrent host threads) race on it and
 * must be serialized by the caller. */
pz_status pz_compress_noalloc(const void *d_in, size_t nbytes, int elem_width,
                              void *d_out, size_t out_capacity,
                              unsigned long long *d_total_bytes,
                              pz_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PLANEZIP_H */
