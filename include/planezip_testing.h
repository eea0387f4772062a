/*
 * planezip_testing.h — test hooks of libplanezip.so. Not part of the codec's
 * API: a program that compresses and decompresses needs only planezip.h.
 * The paper ("PlaneZip: Lossless Bit-Plane Compression of Training
 * Activations Offloaded over PCIe", arXiv:2610.25033v1) has no counterpart;
 * these entry points exist so that the library's bounded device-side waits
 * can be exercised without a GPU fault.
 */
#ifndef PLANEZIP_TESTING_H
#define PLANEZIP_TESTING_H

#include "planezip.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Runs pz_compress's encoder on nbytes (2..4096 chunks) with chunk 0 never
 * taken, so that the look-back of chunk 1 waits on a status word nothing
 * publishes. That wait gives up after its iteration limit (about a second)
 * and the launch ends with *d_total_bytes = UINT64_MAX, the encoder's
 * timeout report; the GPU context stays usable. Arguments and errors as
 * pz_compress (C outside 2..4096 gives PZ_ERR_ARG); the contents of d_out
 * are unspecified afterwards. */
pz_status pz_test_lookback_timeout(const void *d_in, size_t nbytes,
                                   int elem_width, void *d_out,
                                   size_t out_capacity,
                                   unsigned long long *d_total_bytes,
                                   pz_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PLANEZIP_TESTING_H */
