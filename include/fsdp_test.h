/*
 * fsdp_test.h - diagnostic entry points of the GB300 FSDP library.
 *
 * Not part of the method's interface (fsdp.h): these calls exist so that a
 * test can drive the library's failure paths on purpose. They are exported
 * by the same shared library and follow the conventions of fsdp.h.
 */
#ifndef FSDP_GB300_TEST_H
#define FSDP_GB300_TEST_H

#include "fsdp.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Self-test of the bounded waits of the TMA form (the pages have no
 * counterpart; it checks the failure path that fsdp_device_status reports).
 * Launches the TMA form on a copy of `bytes` (>= 16384, <= 2^30, both
 * pointers 16-byte aligned, not overlapping) with block 0's first stage
 * expecting 16 bytes that no copy delivers, and a wait limit of
 * wait_limit_ns (1 ns .. 10 s). The block gives up after the limit, drains its
 * copies and returns; the call synchronizes `stream`, then reads and clears
 * the status word into *status_out (1 when the timeout was seen). dst is
 * partly written. Nothing hangs and the context stays usable.
 * EINVAL: null pointers, sizes or limits out of range, misaligned pointers;
 * EALIAS: dst overlaps src; ECUDA: a CUDA call failed. */
int fsdp_selftest_wait_timeout(const void *src, void *dst, int64_t bytes, int64_t wait_limit_ns,
                               fsdp_stream_t stream, uint32_t *status_out);

#ifdef __cplusplus
}
#endif

#endif /* FSDP_GB300_TEST_H */
