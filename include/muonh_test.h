/*
 * muonh_test.h -- test hooks of libmuonh.  Not part of the optimizer's
 * interface: the pages have no counterpart.  They exist so that tests can
 * exercise the library's failure detection without faulting or hanging a
 * GPU.
 */
#ifndef MUONH_TEST_H
#define MUONH_TEST_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of device workspace muonh_test_gemm_timeout needs. */
#define MUONH_TEST_TIMEOUT_WS_BYTES (512u * 1024u)

/*
 * Launches one Newton-Schulz Gram GEMM (a 256 x 256 tile, K = 256) whose TMA
 * producer issues no copies, so the MMA issuer's first pipeline wait runs out
 * after `timeout_ns` (1e3 .. 1e10 ns) with nothing in flight.  Every wait of
 * the kernel is bounded by the same limit; the kernel sets
 * MUONH_STATUS_KERNEL_TIMEOUT in the device status word (read it with
 * muonh_get_status), frees its TMEM and returns, and the context stays
 * usable.  `flags`: 0 for the CTA-pair kernel, MUONH_FLAG_GEMM_1SM for the
 * 1-SM kernel; no other bit.  `workspace`: device memory of at least
 * MUONH_TEST_TIMEOUT_WS_BYTES, 256-byte aligned; nothing is read from or
 * written to it (it only anchors the TMA descriptors).  Asynchronous on
 * `stream`; returns MUONH_OK once the kernel is launched.
 */
int muonh_test_gemm_timeout(uint32_t flags, uint64_t timeout_ns, void* workspace, size_t ws_bytes,
                            void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MUONH_TEST_H */
