/*
 * det_test_hooks.h -- test hooks of libdet.so.  Not part of any computation:
 * they let a test drive the library's error paths on purpose, from the host,
 * without a GPU fault.  The pages have no counterpart; the error path they
 * exercise is the device-detected error reported to the caller after the
 * launch (Warp user guide "Deterministic Execution", section "Large
 * launches": an overflow found on the device surfaces as an error on the
 * host).
 *
 * Host-side state, one per process, not thread-safe.
 */
#ifndef DET_TEST_HOOKS_H
#define DET_TEST_HOOKS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* det_test_scan_withhold -- while set, every det_scan and global-grid
 * det_segmented_scan call enqueued afterwards computes as usual but never
 * publishes the look-back aggregate of chunk `chunk` (scan order, chunks of
 * DET_SCAN_CHUNK_F32 / _F64 elements), and every on-device wait of those
 * calls gives up after `timeout_ns` nanoseconds instead of 2 s.  The chunks
 * that read that aggregate, and the anchor chain, wait until the limit runs
 * out; the first wait that gives up writes DET_ERR_LOOKBACK_TIMEOUT to the
 * status word, every later wait of the launch gives up at once, and the
 * launch ends.  The host call still returns DET_OK; det_read_status() then
 * reports DET_ERR_LOOKBACK_TIMEOUT, and the output is unspecified.
 *   chunk       >= 0 to set the hook; < 0 clears it (normal publication and
 *               the 2 s limit again)
 *   timeout_ns  1 .. 2e9 when setting; ignored when clearing
 * Returns DET_OK, or DET_ERR_INVALID_ARG for a limit outside that range. */
int det_test_scan_withhold(int64_t chunk, uint64_t timeout_ns);

#ifdef __cplusplus
}
#endif

#endif /* DET_TEST_HOOKS_H */
