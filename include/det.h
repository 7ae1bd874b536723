/*
 * det.h -- deterministic floating-point sum, scatter-add, row scatter-add and
 * prefix scan for one NVIDIA GB300 GPU (sm_103a).
 *
 * Every call adds its floating-point terms in an association order that is a
 * function of element indices only.  The same inputs therefore give the same
 * result bits on every run, for every block size the caller picks, and those
 * bits equal the plain CPU statement of the same order.
 *
 * Conventions shared by every call
 * --------------------------------
 * - dtype is DET_F32 or DET_F64; values, outputs and results have that type.
 *   The arithmetic is IEEE round-to-nearest addition in that type, with no
 *   flush-to-zero.  NaN payloads are not promised to match bit for bit.
 * - Every array pointer is DEVICE memory owned by the caller.  The library
 *   keeps no pointer after a call returns and allocates nothing.
 * - `workspace` is caller-owned device memory of at least the size the
 *   matching *_workspace_bytes() query returns, 256-byte aligned.  Its
 *   contents on entry do not matter; the call zeroes what it needs with
 *   cudaMemsetAsync on `stream`.  Its first bytes hold the device status word
 *   read by det_read_status().  One workspace must not be shared by calls
 *   that may run at the same time.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Work is only enqueued: no call synchronizes, allocates or copies
 *   to the host, so every call that takes a workspace can be captured in a
 *   CUDA graph.
 * - `block_threads` selects the CUDA block size: 0 (the default) or one of
 *   128, 256, 512, 1024.  It changes the launch shape only, never the bits.
 *   The sorts behind the scatter calls use 128-thread CTAs when asked for
 *   128 and 256-thread CTAs otherwise.
 * - Return value: DET_OK, or an error code for a bad argument found on the
 *   host (nothing is enqueued then), or DET_ERR_CUDA if a launch failed.
 *   Errors detected on the device (a look-back wait that gave up) are written
 *   to the status word; read them with det_read_status().
 * - Sizes are int64_t; n = 0 is always valid.
 */
#ifndef DET_H
#define DET_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DET_F32 0
#define DET_F64 1

#define DET_OK 0
#define DET_ERR_INVALID_ARG 1      /* null pointer, negative size, bad flags or block size */
#define DET_ERR_DTYPE 2            /* dtype is not DET_F32 or DET_F64 */
#define DET_ERR_TOO_LARGE 3        /* a size beyond the documented limit */
#define DET_ERR_WORKSPACE 4        /* workspace too small, or misaligned */
#define DET_ERR_LOOKBACK_TIMEOUT 5 /* device: a look-back wait gave up (status word only) */
#define DET_ERR_CUDA 6             /* a CUDA call or launch failed */
#define DET_ERR_COPY_TIMEOUT 7     /* device: a bulk copy into shared memory did not complete in time (status word only) */

/* scan flags */
#define DET_SCAN_INCLUSIVE 0
#define DET_SCAN_EXCLUSIVE 1
#define DET_SCAN_REVERSE 2

/* Frozen scan geometry: a chunk is 32 virtual warps x 32 lanes x E elements,
 * with E = 32 (f32) or 16 (f64); anchor intervals are 32 chunks long. */
#define DET_SCAN_LANE_ELEMS_F32 32
#define DET_SCAN_LANE_ELEMS_F64 16
#define DET_SCAN_CHUNK_F32 32768
#define DET_SCAN_CHUNK_F64 16384
#define DET_SCAN_ANCHOR_INTERVAL 32

/* Largest record count of a scatter call (int32 record slots). */
#define DET_MAX_RECORDS 2147483647LL

/* ------------------------------------------------------------------------
 * det_sum -- out[0] = PT(x[0..n)), the canonical pairwise tree: pad x with
 * absent terms to the next power of two and add pairs (2j, 2j+1) level by
 * level.  The pairing is fixed by element index, not by the grid, so block
 * and grid size cannot change it.  n = 0 gives +0.0.
 *   x   device, n elements of dtype, contiguous, any alignment
 *   out device, 1 element of dtype (written)
 * Follows: Day 68 "Floating point and reproducibility", sections "Contracts
 * from tolerance to fixed bits" (items 1-2) and "Fix the order of every
 * addition" (the atomic tail replaced by a fixed tree).
 */
size_t det_sum_workspace_bytes(int64_t n, int dtype);
int det_sum(const void* x, int64_t n, int dtype, void* out,
            void* workspace, size_t workspace_bytes, int block_threads, void* stream);

/* ------------------------------------------------------------------------
 * det_sum_noalloc -- det_sum without any caller-provided or allocated
 * scratch memory.  (The pages have no counterpart; this entry point exists
 * for callers that cannot allocate.)
 *
 * Some callers cannot call cudaMalloc or hand the library a workspace: a
 * plugin running inside another runtime that owns all device memory and
 * exposes no allocator to it, or a loop that must not allocate after
 * start-up because cudaMalloc can synchronize the device and has unbounded
 * latency.  For them this call keeps its scratch (a 256-byte status/ticket
 * header and up to DET_SUM_NOALLOC_MAX_PARTIALS tile partials) in one
 * statically sized device array inside libdet.so, 256 + 16384 * 8 bytes,
 * which every GPU that loads the library holds until the process exits.
 * The caller still passes the input and the output; the result bits equal
 * det_sum's.
 *   x    device, n elements of dtype
 *   out  device, 1 element of dtype (written)
 * Limit: inputs of at most 2^36 bytes (2^34 f32 or 2^33 f64 elements);
 * larger n returns DET_ERR_TOO_LARGE and enqueues nothing.
 * Set-up: the first call on a device (with that device current) looks up
 * the device address of the static array once; make that first call before
 * any stream capture.  The call allocates nothing and frees nothing.
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents (each call clears the part that must start at zero).
 * Calls whose work can overlap on the GPU -- different streams without
 * ordering between them, or different host threads -- race on that array
 * and must not be made.
 */
#define DET_SUM_NOALLOC_MAX_PARTIALS 16384
int det_sum_noalloc(const void* x, int64_t n, int dtype, void* out, int block_threads, void* stream);

/* ------------------------------------------------------------------------
 * det_scatter_add -- out[bins[i]] += values[i] for every i with
 * 0 <= bins[i] < out_len; other i are skipped.  The records are sorted
 * stably by destination (ascending i inside each destination), each
 * destination's values are added by PT over their rank in that order, and
 * the old value is added once, last: out[b] = out[b] + PT(group b).
 * Destinations that receive nothing keep their bits.
 *   out             device, out_len elements of dtype (read and written)
 *   bins            device, n int32
 *   values          device, n elements of dtype
 *   perm_out        device, n int32 or NULL: the sorted record indices
 *                   (the first seg_offsets[out_len] entries are written)
 *   seg_offsets_out device, out_len + 1 int32 or NULL: group starts;
 *                   seg_offsets_out[out_len] = number of valid records
 * Limits: n <= DET_MAX_RECORDS, out_len <= 2^31 - 1.  out must not overlap
 * the inputs.
 * Follows: Warp user guide "Deterministic Execution", sections "Pattern 1:
 * Accumulation", "Picking the Right Mode" (sort by destination and thread
 * index, then reduce each group) and "Large launches"; out-of-range skipping
 * from "warp.tile_atomic_add_indexed".
 */
size_t det_scatter_add_workspace_bytes(int64_t n, int64_t out_len, int dtype);
int det_scatter_add(void* out, int64_t out_len, const int32_t* bins, const void* values,
                    int64_t n, int dtype, int32_t* perm_out, int32_t* seg_offsets_out,
                    void* workspace, size_t workspace_bytes, int block_threads, void* stream);

/* ------------------------------------------------------------------------
 * det_scatter_add_rows -- the tile row scatter of tile_atomic_add_indexed
 * along axis 0, deterministic: source row s (row_len elements) is added to
 * destination row r = idx[s] + row_offset when 0 <= r < dst_rows (else it
 * is skipped).  Each column is exactly det_scatter_add: rows aimed at one
 * destination are taken in ascending s, added by PT, then added once to the
 * old row.  prev_out[s] receives destination row r as it was before this
 * call (every contributor of one destination sees the same previous row),
 * and +0.0 for skipped rows.
 *   dst      device, dst_rows x row_len, row-major (read and written)
 *   idx      device, src_rows int32
 *   src      device, src_rows x row_len, row-major
 *   prev_out device, src_rows x row_len, or NULL
 * Limits: src_rows, dst_rows <= 2^31 - 1.  dst and prev_out must not
 * overlap the inputs or each other.
 * Follows: Warp language reference "warp.tile_atomic_add_indexed"
 * (parameters, returns, Example).
 */
size_t det_scatter_add_rows_workspace_bytes(int64_t src_rows, int64_t dst_rows, int64_t row_len,
                                            int dtype);
int det_scatter_add_rows(void* dst, int64_t dst_rows, int64_t row_len, const int32_t* idx,
                         int64_t row_offset, const void* src, int64_t src_rows, void* prev_out,
                         int dtype, void* workspace, size_t workspace_bytes, int block_threads,
                         void* stream);

/* ------------------------------------------------------------------------
 * det_scan -- prefix sum by a single-pass decoupled look-back whose
 * look-back is anchored: chunks of DET_SCAN_CHUNK_* elements, intervals of
 * 32 chunks; look-back lane l of chunk c = 32k + j reads the aggregate of
 * chunk c-1-l for l < j and the previous interval's anchor prefix at l = j,
 * and adds them by PT over lanes; only the last chunk of an interval
 * publishes an inclusive prefix.  Inside a chunk: in-lane fold, Kogge-Stone
 * over 32 lanes, Kogge-Stone over 32 virtual warps, then each element is
 * ((Excl + warp prefix) + lane prefix) folded with the lane's elements.
 *   flags      DET_SCAN_INCLUSIVE or DET_SCAN_EXCLUSIVE, optionally | DET_SCAN_REVERSE.
 *              Exclusive output is the inclusive output shifted by one
 *              (first element +0.0); reverse is the scan of the reversed
 *              input, reversed back.
 *   x, y       device, n elements of dtype; y may equal x (in place), other
 *              overlaps are not allowed
 *   total_out  device, 1 element, or NULL: the last inclusive value in scan
 *              order (+0.0 for n = 0)
 * Follows: drjit-core pull request "Make CUDA floating-point prefix sums
 * deterministic", sections "Root cause" and "Implementation" and the
 * author's reworked description (fixed 32-chunk anchor intervals).
 */
size_t det_scan_workspace_bytes(int64_t n, int dtype);
int det_scan(const void* x, void* y, int64_t n, int dtype, int flags, void* total_out,
             void* workspace, size_t workspace_bytes, int block_threads, void* stream);

/* ------------------------------------------------------------------------
 * det_segmented_scan -- det_scan with the segmented operator
 * (fa,a)(+)(fb,b) = (fa|fb, fb ? b : a+b) in every place det_scan adds,
 * left operand always the earlier part; the chunk grid is global.
 * Segment s is [seg_offsets[s], seg_offsets[s+1]); seg_offsets[0] = 0,
 * seg_offsets[num_segments] = n, non-decreasing (empty segments allowed).
 * Exclusive output is +0.0 at each segment's first element.
 *   seg_offsets device, num_segments + 1 int64
 * Follows: the same pull request, "Validation" (full-array and segmented
 * scans, forward/reverse, inclusive/exclusive).
 */
size_t det_segmented_scan_workspace_bytes(int64_t n, int64_t num_segments, int dtype);
int det_segmented_scan(const void* x, void* y, int64_t n, const int64_t* seg_offsets,
                       int64_t num_segments, int dtype, int flags, void* workspace,
                       size_t workspace_bytes, int block_threads, void* stream);

/* ------------------------------------------------------------------------
 * Status.  det_read_status synchronizes `stream`, then copies the device
 * status word out of `workspace` into *device_status: DET_OK,
 * DET_ERR_LOOKBACK_TIMEOUT or DET_ERR_COPY_TIMEOUT (a bounded wait gave up),
 * or DET_ERR_INVALID_ARG (segment offsets found invalid on the device, or a
 * sort position out of range -- the latter cannot happen for a correct
 * ranking and is checked so that no write can leave its buffer).
 * Returns DET_OK or DET_ERR_CUDA.
 */
int det_read_status(const void* workspace, void* stream, int* device_status);
const char* det_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* DET_H */
