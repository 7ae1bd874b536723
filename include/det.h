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
 *   contents on entry do not matter: the call zeroes what it needs with
 *   cudaMemsetAsync on `stream`, or (det_sum) tells its own words apart by a
 *   per-call tag.  Its first bytes hold the device status word read by
 *   det_read_status().  One workspace must not be shared by calls that may
 *   run at the same time.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Work is only enqueued: no call synchronizes, allocates or copies
 *   to the host, so every call that takes a workspace can be captured in a
 *   CUDA graph.  A captured call can be replayed: the state it leaves in the
 *   workspace is cleared by its own captured memsets on the next replay, and
 *   det_sum, which otherwise clears nothing, takes a clearing form on a
 *   capturing stream (its per-call tag would be frozen into the graph).
 * - `block_threads` selects the CUDA block size: 0 (the default) or one of
 *   128, 256, 512, 1024.  It changes the launch shape only, never the bits.
 *   The sorts behind the scatter calls sort tiles of 4,096 records (CTAs of
 *   256 threads) when asked for 128 and tiles of 8,192 (CTAs of 512)
 *   for 256, 512 or 1024; by default they pick the tile from the sizes.
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
#define DET_SCAN_SEGMENT_RESTART 4   /* det_segmented_scan: each segment scanned as det_scan of the segment alone */

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
 * Enqueued work: one launch, which clears nothing (the workspace may hold
 * anything; each call tags its tile partials with a tag of its own).  On a
 * stream under capture the call enqueues a clearing memset of the
 * workspace header and a launch instead, so every replay of the graph
 * starts clean; the bits are the same either way.
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
 * Set-up: the first call in a CUDA context (with its device current) looks
 * up the device address of the static array in that context, and again
 * whenever the current context changes -- another context on the device, or
 * the primary context recreated after cudaDeviceReset (contexts are told
 * apart by their unique ids); make the first call in a context before any
 * stream capture.  The call allocates nothing and frees nothing.
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
 * det_scatter_sub -- the deterministic form of wp.atomic_sub(out, bins[i],
 * values[i]): the values are negated and added in det_scatter_add's order,
 * out[b] = out[b] + PT(-values of group b).  The leaves are negated (not the
 * group's sum), so an exact zero from cancellation is +0.0 as the pages'
 * "negated and added" gives.  Arguments, outputs, limits, workspace
 * (det_scatter_add_workspace_bytes) and errors as det_scatter_add.
 * Follows: Warp user guide "Deterministic Execution", "Pattern 1:
 * Accumulation" (table row atomic_sub).
 */
int det_scatter_sub(void* out, int64_t out_len, const int32_t* bins, const void* values,
                    int64_t n, int dtype, int32_t* perm_out, int32_t* seg_offsets_out,
                    void* workspace, size_t workspace_bytes, int block_threads, void* stream);

/* ------------------------------------------------------------------------
 * det_scatter_min / det_scatter_max -- the deterministic form of
 * wp.atomic_min / wp.atomic_max(out, bins[i], values[i]): for every bin b
 * that receives at least one valid record, out[b] = op(out[b], op over the
 * group), op = IEEE 754-2019 minimum / maximum (a NaN operand gives NaN, -0
 * orders below +0).  That op is associative and commutative, so the result
 * does not depend on any order; the kernels combine exact integer keys with
 * integer atomics.  Bins without valid records are not touched (their bits,
 * NaN payloads included, stay).  NaN results are the canonical quiet NaN.
 *   out     device, out_len elements of dtype (read and written)
 *   bins    device, n int32 (outside [0, out_len): skipped)
 *   values  device, n elements of dtype
 * Workspace: det_scatter_minmax_workspace_bytes(out_len, dtype) bytes.
 * Limits and errors as det_scatter_add.  block_threads 128 gives 128-thread
 * CTAs, any other value 256.
 * Follows: Warp user guide "Deterministic Execution", "Pattern 1:
 * Accumulation" (table rows atomic_min, atomic_max: values are grouped by
 * destination and minimized / maximized).
 */
size_t det_scatter_minmax_workspace_bytes(int64_t out_len, int dtype);
int det_scatter_min(void* out, int64_t out_len, const int32_t* bins, const void* values, int64_t n,
                    int dtype, void* workspace, size_t workspace_bytes, int block_threads, void* stream);
int det_scatter_max(void* out, int64_t out_len, const int32_t* bins, const void* values, int64_t n,
                    int dtype, void* workspace, size_t workspace_bytes, int block_threads, void* stream);

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
 * det_scatter_add_rows_ordered -- det_scatter_add_rows with the other
 * reading of "returns the previous value": the source rows aimed at one
 * destination are applied one at a time in ascending s (atomics in thread
 * order).  prev_out[s] receives the destination row just before row s is
 * added (the running prefix in index order), and the destination ends at the
 * sequential sum old + v_0 + v_1 + ... (left to right).  Arguments, layout,
 * workspace (det_scatter_add_rows_workspace_bytes), limits and errors as
 * det_scatter_add_rows.
 * Follows: Warp language reference "warp.tile_atomic_add_indexed" (returns:
 * the previous values, unspecified under repeats).
 */
int det_scatter_add_rows_ordered(void* dst, int64_t dst_rows, int64_t row_len, const int32_t* idx,
                                 int64_t row_offset, const void* src, int64_t src_rows, void* prev_out,
                                 int dtype, void* workspace, size_t workspace_bytes, int block_threads,
                                 void* stream);

/* ------------------------------------------------------------------------
 * det_scatter_add_vec -- composite values (vec3, mat33, quaternions, ...:
 * `width` components per record) scattered with wp.atomic_add's
 * deterministic form: for every bin b with records and every component c,
 * out[b][c] = out[b][c] + PT(component c of group b), the groups in
 * ascending record index (exactly det_scatter_add per component, and
 * det_scatter_add_rows with row_len = width and no prev).
 *   out     device, out_len x width elements of dtype, row-major (read and written)
 *   bins    device, n int32 (outside [0, out_len): skipped)
 *   values  device, n x width elements of dtype, row-major
 * Workspace: det_scatter_add_vec_workspace_bytes(n, out_len, width, dtype).
 * Limits: n <= DET_MAX_RECORDS, out_len <= 2^31 - 1, width <= 4096.
 * Follows: Warp user guide "Deterministic Execution", "Pattern 1:
 * Accumulation" (vectors, matrices, quaternions and transforms take the
 * segmented reduction path) and "Picking the Right Mode" (composite values).
 */
size_t det_scatter_add_vec_workspace_bytes(int64_t n, int64_t out_len, int64_t width, int dtype);
int det_scatter_add_vec(void* out, int64_t out_len, int64_t width, const int32_t* bins, const void* values,
                        int64_t n, int dtype, void* workspace, size_t workspace_bytes, int block_threads,
                        void* stream);

/* ------------------------------------------------------------------------
 * det_gather_rows -- out[i] = src[idx[i] + row_offset] row by row, +0.0 rows
 * for indices outside [0, src_rows).  Nothing is combined, so the result is
 * schedule-free.  It is the forward of the pages' backward example: its
 * adjoint, grad_src[idx[i]] += grad_out[i], is det_scatter_add_rows
 * (det_scatter_add for row_len 1), which makes the reverse pass
 * deterministic too.
 *   out  device, n x row_len elements of dtype (written)
 *   src  device, src_rows x row_len elements of dtype
 *   idx  device, n int32
 * No workspace.  block_threads 128 gives 128-thread CTAs, any other value 256.
 * Follows: Warp user guide "Deterministic Execution", "Tape and Backward
 * Passes" (gather: out[tid] = values[indices[tid]]).
 */
int det_gather_rows(void* out, const void* src, int64_t src_rows, int64_t row_len, const int32_t* idx,
                    int64_t row_offset, int64_t n, int dtype, int block_threads, void* stream);

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
 * With flags | DET_SCAN_SEGMENT_RESTART every segment is instead scanned
 * exactly as det_scan of the segment alone (its own chunk grid, look-back
 * and anchors from its first element, scan order); one CTA walks each
 * segment, so a single very long segment is slow, and in that mode
 * block_threads is checked and otherwise ignored.  Invalid offsets are
 * reported through the status word (DET_ERR_INVALID_ARG) in both modes.
 *   seg_offsets device, num_segments + 1 int64
 * Follows: the same pull request, "Validation" (full-array and segmented
 * scans, forward/reverse, inclusive/exclusive).
 */
size_t det_segmented_scan_workspace_bytes(int64_t n, int64_t num_segments, int dtype);
int det_segmented_scan(const void* x, void* y, int64_t n, const int64_t* seg_offsets,
                       int64_t num_segments, int dtype, int flags, void* workspace,
                       size_t workspace_bytes, int block_threads, void* stream);

/* ------------------------------------------------------------------------
 * det_scan_i32 -- int32 prefix sum, inclusive (flags 0) or exclusive
 * (flags DET_SCAN_EXCLUSIVE), modulo 2^32 (as int32 atomics wrap); every
 * order of integer additions gives the same bits.  total_out (device, one
 * int32, or NULL) receives the sum of all n values, so the page's "final
 * count is offsets[n-1] + counts[n-1]" is available without a read-back.
 *   x, y    device, n int32 (x == y allowed)
 * Workspace: det_scan_i32_workspace_bytes(n).  Other flags give
 * DET_ERR_INVALID_ARG.  The CTA size is fixed (block_threads is checked and
 * otherwise ignored).
 * Follows: Warp user guide "Deterministic Execution", "Picking the Right
 * Mode" (count_positive -> array_scan(..., inclusive=False) ->
 * write_positive) and "Pattern 2: Slot Allocation" (step 3).
 */
size_t det_scan_i32_workspace_bytes(int64_t n);
int det_scan_i32(const int32_t* x, int32_t* y, int64_t n, int flags, int32_t* total_out,
                 void* workspace, size_t workspace_bytes, int block_threads, void* stream);

/* ------------------------------------------------------------------------
 * det_slot_alloc -- the deterministic form of
 *     slot = wp.atomic_add(counter, index[i], count[i])
 * executed by threads i = 0 .. n-1: per counter element, reservations are
 * served in thread order, so record i gets the element's value before the
 * call plus the requests of the earlier records aimed at the same element,
 * and every element then advances by its records' total.  Pre-existing
 * nonzero counters and repeated (append-style) calls work.  Records whose
 * element index[i] + index_offset is outside [0, num_counters) get slot -1
 * and change nothing.  Arithmetic wraps modulo 2^32.
 *   counter   device, num_counters int32 (read and written)
 *   index     device, n int32
 *   count     device, n int32 (slots requested; may be negative like an
 *             atomic add's operand), or NULL for one slot each
 *   slot_out  device, n int32
 * Workspace: det_slot_alloc_workspace_bytes(n, num_counters).  Limits:
 * n <= DET_MAX_RECORDS, num_counters <= 2^31 - 1.  slot_out must not
 * overlap the inputs.
 * Follows: Warp user guide "Deterministic Execution", "Pattern 2: Slot
 * Allocation" (count, sort by counter element and thread order, segmented
 * prefix scan, slots), "Pattern B: Slot Allocation Counters", and
 * "Counter arrays are allocation counters".
 */
size_t det_slot_alloc_workspace_bytes(int64_t n, int64_t num_counters);
int det_slot_alloc(int32_t* counter, int64_t num_counters, const int32_t* index, int64_t index_offset,
                   const int32_t* count, int64_t n, int32_t* slot_out, void* workspace,
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

/* The last CUDA failure a call of this library met (the step that failed and
 * the CUDA error name), or "" if none: the detail behind DET_ERR_CUDA.  The
 * string lives in library storage until the next failure; calls on other
 * threads may replace it. */
const char* det_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DET_H */
