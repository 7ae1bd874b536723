/*
 * det_baselines.h -- the nondeterministic kernels the deterministic calls are
 * measured against.  Their results depend on the order in which the GPU
 * schedules floating-point atomics or observes look-back states, so their
 * bits may change from run to run; they exist only as overhead baselines.
 * Same conventions as det.h (device pointers, dtype DET_F32 / DET_F64,
 * stream as void*, DET_* return codes).
 */
#ifndef DET_BASELINES_H
#define DET_BASELINES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* out[0] = sum of x: a grid-stride loop and a block tree per CTA, then one
 * floating-point atomicAdd per CTA into out (zeroed first by the call).
 * Day 68 "Floating point and reproducibility", "Fix the order of every
 * addition": the atomic tail of sumSquaresAtomic, without the squaring. */
int det_atomic_sum(const void* x, int64_t n, int dtype, void* out, void* stream);

/* out[bins[i]] += values[i] with one floating-point atomicAdd per record;
 * records with bins[i] outside [0, out_len) are skipped.  Warp user guide
 * "Deterministic Execution", "Pattern A: Accumulation Atomics". */
int det_atomic_scatter_add(void* out, int64_t out_len, const int32_t* bins, const void* values, int64_t n,
                           int dtype, void* stream);

/* Row scatter with one atomicAdd per element; prev_out (may be NULL)
 * receives the value each atomic returned (+0.0 for skipped rows), as
 * "warp.tile_atomic_add_indexed" returns it. */
int det_atomic_scatter_add_rows(void* dst, int64_t dst_rows, int64_t row_len, const int32_t* idx,
                                int64_t row_offset, const void* src, int64_t src_rows, void* prev_out, int dtype,
                                void* stream);

/* slot_out[i] = atomicAdd(&counter[index[i] + index_offset], count[i] or 1)
 * with integer atomics in arrival order (-1 for indices outside the
 * counters): the slot-allocation pattern of Warp user guide "Deterministic
 * Execution", "Pattern 2: Slot Allocation", as it runs without deterministic
 * mode.  The counters' final values are deterministic, the slots are not. */
int det_atomic_slot_alloc(int32_t* counter, int64_t num_counters, const int32_t* index, int64_t index_offset,
                          const int32_t* count, int64_t n, int32_t* slot_out, void* stream);

/* Inclusive forward prefix sum by the unmodified decoupled look-back: each
 * chunk publishes its aggregate (PARTIAL) and then its inclusive prefix
 * (INCLUSIVE); the look-back adds predecessors' values until it meets an
 * INCLUSIVE one, so the association depends on what it observes.
 * drjit-core pull request "Make CUDA floating-point prefix sums
 * deterministic", "Root cause". */
size_t det_dlb_scan_workspace_bytes(int64_t n, int dtype);
int det_dlb_scan(const void* x, void* y, int64_t n, int dtype, void* workspace, size_t workspace_bytes,
                 void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DET_BASELINES_H */
