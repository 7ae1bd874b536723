/*
 * CPU oracle for the deterministic sum / scatter-add / row scatter-add /
 * scan / segmented scan library.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load this code; the library itself never
 * does, and it shares no source with the CUDA path.  Build:
 *
 *   gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared \
 *       det_oracle.c -o liboracle.so
 *
 * Pages followed (cited by title and section):
 *   - Warp user guide "Deterministic Execution": "Pattern 1: Accumulation",
 *     "Picking the Right Mode", "Large launches".
 *   - Day 68 "Floating point and reproducibility": "Contracts from tolerance
 *     to fixed bits", "Fix the order of every addition".
 *   - Warp language reference "warp.tile_atomic_add_indexed": parameters and
 *     Example.
 *   - drjit-core pull request "Make CUDA floating-point prefix sums
 *     deterministic": "Root cause", "Implementation", "Validation".
 *   - Warp user guide "Deterministic Execution": "Pattern 2: Slot
 *     Allocation", "Pattern B: Slot Allocation Counters", "Counter arrays are
 *     allocation counters" (the integer functions at the end of this file).
 *
 * Every function returns 0 on success and a nonzero code on a bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if defined(__FAST_MATH__)
#error "the oracle must be built without fast-math"
#endif

#define T float
#define SFX f32
#define SCAN_E 32
#include "det_oracle_impl.h"
#undef T
#undef SFX
#undef SCAN_E

#define T double
#define SFX f64
#define SCAN_E 16
#include "det_oracle_impl.h"
#undef T
#undef SFX
#undef SCAN_E

/* chunk geometry the scan readings freeze, so tests can place inputs on
 * lane / warp / chunk / interval boundaries */
int64_t oracle_scan_chunk_elems(int is_f64) { return (int64_t)NWARP * NLANE * (is_f64 ? 16 : 32); }
int64_t oracle_scan_lane_elems(int is_f64) { return is_f64 ? 16 : 32; }

/* ---------------------------------------------------------------------- */
/* Integer parts.  int32 arithmetic wraps modulo 2^32 (as an int32 atomic add
 * does), so every order of the additions gives the same bits. */

/* det_scan_i32: inclusive (flags bit 0 clear) or exclusive (bit 0 set) prefix
 * sum of x[0..n); *total_out (may be NULL) = the sum of all n values.  The
 * count-scan-write recipe of Warp "Deterministic Execution", "Picking the
 * Right Mode": offsets = exclusive scan of counts, and the final count is
 * offsets[n-1] + counts[n-1]. */
int oracle_scan_i32(const int32_t* x, int32_t* y, int64_t n, int flags, int32_t* total_out)
{
    if (n < 0 || (n > 0 && (!x || !y))) return 1;
    uint32_t run = 0;
    for (int64_t i = 0; i < n; ++i) {
        const uint32_t v = (uint32_t)x[i];
        if (flags & 1) { y[i] = (int32_t)run; run += v; }
        else { run += v; y[i] = (int32_t)run; }
    }
    if (total_out) *total_out = (int32_t)run;
    return 0;
}

/* det_slot_alloc: the deterministic form of
 *     slot = wp.atomic_add(counter, index[i], count[i])
 * executed by threads i = 0 .. n-1.  Reservations are served in thread order
 * per counter element: record i gets the counter's value before its own
 * request and the counter then advances by count[i] (Warp "Deterministic
 * Execution", "Pattern 2: Slot Allocation": sort reservations by counter
 * element and thread order, then a segmented prefix scan gives each starting
 * slot and each counter's total; "Counter arrays are allocation counters":
 * pre-existing nonzero counters and append-style launches).  count may be
 * NULL (one slot each).  Records whose counter index + index_offset is
 * outside [0, num_counters) are skipped: slot -1, no counter changes. */
int oracle_slot_alloc(int32_t* counter, int64_t num_counters, const int32_t* index, int64_t index_offset,
                      const int32_t* count, int64_t n, int32_t* slot_out)
{
    if (num_counters < 0 || n < 0 || (num_counters > 0 && !counter) || (n > 0 && (!index || !slot_out))) return 1;
    if (n > 2147483647LL || num_counters > 2147483647LL) return 2;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t c = (int64_t)index[i] + index_offset;
        if (c < 0 || c >= num_counters) { slot_out[i] = -1; continue; }
        slot_out[i] = counter[c];
        counter[c] = (int32_t)((uint32_t)counter[c] + (uint32_t)(count ? count[i] : 1));
    }
    return 0;
}
