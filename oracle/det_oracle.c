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
 *
 * Every function returns 0 on success and a nonzero code on a bad argument.
 */
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
