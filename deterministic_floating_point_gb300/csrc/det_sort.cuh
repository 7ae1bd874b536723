// Stable key sort with a validity filter, and the segmented pairwise tree,
// shared by det_scatter_add and det_scatter_add_rows.
//
// Warp user guide "Deterministic Execution", "Pattern 1: Accumulation" and
// "Picking the Right Mode": records are sorted by destination and linear
// thread index, then each destination's group is reduced in a fixed order.
// Here the records are the inputs themselves (key = destination, payload =
// value and/or original index); the sort is an LSD radix sort whose passes
// are stable, so inside a destination the records keep ascending index.
// Destinations outside [0, m) are dropped by the first pass, as
// "warp.tile_atomic_add_indexed" skips negative and past-the-end indices.
#pragma once

#include "det_common.cuh"

namespace det {

// Layout and plan of one sort, computed on the host from sizes only.
struct SortPlan {
  long long n = 0;          // records
  long long m = 0;          // destinations
  int passes = 1;           // LSD passes
  int digit_bits = 1;       // bits per pass (<= 10)
  int threads = 512;        // CTA size of the passes
  int ipt = 16;             // records per thread per tile
  long long tiles = 0;      // tiles per pass
  int value_bytes = 0;      // payload value size (0, 4 or 8)
  bool need_idx = false;    // carry the original index
  // workspace offsets (bytes from the workspace start)
  size_t totals = 0, counts = 0, keys[2] = {0, 0}, vals[2] = {0, 0}, idx[2] = {0, 0};
  size_t seg = 0, blocks = 0, lsegs = 0, nodes = 0, total = 0;
  long long max_blocks = 0, max_lsegs = 0;
  // Wide records (set by the caller on a one-pass plan without values or
  // indices): `wide` components of wide_elem bytes per record, moved by the
  // pass into one array per component (enqueue_sort's comp_out).
  int wide = 0, wide_elem = 0;
};

// Header fields of a sort workspace (overlays the first 256 bytes).
struct SortHdr {
  unsigned int status;
  unsigned int n_valid;
  unsigned int long_blocks;
  unsigned int long_segs;
};

constexpr int kSegBlock = 4096;   // rank-aligned block of the segmented tree

SortPlan make_sort_plan(long long n, long long m, int value_bytes, bool need_idx, int block_threads);

// Enqueue the whole sort: histogram, digit starts, passes, segment starts.
// Results: sorted values at plan.vals[final], sorted indices at
// perm_out (if not null) else plan.idx[final], segment starts (m+1 int32)
// at plan.seg.  With rank_out (one-pass plans without values or indices
// only) the pass writes each valid record's sorted position to rank_out[i],
// in input order, and moves nothing else.  Returns DET_OK or DET_ERR_CUDA.
// With plan.wide, the values are row-major records and component c of the
// record at sorted position q goes to comp_out[c * n + q].
int enqueue_sort(const SortPlan& p, void* ws, const int32_t* keys, long long key_offset, const void* values,
                 int32_t* perm_out, cudaStream_t s, int* final_buf, int32_t* rank_out = nullptr,
                 void* comp_out = nullptr);

// Segmented pairwise tree: out[b] = out[b] + PT(vals[seg[b] .. seg[b+1]))
// for every non-empty b.  T is float or double.
template <typename T>
// out[b * ostride] receives bin b; reset_counters clears the long-bin
// counters of the header (needed when the same sort feeds several trees).
int enqueue_segmented_tree(const SortPlan& p, void* ws, const T* sorted_vals, T* out, cudaStream_t s,
                           bool negate = false, long long ostride = 1, bool reset_counters = false);

}  // namespace det
