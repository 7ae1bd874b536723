// det_scatter_add_rows: deterministic form of the tile row scatter of
// "warp.tile_atomic_add_indexed" along axis 0.
//
// The page's primitive adds element c of the tile to a[offset + indices[c_0],
// c_1] atomically, skips destinations outside the array, lets repeated
// indices accumulate and returns each destination's previous value -- with
// the order (and so the rounding and the returned values) unspecified under
// repeats.  Here:
//   1. the row indices are sorted stably (payload: the source row id), so
//      the rows aimed at one destination are in ascending source order;
//   2. one warp per destination row reads the old row, then reduces the rows
//      column by column with the pairwise tree over their rank (rounds of 8
//      rows in registers, each a level-3 node; up to four such nodes
//      combined by a fixed tree, a binary counter beyond), writes the old row
//      to prev for every contributor as it goes, and stores old + tree.
//      Where every row starts on a pair boundary a lane moves two adjacent
//      columns as one access.  (Measured on this chip and dropped: rounds of
//      16 rows, which need registers that cost resident warps; contributor
//      rows staged in shared memory by bulk copies, with or without a
//      persistent warp pipelining two destinations: all slower, as the
//      kernel is bound by the latency chain of each warp's loads and by how
//      many warps an SM holds.)
//   3. skipped source rows get prev = +0.0.
#include "det_sort.cuh"

namespace det {
namespace {

constexpr int kCPL = 2;   // columns per lane per pass over the row (64 columns per warp pass)
constexpr int kRR = 8;    // contributor rows per round, all loads in flight together

template <typename T> struct Pair;
template <> struct Pair<float> { using V = float2; };
template <> struct Pair<double> { using V = double2; };

// Columns of one lane in the warp pass starting at column c0.  VEC (even W,
// pair-aligned arrays): the two adjacent columns c0 + 2 lane + {0, 1}, moved
// as one 8- or 16-byte access, so a warp reads a 64-column row slice in one
// request; otherwise c0 + lane and c0 + 32 + lane.  Only the memory
// accesses differ: each column is reduced on its own either way.
template <typename T, bool VEC>
struct RowCols {
  using V = typename Pair<T>::V;
  long long col[kCPL];
  bool ok[kCPL];
  __device__ __forceinline__ RowCols(long long c0, long long W, int lane) {
#pragma unroll
    for (int c = 0; c < kCPL; ++c) {
      col[c] = VEC ? c0 + 2 * lane + c : c0 + c * 32 + lane;
      ok[c] = col[c] < W;
    }
  }
  // the lane's columns of row `row` (absent fill where a column or the row is missing)
  __device__ __forceinline__ void load(T (&x)[kCPL], const T* __restrict__ a, long long row, long long W,
                                       bool have, T fill) const {
    if (VEC) {
      const bool in = have && ok[0];
      V q;
      if (in) q = __ldg(reinterpret_cast<const V*>(a + row * W + col[0]));
      x[0] = in ? q.x : fill;
      x[1] = in ? q.y : fill;
    } else {
#pragma unroll
      for (int c = 0; c < kCPL; ++c) x[c] = (have && ok[c]) ? __ldg(a + row * W + col[c]) : fill;
    }
  }
  __device__ __forceinline__ void store(T* a, long long row, long long W, const T (&x)[kCPL]) const {
    if (VEC) {
      if (ok[0]) {
        V q;
        q.x = x[0];
        q.y = x[1];
        *reinterpret_cast<V*>(a + row * W + col[0]) = q;
      }
    } else {
#pragma unroll
      for (int c = 0; c < kCPL; ++c)
        if (ok[c]) a[row * W + col[c]] = x[c];
    }
  }
};

// Source row of contributor k of the destination's group, -1 past its end.
// Every lane loads the same entry (one broadcast request); handing a group
// of 32 entries to the warp by shuffles measured far slower on this chip.
__device__ __forceinline__ int group_perm(const int32_t* __restrict__ perm, long long lo, long long k, long long L,
                                          long long src_rows) {
  int sv = k < L ? perm[lo + k] : -1;
  if ((long long)sv >= src_rows) sv = -1;   // cannot happen for a correct sort
  return sv;
}

// Registers capped so that four (f32) or three (f64) CTAs share an SM: the
// kernel is bound by each warp's chain of dependent loads, so resident warps
// count (f64 measured 13 % faster at three CTAs than at two, despite a few
// spilled bytes).
template <typename T, bool VEC>
__global__ void __launch_bounds__(256, sizeof(T) == 8 ? 3 : 4)
rows_kernel(T* __restrict__ dst, long long R, long long W, const T* __restrict__ src, const int32_t* __restrict__ perm,
            const int32_t* __restrict__ seg, const unsigned int* __restrict__ n_valid, T* __restrict__ prev,
            long long src_rows) {
  const long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= R) return;
  const long long N = *n_valid;
  const long long hi = min((long long)seg[r + 1], N), lo = max(0LL, min((long long)seg[r], hi));
  const long long L = hi - lo;
  if (L <= 0) return;
  const bool small = L <= 32;   // at most four level-3 nodes: combined by a fixed tree
  for (long long c0 = 0; c0 < W; c0 += 32 * kCPL) {
    const RowCols<T, VEC> rc(c0, W, lane);
    T old[kCPL];   // the row before the call: every contributor's prev
    rc.load(old, dst, r, W, true, T(0));
    T n4[kCPL][4];
#pragma unroll
    for (int c = 0; c < kCPL; ++c)
#pragma unroll
      for (int q = 0; q < 4; ++q) n4[c][q] = absent<T>();
    NodeCounter<T, 1> nc[kCPL];   // groups of more than 32 rows only (rare): deeper levels in local memory
    for (long long k0 = 0; k0 < L; k0 += kRR) {
      int sr[kRR];
      T v[kCPL][kRR];
#pragma unroll
      for (int e = 0; e < kRR; ++e) {
        sr[e] = group_perm(perm, lo, k0 + e, L, src_rows);
        T x[kCPL];
        rc.load(x, src, sr[e], W, sr[e] >= 0, absent<T>());
#pragma unroll
        for (int c = 0; c < kCPL; ++c) v[c][e] = x[c];
      }
      if (prev) {
#pragma unroll
        for (int e = 0; e < kRR; ++e)
          if (sr[e] >= 0) rc.store(prev, sr[e], W, old);
      }
      // two level-3 nodes (8 rows each) per round, in rank order
      const int q = (int)(k0 >> 3);
#pragma unroll
      for (int c = 0; c < kCPL; ++c) {
#pragma unroll
        for (int h = 0; h < kRR / 8; ++h) {
          T leaf[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) leaf[e] = v[c][8 * h + e];
          const T node = thread_pt(leaf);
          if (small) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (j == q + h) n4[c][j] = node;
          } else {
            nc[c].push(node);
          }
        }
      }
    }
    T out[kCPL];
#pragma unroll
    for (int c = 0; c < kCPL; ++c)
      out[c] = old[c] + (small ? (n4[c][0] + n4[c][1]) + (n4[c][2] + n4[c][3]) : nc[c].result());
    rc.store(dst, r, W, out);
  }
}

// Ordered reading: per destination row and column the contributors are
// added one at a time in ascending source row, each getting the running
// value before its own add as prev (atomics applied in thread order).
template <typename T, bool VEC>
__global__ void __launch_bounds__(256, sizeof(T) == 8 ? 3 : 4)
rows_ordered_kernel(T* __restrict__ dst, long long R, long long W, const T* __restrict__ src,
                    const int32_t* __restrict__ perm, const int32_t* __restrict__ seg,
                    const unsigned int* __restrict__ n_valid, T* __restrict__ prev, long long src_rows) {
  const long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= R) return;
  const long long N = *n_valid;
  const long long hi = min((long long)seg[r + 1], N), lo = max(0LL, min((long long)seg[r], hi));
  const long long L = hi - lo;
  if (L <= 0) return;
  for (long long c0 = 0; c0 < W; c0 += 32 * kCPL) {
    const RowCols<T, VEC> rc(c0, W, lane);
    T acc[kCPL];
    rc.load(acc, dst, r, W, true, T(0));
    for (long long k0 = 0; k0 < L; k0 += kRR) {
      int sr[kRR];
      T v[kCPL][kRR];
#pragma unroll
      for (int e = 0; e < kRR; ++e) {   // the round's rows in flight, then applied in order
        sr[e] = group_perm(perm, lo, k0 + e, L, src_rows);
        T x[kCPL];
        rc.load(x, src, sr[e], W, sr[e] >= 0, T(0));
#pragma unroll
        for (int c = 0; c < kCPL; ++c) v[c][e] = x[c];
      }
#pragma unroll
      for (int e = 0; e < kRR; ++e) {
        if (sr[e] < 0) continue;
        if (prev) rc.store(prev, sr[e], W, acc);
#pragma unroll
        for (int c = 0; c < kCPL; ++c) acc[c] = acc[c] + v[c][e];
      }
    }
    rc.store(dst, r, W, acc);
  }
}

// prev = +0.0 for source rows whose destination is outside [0, R).
template <typename T>
__global__ void rows_prev_skipped_kernel(const int32_t* __restrict__ idx, long long src_rows, long long offset,
                                         long long R, long long W, T* __restrict__ prev) {
  const long long s = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= src_rows) return;
  const long long r = (long long)idx[s] + offset;
  if (r >= 0 && r < R) return;
  for (long long j = 0; j < W; ++j) prev[s * W + j] = T(0);
}

}  // namespace
}  // namespace det

using namespace det;

extern "C" size_t det_scatter_add_rows_workspace_bytes(int64_t src_rows, int64_t dst_rows, int64_t row_len,
                                                       int dtype) {
  if (src_rows < 0 || dst_rows < 0 || row_len < 0 || !valid_dtype(dtype)) return 0;
  return make_sort_plan(src_rows, dst_rows, 0, true, 128).total;
}

template <typename T>
static int rows_impl(T* dst, long long R, long long W, const int32_t* idx, long long off, const T* src, long long M,
                     T* prev, void* ws, size_t ws_bytes, int bt, cudaStream_t s, bool ordered) {
  const SortPlan p = make_sort_plan(M, R, 0, true, bt);
  if (ws_bytes < p.total) return DET_ERR_WORKSPACE;
  if (M == 0 || W == 0) return cudaMemsetAsync(ws, 0, kHeaderBytes, s) == cudaSuccess ? DET_OK : DET_ERR_CUDA;
  int fb = 0;
  int rc = enqueue_sort(p, ws, idx, off, nullptr, nullptr, s, &fb);
  if (rc != DET_OK) return rc;
  char* w = reinterpret_cast<char*>(ws);
  SortHdr* h = reinterpret_cast<SortHdr*>(ws);
  if (prev) {
    launch_begin("det_rows_prev_skipped", s);
    rows_prev_skipped_kernel<T><<<(unsigned)((M + 255) / 256), 256, 0, s>>>(idx, M, off, R, W, prev);
    launch_end(s);
  }
  if (R > 0) {
    const int32_t* perm = reinterpret_cast<const int32_t*>(w + p.idx[fb]);
    const int32_t* seg = reinterpret_cast<const int32_t*>(w + p.seg);
    // pair accesses when every row starts on a pair boundary
    const uintptr_t pa = 2 * sizeof(T) - 1;
    const bool vec = W % 2 == 0 && (reinterpret_cast<uintptr_t>(dst) & pa) == 0 &&
                     (reinterpret_cast<uintptr_t>(src) & pa) == 0 && (reinterpret_cast<uintptr_t>(prev) & pa) == 0;
    const unsigned grid = (unsigned)((R * 32 + 255) / 256);
    launch_begin(ordered ? "det_rows_ordered" : "det_rows", s);
    if (ordered) {
      if (vec)
        rows_ordered_kernel<T, true><<<grid, 256, 0, s>>>(dst, R, W, src, perm, seg, &h->n_valid, prev, M);
      else
        rows_ordered_kernel<T, false><<<grid, 256, 0, s>>>(dst, R, W, src, perm, seg, &h->n_valid, prev, M);
    } else {
      if (vec)
        rows_kernel<T, true><<<grid, 256, 0, s>>>(dst, R, W, src, perm, seg, &h->n_valid, prev, M);
      else
        rows_kernel<T, false><<<grid, 256, 0, s>>>(dst, R, W, src, perm, seg, &h->n_valid, prev, M);
    }
    launch_end(s);
  }
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

static int rows_entry(void* dst, int64_t dst_rows, int64_t row_len, const int32_t* idx, int64_t row_offset,
                      const void* src, int64_t src_rows, void* prev_out, int dtype, void* workspace,
                      size_t workspace_bytes, int block_threads, void* stream, bool ordered) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (dst_rows < 0 || row_len < 0 || src_rows < 0 || !workspace || !valid_block_threads(block_threads))
    return DET_ERR_INVALID_ARG;
  if (src_rows > DET_MAX_RECORDS || dst_rows > 2147483647LL) return DET_ERR_TOO_LARGE;
  if (src_rows > 0 && (!idx || (row_len > 0 && !src))) return DET_ERR_INVALID_ARG;
  if (dst_rows > 0 && row_len > 0 && !dst) return DET_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return DET_ERR_WORKSPACE;
  if (dtype == DET_F32)
    return rows_impl<float>((float*)dst, dst_rows, row_len, idx, row_offset, (const float*)src, src_rows,
                            (float*)prev_out, workspace, workspace_bytes, block_threads, as_stream(stream), ordered);
  return rows_impl<double>((double*)dst, dst_rows, row_len, idx, row_offset, (const double*)src, src_rows,
                           (double*)prev_out, workspace, workspace_bytes, block_threads, as_stream(stream), ordered);
}

extern "C" int det_scatter_add_rows(void* dst, int64_t dst_rows, int64_t row_len, const int32_t* idx,
                                    int64_t row_offset, const void* src, int64_t src_rows, void* prev_out, int dtype,
                                    void* workspace, size_t workspace_bytes, int block_threads, void* stream) {
  return rows_entry(dst, dst_rows, row_len, idx, row_offset, src, src_rows, prev_out, dtype, workspace,
                    workspace_bytes, block_threads, stream, false);
}

// The ordered reading of "returns the previous value": source rows applied
// one at a time in ascending order (Warp language reference
// "warp.tile_atomic_add_indexed", returns).
extern "C" int det_scatter_add_rows_ordered(void* dst, int64_t dst_rows, int64_t row_len, const int32_t* idx,
                                            int64_t row_offset, const void* src, int64_t src_rows, void* prev_out,
                                            int dtype, void* workspace, size_t workspace_bytes, int block_threads,
                                            void* stream) {
  return rows_entry(dst, dst_rows, row_len, idx, row_offset, src, src_rows, prev_out, dtype, workspace,
                    workspace_bytes, block_threads, stream, true);
}
