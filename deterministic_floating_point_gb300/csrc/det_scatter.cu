// det_scatter_add: out[bins[i]] += values[i] with a fixed association order.
//
// Warp user guide "Deterministic Execution", "Pattern 1: Accumulation":
// instead of a floating-point atomic per record, the records are sorted
// stably by destination (ascending index inside a destination, as in
// "Picking the Right Mode") and each destination's group is reduced.  The
// group reduction here is the pairwise tree over the rank inside the group
// (not a sequential walk), and the old value is added once, last.
#include "det_sort.cuh"

using namespace det;

extern "C" size_t det_scatter_add_workspace_bytes(int64_t n, int64_t out_len, int dtype) {
  if (n < 0 || out_len < 0 || !valid_dtype(dtype)) return 0;
  // the largest plan: smallest tiles (128 threads) and the index payload
  return make_sort_plan(n, out_len, elem_size(dtype), true, 128).total;
}

template <typename T>
static int scatter_impl(T* out, long long m, const int32_t* bins, const T* values, long long n, int32_t* perm_out,
                        int32_t* seg_out, void* ws, size_t ws_bytes, int bt, cudaStream_t s, bool negate) {
  const SortPlan p = make_sort_plan(n, m, sizeof(T), perm_out != nullptr, bt);
  if (ws_bytes < p.total) return DET_ERR_WORKSPACE;
  int fb = 0;
  int rc = enqueue_sort(p, ws, bins, 0, values, perm_out, s, &fb);
  if (rc != DET_OK) return rc;
  const T* sorted = reinterpret_cast<const T*>(reinterpret_cast<char*>(ws) + p.vals[fb]);
  rc = enqueue_segmented_tree<T>(p, ws, sorted, out, s, negate);
  if (rc != DET_OK) return rc;
  if (seg_out && cudaMemcpyAsync(seg_out, reinterpret_cast<char*>(ws) + p.seg, (size_t)(m + 1) * 4,
                                 cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return DET_ERR_CUDA;
  return DET_OK;
}

static int scatter_entry(void* out, int64_t out_len, const int32_t* bins, const void* values, int64_t n, int dtype,
                         int32_t* perm_out, int32_t* seg_offsets_out, void* workspace, size_t workspace_bytes,
                         int block_threads, void* stream, bool negate) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (n < 0 || out_len < 0 || !workspace || !valid_block_threads(block_threads)) return DET_ERR_INVALID_ARG;
  if (n > DET_MAX_RECORDS || out_len > 2147483647LL) return DET_ERR_TOO_LARGE;
  if ((out_len > 0 && !out) || (n > 0 && (!bins || !values))) return DET_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return DET_ERR_WORKSPACE;
  if (dtype == DET_F32)
    return scatter_impl<float>((float*)out, out_len, bins, (const float*)values, n, perm_out, seg_offsets_out,
                               workspace, workspace_bytes, block_threads, as_stream(stream), negate);
  return scatter_impl<double>((double*)out, out_len, bins, (const double*)values, n, perm_out, seg_offsets_out,
                              workspace, workspace_bytes, block_threads, as_stream(stream), negate);
}

extern "C" int det_scatter_add(void* out, int64_t out_len, const int32_t* bins, const void* values, int64_t n,
                               int dtype, int32_t* perm_out, int32_t* seg_offsets_out, void* workspace,
                               size_t workspace_bytes, int block_threads, void* stream) {
  return scatter_entry(out, out_len, bins, values, n, dtype, perm_out, seg_offsets_out, workspace, workspace_bytes,
                       block_threads, stream, false);
}

// det_scatter_sub: the values negated and added in det_scatter_add's order
// (Warp "Deterministic Execution", "Pattern 1: Accumulation", atomic_sub).
extern "C" int det_scatter_sub(void* out, int64_t out_len, const int32_t* bins, const void* values, int64_t n,
                               int dtype, int32_t* perm_out, int32_t* seg_offsets_out, void* workspace,
                               size_t workspace_bytes, int block_threads, void* stream) {
  return scatter_entry(out, out_len, bins, values, n, dtype, perm_out, seg_offsets_out, workspace, workspace_bytes,
                       block_threads, stream, true);
}
