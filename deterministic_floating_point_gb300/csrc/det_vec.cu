// det_scatter_add_vec: composite values (vec3, mat33, ...: `width`
// components per record) scattered with wp.atomic_add's deterministic form.
// Warp user guide "Deterministic Execution", "Pattern 1: Accumulation":
// vectors, matrices, quaternions and transforms take the same segmented
// reduction path as scalars, component by component.  Here: one stable sort
// of the records by destination that lays each component out in sorted
// order, then per component the scalar segmented tree:
// out[b][c] = out[b][c] + PT(component c of group b).  A one-pass sort of
// records of at most 16 bytes carries the whole record through the pass;
// otherwise the sort carries the record index and a gather follows.
#include "det_sort.cuh"

#include <algorithm>

namespace det {
namespace {

// comp[c * n + p] = values[perm[p] * width + c] for sorted positions p.
template <typename T>
__global__ void __launch_bounds__(256)
vec_gather_kernel(const T* __restrict__ values, long long width, const int32_t* __restrict__ perm,
                  const unsigned int* __restrict__ n_valid, long long n, T* __restrict__ comp) {
  const long long N = min((long long)*n_valid, n);
  for (long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x; p < N; p += (long long)gridDim.x * blockDim.x) {
    const long long r = perm[p];
    if (r < 0 || r >= n) continue;   // cannot happen for a correct sort
    for (long long c = 0; c < width; ++c) comp[c * n + p] = __ldg(values + r * width + c);
  }
}

struct VecLayout {
  SortPlan plan;
  size_t comp = 0, total = 0;
};

VecLayout vec_layout(long long n, long long m, long long width, int elem, int bt) {
  VecLayout L;
  L.plan = make_sort_plan(n, m, 0, true, bt);
  L.comp = align_up(L.plan.total, 256);
  L.total = align_up(L.comp + (size_t)width * n * elem, 256);
  return L;
}

template <typename T>
int vec_impl(T* out, long long m, long long width, const int32_t* bins, const T* values, long long n, void* ws,
             size_t ws_bytes, int bt, cudaStream_t s) {
  const VecLayout L = vec_layout(n, m, width, sizeof(T), bt);
  if (ws_bytes < L.total) return DET_ERR_WORKSPACE;
  if (n == 0 || m == 0 || width == 0)
    return cudaMemsetAsync(ws, 0, kHeaderBytes, s) == cudaSuccess ? DET_OK : DET_ERR_CUDA;
  char* w = reinterpret_cast<char*>(ws);
  SortHdr* h = reinterpret_cast<SortHdr*>(ws);
  T* comp = reinterpret_cast<T*>(w + L.comp);
  int fb = 0;
  SortPlan q = make_sort_plan(n, m, 0, false, 128);   // tiles of 4,096: the records fill shared memory
  if (q.passes == 1 && width * (long long)sizeof(T) <= 16 && q.total <= L.comp) {
    // records through the pass: no index, no gather (the plan's workspace
    // ends before the component arrays at L.comp)
    q.wide = (int)width;
    q.wide_elem = (int)sizeof(T);
    int rc = enqueue_sort(q, ws, bins, 0, values, nullptr, s, &fb, nullptr, comp);
    if (rc != DET_OK) return rc;
    for (long long c = 0; c < width; ++c) {
      rc = enqueue_segmented_tree<T>(q, ws, comp + c * n, out + c, s, false, width, c > 0);
      if (rc != DET_OK) return rc;
    }
    return DET_OK;
  }
  const SortPlan& p = L.plan;
  int rc = enqueue_sort(p, ws, bins, 0, nullptr, nullptr, s, &fb);
  if (rc != DET_OK) return rc;
  // one thread per record: many independent gathers in flight
  const long long grid = std::max(1LL, (long long)((n + 255) / 256));
  launch_begin("det_vec_gather", s);
  vec_gather_kernel<T><<<(unsigned)grid, 256, 0, s>>>(values, width, reinterpret_cast<const int32_t*>(w + p.idx[fb]),
                                                       &h->n_valid, n, comp);
  launch_end(s);
  if (cudaGetLastError() != cudaSuccess) return DET_ERR_CUDA;
  for (long long c = 0; c < width; ++c) {
    rc = enqueue_segmented_tree<T>(p, ws, comp + c * n, out + c, s, false, width, c > 0);
    if (rc != DET_OK) return rc;
  }
  return DET_OK;
}

}  // namespace
}  // namespace det

using namespace det;

extern "C" size_t det_scatter_add_vec_workspace_bytes(int64_t n, int64_t out_len, int64_t width, int dtype) {
  if (n < 0 || out_len < 0 || width < 0 || !valid_dtype(dtype)) return 0;
  return vec_layout(n, out_len, width, elem_size(dtype), 128).total;   // the largest plan: 128-thread tiles
}

extern "C" int det_scatter_add_vec(void* out, int64_t out_len, int64_t width, const int32_t* bins, const void* values,
                                   int64_t n, int dtype, void* workspace, size_t workspace_bytes, int block_threads,
                                   void* stream) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (n < 0 || out_len < 0 || width < 0 || !workspace || !valid_block_threads(block_threads))
    return DET_ERR_INVALID_ARG;
  if (n > DET_MAX_RECORDS || out_len > 2147483647LL || width > 4096) return DET_ERR_TOO_LARGE;
  if ((out_len > 0 && width > 0 && !out) || (n > 0 && (!bins || (width > 0 && !values)))) return DET_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return DET_ERR_WORKSPACE;
  if (dtype == DET_F32)
    return vec_impl<float>((float*)out, out_len, width, bins, (const float*)values, n, workspace, workspace_bytes,
                           block_threads, as_stream(stream));
  return vec_impl<double>((double*)out, out_len, width, bins, (const double*)values, n, workspace, workspace_bytes,
                          block_threads, as_stream(stream));
}
