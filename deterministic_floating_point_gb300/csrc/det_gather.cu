// det_gather_rows: out[i] = src[idx[i] + row_offset] row by row (+0.0 rows
// for indices outside src).  No element is combined with another, so any
// schedule gives the same bits.  It is the forward pass of Warp user guide
// "Deterministic Execution", "Tape and Backward Passes" (out[tid] =
// values[indices[tid]]); the deterministic adjoint is det_scatter_add_rows
// (det_scatter_add for width 1) of the output gradient.
#include "det_common.cuh"

#include <algorithm>

namespace det {
namespace {

// One warp per output row, lanes over columns (scalar gathers: one thread per element).
template <typename T>
__global__ void __launch_bounds__(256)
gather_rows_kernel(T* __restrict__ out, const T* __restrict__ src, long long src_rows, long long W,
                   const int32_t* __restrict__ idx, long long off, long long n) {
  if (W == 1) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
      const long long r = (long long)__ldg(idx + i) + off;
      out[i] = (r >= 0 && r < src_rows) ? __ldg(src + r) : T(0);
    }
    return;
  }
  const int lane = threadIdx.x & 31;
  const long long nw = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long i = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < n; i += nw) {
    const long long r = (long long)__ldg(idx + i) + off;
    const bool ok = r >= 0 && r < src_rows;
    for (long long j = lane; j < W; j += 32) out[i * W + j] = ok ? __ldg(src + r * W + j) : T(0);
  }
}

}  // namespace
}  // namespace det

using namespace det;

extern "C" int det_gather_rows(void* out, const void* src, int64_t src_rows, int64_t row_len, const int32_t* idx,
                               int64_t row_offset, int64_t n, int dtype, int block_threads, void* stream) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (src_rows < 0 || row_len < 0 || n < 0 || !valid_block_threads(block_threads)) return DET_ERR_INVALID_ARG;
  if (n > 0 && row_len > 0 && (!out || !idx || (src_rows > 0 && !src))) return DET_ERR_INVALID_ARG;
  if (n == 0 || row_len == 0) return DET_OK;
  const cudaStream_t s = as_stream(stream);
  const int threads = block_threads == 128 ? 128 : 256;   // the kernel is built for at most 256 threads
  const long long per_cta = row_len == 1 ? threads : threads / 32;
  const long long grid = std::max(1LL, std::min((long long)((n + per_cta - 1) / per_cta), 16LL * std::max(device_sm_count(), 1)));
  launch_begin("det_gather_rows", s);
  if (dtype == DET_F32)
    gather_rows_kernel<float><<<(unsigned)grid, threads, 0, s>>>((float*)out, (const float*)src, src_rows, row_len,
                                                                 idx, row_offset, n);
  else
    gather_rows_kernel<double><<<(unsigned)grid, threads, 0, s>>>((double*)out, (const double*)src, src_rows,
                                                                  row_len, idx, row_offset, n);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}
