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

template <typename T> struct Pair2;
template <> struct Pair2<float> { using V = float2; };
template <> struct Pair2<double> { using V = double2; };

// W = 1: one thread per element.  Otherwise a warp takes 8 consecutive
// output rows at a time: the 8 row indices are loaded together (one round
// trip), then every lane's part of the 8 source rows, then the stores; with
// VEC (even W, pair-aligned arrays) a lane moves two adjacent columns as one
// access, so a warp covers 64 columns of a row per request.
constexpr int kGatherRows = 8;

template <typename T, bool VEC>
__global__ void __launch_bounds__(256)
gather_rows_kernel(T* __restrict__ out, const T* __restrict__ src, long long src_rows, long long W,
                   const int32_t* __restrict__ idx, long long off, long long n) {
  using V = typename Pair2<T>::V;
  if (W == 1) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
      const long long r = (long long)__ldg(idx + i) + off;
      out[i] = (r >= 0 && r < src_rows) ? __ldg(src + r) : T(0);
    }
    return;
  }
  constexpr int RB = kGatherRows;
  const int lane = threadIdx.x & 31;
  const long long nw = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long i0 = ((long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RB; i0 < n; i0 += nw * RB) {
    long long r[RB];
    bool ok[RB];
#pragma unroll
    for (int e = 0; e < RB; ++e) {
      const bool in = i0 + e < n;
      r[e] = in ? (long long)__ldg(idx + i0 + e) + off : -1;
      ok[e] = in && r[e] >= 0 && r[e] < src_rows;
    }
    if (VEC) {
      for (long long c = 2 * lane; c < W; c += 64) {
        V v[RB];
#pragma unroll
        for (int e = 0; e < RB; ++e) {
          if (ok[e]) {
            v[e] = __ldg(reinterpret_cast<const V*>(src + r[e] * W + c));
          } else {
            v[e].x = T(0);
            v[e].y = T(0);
          }
        }
#pragma unroll
        for (int e = 0; e < RB; ++e)
          if (i0 + e < n) *reinterpret_cast<V*>(out + (i0 + e) * W + c) = v[e];
      }
    } else {
      for (long long j = lane; j < W; j += 32) {
        T v[RB];
#pragma unroll
        for (int e = 0; e < RB; ++e) v[e] = ok[e] ? __ldg(src + r[e] * W + j) : T(0);
#pragma unroll
        for (int e = 0; e < RB; ++e)
          if (i0 + e < n) out[(i0 + e) * W + j] = v[e];
      }
    }
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
  const long long per_cta = row_len == 1 ? threads : (threads / 32) * kGatherRows;
  const long long grid = std::max(1LL, std::min((long long)((n + per_cta - 1) / per_cta), 16LL * std::max(device_sm_count(), 1)));
  const size_t es = dtype == DET_F32 ? 4 : 8;
  const bool vec = row_len % 2 == 0 && reinterpret_cast<uintptr_t>(out) % (2 * es) == 0 &&
                   (src_rows == 0 || reinterpret_cast<uintptr_t>(src) % (2 * es) == 0);
  launch_begin("det_gather_rows", s);
  if (dtype == DET_F32) {
    if (vec)
      gather_rows_kernel<float, true><<<(unsigned)grid, threads, 0, s>>>((float*)out, (const float*)src, src_rows,
                                                                         row_len, idx, row_offset, n);
    else
      gather_rows_kernel<float, false><<<(unsigned)grid, threads, 0, s>>>((float*)out, (const float*)src, src_rows,
                                                                          row_len, idx, row_offset, n);
  } else {
    if (vec)
      gather_rows_kernel<double, true><<<(unsigned)grid, threads, 0, s>>>((double*)out, (const double*)src, src_rows,
                                                                          row_len, idx, row_offset, n);
    else
      gather_rows_kernel<double, false><<<(unsigned)grid, threads, 0, s>>>((double*)out, (const double*)src, src_rows,
                                                                           row_len, idx, row_offset, n);
  }
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}
