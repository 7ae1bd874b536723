// det_scan_i32: reduce-then-scan over 4,096-element tiles.  Integer addition
// modulo 2^32 is associative, so the tiling does not change the result.
#include "det_iscan.cuh"

namespace det {
namespace {

constexpr int kPer = 16;   // elements per thread

// Load this thread's kPer consecutive elements of tile t (zeros past n).
__device__ __forceinline__ void load16(const int32_t* __restrict__ x, long long n, long long i0, unsigned (&v)[kPer]) {
  if (i0 + kPer <= n && (reinterpret_cast<uintptr_t>(x + i0) & 15) == 0) {
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q) {
      const int4 w = __ldg(reinterpret_cast<const int4*>(x + i0) + q);
      v[4 * q] = (unsigned)w.x;
      v[4 * q + 1] = (unsigned)w.y;
      v[4 * q + 2] = (unsigned)w.z;
      v[4 * q + 3] = (unsigned)w.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < kPer; ++e) v[e] = i0 + e < n ? (unsigned)__ldg(x + i0 + e) : 0u;
  }
}

// Exclusive scan of one value per thread over a CTA of 256 threads; also
// returns the CTA total.
__device__ __forceinline__ unsigned cta_exclusive(unsigned v, unsigned* wsum, unsigned& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned o = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += o;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned w = lane < nw ? wsum[lane] : 0u;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const unsigned o = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += o;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  total = wsum[nw - 1];
  const unsigned r = (warp ? wsum[warp - 1] : 0u) + x - v;
  __syncthreads();   // wsum may be reused
  return r;
}

__global__ void __launch_bounds__(256) iscan_tile_sums(const int32_t* __restrict__ x, long long n,
                                                       unsigned* __restrict__ tsum) {
  __shared__ unsigned wsum[32];
  unsigned v[kPer];
  load16(x, n, blockIdx.x * kIScanTile + (long long)threadIdx.x * kPer, v);
  unsigned s = 0;
#pragma unroll
  for (int e = 0; e < kPer; ++e) s += v[e];
  unsigned total;
  cta_exclusive(s, wsum, total);
  if (threadIdx.x == 0) tsum[blockIdx.x] = total;
}

// One CTA of 1024 threads: exclusive scan of the tile sums in place.
__global__ void __launch_bounds__(1024) iscan_tile_prefix(unsigned* __restrict__ tsum, long long T,
                                                          int32_t* __restrict__ total_out) {
  __shared__ unsigned wsum[32];
  const long long per = (T + blockDim.x - 1) / blockDim.x;
  const long long t0 = threadIdx.x * per, t1 = min(T, t0 + per);
  unsigned s = 0;
  for (long long t = t0; t < t1; ++t) s += tsum[t];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned x = s;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned o = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += o;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned w = wsum[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const unsigned o = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += o;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  unsigned run = (warp ? wsum[warp - 1] : 0u) + x - s;
  for (long long t = t0; t < t1; ++t) {
    const unsigned v = tsum[t];
    tsum[t] = run;
    run += v;
  }
  if (threadIdx.x == blockDim.x - 1 && total_out) *total_out = (int32_t)run;
}

__global__ void __launch_bounds__(256) iscan_tiles(const int32_t* x, int32_t* y, long long n,
                                                   const unsigned* __restrict__ tpre, int exclusive) {
  __shared__ unsigned wsum[32];
  const long long i0 = blockIdx.x * kIScanTile + (long long)threadIdx.x * kPer;
  unsigned v[kPer];
  load16(x, n, i0, v);   // the whole tile is read before any of it is written (x may be y)
  unsigned s = 0;
#pragma unroll
  for (int e = 0; e < kPer; ++e) s += v[e];
  unsigned total;
  unsigned run = tpre[blockIdx.x] + cta_exclusive(s, wsum, total);
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const unsigned inc = run + v[e];
    v[e] = exclusive ? run : inc;
    run = inc;
  }
  if (i0 + kPer <= n && (reinterpret_cast<uintptr_t>(y + i0) & 15) == 0) {
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q)
      reinterpret_cast<int4*>(y + i0)[q] =
          make_int4((int)v[4 * q], (int)v[4 * q + 1], (int)v[4 * q + 2], (int)v[4 * q + 3]);
  } else {
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      if (i0 + e < n) y[i0 + e] = (int32_t)v[e];
  }
}

}  // namespace

size_t iscan_ws_bytes(long long n) {
  const long long T = (n + kIScanTile - 1) / kIScanTile;
  return align_up((size_t)(T + 1) * 4, 256);
}

int enqueue_scan_i32(const int32_t* x, int32_t* y, long long n, bool exclusive, int32_t* total, void* ws,
                     cudaStream_t s) {
  if (n == 0) {
    if (total && cudaMemsetAsync(total, 0, 4, s) != cudaSuccess) return DET_ERR_CUDA;
    return DET_OK;
  }
  const long long T = (n + kIScanTile - 1) / kIScanTile;
  unsigned* tsum = reinterpret_cast<unsigned*>(ws);
  launch_begin("det_iscan_sums", s);
  iscan_tile_sums<<<(unsigned)T, 256, 0, s>>>(x, n, tsum);
  launch_end(s);
  launch_begin("det_iscan_prefix", s);
  iscan_tile_prefix<<<1, 1024, 0, s>>>(tsum, T, total);
  launch_end(s);
  launch_begin("det_iscan_tiles", s);
  iscan_tiles<<<(unsigned)T, 256, 0, s>>>(x, y, n, tsum, exclusive ? 1 : 0);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

}  // namespace det

using namespace det;

extern "C" size_t det_scan_i32_workspace_bytes(int64_t n) {
  if (n < 0) return 0;
  return kHeaderBytes + iscan_ws_bytes(n);
}

extern "C" int det_scan_i32(const int32_t* x, int32_t* y, int64_t n, int flags, int32_t* total_out, void* workspace,
                            size_t workspace_bytes, int block_threads, void* stream) {
  if (n < 0 || !workspace || (flags & ~DET_SCAN_EXCLUSIVE) || !valid_block_threads(block_threads))
    return DET_ERR_INVALID_ARG;
  if (n > 0 && (!x || !y)) return DET_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return DET_ERR_WORKSPACE;
  if (workspace_bytes < det_scan_i32_workspace_bytes(n)) return DET_ERR_WORKSPACE;
  const cudaStream_t s = as_stream(stream);
  if (cudaMemsetAsync(workspace, 0, kHeaderBytes, s) != cudaSuccess) return DET_ERR_CUDA;
  return enqueue_scan_i32(x, y, n, (flags & DET_SCAN_EXCLUSIVE) != 0, total_out,
                          reinterpret_cast<char*>(workspace) + kHeaderBytes, s);
}
