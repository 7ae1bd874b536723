// det_scan_i32: reduce-then-scan over 4,096-element tiles.  Integer addition
// modulo 2^32 is associative, so the tiling does not change the result.
#include "det_iscan.cuh"

namespace det {

__global__ void __launch_bounds__(1024) iscan_tile_prefix(unsigned* __restrict__ tsum, long long T,
                                                          int32_t* __restrict__ total_out) {
  __shared__ unsigned wsum[32];
  const long long per = (T + blockDim.x - 1) / blockDim.x;
  const long long t0 = threadIdx.x * per, t1 = min(T, t0 + per);
  unsigned s = 0;
  for (long long t = t0; t < t1; ++t) s += tsum[t];
  unsigned total;
  unsigned run = iscan_cta_exclusive(s, wsum, total);
  for (long long t = t0; t < t1; ++t) {
    const unsigned v = tsum[t];
    tsum[t] = run;
    run += v;
  }
  if (threadIdx.x == 0 && total_out) *total_out = (int32_t)total;
}

namespace {

// Plain int32 array: 16 consecutive values per thread (16-byte loads when aligned).
struct I32Src {
  const int32_t* x;
  __device__ __forceinline__ void load(long long i0, long long n, unsigned (&v)[kIScanPer]) const {
    if (i0 + kIScanPer <= n && (reinterpret_cast<uintptr_t>(x + i0) & 15) == 0) {
#pragma unroll
      for (int q = 0; q < kIScanPer / 4; ++q) {
        const int4 w = __ldg(reinterpret_cast<const int4*>(x + i0) + q);
        v[4 * q] = (unsigned)w.x;
        v[4 * q + 1] = (unsigned)w.y;
        v[4 * q + 2] = (unsigned)w.z;
        v[4 * q + 3] = (unsigned)w.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < kIScanPer; ++e) v[e] = i0 + e < n ? (unsigned)__ldg(x + i0 + e) : 0u;
    }
  }
};

struct I32Dst {
  int32_t* y;
  int exclusive;
  __device__ __forceinline__ void store(long long i0, long long n, const unsigned (&ex)[kIScanPer],
                                        const unsigned (&v)[kIScanPer]) const {
    unsigned o[kIScanPer];
#pragma unroll
    for (int e = 0; e < kIScanPer; ++e) o[e] = exclusive ? ex[e] : ex[e] + v[e];
    if (i0 + kIScanPer <= n && (reinterpret_cast<uintptr_t>(y + i0) & 15) == 0) {
#pragma unroll
      for (int q = 0; q < kIScanPer / 4; ++q)
        reinterpret_cast<int4*>(y + i0)[q] =
            make_int4((int)o[4 * q], (int)o[4 * q + 1], (int)o[4 * q + 2], (int)o[4 * q + 3]);
    } else {
#pragma unroll
      for (int e = 0; e < kIScanPer; ++e)
        if (i0 + e < n) y[i0 + e] = (int32_t)o[e];
    }
  }
};

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
  return enqueue_iscan(I32Src{x}, I32Dst{y, exclusive ? 1 : 0}, n, total, reinterpret_cast<unsigned*>(ws), s);
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
