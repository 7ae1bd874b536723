// int32 prefix sums (modular, so every order of the additions gives the same
// bits): the count -> exclusive scan -> write step of deterministic slot
// allocation (Warp user guide "Deterministic Execution", "Pattern 2: Slot
// Allocation" and "Picking the Right Mode").
//
// Reduce-then-scan over tiles of 4,096 elements (256 threads x 16): tile
// sums, one CTA scanning the tile sums, then each tile's exclusive prefixes.
// The tile kernels read their values through a source and hand the exclusive
// prefixes to a sink, so the same scan serves a plain int32 array and the
// slot requests of a single allocation counter.
#pragma once
#include "det_common.cuh"

namespace det {

constexpr long long kIScanTile = 4096;   // elements per CTA of 256 threads
constexpr int kIScanPer = 16;            // elements per thread

// Workspace bytes of the tile sums for n elements (no header).
size_t iscan_ws_bytes(long long n);

// y[i] = x[0] + ... + x[i] (inclusive) or x[0] + ... + x[i-1] (exclusive),
// modulo 2^32; *total (device, may be null) = the sum of all n values.
// x may equal y.  ws: iscan_ws_bytes(n) bytes, 256-byte aligned.
int enqueue_scan_i32(const int32_t* x, int32_t* y, long long n, bool exclusive, int32_t* total, void* ws,
                     cudaStream_t s);

// Exclusive scan of one value per thread over the CTA; also the CTA total.
__device__ __forceinline__ unsigned iscan_cta_exclusive(unsigned v, unsigned* wsum, unsigned& total) {
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

// tsum[t] = sum of the source's values in tile t.
template <class Src>
__global__ void __launch_bounds__(256) iscan_tile_sums(Src src, long long n, unsigned* __restrict__ tsum) {
  __shared__ unsigned wsum[32];
  unsigned v[kIScanPer];
  src.load(blockIdx.x * kIScanTile + (long long)threadIdx.x * kIScanPer, n, v);
  unsigned s = 0;
#pragma unroll
  for (int e = 0; e < kIScanPer; ++e) s += v[e];
  unsigned total;
  iscan_cta_exclusive(s, wsum, total);
  if (threadIdx.x == 0) tsum[blockIdx.x] = total;
}

// One CTA of 1024 threads: exclusive scan of the tile sums in place; the sum
// of all tiles goes to *total_out (if not null).
__global__ void __launch_bounds__(1024) iscan_tile_prefix(unsigned* __restrict__ tsum, long long T,
                                                          int32_t* __restrict__ total_out);

// Each tile: its values' exclusive prefixes (plus the tile's prefix) to the sink.
template <class Src, class Dst>
__global__ void __launch_bounds__(256) iscan_tiles(Src src, Dst dst, long long n, const unsigned* __restrict__ tpre) {
  __shared__ unsigned wsum[32];
  const long long i0 = blockIdx.x * kIScanTile + (long long)threadIdx.x * kIScanPer;
  unsigned v[kIScanPer];
  src.load(i0, n, v);   // the whole tile is read before any of it is written (in-place use)
  unsigned s = 0;
#pragma unroll
  for (int e = 0; e < kIScanPer; ++e) s += v[e];
  unsigned total;
  unsigned run = tpre[blockIdx.x] + iscan_cta_exclusive(s, wsum, total);
  unsigned ex[kIScanPer];
#pragma unroll
  for (int e = 0; e < kIScanPer; ++e) {
    ex[e] = run;
    run += v[e];
  }
  dst.store(i0, n, ex, v);
}

// Launch the three kernels over n elements (tsum: iscan_ws_bytes(n) bytes).
template <class Src, class Dst>
int enqueue_iscan(Src src, Dst dst, long long n, int32_t* total, unsigned* tsum, cudaStream_t s) {
  const long long T = (n + kIScanTile - 1) / kIScanTile;
  launch_begin("det_iscan_sums", s);
  iscan_tile_sums<Src><<<(unsigned)T, 256, 0, s>>>(src, n, tsum);
  launch_end(s);
  launch_begin("det_iscan_prefix", s);
  iscan_tile_prefix<<<1, 1024, 0, s>>>(tsum, T, total);
  launch_end(s);
  launch_begin("det_iscan_tiles", s);
  iscan_tiles<Src, Dst><<<(unsigned)T, 256, 0, s>>>(src, dst, n, tsum);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

}  // namespace det
