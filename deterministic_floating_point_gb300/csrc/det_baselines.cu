// Nondeterministic overhead baselines (see include/det_baselines.h).  Their
// association order is left to the scheduler on purpose; the deterministic
// calls are measured against them.
#include "det_common.cuh"
#include "../../include/det_baselines.h"

namespace det {
namespace {

template <typename T>
__device__ __forceinline__ T block_sum(T v, T* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) v += __shfl_down_sync(0xffffffffu, v, s);
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  T r = T(0);
  if (warp == 0) {
    r = lane < nw ? sh[lane] : T(0);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) r += __shfl_down_sync(0xffffffffu, r, s);
  }
  return r;
}

template <typename T>
__global__ void __launch_bounds__(256) atomic_sum_kernel(const T* __restrict__ x, long long n, T* out) {
  __shared__ T sh[32];
  T acc = T(0);
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) acc += x[i];
  const T bs = block_sum(acc, sh);
  if (threadIdx.x == 0) atomicAdd(out, bs);   // arrival order decides the addition order
}

template <typename T>
__global__ void atomic_scatter_kernel(T* out, long long m, const int32_t* __restrict__ bins,
                                      const T* __restrict__ values, long long n) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const long long b = bins[i];
    if (b >= 0 && b < m) atomicAdd(out + b, values[i]);
  }
}

__global__ void atomic_slot_kernel(int32_t* counter, long long C, const int32_t* __restrict__ index, long long off,
                                   const int32_t* __restrict__ count, long long n, int32_t* __restrict__ slot_out) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const long long c = (long long)index[i] + off;
    slot_out[i] = (c >= 0 && c < C) ? atomicAdd(counter + c, count ? count[i] : 1) : -1;
  }
}

template <typename T>
__global__ void atomic_rows_kernel(T* dst, long long R, long long W, const int32_t* __restrict__ idx, long long off,
                                   const T* __restrict__ src, long long M, T* prev) {
  const long long total = M * W;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
    const long long s = e / W, j = e - s * W;
    const long long r = (long long)idx[s] + off;
    T old = T(0);
    if (r >= 0 && r < R) old = atomicAdd(dst + r * W + j, src[e]);
    if (prev) prev[e] = old;
  }
}

// ---- plain decoupled look-back
template <typename T> struct DBits;
template <> struct DBits<float> {
  using U = unsigned int;
  static constexpr U S = 0xffffffffu;
};
template <> struct DBits<double> {
  using U = unsigned long long;
  static constexpr U S = 0xffffffffffffffffull;
};
__device__ __forceinline__ unsigned int dl_ld(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long dl_ld(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void dl_st(unsigned int* p, float v) {
  unsigned int b = __float_as_uint(v);
  if (b == 0xffffffffu) b = 0x7fc00000u;
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(b) : "memory");
}
__device__ __forceinline__ void dl_st(unsigned long long* p, double v) {
  unsigned long long b = (unsigned long long)__double_as_longlong(v);
  if (b == 0xffffffffffffffffull) b = 0x7ff8000000000000ull;
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(b) : "memory");
}
__device__ __forceinline__ float dl_val(unsigned int b) { return __uint_as_float(b); }
__device__ __forceinline__ double dl_val(unsigned long long b) { return __longlong_as_double((long long)b); }

constexpr int kDlbItems = 16;
constexpr int kDlbThreads = 256;
constexpr int kDlbChunk = kDlbItems * kDlbThreads;

template <typename T>
__global__ void __launch_bounds__(kDlbThreads) dlb_scan_kernel(const T* __restrict__ x, T* __restrict__ y, long long n,
                                                              typename DBits<T>::U* agg, typename DBits<T>::U* incl,
                                                              unsigned int* ticket, unsigned int* status) {
  using U = typename DBits<T>::U;
  __shared__ T wtot[kDlbThreads / 32];
  __shared__ T s_excl;
  __shared__ long long s_c;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_c = atomicAdd(ticket, 1u);
  __syncthreads();
  const long long c = s_c;
  const long long base = c * kDlbChunk + (long long)tid * kDlbItems;
  T v[kDlbItems];
  T tsum = T(0);
#pragma unroll
  for (int e = 0; e < kDlbItems; ++e) {
    v[e] = base + e < n ? x[base + e] : T(0);
    tsum += v[e];
  }
  T inc = tsum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const T o = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += o;
  }
  if (lane == 31) wtot[warp] = inc;
  __syncthreads();
  T wex = T(0), total = T(0);
  for (int w = 0; w < kDlbThreads / 32; ++w) {
    if (w < warp) wex += wtot[w];
    total += wtot[w];
  }
  if (warp == 0) {
    if (lane == 0) dl_st(agg + c, total);
    T run = T(0);
    long long q0 = c - 1;
    bool done = q0 < 0;
    const unsigned long long t0 = clock64();
    while (!done) {
      const long long q = q0 - lane;
      T val = T(0);
      bool isinc = true;
      if (q >= 0) {
        while (true) {
          const U bi = dl_ld(incl + q);
          if (bi != DBits<T>::S) {
            val = dl_val(bi);
            isinc = true;
            break;
          }
          const U ba = dl_ld(agg + q);
          if (ba != DBits<T>::S) {
            val = dl_val(ba);
            isinc = false;
            break;
          }
          if (clock64() - t0 > (1ull << 34)) {   // give up after a few seconds
            set_status(status, DET_ERR_LOOKBACK_TIMEOUT);
            break;
          }
        }
      }
      const unsigned im = __ballot_sync(0xffffffffu, isinc);
      const int f = __ffs(im) - 1;            // nearest inclusive predecessor in this window
      const int last = f < 0 ? 31 : f;        // no inclusive one: the whole window is partial
      T part = lane <= last ? val : T(0);
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) part += __shfl_xor_sync(0xffffffffu, part, s);
      run += part;
      done = true;
      if (f < 0) {
        done = false;
        q0 -= 32;
      }
    }
    if (lane == 0) {
      s_excl = run;
      dl_st(incl + c, run + total);
    }
  }
  __syncthreads();
  T acc = s_excl + wex + (inc - tsum);
#pragma unroll
  for (int e = 0; e < kDlbItems; ++e) {
    acc += v[e];
    if (base + e < n) y[base + e] = acc;
  }
}

}  // namespace
}  // namespace det

using namespace det;

static unsigned blocks_for(long long n, int threads) {
  long long b = (n + threads - 1) / threads;
  if (b > 4 * 152) b = 4 * 152;
  return (unsigned)(b < 1 ? 1 : b);
}

extern "C" int det_atomic_sum(const void* x, int64_t n, int dtype, void* out, void* stream) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (n < 0 || !out || (n > 0 && !x)) return DET_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  if (cudaMemsetAsync(out, 0, elem_size(dtype), s) != cudaSuccess) return DET_ERR_CUDA;
  if (n == 0) return DET_OK;
  launch_begin("atomic_sum", s);
  if (dtype == DET_F32)
    atomic_sum_kernel<float><<<blocks_for(n, 256), 256, 0, s>>>((const float*)x, n, (float*)out);
  else
    atomic_sum_kernel<double><<<blocks_for(n, 256), 256, 0, s>>>((const double*)x, n, (double*)out);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

extern "C" int det_atomic_scatter_add(void* out, int64_t out_len, const int32_t* bins, const void* values, int64_t n,
                                      int dtype, void* stream) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (n < 0 || out_len < 0 || (out_len > 0 && !out) || (n > 0 && (!bins || !values))) return DET_ERR_INVALID_ARG;
  if (n == 0) return DET_OK;
  cudaStream_t s = as_stream(stream);
  const unsigned g = (unsigned)min((long long)(n + 255) / 256, 16LL * 152);
  launch_begin("atomic_scatter_add", s);
  if (dtype == DET_F32)
    atomic_scatter_kernel<float><<<g, 256, 0, s>>>((float*)out, out_len, bins, (const float*)values, n);
  else
    atomic_scatter_kernel<double><<<g, 256, 0, s>>>((double*)out, out_len, bins, (const double*)values, n);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

extern "C" int det_atomic_scatter_add_rows(void* dst, int64_t dst_rows, int64_t row_len, const int32_t* idx,
                                           int64_t row_offset, const void* src, int64_t src_rows, void* prev_out,
                                           int dtype, void* stream) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (dst_rows < 0 || row_len < 0 || src_rows < 0) return DET_ERR_INVALID_ARG;
  if (src_rows > 0 && (!idx || (row_len > 0 && !src))) return DET_ERR_INVALID_ARG;
  if (dst_rows > 0 && row_len > 0 && !dst) return DET_ERR_INVALID_ARG;
  const long long total = src_rows * row_len;
  if (total == 0) return DET_OK;
  cudaStream_t s = as_stream(stream);
  const unsigned g = (unsigned)min((total + 255) / 256, 16LL * 152);
  launch_begin("atomic_scatter_add_rows", s);
  if (dtype == DET_F32)
    atomic_rows_kernel<float><<<g, 256, 0, s>>>((float*)dst, dst_rows, row_len, idx, row_offset, (const float*)src,
                                                src_rows, (float*)prev_out);
  else
    atomic_rows_kernel<double><<<g, 256, 0, s>>>((double*)dst, dst_rows, row_len, idx, row_offset,
                                                 (const double*)src, src_rows, (double*)prev_out);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

extern "C" size_t det_dlb_scan_workspace_bytes(int64_t n, int dtype) {
  if (n < 0 || !valid_dtype(dtype)) return 0;
  const long long nch = (n + kDlbChunk - 1) / kDlbChunk;
  return kHeaderBytes + 2 * align_up((size_t)(nch + 1) * elem_size(dtype), 256);
}

extern "C" int det_dlb_scan(const void* x, void* y, int64_t n, int dtype, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (n < 0 || !workspace || (n > 0 && (!x || !y))) return DET_ERR_INVALID_ARG;
  if (workspace_bytes < det_dlb_scan_workspace_bytes(n, dtype)) return DET_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  char* w = (char*)workspace;
  if (cudaMemsetAsync(w, 0, kHeaderBytes, s) != cudaSuccess) return DET_ERR_CUDA;
  if (n == 0) return DET_OK;
  const long long nch = (n + kDlbChunk - 1) / kDlbChunk;
  const size_t arr = align_up((size_t)(nch + 1) * elem_size(dtype), 256);
  if (cudaMemsetAsync(w + kHeaderBytes, 0xff, 2 * arr, s) != cudaSuccess) return DET_ERR_CUDA;
  WsHeader* h = reinterpret_cast<WsHeader*>(w);
  launch_begin("dlb_scan", s);
  if (dtype == DET_F32)
    dlb_scan_kernel<float><<<(unsigned)nch, kDlbThreads, 0, s>>>(
        (const float*)x, (float*)y, n, (unsigned int*)(w + kHeaderBytes), (unsigned int*)(w + kHeaderBytes + arr),
        &h->ticket, &h->status);
  else
    dlb_scan_kernel<double><<<(unsigned)nch, kDlbThreads, 0, s>>>(
        (const double*)x, (double*)y, n, (unsigned long long*)(w + kHeaderBytes),
        (unsigned long long*)(w + kHeaderBytes + arr), &h->ticket, &h->status);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

extern "C" int det_atomic_slot_alloc(int32_t* counter, int64_t num_counters, const int32_t* index, int64_t index_offset,
                                     const int32_t* count, int64_t n, int32_t* slot_out, void* stream) {
  if (n < 0 || num_counters < 0 || (num_counters > 0 && !counter) || (n > 0 && (!index || !slot_out)))
    return DET_ERR_INVALID_ARG;
  if (n == 0) return DET_OK;
  cudaStream_t s = as_stream(stream);
  const unsigned g = (unsigned)min((long long)((n + 255) / 256), 16LL * 152);
  launch_begin("det_atomic_slot_alloc", s);
  atomic_slot_kernel<<<g, 256, 0, s>>>(counter, num_counters, index, index_offset, count, n, slot_out);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}
