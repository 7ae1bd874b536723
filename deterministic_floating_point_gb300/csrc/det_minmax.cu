// det_scatter_min / det_scatter_max: out[b] = minimum(out[b], values of
// group b) (maximum), for the bins that receive at least one record.
//
// Warp user guide "Deterministic Execution", "Pattern 1: Accumulation": the
// atomic_min / atomic_max rows group the values by destination and minimize
// (maximize) them.  The pages leave signed zeros and NaN open; here the
// operation is IEEE 754-2019 minimum / maximum (a NaN operand gives NaN,
// -0 orders below +0).  That operation is associative and commutative, so
// every order of combination gives the same bits and no sort is needed: each
// value is mapped to an unsigned key whose integer order is that total order
// (NaN mapped to the key that always wins), and integer atomics, exact and
// order-free, combine the keys.  NaN results are the canonical quiet NaN
// (payloads are not promised); bins without records keep their bits.
#include "det_common.cuh"

#include <algorithm>

namespace det {
namespace {

template <typename T> struct KeyOf;
template <> struct KeyOf<float> { using U = unsigned int; };
template <> struct KeyOf<double> { using U = unsigned long long; };

// Largest bin count whose keys a CTA keeps in shared memory.
constexpr long long kSmemBins = 8192;

template <typename T, bool MAX>
__device__ __forceinline__ typename KeyOf<T>::U to_key(T x) {
  using U = typename KeyOf<T>::U;
  constexpr U kSign = U(1) << (8 * sizeof(U) - 1);
  if (x != x) return MAX ? ~U(0) : U(0);   // no other value maps to these keys
  U u;
  memcpy(&u, &x, sizeof(u));
  return (u & kSign) ? ~u : (u | kSign);
}

template <typename T, bool MAX>
__device__ __forceinline__ T from_key(typename KeyOf<T>::U k) {
  using U = typename KeyOf<T>::U;
  constexpr U kSign = U(1) << (8 * sizeof(U) - 1);
  U u;
  if (k == (MAX ? ~U(0) : U(0)))
    u = sizeof(T) == 4 ? U(0x7fc00000u) : U(0x7ff8000000000000ull);   // canonical quiet NaN
  else
    u = (k & kSign) ? (k & ~kSign) : ~k;
  T x;
  memcpy(&x, &u, sizeof(x));
  return x;
}

// The key no value maps to: the identity of the combination.
template <typename T, bool MAX>
__device__ __forceinline__ typename KeyOf<T>::U identity_key() {
  using U = typename KeyOf<T>::U;
  return MAX ? U(0) : ~U(0);
}

template <bool MAX>
__device__ __forceinline__ unsigned int key_atomic(unsigned int* p, unsigned int k) {
  return MAX ? atomicMax(p, k) : atomicMin(p, k);
}
template <bool MAX>
__device__ __forceinline__ unsigned long long key_atomic(unsigned long long* p, unsigned long long k) {
  return MAX ? atomicMax(p, k) : atomicMin(p, k);
}

// Each lane takes 16 consecutive records per step (16-byte loads, all in
// flight before any is combined; the order of combination is free) and
// combines each run of one bin among them in registers, applying one atomic
// per run: a hot bin (every record in one bin) costs one atomic per 16
// records instead of one per record.  (A warp-wide grouping of the lanes
// that share lane 0's bin, by a shuffle and a ballot per record, measured 2 %
// slower on 1,024 uniform bins and 15 % slower with every record in one bin.)  m <= kSmemBins keeps the bins'
// keys in shared memory per CTA and folds them into the global keys at the end.
constexpr int kPerLane = 16;

template <typename T, bool MAX, bool SMEM>
__global__ void __launch_bounds__(256)
minmax_scatter_kernel(const int32_t* __restrict__ bins, const T* __restrict__ values, long long n, long long m,
                      typename KeyOf<T>::U* __restrict__ gkeys) {
  using U = typename KeyOf<T>::U;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  U* skeys = reinterpret_cast<U*>(smem_raw);
  if (SMEM) {
    for (long long b = threadIdx.x; b < m; b += blockDim.x) skeys[b] = identity_key<T, MAX>();
    __syncthreads();
  }
  U* keys = SMEM ? skeys : gkeys;
  const int lane = threadIdx.x & 31;
  const long long wchunk = 32LL * kPerLane;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (long long base = wid * wchunk; base < n; base += nwarps * wchunk) {   // whole warps step together
    const long long i0 = base + (long long)lane * kPerLane;
    int32_t bb[kPerLane];
    T vv[kPerLane];
    if (i0 + kPerLane <= n && (reinterpret_cast<uintptr_t>(bins + i0) & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(values + i0) & 15) == 0) {
#pragma unroll
      for (int q = 0; q < kPerLane / 4; ++q) {
        const int4 w = __ldg(reinterpret_cast<const int4*>(bins + i0) + q);
        bb[4 * q] = w.x, bb[4 * q + 1] = w.y, bb[4 * q + 2] = w.z, bb[4 * q + 3] = w.w;
      }
      if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int q = 0; q < kPerLane / 4; ++q) {
          const float4 w = __ldg(reinterpret_cast<const float4*>(values + i0) + q);
          vv[4 * q] = w.x, vv[4 * q + 1] = w.y, vv[4 * q + 2] = w.z, vv[4 * q + 3] = w.w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < kPerLane / 2; ++q) {
          const double2 w = __ldg(reinterpret_cast<const double2*>(values + i0) + q);
          vv[2 * q] = w.x, vv[2 * q + 1] = w.y;
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < kPerLane; ++e) {
        const bool in = i0 + e < n;
        bb[e] = in ? __ldg(bins + i0 + e) : -1;
        vv[e] = in ? __ldg(values + i0 + e) : T(0);
      }
    }
    // runs of one bin among the lane's consecutive records are combined in
    // registers first: one atomic per run
    int cb = bb[0];
    U acc = to_key<T, MAX>(vv[0]);
#pragma unroll
    for (int e = 1; e < kPerLane; ++e) {
      const U k = to_key<T, MAX>(vv[e]);
      if (bb[e] == cb) {
        acc = MAX ? (acc > k ? acc : k) : (acc < k ? acc : k);
      } else {
        if (cb >= 0 && (long long)cb < m) key_atomic<MAX>(keys + cb, acc);
        cb = bb[e];
        acc = k;
      }
    }
    if (cb >= 0 && (long long)cb < m) key_atomic<MAX>(keys + cb, acc);
  }
  if (SMEM) {
    __syncthreads();
    for (long long b = threadIdx.x; b < m; b += blockDim.x)
      if (skeys[b] != identity_key<T, MAX>()) key_atomic<MAX>(gkeys + b, skeys[b]);
  }
}

// out[b] = op(out[b], group) for the bins that received a record.
template <typename T, bool MAX>
__global__ void minmax_finish_kernel(T* __restrict__ out, long long m, const typename KeyOf<T>::U* __restrict__ gkeys) {
  const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= m) return;
  const auto k = gkeys[b];
  if (k == identity_key<T, MAX>()) return;
  const auto ko = to_key<T, MAX>(out[b]);
  out[b] = from_key<T, MAX>(MAX ? (ko > k ? ko : k) : (ko < k ? ko : k));
}

template <typename T, bool MAX>
int minmax_impl(T* out, long long m, const int32_t* bins, const T* values, long long n, void* ws, int bt,
                cudaStream_t s) {
  using U = typename KeyOf<T>::U;
  U* gkeys = reinterpret_cast<U*>(reinterpret_cast<char*>(ws) + kHeaderBytes);
  if (cudaMemsetAsync(ws, 0, kHeaderBytes, s) != cudaSuccess) return DET_ERR_CUDA;
  if (m == 0) return DET_OK;
  if (cudaMemsetAsync(gkeys, MAX ? 0x00 : 0xff, (size_t)m * sizeof(U), s) != cudaSuccess) return DET_ERR_CUDA;
  const int sms = device_sm_count();
  const int threads = bt == 128 ? 128 : 256;   // the kernel is built for at most 256 threads
  if (n > 0) {
    const bool smem = m <= kSmemBins;
    const long long want = (n + (long long)threads * 64 - 1) / ((long long)threads * 64);   // >= 64 records per thread
    const long long grid = std::max(1LL, std::min(want, 4LL * std::max(sms, 1)));
    const size_t sb = smem ? (size_t)m * sizeof(U) : 0;   // up to 64 KB: above the default 48 KB for f64
    if (smem && ensure_dyn_smem((const void*)minmax_scatter_kernel<T, MAX, true>, sb) != cudaSuccess)
      return DET_ERR_CUDA;
    launch_begin("det_minmax_scatter", s);
    if (smem)
      minmax_scatter_kernel<T, MAX, true><<<(unsigned)grid, threads, sb, s>>>(bins, values, n, m, gkeys);
    else
      minmax_scatter_kernel<T, MAX, false><<<(unsigned)grid, threads, 0, s>>>(bins, values, n, m, gkeys);
    launch_end(s);
  }
  launch_begin("det_minmax_finish", s);
  minmax_finish_kernel<T, MAX><<<(unsigned)((m + 255) / 256), 256, 0, s>>>(out, m, gkeys);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

int minmax_entry(void* out, int64_t out_len, const int32_t* bins, const void* values, int64_t n, int dtype,
                 void* workspace, size_t workspace_bytes, int block_threads, void* stream, bool is_max) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (n < 0 || out_len < 0 || !workspace || !valid_block_threads(block_threads)) return DET_ERR_INVALID_ARG;
  if (n > DET_MAX_RECORDS || out_len > 2147483647LL) return DET_ERR_TOO_LARGE;
  if ((out_len > 0 && !out) || (n > 0 && (!bins || !values))) return DET_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return DET_ERR_WORKSPACE;
  if (workspace_bytes < kHeaderBytes + (size_t)out_len * elem_size(dtype)) return DET_ERR_WORKSPACE;
  const cudaStream_t s = as_stream(stream);
  if (dtype == DET_F32)
    return is_max ? minmax_impl<float, true>((float*)out, out_len, bins, (const float*)values, n, workspace,
                                             block_threads, s)
                  : minmax_impl<float, false>((float*)out, out_len, bins, (const float*)values, n, workspace,
                                              block_threads, s);
  return is_max ? minmax_impl<double, true>((double*)out, out_len, bins, (const double*)values, n, workspace,
                                            block_threads, s)
                : minmax_impl<double, false>((double*)out, out_len, bins, (const double*)values, n, workspace,
                                             block_threads, s);
}

}  // namespace
}  // namespace det

using namespace det;

extern "C" size_t det_scatter_minmax_workspace_bytes(int64_t out_len, int dtype) {
  if (out_len < 0 || !valid_dtype(dtype)) return 0;
  return align_up(kHeaderBytes + (size_t)out_len * elem_size(dtype), 256);
}

extern "C" int det_scatter_min(void* out, int64_t out_len, const int32_t* bins, const void* values, int64_t n,
                               int dtype, void* workspace, size_t workspace_bytes, int block_threads, void* stream) {
  return minmax_entry(out, out_len, bins, values, n, dtype, workspace, workspace_bytes, block_threads, stream, false);
}

extern "C" int det_scatter_max(void* out, int64_t out_len, const int32_t* bins, const void* values, int64_t n,
                               int dtype, void* workspace, size_t workspace_bytes, int block_threads, void* stream) {
  return minmax_entry(out, out_len, bins, values, n, dtype, workspace, workspace_bytes, block_threads, stream, true);
}
