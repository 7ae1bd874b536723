// Arithmetic-rate probe for the measurement hooks (det_profile.h): how many
// floating-point adds per second the SMs retire when nothing else limits
// them.  The f64 sum and scan can be bound by GB300's FP64 add rate rather
// than by HBM; this gives the measured rate to set beside the nominal one.
//
// Each thread runs kChains independent chains of dependent adds of a tiny
// increment, from registers only (no memory traffic), so the add pipe is the
// only resource the launch exercises.
#include "det_common.cuh"
#include "../../include/det_profile.h"

namespace det {
namespace {

constexpr int kChains = 8;
constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 8;

template <typename T>
__global__ void __launch_bounds__(kThreads) add_rate_kernel(T* sink, int iters, T inc) {
  T v[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) v[c] = T(threadIdx.x + c);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) v[c] = v[c] + inc;
  }
  T s = v[0];
#pragma unroll
  for (int c = 1; c < kChains; ++c) s = s + v[c];
  if (s == T(-1)) sink[0] = s;   // never true; keeps every chain live
}

}  // namespace
}  // namespace det

using namespace det;

extern "C" int det_profile_add_rate_probe(int dtype, int iters, void* sink, void* stream,
                                          unsigned long long* adds_out) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (iters <= 0 || !sink || !adds_out) return DET_ERR_INVALID_ARG;
  const int sms = device_sm_count();
  if (sms <= 0) return DET_ERR_CUDA;
  const unsigned blocks = (unsigned)(sms * kBlocksPerSm);
  const cudaStream_t s = as_stream(stream);
  launch_begin("det_add_rate_probe", s);
  if (dtype == DET_F32)
    add_rate_kernel<float><<<blocks, kThreads, 0, s>>>((float*)sink, iters, 1e-9f);
  else
    add_rate_kernel<double><<<blocks, kThreads, 0, s>>>((double*)sink, iters, 1e-9);
  launch_end(s);
  *adds_out = (unsigned long long)blocks * kThreads * (unsigned long long)iters * kChains;
  return check_launch("det_profile_add_rate_probe");
}
