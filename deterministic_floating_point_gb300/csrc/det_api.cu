// Status reporting and measurement hooks for the C ABI.
#include "det_common.cuh"

#include <atomic>
#include <cstdio>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>
#include "../../include/det_profile.h"

namespace {
struct Profile {
  cudaEvent_t* events = nullptr;
  int capacity = 0;
  int count = 0;
  int open = 0;
  const char* names[4096];
};
Profile g_prof;
unsigned long long g_launches = 0;
}  // namespace

namespace det {
namespace {
constexpr int kAttrDevices = 64;
std::atomic<int> g_sms[kAttrDevices];
std::atomic<int> g_smem[kAttrDevices];
std::mutex g_dyn_mu;
std::map<std::pair<const void*, int>, size_t> g_dyn;

int cached_attr(std::atomic<int>* cache, cudaDeviceAttr attr) {
  int dev = 0;
  cudaGetDevice(&dev);
  int v = (dev >= 0 && dev < kAttrDevices) ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (v == 0) {
    cudaDeviceGetAttribute(&v, attr, dev);
    if (dev >= 0 && dev < kAttrDevices && v > 0) cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}
}  // namespace

namespace {
std::mutex g_err_mu;
char g_err[256] = "";
}  // namespace

int cuda_fail(cudaError_t e, const char* where) {
  std::lock_guard<std::mutex> lk(g_err_mu);
  snprintf(g_err, sizeof(g_err), "%s: %s", where, cudaGetErrorName(e));
  return DET_ERR_CUDA;
}

const char* last_cuda_error() { return g_err; }

int device_sm_count() { return cached_attr(g_sms, cudaDevAttrMultiProcessorCount); }
int device_max_smem_optin() { return cached_attr(g_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin); }

cudaError_t ensure_dyn_smem(const void* kernel, size_t bytes) {
  // within the default limit even with a kernel's static shared arrays (the
  // 48 KB default covers static + dynamic bytes)
  if (bytes <= 32 * 1024) return cudaSuccess;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(g_dyn_mu);
  size_t& cur = g_dyn[{kernel, dev}];
  if (bytes <= cur) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) cur = bytes;
  return e;
}

int kernel_occupancy(const void* kernel, int threads, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, size_t>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_tuple(kernel, dev, threads, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess) return -1;
  cache[key] = per_sm;
  return per_sm;
}

void launch_begin(const char* name, cudaStream_t s) {
  ++g_launches;
  if (g_prof.events && g_prof.count < g_prof.capacity && g_prof.count < 4096) {
    cudaEventRecord(g_prof.events[2 * g_prof.count], s);
    g_prof.names[g_prof.count] = name;
    g_prof.open = 1;
  }
}
void launch_end(cudaStream_t s) {
  if (g_prof.open) {
    cudaEventRecord(g_prof.events[2 * g_prof.count + 1], s);
    ++g_prof.count;
    g_prof.open = 0;
  }
}
}  // namespace det

extern "C" int det_profile_set_events(void* const* events, int capacity) {
  g_prof.events = (events && capacity > 0) ? (cudaEvent_t*)events : nullptr;
  g_prof.capacity = g_prof.events ? capacity : 0;
  g_prof.count = 0;
  g_prof.open = 0;
  return 0;
}
extern "C" int det_profile_event_count(void) { return g_prof.count; }
extern "C" const char* det_profile_event_name(int i) {
  return (i >= 0 && i < g_prof.count) ? g_prof.names[i] : nullptr;
}
extern "C" unsigned long long det_launch_count(void) { return g_launches; }

extern "C" int det_read_status(const void* workspace, void* stream, int* device_status) {
  if (!workspace || !device_status) return DET_ERR_INVALID_ARG;
  cudaStream_t s = det::as_stream(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return DET_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DET_ERR_CUDA;
  *device_status = (int)v;
  return DET_OK;
}

extern "C" const char* det_last_cuda_error(void) { return det::last_cuda_error(); }

extern "C" const char* det_status_string(int status) {
  switch (status) {
    case DET_OK: return "ok";
    case DET_ERR_INVALID_ARG: return "invalid argument";
    case DET_ERR_DTYPE: return "unsupported dtype (use DET_F32 or DET_F64)";
    case DET_ERR_TOO_LARGE: return "size beyond the documented limit";
    case DET_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    case DET_ERR_LOOKBACK_TIMEOUT: return "device: a look-back wait gave up";
    case DET_ERR_CUDA: return "CUDA call or launch failed";
    case DET_ERR_COPY_TIMEOUT: return "device: a bulk copy into shared memory did not complete in time";
    default: return "unknown status";
  }
}
