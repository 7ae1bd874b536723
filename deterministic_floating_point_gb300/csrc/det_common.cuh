// Shared device helpers for the deterministic reductions (sm_103a).
//
// Only IEEE round-to-nearest additions of the data type touch values.  The
// build uses no fast-math and leaves flush-to-zero off; there are no
// multiplies on any value path, so FMA contraction cannot arise.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/det.h"

namespace det {

constexpr int kWarp = 32;

// Workspace header: the first 256 bytes of every workspace.
struct WsHeader {
  unsigned int status;     // DET_OK or a device-detected error code
  unsigned int ticket;     // per-call integer ticket (order-safe: integer adds)
  unsigned int ticket2;
  unsigned int pad_[61];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");
constexpr size_t kHeaderBytes = 256;

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// "absent" term: x + (-0.0) == x for every x under round to nearest.
template <typename T> __device__ __forceinline__ T absent() { return T(-0.0); }

// ---------------------------------------------------------------------------
// 256-bit loads (one 32-byte sector per lane).  The pointer must be 32-byte
// aligned.  Read-only path; the data are not written by the same kernel.
// Bulk prefetch of the byte range [p, p + bytes) into L2 by the copy engine
// (cp.async.bulk.prefetch.L2), in 4 KB pieces spread over threads
// [0, nthreads) of the caller's group.  Both ends are widened to 16-byte
// boundaries; every widened block still holds a byte of the range, so it lies
// in mapped memory.  A prefetch changes no data, only where it is cached.
__device__ __forceinline__ void prefetch_l2(const void* p, size_t bytes, int me, int nthreads) {
  if (bytes == 0) return;
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p) & ~(uintptr_t)15;
  const uintptr_t hi = (reinterpret_cast<uintptr_t>(p) + bytes + 15) & ~(uintptr_t)15;
  for (uintptr_t q = lo + (uintptr_t)me * 4096; q < hi; q += (uintptr_t)nthreads * 4096) {
    const unsigned sz = (unsigned)((hi - q) < 4096 ? (hi - q) : 4096);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(q), "r"(sz) : "memory");
  }
}

__device__ __forceinline__ void ld_nc_256(const float* p, float (&v)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
                 "=f"(v[6]), "=f"(v[7])
               : "l"(p));
}
__device__ __forceinline__ void ld_nc_256(const double* p, double (&v)[4]) {
  asm volatile("ld.global.nc.L1::no_allocate.v4.f64 {%0,%1,%2,%3}, [%4];"
               : "=d"(v[0]), "=d"(v[1]), "=d"(v[2]), "=d"(v[3])
               : "l"(p));
}

__device__ __forceinline__ void st_256(float* p, const float (&v)[8]) {
  asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(v[0]),
               "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}
__device__ __forceinline__ void st_256(double* p, const double (&v)[4]) {
  asm volatile("st.global.v4.f64 [%0], {%1,%2,%3,%4};" ::"l"(p), "d"(v[0]), "d"(v[1]),
               "d"(v[2]), "d"(v[3])
               : "memory");
}

template <typename T> struct Vec256;
template <> struct Vec256<float> { static constexpr int N = 8; };
template <> struct Vec256<double> { static constexpr int N = 4; };

// ---------------------------------------------------------------------------
// Canonical pairwise tree over N (a power of two) values held in registers:
// level by level, v[i] = v[i] + v[i + s] for i a multiple of 2s.
template <typename T, int N>
__device__ __forceinline__ T thread_pt(T (&v)[N]) {
  static_assert((N & (N - 1)) == 0, "N must be a power of two");
#pragma unroll
  for (int s = 1; s < N; s <<= 1) {
#pragma unroll
    for (int i = 0; i < N; i += 2 * s) v[i] = v[i] + v[i + s];
  }
  return v[0];
}

// Five tree levels across the 32 lanes of a warp: at level s lane l adds the
// value of lane l ^ s.  For the lower lane of each pair this is the pair
// (2j, 2j+1) of the tree, and IEEE addition is commutative, so every lane ends
// with the bits of PT over lanes 0..31.
template <typename T>
__device__ __forceinline__ T warp_pt(T v) {
#pragma unroll
  for (int s = 1; s < kWarp; s <<= 1) v = v + __shfl_xor_sync(0xffffffffu, v, s);
  return v;
}

// Binary counter of pairwise-tree nodes.  push() takes the nodes of
// consecutive aligned blocks (all of one level) in order and merges equal
// levels as a binary counter does: the new node is added to the pending node
// of each lower level it completes, the earlier node always the left operand.
// result() folds the pending nodes from the smallest upwards, which is the
// pairwise tree over all blocks with absent padding.  Levels below L live in
// registers and are indexed only statically; deeper levels (more than 2^L
// blocks) use a small local array.
template <typename T, int L>
struct NodeCounter {
  T st[L];
  T deep[40 - L];
  unsigned long long cnt = 0;

  __device__ __forceinline__ void push(T node) {
    const int z = __ffsll((long long)~cnt) - 1;   // levels completed by this node
#pragma unroll
    for (int l = 0; l < L; ++l)
      if (l < z) node = st[l] + node;
    for (int l = L; l < z; ++l) node = deep[l - L] + node;
#pragma unroll
    for (int l = 0; l < L; ++l)
      if (l == z) st[l] = node;
    if (z >= L) deep[z - L] = node;
    ++cnt;
  }

  __device__ __forceinline__ T result() const {
    T res = absent<T>();
    bool have = false;
#pragma unroll
    for (int l = 0; l < L; ++l)
      if ((cnt >> l) & 1ull) {
        res = have ? st[l] + res : st[l];
        have = true;
      }
    for (int l = L; l < 40; ++l)
      if ((cnt >> l) & 1ull) {
        res = have ? deep[l - L] + res : deep[l - L];
        have = true;
      }
    return res;
  }
};

// ---------------------------------------------------------------------------
// Memory-model helpers for published values.
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// A relaxed 16-byte load of words that carry their own payload (nothing else
// is read on their strength), so several can be in flight at once.
__device__ __forceinline__ void ld_relaxed_v2u64(const unsigned long long* p, unsigned long long& a,
                                                 unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// Record a device-detected error in the status word (first error wins).
// Record a failed CUDA call (`where` = the step) for det_last_cuda_error and
// return DET_ERR_CUDA.  check_launch does the same for the last launch.
int cuda_fail(cudaError_t e, const char* where);
inline int check_launch(const char* where) {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DET_OK : cuda_fail(e, where);
}

__device__ __forceinline__ void set_status(unsigned int* status, unsigned int code) {
  atomicCAS(status, 0u, code);
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded on-device waits give up after this long (nanoseconds).
constexpr unsigned long long kWaitNs = 2000000000ull;

// ---------------------------------------------------------------------------
// Bulk copies global -> shared by the copy engine, completed on an mbarrier
// (CTA scope; a launch without clusters is a cluster of one CTA).
__device__ __forceinline__ unsigned smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Arrive on bar (count 1) and add `bytes` to the transfer it waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, unsigned bytes, unsigned long long* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// L2 eviction priority evict_first, for data a kernel reads for the last
// time.  A priority only changes what L2 keeps, never the data.
__device__ __forceinline__ unsigned long long l2_evict_first() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// bulk_copy_g2s with an L2 eviction priority for the source.
__device__ __forceinline__ void bulk_copy_g2s_hint(void* dst, const void* src, unsigned bytes, unsigned long long* bar,
                                                   unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Wait until phase `parity` of bar has completed, for at most timeout_ns;
// false if the wait gave up.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned parity, unsigned long long timeout_ns) {
  const unsigned long long t0 = globaltimer();
  unsigned polls = 0;
  while (!mbar_try_wait(bar, parity))
    if ((++polls & 255u) == 0 && globaltimer() - t0 > timeout_ns) return false;
  return true;
}

// Programmatic dependent launch.  A kernel launched with launch_dep() may be
// launched while the previous kernel of the stream is still running; it
// calls dep_wait() before any global memory access, which returns once that
// kernel has completed and its writes are visible.  What overlaps is the
// launch itself (the CTAs are already resident when the wait returns), not
// the work.  For a kernel launched the ordinary way dep_wait() is a no-op.
__device__ __forceinline__ void dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Host-side helpers -----------------------------------------------------------
inline bool valid_block_threads(int bt) {
  return bt == 0 || bt == 128 || bt == 256 || bt == 512 || bt == 1024;
}
inline int elem_size(int dtype) { return dtype == DET_F32 ? 4 : 8; }
inline bool valid_dtype(int dtype) { return dtype == DET_F32 || dtype == DET_F64; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Attributes of the current device, queried once per device and cached.
int device_sm_count();
int device_max_smem_optin();
// Raise `kernel`'s dynamic shared-memory limit to at least `bytes` on the
// current device; the attribute is set once per kernel and device.
cudaError_t ensure_dyn_smem(const void* kernel, size_t bytes);
// Resident CTAs per SM of `kernel` at this CTA size and dynamic shared
// memory, cached per kernel and device; -1 if the query failed.
int kernel_occupancy(const void* kernel, int threads, size_t smem);

// Launch bookkeeping for the measurement hooks of det_profile.h.  Every
// kernel launch of the library goes through launch_begin / launch_end.
void launch_begin(const char* name, cudaStream_t s);
void launch_end(cudaStream_t s);

// Launch `kernel` with programmatic stream serialization: it may be launched
// before the previous kernel in the stream completes, and waits for it in
// dep_wait().
template <typename... KArgs, typename... Args>
cudaError_t launch_dep(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace det
