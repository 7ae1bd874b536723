// det_sum: the canonical pairwise tree over element index, in one launch.
//
// Day 68 "Floating point and reproducibility" ("Contracts from tolerance to
// fixed bits", items 1-2; "Fix the order of every addition") replaces the
// scheduler-ordered atomic tail with a fixed tree, but its tree is a function
// of the grid.  Here the tree is PT over element index: node (level k, j)
// covers elements [j 2^k, (j+1) 2^k).  Any split of the input into aligned
// power-of-two tiles, followed by PT over the tile results, gives exactly
// those nodes, so neither the block size nor the grid enters the bits.
//
// Layout of the work:
//   lane       32 contiguous f32 (128 bytes) or 64 f64 (four 128-byte
//              chunks) by 256-bit loads, reduced in registers by PT
//                                                          -> level 5 / 6 node
//   warp-block 32 lanes = 4 KB / 16 KB, five xor-shuffle levels -> level 10 / 11
//   tile       2^tb warp-blocks per CTA (host-chosen power of two), nodes
//              staged in shared memory and reduced by PT
//   final      PT over the tile partials, by one CTA.  det_sum: each tile
//              publishes its partial in words tagged with this call's 64-bit
//              tag; the last CTA of the grid waits for every tile's words, so
//              nothing is cleared between calls and a call is one launch.
//              det_sum_noalloc: the last CTA to finish, by an integer ticket
//              cleared before the launch.
#include <cuda.h>

#include <atomic>
#include <chrono>
#include <random>
#include <mutex>

#include "det_common.cuh"

namespace det {
namespace {

template <typename T> struct SumGeom {
  static constexpr int CE = 128 / sizeof(T);   // elements per 128-byte lane chunk
  static constexpr int LE = sizeof(T) == 4 ? 32 : 64;   // elements per lane
  static constexpr int WB = kWarp * LE;        // elements per warp-block
  static constexpr int V = Vec256<T>::N;       // elements per 256-bit load
};

// The lane's node over LE contiguous elements at p (absent past n): PT of
// each 128-byte chunk in registers, then PT over the chunk nodes.  For f64 a
// lane takes four chunks, so that only one add in sixteen runs at the
// warp-shuffle levels, where every lane of the warp issues it.
template <typename T, bool VEC>
__device__ __forceinline__ T lane_node(const T* __restrict__ x, long long base, long long n) {
  using G = SumGeom<T>;
  constexpr int NC = G::LE / G::CE;
  T cn[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const long long cb = base + c * G::CE;
    T v[G::CE];
    if (VEC && cb + G::CE <= n) {
#pragma unroll
      for (int q = 0; q < G::CE / G::V; ++q) {
        T w[G::V];
        ld_nc_256(x + cb + q * G::V, w);
#pragma unroll
        for (int e = 0; e < G::V; ++e) v[q * G::V + e] = w[e];
      }
    } else {
#pragma unroll
      for (int e = 0; e < G::CE; ++e) v[e] = (cb + e < n) ? x[cb + e] : absent<T>();
    }
    cn[c] = thread_pt(v);
  }
  return thread_pt(cn);
}

// PT over p[0..L) by a whole CTA; the result is returned to thread 0.
// Thread t reduces the aligned group [t g, (t+1) g) with g = max(1, P / T)
// (P = next power of two >= L): chunks of 8 leaves, their loads all in
// flight, each reduced in registers (a level-3 node, absent terms past the
// group or the end), the chunk nodes merged by a binary counter.  The thread
// nodes are then reduced by warp_pt and a final PT over the warp nodes.
template <typename T>
__device__ T cta_pt_global(const T* p, long long L, T* smem_warp) {
  const int nthreads = blockDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  long long P = 1;
  while (P < L) P <<= 1;
  long long g = P / nthreads;
  if (g < 1) g = 1;
  T node;
  {
    const long long lo = (long long)tid * g;
    NodeCounter<T, 6> nc;
#pragma unroll 2
    for (long long c = 0; c < g; c += 8) {
      T v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const long long idx = lo + c + i;
        v[i] = (c + i < g && idx < L) ? __ldcg(p + idx) : absent<T>();
      }
      nc.push(thread_pt(v));
    }
    // g < 8: one chunk, PT over g leaves padded to 8; otherwise g / 8 (a
    // power of two) chunk nodes, so the counter ends with one full node
    node = nc.result();
  }
  node = warp_pt(node);
  if (lane == 0) smem_warp[warp] = node;
  __syncthreads();
  T r = absent<T>();
  if (warp == 0) {
    T v = lane < nwarps ? smem_warp[lane] : absent<T>();
    r = warp_pt(v);
  }
  __syncthreads();
  return r;
}

// Tagged partials: a tile's partial sum travels in two 64-bit words, read by
// one 16-byte load.  Their high halves hold the two halves of the call's
// 64-bit tag; their low halves hold the value's bits (f64: low then high 32
// bits; f32: the value in both).  The workspace may hold anything from
// earlier use -- other calls' words, or any other data -- so a tile counts
// as published only when both halves carry this call's tag.  Tags are
// distinct for every call of the process (a bijective mix of a call counter
// and a per-process seed), with neither half zero: earlier calls' words
// never match, and other contents match a given tag by chance only (2^-64
// per word for data that is not itself such a word).
template <typename T> struct Tagged {
  static constexpr int W = 2;
  __device__ static void put(unsigned long long* p, T v, unsigned long long tag) {
    unsigned long long lo, hi;
    if (sizeof(T) == 8) {
      const unsigned long long b = (unsigned long long)__double_as_longlong((double)v);
      lo = b & 0xffffffffull;
      hi = b >> 32;
    } else {
      lo = hi = __float_as_uint((float)v);
    }
    st_release_u64(p, (tag & 0xffffffff00000000ull) | lo);
    st_release_u64(p + 1, (tag << 32) | hi);
  }
  // the value travels in the tagged words themselves: relaxed loads suffice
  __device__ static bool get(const unsigned long long* p, unsigned long long tag, T& v) {
    unsigned long long w0, w1;
    ld_relaxed_v2u64(p, w0, w1);
    if (sizeof(T) == 8)
      v = (T)__longlong_as_double((long long)(((w1 & 0xffffffffull) << 32) | (w0 & 0xffffffffull)));
    else
      v = (T)__uint_as_float((unsigned)w0);
    return (w0 >> 32) == (tag >> 32) && (w1 >> 32) == (tag & 0xffffffffull);
  }
};

// PT over the L tagged partials by a whole CTA (the same groups, chunks and
// trees as cta_pt_global), each partial waited for until it carries `tag`;
// *ok turns false (in every thread) if a wait gave up.
template <typename T>
__device__ T cta_pt_tagged(const unsigned long long* words, long long L, unsigned long long tag, T* smem_warp,
                           bool* ok) {
  const int nthreads = blockDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  long long P = 1;
  while (P < L) P <<= 1;
  long long g = P / nthreads;
  if (g < 1) g = 1;
  const unsigned long long t0 = globaltimer();
  bool fine = true;
  T node;
  {
    const long long lo = (long long)tid * g;
    NodeCounter<T, 6> nc;
    for (long long c = 0; c < g; c += 8) {
      T v[8];
      bool got[8];
      // first look at all eight words (loads in flight together), then wait
      // only for those not yet tagged with this call
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const long long idx = lo + c + i;
        v[i] = absent<T>();
        got[i] = !(c + i < g && idx < L) || Tagged<T>::get(words + Tagged<T>::W * idx, tag, v[i]);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        unsigned polls = 0;
        while (!got[i] && fine) {
          got[i] = Tagged<T>::get(words + Tagged<T>::W * (lo + c + i), tag, v[i]);
          if ((++polls & 63u) == 0 && globaltimer() - t0 > kWaitNs) fine = false;
        }
      }
      nc.push(thread_pt(v));
    }
    node = nc.result();
  }
  *ok = __syncthreads_and(fine);
  node = warp_pt(node);
  if (lane == 0) smem_warp[warp] = node;
  __syncthreads();
  T r = absent<T>();
  if (warp == 0) {
    T v = lane < nwarps ? smem_warp[lane] : absent<T>();
    r = warp_pt(v);
  }
  __syncthreads();
  return r;
}

// FLAGS: tile t publishes its partial as words tagged with this call's tag;
// the grid's last CTA waits (bounded in time) for every tile's words, forms
// the final tree and writes the status word itself.  CTAs start in index
// order, so when the last one runs every other tile has started and only
// needs to finish; words of earlier calls carry other tags, so nothing
// needs clearing between calls.  Otherwise (the ticket form): each tile
// stores its partial, and the CTA that takes the last ticket of a counter
// cleared before the launch forms the final tree.
template <typename T, bool VEC, bool FLAGS>
__global__ void __launch_bounds__(1024)
sum_kernel(const T* __restrict__ x, long long n, int tb_log2, long long ntiles, T* __restrict__ partials,
           unsigned int* __restrict__ ticket, T* __restrict__ out, unsigned long long* __restrict__ tagged,
           unsigned tag, unsigned int* __restrict__ status) {
  using G = SumGeom<T>;
  __shared__ T nodes[1024];
  __shared__ T warp_nodes[32];
  __shared__ int is_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int TB = 1 << tb_log2;
  const long long tile_base = (long long)blockIdx.x * TB * G::WB;

  for (int b = warp; b < TB; b += nwarps) {
    const long long base = tile_base + (long long)b * G::WB + (long long)lane * G::LE;
    T node = warp_pt(lane_node<T, VEC>(x, base, n));
    if (lane == 0) nodes[b] = node;
  }
  __syncthreads();

  // PT over the TB warp-block nodes of this tile, by warp 0.
  if (warp == 0) {
    const int per = TB > 32 ? TB / 32 : 1;   // aligned group per lane
    T acc[32];
    T node;
    if (per == 1) {
      node = lane < TB ? nodes[lane] : absent<T>();
    } else {
      // per is a power of two <= 32: level-by-level PT over the lane's group
      for (int i = 0; i < per; ++i) acc[i] = nodes[lane * per + i];
      for (int s = 1; s < per; s <<= 1)
        for (int i = 0; i < per; i += 2 * s) acc[i] = acc[i] + acc[i + s];
      node = acc[0];
    }
    node = warp_pt(node);
    if (lane == 0) {
      if (FLAGS) {
        Tagged<T>::put(tagged + Tagged<T>::W * blockIdx.x, node, tag);
        is_last = blockIdx.x == ntiles - 1;
      } else {
        partials[blockIdx.x] = node;
        __threadfence();
        unsigned int t = atomicAdd(ticket, 1u);
        is_last = (t == (unsigned int)(ntiles - 1));
      }
    }
  }
  __syncthreads();
  if (!is_last) return;
  if (FLAGS) {
    // the tree over every tile's tagged partial (bounded waits)
    bool ok = true;
    const T r = cta_pt_tagged<T>(tagged, ntiles, tag, warp_nodes, &ok);
    if (threadIdx.x == 0) {
      if (ok) *out = r;
      *status = ok ? (unsigned)DET_OK : (unsigned)DET_ERR_LOOKBACK_TIMEOUT;
    }
    return;
  }
  __threadfence();
  // Partials were written by other CTAs: read them through L2 (volatile).
  T r = cta_pt_global<T>((const T*)partials, ntiles, warp_nodes);
  if (threadIdx.x == 0) *out = r;
}

}  // namespace

// Tile size: a power of two number of warp-blocks (32 lanes' nodes) chosen
// from n only (the bits do not depend on it; only the grid does).  Large
// inputs get 2,400 to 4,800 tiles (at most 1,024 warp-blocks each), several
// per resident CTA, so that the last, partly filled wave of CTAs is a small
// share of the launch (at 2^28 elements measured 2 % (f32) and 4 % (f64)
// faster than about 600 tiles, which leave 1.7 waves); inputs below 4,800
// warp-blocks get at least 128 larger tiles, so that the launch and the
// final tree over the tile partials stay short.
static int sum_tile_log2(long long nblocks) {
  long long want = nblocks >= 4800 ? nblocks / 2400 : nblocks / 128;
  int t = 0;
  while (t < 10 && (2LL << t) <= want) ++t;
  return t;
}

template <typename T>
static long long sum_ntiles(long long n, int* tb_log2) {
  long long nblocks = (n + SumGeom<T>::WB - 1) / SumGeom<T>::WB;
  int t = sum_tile_log2(nblocks);
  if (tb_log2) *tb_log2 = t;
  return (nblocks + (1LL << t) - 1) >> t;
}

}  // namespace det

using namespace det;

// Per-call tags of the single-launch path: the splitmix64 finalizer (Steele,
// Lea and Flood, "Fast splittable pseudorandom number generators", 2014; a
// bijection of 64-bit words) of a call counter XOR a per-process seed, so no
// two calls of the process share a tag; tags with a zero half are skipped.
static std::atomic<unsigned long long> g_sum_gen{0};

static unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

static unsigned long long process_seed() {
  static const unsigned long long seed = [] {
    unsigned long long v = 0;
    try {
      std::random_device rd;
      v = ((unsigned long long)rd() << 32) ^ rd();
    } catch (...) {
    }
    // mixed with the clock and an address of this process as well
    v ^= (unsigned long long)std::chrono::high_resolution_clock::now().time_since_epoch().count();
    v ^= (unsigned long long)reinterpret_cast<uintptr_t>(&g_sum_gen) << 7;
    return v;
  }();
  return seed;
}

static unsigned long long next_sum_tag() {
  const unsigned long long seed = process_seed();
  for (;;) {
    const unsigned long long t = mix64(++g_sum_gen ^ seed);
    if ((t >> 32) != 0 && (t & 0xffffffffull) != 0) return t;
  }
}

// Workspace: the header, then the tiles' tagged partials (16 bytes a tile).
extern "C" size_t det_sum_workspace_bytes(int64_t n, int dtype) {
  if (n < 0 || !valid_dtype(dtype)) return 0;
  long long nt = dtype == DET_F32 ? sum_ntiles<float>(n, nullptr) : sum_ntiles<double>(n, nullptr);
  return kHeaderBytes + align_up((size_t)nt * 16, 256);
}

template <typename T>
static int det_sum_impl(const T* x, long long n, T* out, void* ws, size_t ws_bytes, int bt,
                        cudaStream_t s) {
  int tb;
  long long nt = sum_ntiles<T>(n, &tb);
  if (ws_bytes < det_sum_workspace_bytes(n, sizeof(T) == 4 ? DET_F32 : DET_F64)) return DET_ERR_WORKSPACE;
  WsHeader* h = reinterpret_cast<WsHeader*>(ws);
  if (n == 0) {
    if (cudaMemsetAsync(h, 0, kHeaderBytes, s) != cudaSuccess) return DET_ERR_CUDA;
    if (cudaMemsetAsync(out, 0, sizeof(T), s) != cudaSuccess) return DET_ERR_CUDA;
    return DET_OK;
  }
  unsigned long long* tagged = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(ws) + kHeaderBytes);
  const int threads = bt ? bt : (tb >= 3 ? 256 : 32 << tb);
  const bool vec = (reinterpret_cast<uintptr_t>(x) % 32) == 0;
  // Under stream capture the tag would be fixed into the graph and shared by
  // every replay, and a replay could take an earlier replay's partials for
  // its own: there the call is a clearing memset of the header (captured
  // too, so it runs on every replay) and the ticket form of the kernel.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    cudaGetLastError();   // not a launch failure: take the form that is safe either way
    cap = cudaStreamCaptureStatusActive;
  }
  if (cap != cudaStreamCaptureStatusNone) {
    if (cudaMemsetAsync(h, 0, kHeaderBytes, s) != cudaSuccess) return DET_ERR_CUDA;
    T* partials = reinterpret_cast<T*>(tagged);
    launch_begin("det_sum", s);
    if (vec)
      sum_kernel<T, true, false><<<(unsigned)nt, threads, 0, s>>>(x, n, tb, nt, partials, &h->ticket, out, nullptr,
                                                                   0ull, &h->status);
    else
      sum_kernel<T, false, false><<<(unsigned)nt, threads, 0, s>>>(x, n, tb, nt, partials, &h->ticket, out, nullptr,
                                                                    0ull, &h->status);
    launch_end(s);
    return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
  }
  // one launch: the grid's last CTA forms the final tree once every tile's
  // partial carries this call's tag
  const unsigned long long tag = next_sum_tag();
  launch_begin("det_sum", s);
  if (vec)
    sum_kernel<T, true, true><<<(unsigned)nt, threads, 0, s>>>(x, n, tb, nt, nullptr, &h->ticket, out, tagged, tag,
                                                                &h->status);
  else
    sum_kernel<T, false, true><<<(unsigned)nt, threads, 0, s>>>(x, n, tb, nt, nullptr, &h->ticket, out, tagged, tag,
                                                                 &h->status);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

extern "C" int det_sum(const void* x, int64_t n, int dtype, void* out, void* workspace,
                       size_t workspace_bytes, int block_threads, void* stream) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (n < 0 || !out || !workspace || (n > 0 && !x) || !valid_block_threads(block_threads))
    return DET_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return DET_ERR_WORKSPACE;
  if (dtype == DET_F32)
    return det_sum_impl<float>((const float*)x, n, (float*)out, workspace, workspace_bytes,
                               block_threads, as_stream(stream));
  return det_sum_impl<double>((const double*)x, n, (double*)out, workspace, workspace_bytes,
                              block_threads, as_stream(stream));
}

// ---------------------------------------------------------------------------
// det_sum_noalloc: det_sum whose scratch (header + tile partials) lives in a
// statically sized device array of this file instead of a workspace, for
// callers that cannot allocate device memory.  The kernel is det_sum's.

static __device__ __align__(256) unsigned char g_sum_noalloc_scratch[kHeaderBytes +
                                                                     (size_t)DET_SUM_NOALLOC_MAX_PARTIALS *
                                                                         sizeof(double)];

namespace {
constexpr int kMaxDevices = 128;
std::mutex g_noalloc_mutex;
struct NoallocScratch {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;   // the context the address belongs to (0: not known)
};
NoallocScratch g_noalloc_scratch[kMaxDevices];

// Unique id of the current CUDA context (never reused within the process), or
// 0 when the driver does not provide one.  A device reset or another context
// on the same device gets a new id, and with it a new lookup below.
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS) return id;
  return 0;
}

// Device address of the static array in the current device's current
// context, looked up on the first call there (and again whenever the context
// changes).  In host code g_sum_noalloc_scratch names a host-side stand-in,
// never device memory, so only this address may be handed to a kernel.
int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DET_ERR_CUDA;
  const unsigned long long ctx = current_context_id();   // 0 before any context is current: look up again
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoallocScratch& e = g_noalloc_scratch[dev];
  if (!e.ptr || ctx == 0 || e.ctx_id != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sum_noalloc_scratch) != cudaSuccess || !p) return DET_ERR_CUDA;
    e.ptr = p;
    e.ctx_id = ctx;
  }
  *out = e.ptr;
  return DET_OK;
}

template <typename T>
int det_sum_noalloc_impl(const T* x, long long n, T* out, int bt, cudaStream_t s) {
  int tb;
  const long long nt = sum_ntiles<T>(n, &tb);
  if (nt > DET_SUM_NOALLOC_MAX_PARTIALS) return DET_ERR_TOO_LARGE;
  void* scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != DET_OK) return rc;
  WsHeader* h = reinterpret_cast<WsHeader*>(scratch);
  // the ticket must start at zero; the partials are written before they are read
  if (cudaMemsetAsync(h, 0, kHeaderBytes, s) != cudaSuccess) return DET_ERR_CUDA;
  if (n == 0) return cudaMemsetAsync(out, 0, sizeof(T), s) == cudaSuccess ? DET_OK : DET_ERR_CUDA;
  T* partials = reinterpret_cast<T*>(reinterpret_cast<char*>(scratch) + kHeaderBytes);
  const int threads = bt ? bt : (tb >= 3 ? 256 : 32 << tb);
  const bool vec = (reinterpret_cast<uintptr_t>(x) % 32) == 0;
  launch_begin("det_sum_noalloc", s);
  if (vec)
    sum_kernel<T, true, false><<<(unsigned)nt, threads, 0, s>>>(x, n, tb, nt, partials, &h->ticket, out, nullptr,
                                                                 0u, nullptr);
  else
    sum_kernel<T, false, false><<<(unsigned)nt, threads, 0, s>>>(x, n, tb, nt, partials, &h->ticket, out, nullptr,
                                                                  0u, nullptr);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}
}  // namespace

extern "C" int det_sum_noalloc(const void* x, int64_t n, int dtype, void* out, int block_threads,
                               void* stream) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (n < 0 || !out || (n > 0 && !x) || !valid_block_threads(block_threads)) return DET_ERR_INVALID_ARG;
  if (dtype == DET_F32)
    return det_sum_noalloc_impl<float>((const float*)x, n, (float*)out, block_threads, as_stream(stream));
  return det_sum_noalloc_impl<double>((const double*)x, n, (double*)out, block_threads, as_stream(stream));
}
