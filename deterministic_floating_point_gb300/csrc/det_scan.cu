// det_scan / det_segmented_scan: single-pass decoupled look-back prefix sum
// whose look-back is anchored, so the association order never depends on
// which predecessors a chunk happens to observe as finished.
//
// drjit-core pull request "Make CUDA floating-point prefix sums
// deterministic": "Root cause" (a block observing PARTIAL/INCLUSIVE states in
// scheduling-dependent ways changes the association) and "Implementation"
// (fixed warp-sized anchor intervals; each lane examines a fixed predecessor,
// waits for the interval anchor's inclusive prefix, and a fixed-order warp
// reduction runs through that anchor; only anchor chunks publish inclusive
// prefixes).
//
// Frozen order (identical for every block size):
//   chunk c       C = 32 virtual warps x 32 lanes x E elements (E = 32 f32,
//                 16 f64); virtual lane (w, l) owns t = w*32E + l*E + e.
//   lane          LT = in-lane fold x0 + x1 + ... (left to right)
//   lanes         Kogge-Stone over l: K[l] = K[l-2^r] + K[l]; LX[l] = K[l-1]
//   warps         the same over w on the warp totals: WX[w], Agg(c) = K[31]
//   look-back     c = 32k + j; lane L reads Agg(c-1-L) for L < j and the
//                 anchor prefix A(k-1) for L = j; Excl(c) = PT over lanes
//   anchor        j = 31 publishes A(k) = Excl(c) + Agg(c)
//   element       y = (Excl + WX[w]) + LX[l], then y = y + x_e for each e
// Segmented: every '+' becomes (fa,a)(+)(fb,b) = (fa|fb, fb ? b : a+b) with
// the earlier part as left operand.  Exclusive output is the inclusive
// output shifted by one (first element +0.0; +0.0 at segment heads).
// Reverse is the scan of the reversed input (and reversed segmentation).
//
// Execution: one CTA per chunk in ticket order (an integer atomic), so every
// predecessor of a chunk has already started; the chunk is staged in shared
// memory with 144-byte rows (one virtual lane per row, padded so that rows
// read by a warp hit distinct banks); warp 0 does the look-back.  Every wait
// has a time limit: on expiry the status word gets DET_ERR_LOOKBACK_TIMEOUT
// and all later waits of the launch give up at once.
#include "det_common.cuh"
#include "../../include/det_test_hooks.h"

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

namespace det {
namespace {

template <typename T> struct Bits;
template <> struct Bits<float> {
  using U = unsigned int;
  static constexpr U kSentinel = 0xffffffffu;
  static constexpr U kQNaN = 0x7fc00000u;
};
template <> struct Bits<double> {
  using U = unsigned long long;
  static constexpr U kSentinel = 0xffffffffffffffffull;
  static constexpr U kQNaN = 0x7ff8000000000000ull;
};

template <typename T> __device__ __forceinline__ typename Bits<T>::U to_bits(T v);
template <> __device__ __forceinline__ unsigned int to_bits<float>(float v) { return __float_as_uint(v); }
template <> __device__ __forceinline__ unsigned long long to_bits<double>(double v) {
  return (unsigned long long)__double_as_longlong(v);
}
__device__ __forceinline__ float from_bits(unsigned int b) { return __uint_as_float(b); }
__device__ __forceinline__ double from_bits(unsigned long long b) { return __longlong_as_double((long long)b); }

__device__ __forceinline__ void st_relaxed(unsigned int* p, unsigned int v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned int ld_relaxed(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Published words hold the complement of the value's bits, so the all-zero
// word -- what the call's one clearing memset leaves -- marks "not yet
// published".  The only value whose complement is zero is the all-ones NaN,
// which is published as the canonical quiet NaN instead (NaN payloads are
// outside the bit-exact promise).
template <typename T>
__device__ __forceinline__ void publish(typename Bits<T>::U* p, T v) {
  typename Bits<T>::U b = to_bits<T>(v);
  if (b == Bits<T>::kSentinel) b = Bits<T>::kQNaN;
  st_relaxed(p, ~b);
}
template <typename U> __device__ __forceinline__ bool is_published(U w) { return w != U(0); }
__device__ __forceinline__ float decode(unsigned int w) { return from_bits(~w); }
__device__ __forceinline__ double decode(unsigned long long w) { return from_bits(~w); }

// Wait (bounded in time) for a published value word.  Returns false if the
// launch has given up (this wait timed out, or another one did).
template <typename T>
__device__ bool wait_value(const typename Bits<T>::U* p, T& out, unsigned int* status,
                           unsigned long long timeout_ns) {
  typename Bits<T>::U b = ld_relaxed(p);
  if (is_published(b)) {
    out = decode(b);
    return true;
  }
  const unsigned long long t0 = globaltimer();
  unsigned int polls = 0;
  while (true) {
    b = ld_relaxed(p);
    if (is_published(b)) {
      out = decode(b);
      return true;
    }
    if ((++polls & 63u) == 0) {
      if (ld_relaxed(status) != 0u) break;
      if (globaltimer() - t0 > timeout_ns) {
        set_status(status, DET_ERR_LOOKBACK_TIMEOUT);
        break;
      }
    }
  }
  out = absent<T>();
  return false;
}

// Segmented operator on (flag, value); a is the earlier part.
template <typename T, bool SEG>
__device__ __forceinline__ void segop(bool fa, T a, bool fb, T b, bool& fr, T& r) {
  if (SEG) {
    fr = fa | fb;
    r = fb ? b : a + b;
  } else {
    fr = false;
    r = a + b;
  }
}

template <typename T> struct ScanGeom {
  static constexpr int E = sizeof(T) == 4 ? 32 : 16;         // elements per virtual lane
  static constexpr int C = 1024 * E;                          // elements per chunk
  static constexpr int ROW = E + 16 / (int)sizeof(T);         // padded row (elements)
  static constexpr size_t kStageBytes = (size_t)1024 * ROW * sizeof(T);
};

// Copy one padded stage row (E elements, 16-byte aligned) into registers
// with 16-byte shared loads; reversed order for reverse scans.
template <typename T, int E, bool REVERSED>
__device__ __forceinline__ void row_to_regs(const T* row, T (&x)[E]) {
  constexpr int P = 16 / sizeof(T);
#pragma unroll
  for (int q = 0; q < E / P; ++q) {
    const float4 v = reinterpret_cast<const float4*>(row)[q];
    const T* pv = reinterpret_cast<const T*>(&v);
#pragma unroll
    for (int k = 0; k < P; ++k) {
      if (REVERSED)
        x[E - 1 - (q * P + k)] = pv[k];
      else
        x[q * P + k] = pv[k];
    }
  }
}

// Store E elements of a lane (32 B at a time, one full sector per lane per
// instruction).  p must be 32-byte aligned.
template <typename T, int E, bool REVERSED>
__device__ __forceinline__ void regs_to_global_256(T* p, const T (&x)[E]) {
  constexpr int P = 32 / sizeof(T);
#pragma unroll
  for (int q = 0; q < E / P; ++q) {
    T v[P];
#pragma unroll
    for (int k = 0; k < P; ++k) v[k] = REVERSED ? x[E - 1 - (q * P + k)] : x[q * P + k];
    st_256(p + q * P, v);
  }
}

// Store a warp's 32 lanes x E elements (each lane E consecutive elements of
// y, the lanes' rows adjacent: the warp's span [ylo, ylo + 32 E) of y) with
// coalesced 16-byte stores, through a 2 KB buffer of the warp: 16 lane rows
// at a time, rows written with their 16-byte chunks XOR-swizzled by the row
// (conflict-free), then read back as consecutive chunks.  REVERSED: the
// lanes' rows and the elements inside a row are in descending address order.
// ylo must be 16-byte aligned.
template <typename T, int E, bool REVERSED>
__device__ __forceinline__ void warp_store_staged(T* __restrict__ buf, const T (&x)[E], T* __restrict__ ylo,
                                                  int lane) {
  constexpr int P = 16 / (int)sizeof(T);   // elements per 16-byte chunk
  constexpr int CH = E / P;                // chunks per lane row
  static_assert(CH == 8, "a lane row is one 128-byte line");
  const int pos = REVERSED ? 31 - lane : lane;   // the lane row's place in the span
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if ((pos >> 4) == h) {
      const int r = pos & 15;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        T v[P];
#pragma unroll
        for (int k = 0; k < P; ++k) v[k] = REVERSED ? x[E - 1 - (c * P + k)] : x[c * P + k];
        *reinterpret_cast<float4*>(buf + (r * CH + (c ^ (r & 7))) * P) = *reinterpret_cast<const float4*>(v);
      }
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 16 * CH / 32; ++k) {
      const int i = lane + 32 * k, r = i / CH, c = i % CH;
      const float4 v = *reinterpret_cast<const float4*>(buf + (r * CH + (c ^ (r & 7))) * P);
      __stcs(reinterpret_cast<float4*>(ylo + (h * 16 + r) * E + c * P), v);
    }
    __syncwarp();
  }
}

template <typename T> struct ScanArgs {
  const T* x;
  T* y;
  long long n;
  long long nchunks;
  typename Bits<T>::U* desc;     // Agg(c)
  typename Bits<T>::U* anchors;  // A(k)
  typename Bits<T>::U* tails;    // last inclusive value of chunk c (exclusive scans)
  const unsigned int* head_bits; // segmented: head bitmap over scan-order positions
  const unsigned char* has_head; // segmented: chunk contains a head
  unsigned int* ticket;
  unsigned int* role;             // first CTA to start runs the anchor chain
  unsigned int* status;
  T* total_out;
  unsigned long long timeout_ns;
  long long withhold;             // chunk whose aggregate is never published (test hook), else -1
};

// Shared memory of one CTA (dynamic): stage rows, then the small arrays.
template <typename T> struct ScanSmem {
  T lx[1024];
  unsigned int lxf[32];   // segmented flags of lx (bit l of word w)
  T wt[32];
  T wx[32];
  unsigned int wtf, wxf;  // flags of wt / wx (bit w)
  T excl;
  int exclf;
  long long chunk;
  unsigned int heads[ScanGeom<T>::C / 32];
};

// The anchor chain, computed by one warp of one CTA of the launch.
//
// A(k) is the anchor chunk's own formula -- Excl(32k+31) + Agg(32k+31) with
// Excl(32k+31) = PT over lanes of Agg(32k+30-L) for L < 31 and A(k-1) in lane
// 31 -- so the bits are the same whoever computes it.  Holding A(k-1) in a
// register, this warp only waits for each interval's aggregates (published
// by the chunks without waiting on anything) instead of a cross-SM round
// trip per interval; chunks read A(k-1) once from the published array.
template <typename T, bool SEG>
__device__ void anchor_chain(const ScanArgs<T>& a) {
  using U = typename Bits<T>::U;
  constexpr int kAhead = 4;                // intervals whose aggregates are loaded at once
  const int lane = threadIdx.x & 31;
  const long long nint = a.nchunks / 32;   // complete intervals
  T prev = absent<T>();                    // A(k-1), in every lane
  for (long long kb = 0; kb < nint; kb += kAhead) {
    // lane L holds Agg(32k + L) of intervals kb .. kb+kAhead-1 (one round trip)
    U b[kAhead];
#pragma unroll
    for (int q = 0; q < kAhead; ++q)
      b[q] = (kb + q < nint) ? ld_relaxed(a.desc + 32 * (kb + q) + lane) : U(0);
#pragma unroll
    for (int q = 0; q < kAhead; ++q) {
      const long long k = kb + q;
      if (k >= nint) break;
      T mine;
      if (is_published(b[q]))
        mine = decode(b[q]);
      else
        wait_value<T>(a.desc + 32 * k + lane, mine, a.status, a.timeout_ns);
      const bool minef = SEG && a.has_head[32 * k + lane];
      // tree lane t < 31 takes Agg(32k + 30 - t) (held by lane 30 - t); lane 31 takes A(k-1)
      const int srcl = lane < 31 ? 30 - lane : 31;
      T v = __shfl_sync(0xffffffffu, mine, srcl);
      bool vf = __shfl_sync(0xffffffffu, (int)minef, srcl);
      if (lane == 31) {
        v = (k > 0) ? prev : absent<T>();
        vf = SEG && k > 0;
      }
#pragma unroll
      for (int s = 1; s < 32; s <<= 1) {
        const T o = __shfl_xor_sync(0xffffffffu, v, s);
        const bool of = __shfl_xor_sync(0xffffffffu, (int)vf, s);
        bool fr;
        if (lane & s)
          segop<T, SEG>(vf, v, of, o, fr, v);
        else
          segop<T, SEG>(of, o, vf, v, fr, v);
        vf = fr;
      }
      const T agg = __shfl_sync(0xffffffffu, mine, 31);
      const bool aggf = __shfl_sync(0xffffffffu, (int)minef, 31);
      T an;
      bool anf;
      segop<T, SEG>(vf, v, aggf, agg, anf, an);
      if (lane == 0) publish<T>(a.anchors + k, an);
      prev = an;
    }
  }
}

// ---------------------------------------------------------------------------
// Small scans in one thread-block cluster.  When an f64 input has at most
// kClusterChunks chunks, one cluster holds a CTA per chunk (CTA c = chunk c,
// 1,024 threads, one virtual lane each).  The chunks' aggregates, and for
// exclusive scans the chunks' last inclusive values, are exchanged through
// distributed shared memory across cluster barriers: no descriptor in global
// memory, nothing to clear, one launch.  The association order is the
// anchored look-back's: below 32 chunks there is no anchor, and Excl(c) is
// the tree over lanes L < c holding Agg(c - 1 - L), exactly as above.
constexpr int kClusterChunks = 16;

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The value at `local` in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ float ld_dsmem(const float* local, unsigned rank) {
  unsigned r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
  return v;
}
__device__ __forceinline__ double ld_dsmem(const double* local, unsigned rank) {
  unsigned r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(r) : "memory");
  return v;
}

template <typename T, bool REV, bool EXCL>
__global__ void __launch_bounds__(1024, 1) scan_cluster_kernel(const T* __restrict__ x, T* y, long long n,
                                                               T* total_out, unsigned int* status) {
  using G = ScanGeom<T>;
  constexpr int E = G::E, C = G::C, ROW = G::ROW;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T* stage = reinterpret_cast<T*>(smem_raw);
  __shared__ T wt[32], wx[32], last[32];
  __shared__ T agg_s, tail_s, excl_s;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const long long c = blockIdx.x;   // the grid is one cluster: block index = cluster rank = chunk
  const long long base = c * C, nvalid = min((long long)C, n - base);
  auto gidx = [&](long long t) -> long long { return REV ? n - 1 - (base + t) : base + t; };
  if (c == 0 && tid == 0) *status = DET_OK;   // no wait here can give up: the call's status is ok

  // ---- stage the chunk (scan order): element t -> row t / E, column t % E
  const bool vec = !REV && nvalid == C && ((reinterpret_cast<uintptr_t>(x + base) & 15) == 0) &&
                   ((reinterpret_cast<uintptr_t>(y + base) & 15) == 0);
  constexpr int PER16 = 16 / sizeof(T), NV = C / PER16 / 1024;
  if (vec) {
    float4 v[NV];   // every load in flight before the first store
#pragma unroll
    for (int k = 0; k < NV; ++k) v[k] = __ldcs(reinterpret_cast<const float4*>(x + base) + tid + k * 1024);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int t = (tid + k * 1024) * PER16;
      *reinterpret_cast<float4*>(stage + (t / E) * ROW + (t % E)) = v[k];
    }
  } else {
    T v[E];
#pragma unroll
    for (int k = 0; k < E; ++k) {
      const int t = tid + k * 1024;
      v[k] = t < nvalid ? x[gidx(t)] : absent<T>();
    }
#pragma unroll
    for (int k = 0; k < E; ++k) {
      const int t = tid + k * 1024;
      stage[(t / E) * ROW + (t % E)] = v[k];
    }
  }
  __syncthreads();

  // ---- phase 1: lane fold, Kogge-Stone over lanes, then over warps (warp 0)
  T xr[E];
  row_to_regs<T, E, false>(stage + tid * ROW, xr);
  T acc = xr[0];
#pragma unroll
  for (int e = 1; e < E; ++e) acc = acc + xr[e];
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const T o = __shfl_up_sync(0xffffffffu, acc, d);
    if (lane >= d) acc = o + acc;
  }
  T lx = __shfl_up_sync(0xffffffffu, acc, 1);
  if (lane == 0) lx = absent<T>();
  if (lane == 31) wt[w] = acc;
  __syncthreads();
  if (w == 0) {
    T wa = wt[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const T o = __shfl_up_sync(0xffffffffu, wa, d);
      if (lane >= d) wa = o + wa;
    }
    const T ex = __shfl_up_sync(0xffffffffu, wa, 1);
    wx[lane] = lane == 0 ? absent<T>() : ex;
    if (lane == 31) agg_s = wa;   // Agg(c)
  }
  cluster_sync_all();   // every chunk's aggregate is visible in the cluster

  // ---- Excl(c): PT over lanes, lane L < c holding Agg(c - 1 - L)
  if (w == 0) {
    T v = lane < c ? ld_dsmem(&agg_s, (unsigned)(c - 1 - lane)) : absent<T>();
    v = warp_pt(v);   // the look-back tree (commutative pairs: the same bits)
    if (lane == 0) excl_s = v;
  }
  __syncthreads();

  // ---- phase 2: element values
  {
    T yv = (excl_s + wx[w]) + lx;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      yv = yv + xr[e];
      xr[e] = yv;
    }
  }
  if (total_out && c == gridDim.x - 1) {
    const long long tl = nvalid - 1;   // the last element in scan order
    if (tid == tl / E) {
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (e == tl % E) *total_out = xr[e];
    }
  }
  if (EXCL) {
    // previous inclusive value of each lane's first element; the chunk's
    // first takes the previous chunk's last inclusive value
    if (lane == 31) last[w] = xr[E - 1];
    if (tid == 1023) tail_s = xr[E - 1];
    T pl = __shfl_up_sync(0xffffffffu, xr[E - 1], 1);
    cluster_sync_all();   // last[] and every chunk's tail visible
    if (lane == 0) pl = w > 0 ? last[w - 1] : (c > 0 ? ld_dsmem(&tail_s, (unsigned)(c - 1)) : T(0.0));
#pragma unroll
    for (int e = E - 1; e > 0; --e) xr[e] = xr[e - 1];
    xr[0] = pl;
  }
  // ---- outputs through the stage rows (each thread rewrites its own row)
  {
    T* row = stage + tid * ROW;
#pragma unroll
    for (int q = 0; q < E / PER16; ++q) reinterpret_cast<float4*>(row)[q] = reinterpret_cast<const float4*>(xr)[q];
  }
  __syncthreads();
  if (vec) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int t = (tid + k * 1024) * PER16;
      __stcs(reinterpret_cast<float4*>(y + base + t), *reinterpret_cast<const float4*>(stage + (t / E) * ROW + (t % E)));
    }
  } else {
    for (int t = tid; t < nvalid; t += 1024) y[gidx(t)] = stage[(t / E) * ROW + (t % E)];
  }
  cluster_sync_all();   // no CTA leaves while another may still read its shared memory
}

template <typename T, bool SEG, bool REV, bool EXCL>
__global__ void __launch_bounds__(1024, 1) scan_kernel(ScanArgs<T> a) {
  using G = ScanGeom<T>;
  constexpr int E = G::E, C = G::C, ROW = G::ROW;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T* stage = reinterpret_cast<T*>(smem_raw);
  ScanSmem<T>& sm = *reinterpret_cast<ScanSmem<T>*>(smem_raw + G::kStageBytes);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads >> 5, R = 32 / nwarps;

  if (tid == 0) {
    // the first CTA to start runs the anchor chain; the others take chunks
    sm.chunk = atomicAdd(a.role, 1u) == 0u ? -1LL : (long long)atomicAdd(a.ticket, 1u);
    sm.wtf = 0u;
  }
  __syncthreads();
  const long long c = sm.chunk;
  if (c < 0) {
    if (warp == 0) anchor_chain<T, SEG>(a);
    return;
  }
  if (c >= a.nchunks) return;
  const long long base = c * C;                      // scan-order position of element 0
  const long long nvalid = min((long long)C, a.n - base);

  // ---- stage the chunk: scan-order element t -> row t/E, column t%E
  auto gidx = [&](long long t) -> long long { return REV ? a.n - 1 - (base + t) : base + t; };
  const bool vec_in = !REV && nvalid == C && ((reinterpret_cast<uintptr_t>(a.x + base) & 15) == 0);
  if (vec_in) {
    constexpr int PER16 = 16 / sizeof(T);
    for (int i = tid; i < C / PER16; i += nthreads) {
      const int t = i * PER16;
      const float4 v = __ldcs(reinterpret_cast<const float4*>(a.x + base + t));
      *reinterpret_cast<float4*>(stage + (t / E) * ROW + (t % E)) = v;
    }
  } else {
    for (int t = tid; t < C; t += nthreads) {
      T v = t < nvalid ? a.x[gidx(t)] : absent<T>();
      stage[(t / E) * ROW + (t % E)] = v;
    }
  }
  if (SEG) {
    // head bits of this chunk (bit t of the chunk's window); the bitmap covers
    // ceil(n/32) words, positions past n read as "no head"
    const long long w0 = base / 32;
    const long long nwords = (a.n + 31) / 32;
    for (int i = tid; i < C / 32; i += nthreads)
      sm.heads[i] = (w0 + i < nwords) ? a.head_bits[w0 + i] : 0u;
  }
  __syncthreads();
  auto head = [&](int t) -> bool { return SEG && ((sm.heads[t >> 5] >> (t & 31)) & 1u); };

  // ---- phase 1: lane folds, Kogge-Stone over lanes, per virtual warp
  for (int r = 0; r < R; ++r) {
    const int v = warp * R + r;
    const int t0 = v * 32 * E + lane * E;
    T xr[E];
    row_to_regs<T, E, false>(stage + (v * 32 + lane) * ROW, xr);
    T acc = xr[0];
    bool f = head(t0);
#pragma unroll
    for (int e = 1; e < E; ++e) {
      bool fr;
      segop<T, SEG>(f, acc, head(t0 + e), xr[e], fr, acc);
      f = fr;
    }
    // inclusive Kogge-Stone over the 32 lanes
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      T o = __shfl_up_sync(0xffffffffu, acc, d);
      bool of = __shfl_up_sync(0xffffffffu, (int)f, d);
      if (lane >= d) {
        bool fr;
        segop<T, SEG>(of, o, f, acc, fr, acc);
        f = fr;
      }
    }
    T lx = __shfl_up_sync(0xffffffffu, acc, 1);
    bool lxf = __shfl_up_sync(0xffffffffu, (int)f, 1);
    if (lane == 0) {
      lx = absent<T>();
      lxf = false;
    }
    sm.lx[v * 32 + lane] = lx;
    unsigned int fm = __ballot_sync(0xffffffffu, lxf);
    if (lane == 31) {
      sm.wt[v] = acc;
      sm.lxf[v] = fm;
    }
    // the virtual warp's total carries the flag of lane 31's inclusive value
    const unsigned int wf = __ballot_sync(0xffffffffu, f);
    if (SEG && lane == 0 && ((wf >> 31) & 1u)) atomicOr(&sm.wtf, 1u << v);
  }
  __syncthreads();

  // ---- chunk aggregate, publication, anchored look-back (warp 0)
  if (warp == 0) {
    T acc = sm.wt[lane];
    bool f = SEG && ((sm.wtf >> lane) & 1u);
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      T o = __shfl_up_sync(0xffffffffu, acc, d);
      bool of = __shfl_up_sync(0xffffffffu, (int)f, d);
      if (lane >= d) {
        bool fr;
        segop<T, SEG>(of, o, f, acc, fr, acc);
        f = fr;
      }
    }
    T wx = __shfl_up_sync(0xffffffffu, acc, 1);
    bool wxf = __shfl_up_sync(0xffffffffu, (int)f, 1);
    if (lane == 0) {
      wx = absent<T>();
      wxf = false;
    }
    sm.wx[lane] = wx;
    const unsigned int wxm = __ballot_sync(0xffffffffu, wxf);
    const T agg = __shfl_sync(0xffffffffu, acc, 31);
    const bool aggf = __shfl_sync(0xffffffffu, (int)f, 31);
    if (lane == 0) {
      sm.wxf = wxm;
      if (c != a.withhold) publish<T>(a.desc + c, agg);
    }
    // look-back
    const long long k = c / 32;
    const int j = (int)(c % 32);
    T v = absent<T>();
    bool vf = false;
    if (lane < j) {
      const long long q = c - 1 - lane;
      wait_value<T>(a.desc + q, v, a.status, a.timeout_ns);
      vf = SEG && a.has_head[q];
    } else if (lane == j && k > 0) {
      wait_value<T>(a.anchors + (k - 1), v, a.status, a.timeout_ns);
      vf = SEG;  // position 0 is a head, so every anchor prefix carries the flag
    }
    // PT over lanes; higher lanes hold earlier chunks (left operand)
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      T o = __shfl_xor_sync(0xffffffffu, v, s);
      bool of = __shfl_xor_sync(0xffffffffu, (int)vf, s);
      bool fr;
      if (lane & s)
        segop<T, SEG>(vf, v, of, o, fr, v);
      else
        segop<T, SEG>(of, o, vf, v, fr, v);
      vf = fr;
    }
    if (lane == 0) {
      sm.excl = v;
      sm.exclf = vf;
    }
    (void)aggf;
  }
  __syncthreads();

  // ---- phase 2: element values, written back into the stage rows
  const T excl = sm.excl;
  const bool exclf = SEG && sm.exclf;
  for (int r = 0; r < R; ++r) {
    const int v = warp * R + r;
    T* row = stage + (v * 32 + lane) * ROW;
    const int t0 = v * 32 * E + lane * E;
    bool f1;
    T y;
    segop<T, SEG>(exclf, excl, SEG && ((sm.wxf >> v) & 1u), sm.wx[v], f1, y);
    bool f2;
    segop<T, SEG>(f1, y, SEG && ((sm.lxf[v] >> lane) & 1u), sm.lx[v * 32 + lane], f2, y);
    T xr[E];
    row_to_regs<T, E, false>(row, xr);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      y = (SEG && head(t0 + e)) ? xr[e] : y + xr[e];
      xr[e] = y;
    }
    constexpr int P = 16 / sizeof(T);
#pragma unroll
    for (int q = 0; q < E / P; ++q) reinterpret_cast<float4*>(row)[q] = reinterpret_cast<const float4*>(xr)[q];
  }
  __syncthreads();

  // ---- outputs
  const T* st = stage;
  auto sval = [&](int t) -> T { return st[(t / E) * ROW + (t % E)]; };
  if (EXCL && tid == 0 && c + 1 < a.nchunks) publish<T>(a.tails + c, sval(C - 1));
  if (tid == 0 && a.total_out && base + nvalid == a.n) *a.total_out = sval((int)nvalid - 1);
  if (!EXCL) {
    const bool vec_out = !REV && nvalid == C && ((reinterpret_cast<uintptr_t>(a.y + base) & 15) == 0);
    if (vec_out) {
      constexpr int PER16 = 16 / sizeof(T);
      for (int i = tid; i < C / PER16; i += nthreads) {
        const int t = i * PER16;
        const float4 v = *reinterpret_cast<const float4*>(stage + (t / E) * ROW + (t % E));
        __stcs(reinterpret_cast<float4*>(a.y + base + t), v);
      }
    } else {
      for (int t = tid; t < nvalid; t += nthreads) a.y[gidx(t)] = sval(t);
    }
  } else {
    for (int t = tid + 1; t < nvalid; t += nthreads) a.y[gidx(t)] = (SEG && head(t)) ? T(0.0) : sval(t - 1);
    if (tid == 0) {
      T first = T(0.0);
      if (c > 0 && !(SEG && head(0))) wait_value<T>(a.tails + (c - 1), first, a.status, a.timeout_ns);
      a.y[gidx(0)] = first;
    }
  }
}

// ---------------------------------------------------------------------------
// Persistent variant for 1024-thread CTAs: one virtual lane per thread, the
// current chunk held in registers, the next chunk (and its head bits)
// prefetched into the padded shared stage with cp.async while the current
// one publishes, looks back and writes.  Same association order as
// scan_kernel, so the same bits.

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <typename T> struct KeepSmem {
  T wt[32];
  T wx[2][32];            // warp prefixes of the current / next chunk (by parity)
  T last[32];
  unsigned int wtf;
  unsigned int wxf[2];
  T excl;
  int exclf;
  alignas(16) unsigned int heads[2][ScanGeom<T>::C / 32];   // cp.async destinations: 16-byte aligned
};

// Software-pipelined by one chunk: in iteration i a CTA runs phase 1 of its
// next chunk (from the stage) and publishes that chunk's aggregate before it
// waits in the look-back of its current chunk, so every aggregate -- and the
// anchor chain built on them -- is published about one round before anyone
// needs it.
template <typename T, bool SEG, bool REV, bool EXCL>
__global__ void __launch_bounds__(1024, 1) scan_keep_kernel(ScanArgs<T> a) {
  using G = ScanGeom<T>;
  constexpr int E = G::E, C = G::C, ROW = G::ROW, PER16 = 16 / (int)sizeof(T);
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T* stage = reinterpret_cast<T*>(smem_raw);
  KeepSmem<T>& sm = *reinterpret_cast<KeepSmem<T>*>(smem_raw + G::kStageBytes);
  // per-warp 2 KB output buffers (coalesced stores)
  T* obuf = reinterpret_cast<T*>(smem_raw + G::kStageBytes + align_up(sizeof(KeepSmem<T>), 16)) +
            (threadIdx.x >> 5) * (2048 / sizeof(T));
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int t0 = tid * E;   // first element of this thread's virtual lane (w = warp, l = lane)

  auto gidx = [&](long long c, long long t) -> long long { return REV ? a.n - 1 - (c * C + t) : c * C + t; };
  auto can_prefetch = [&](long long c) -> bool {
    if ((c + 1) * C > a.n) return false;
    const long long g0 = REV ? a.n - (c + 1) * C : c * C;
    return (reinterpret_cast<uintptr_t>(a.x + g0) & 15) == 0;
  };
  // copies of chunk c (and its head bits) into the stage, by threads [first, 1024)
  auto prefetch = [&](long long c, int hb, int first) {
    const long long g0 = REV ? a.n - (c + 1) * C : c * C;
    const T* src = a.x + g0;
    const int nthr = 1024 - first, me = tid - first;
    if (me < 0) return;
    for (int i = me; i < C / PER16; i += nthr) {
      const int j0 = i * PER16;
      const int r = REV ? (C - 1 - j0) / E : j0 / E;
      const int col = REV ? j0 - (C - (r + 1) * E) : j0 - r * E;
      cp_async16(stage + r * ROW + col, src + j0);
    }
    if (SEG) {
      const unsigned int* hsrc = a.head_bits + (c * C) / 32;
      for (int i = me; i < C / 32 / 4; i += nthr) cp_async16(&sm.heads[hb][i * 4], hsrc + i * 4);
    }
    cp_async_commit();
  };
  // head bits of a chunk loaded directly (chunks that are not prefetched)
  auto load_heads = [&](long long c, int hb) {
    if (!SEG) return;
    const long long w0 = (c * C) / 32, nwords = (a.n + 31) / 32;
    for (int i = tid; i < C / 32; i += 1024) sm.heads[hb][i] = (w0 + i < nwords) ? a.head_bits[w0 + i] : 0u;
  };
  auto head_of = [&](int hb, int t) -> bool { return SEG && ((sm.heads[hb][t >> 5] >> (t & 31)) & 1u); };
  // this lane's E head bits (bit e: position t0 + e), read once: E divides 32
  auto lane_heads = [&](int hb) -> unsigned {
    return SEG ? (sm.heads[hb][t0 >> 5] >> (t0 & 31)) & (E == 32 ? 0xffffffffu : ((1u << E) - 1u)) : 0u;
  };

  // Phase 1 after the lane fold: Kogge-Stone over lanes (-> lx), then over
  // warps by warp 0 (-> wx[set]) and publication of Agg(c).  Ends with the
  // warp prefixes in shared memory once the caller synchronises.
  auto finish_phase1 = [&](T acc, bool f, int set, long long c, T& lx, bool& lxf) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const T o = __shfl_up_sync(0xffffffffu, acc, d);
      const bool of = __shfl_up_sync(0xffffffffu, (int)f, d);
      if (lane >= d) {
        bool fr;
        segop<T, SEG>(of, o, f, acc, fr, acc);
        f = fr;
      }
    }
    lx = __shfl_up_sync(0xffffffffu, acc, 1);
    lxf = __shfl_up_sync(0xffffffffu, (int)f, 1);
    if (lane == 0) {
      lx = absent<T>();
      lxf = false;
    }
    if (lane == 31) sm.wt[w] = acc;
    if (SEG && lane == 31 && f) atomicOr(&sm.wtf, 1u << w);
    __syncthreads();
    if (w == 0) {
      T wa = sm.wt[lane];
      bool wf = SEG && ((sm.wtf >> lane) & 1u);
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const T o = __shfl_up_sync(0xffffffffu, wa, d);
        const bool of = __shfl_up_sync(0xffffffffu, (int)wf, d);
        if (lane >= d) {
          bool fr;
          segop<T, SEG>(of, o, wf, wa, fr, wa);
          wf = fr;
        }
      }
      T wx = __shfl_up_sync(0xffffffffu, wa, 1);
      bool wxf = __shfl_up_sync(0xffffffffu, (int)wf, 1);
      if (lane == 0) {
        wx = absent<T>();
        wxf = false;
      }
      sm.wx[set][lane] = wx;
      const unsigned int wxm = __ballot_sync(0xffffffffu, wxf);
      const T agg = __shfl_sync(0xffffffffu, wa, 31);
      if (lane == 0) {
        sm.wxf[set] = wxm;
        sm.wtf = 0u;   // read above; reset for the next phase 1
        if (c != a.withhold) publish<T>(a.desc + c, agg);
      }
    }
  };

  if (blockIdx.x == 0) {   // CTA 0 runs the anchor chain
    if (w == 0) anchor_chain<T, SEG>(a);
    return;
  }
  // worker CTA i takes chunks i-1, i-1+(G-1), ... (cooperative launch: all resident)
  const long long stride = gridDim.x - 1;
  long long c = blockIdx.x - 1;
  if (c >= a.nchunks) return;

  T x[E];
  int hb = 0, set = 0;
  T lx;
  bool lxf;
  if (tid == 0) sm.wtf = 0u;
  // ---- prologue: chunk c into registers, its phase 1
  if (can_prefetch(c)) {
    prefetch(c, hb, 0);
    cp_async_wait_all();
    __syncthreads();
    row_to_regs<T, E, REV>(stage + tid * ROW, x);
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const long long t = (long long)c * C + t0 + e;
      x[e] = t < a.n ? a.x[gidx(c, t0 + e)] : absent<T>();
    }
    load_heads(c, hb);
  }
  __syncthreads();
  {
    T acc = x[0];
    const unsigned hw = lane_heads(hb);
    bool f = hw & 1u;
#pragma unroll
    for (int e = 1; e < E; ++e) {
      bool fr;
      segop<T, SEG>(f, acc, (hw >> e) & 1u, x[e], fr, acc);
      f = fr;
    }
    finish_phase1(acc, f, set, c, lx, lxf);
  }
  long long cn = c + stride;
  bool next_staged = cn < a.nchunks && can_prefetch(cn);
  if (next_staged) prefetch(cn, hb ^ 1, 0);
  long long pend_pos = -1, pend_chunk = 0;   // deferred first element of an exclusive chunk (thread 0)

  while (true) {
    const bool have_next = cn < a.nchunks;
    T lxn = absent<T>();
    bool lxfn = false;
    {
      // the chunk after next is copied into the stage only at the end of this
      // iteration; move it from HBM into L2 now (warp 1: warp 0 runs the look-back)
      const long long cn2 = cn + stride;
      if (cn2 < a.nchunks && w == 1) {
        const long long lo = cn2 * C, hi = min(a.n, lo + C);
        prefetch_l2(a.x + (REV ? a.n - hi : lo), (size_t)(hi - lo) * sizeof(T), lane, 32);
        if (SEG) prefetch_l2(a.head_bits + lo / 32, (size_t)((hi - lo + 31) / 32) * 4, lane, 32);
      }
    }
    // ---- anchored look-back of the current chunk (warp 0).  Its inputs were
    // published during the previous iteration; it runs while the stage fills.
    if (w == 0) {
      const long long k = c / 32;
      const int j = (int)(c % 32);
      T v = absent<T>();
      bool vf = false;
      if (lane < j) {
        const long long q = c - 1 - lane;
        wait_value<T>(a.desc + q, v, a.status, a.timeout_ns);
        vf = SEG && a.has_head[q];
      } else if (lane == j && k > 0) {
        wait_value<T>(a.anchors + (k - 1), v, a.status, a.timeout_ns);
        vf = SEG;
      }
#pragma unroll
      for (int s2 = 1; s2 < 32; s2 <<= 1) {
        const T o = __shfl_xor_sync(0xffffffffu, v, s2);
        const bool of = __shfl_xor_sync(0xffffffffu, (int)vf, s2);
        bool fr;
        if (lane & s2)
          segop<T, SEG>(vf, v, of, o, fr, v);
        else
          segop<T, SEG>(of, o, vf, v, fr, v);
        vf = fr;
      }
      if (lane == 0) {
        sm.excl = v;
        sm.exclf = vf;
      }
    }

    // ---- phase 1 of the next chunk, straight from the stage (or global)
    if (have_next) {
      if (next_staged) {
        cp_async_wait_all();
      } else {
        load_heads(cn, hb ^ 1);
      }
      __syncthreads();
      T acc = absent<T>();
      bool f = false;
      const unsigned hwn = lane_heads(hb ^ 1);
      if (next_staged) {
        const T* row = stage + tid * ROW;
        // FL: the segmented operator; a warp whose lanes hold no head folds
        // with plain additions (the same values: no flag is ever set)
        auto fold = [&](auto flagged) {
          constexpr bool FL = decltype(flagged)::value;
#pragma unroll
          for (int q = 0; q < E / PER16; ++q) {
            const int qq = REV ? E / PER16 - 1 - q : q;
            const float4 v4 = reinterpret_cast<const float4*>(row)[qq];
            const T* pv = reinterpret_cast<const T*>(&v4);
#pragma unroll
            for (int k = 0; k < PER16; ++k) {
              const int e = q * PER16 + k;
              const T xe = REV ? pv[PER16 - 1 - k] : pv[k];
              if (e == 0) {
                acc = xe;
                f = FL && (hwn & 1u);
              } else {
                bool fr;
                segop<T, FL>(f, acc, (hwn >> e) & 1u, xe, fr, acc);
                f = fr;
              }
            }
          }
        };
        // (f32 only: f64 scans are bound by the FP64 adds, which both paths issue alike)
        if (SEG && (sizeof(T) == 8 || __any_sync(0xffffffffu, hwn != 0u)))
          fold(std::integral_constant<bool, SEG>{});
        else
          fold(std::integral_constant<bool, false>{});
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const long long t = (long long)cn * C + t0 + e;
          const T xe = t < a.n ? a.x[gidx(cn, t0 + e)] : absent<T>();
          if (e == 0) {
            acc = xe;
            f = hwn & 1u;
          } else {
            bool fr;
            segop<T, SEG>(f, acc, (hwn >> e) & 1u, xe, fr, acc);
            f = fr;
          }
        }
      }
      finish_phase1(acc, f, set ^ 1, cn, lxn, lxfn);
    }

    __syncthreads();   // Excl(c) and the warp prefixes of c visible

    // ---- phase 2 of the current chunk: element values, in place in x
    const long long base = c * C;
    const long long nvalid = min((long long)C, a.n - base);
    // f64 scans interleave the output additions, the
    // stores and the move of the next chunk into registers, a 32-byte group
    // at a time: the FP64 add rate bounds them, and this keeps the add pipe
    // busy while stores and shared-memory reads are in flight (one barrier
    // fewer per chunk).  Same values: only the instruction order changes.
    // The interleaved form is for f64 only: f32 scans, bound by HBM rather
    // than by their additions, measured slower with it (e.g. 477 -> 567 us
    // forward exclusive at 2^28).
    constexpr bool kMergedPath = sizeof(T) == 8;
    // (the forward inclusive full scan written out on its own: measured 11 %
    // faster than the general form below, which is faster for the others)
    if constexpr (sizeof(T) == 8 && !SEG && !REV && !EXCL) {
      constexpr int P = 32 / (int)sizeof(T);   // elements per 32-byte group
      bool f1, f2;
      T y;
      segop<T, SEG>(SEG && sm.exclf, sm.excl, SEG && ((sm.wxf[set] >> w) & 1u), sm.wx[set][w], f1, y);
      segop<T, SEG>(f1, y, lxf, lx, f2, y);
      const unsigned hw = lane_heads(hb);
      const long long g0 = base + t0;
      const bool vstore = nvalid == C && (reinterpret_cast<uintptr_t>(a.y + g0) & 31) == 0;
      const bool promote = have_next && next_staged;
      const T* row = stage + tid * ROW;
      const long long want = a.n - 1 - base - t0;   // the last element of the scan, if in this lane
      const bool has_total = a.total_out && want >= 0 && want < E;
      T tv = absent<T>();
#pragma unroll
      for (int q = 0; q < E / P; ++q) {
#pragma unroll
        for (int k = 0; k < P; ++k) {
          const int e = q * P + k;
          y = (SEG && ((hw >> e) & 1u)) ? x[e] : y + x[e];
          x[e] = y;
          if (e == want) tv = y;
        }
        if (vstore) {
          asm volatile("st.global.v4.f64 [%0], {%1,%2,%3,%4};" ::"l"(a.y + g0 + q * P), "d"(x[q * P]),
                       "d"(x[q * P + 1]), "d"(x[q * P + 2]), "d"(x[q * P + 3])
                       : "memory");
        } else {
#pragma unroll
          for (int k = 0; k < P; ++k)
            if (t0 + q * P + k < nvalid) a.y[g0 + q * P + k] = x[q * P + k];
        }
        if (promote) {   // x[q P .. q P + P) now free: the next chunk's elements there
#pragma unroll
          for (int h = 0; h < P / 2; ++h) {
            const double2 v2 = reinterpret_cast<const double2*>(row)[q * (P / 2) + h];
            x[q * P + 2 * h] = v2.x;
            x[q * P + 2 * h + 1] = v2.y;
          }
        }
      }
      if (has_total) *a.total_out = tv;
      if (!have_next) break;
      if (!next_staged) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const long long t = (long long)cn * C + t0 + e;
          x[e] = t < a.n ? a.x[gidx(cn, t0 + e)] : absent<T>();
        }
      }
      __syncthreads();   // this chunk's shared data and the stage no longer read
      c = cn;
      hb ^= 1;
      set ^= 1;
      lx = lxn;
      lxf = lxfn;
      cn = c + stride;
      next_staged = cn < a.nchunks && can_prefetch(cn);
      if (next_staged) prefetch(cn, hb ^ 1, 0);
      continue;
    }
    if constexpr (kMergedPath) {
      constexpr int P = 32 / (int)sizeof(T);   // elements per 32-byte group
      constexpr int Q = 16 / (int)sizeof(T);   // elements per 16-byte chunk of a stage row
      bool f1, f2;
      T y;
      segop<T, SEG>(SEG && sm.exclf, sm.excl, SEG && ((sm.wxf[set] >> w) & 1u), sm.wx[set][w], f1, y);
      segop<T, SEG>(f1, y, lxf, lx, f2, y);
      const unsigned hw = lane_heads(hb);
      // the lane's E elements occupy y[g0, g0 + E) (descending scan order when REV)
      const long long g0 = REV ? a.n - base - t0 - E : base + t0;
      const bool vstore = nvalid == C && (reinterpret_cast<uintptr_t>(a.y + g0) & 31) == 0;
      const bool promote = have_next && next_staged;
      const T* row = stage + tid * ROW;
      const long long want = a.n - 1 - base - t0;   // the last element of the scan, if in this lane
      const bool has_total = a.total_out && want >= 0 && want < E;
      T tv = absent<T>();
      // outputs o[] of group q (scan order) to memory
      auto store_group = [&](int q, const T (&o)[P]) {
        if (vstore) {
          if (REV) {   // group q lands at the mirrored group, its elements reversed
            T r[P];
#pragma unroll
            for (int k = 0; k < P; ++k) r[k] = o[P - 1 - k];
            st_256(a.y + g0 + (E / P - 1 - q) * P, r);
          } else {
            st_256(a.y + g0 + q * P, o);
          }
        } else {
#pragma unroll
          for (int k = 0; k < P; ++k)
            if (t0 + q * P + k < nvalid) a.y[gidx(c, t0 + q * P + k)] = o[k];
        }
      };
      // x[q P .. q P + P) is free: the next chunk's elements there
      auto promote_group = [&](int q) {
        if (!promote) return;
#pragma unroll
        for (int h = 0; h < P / Q; ++h) {
          T v[Q];
          if (REV) {   // scan element e of the row sits at row index E - 1 - e
            *reinterpret_cast<float4*>(v) = reinterpret_cast<const float4*>(row)[(E - q * P - P) / Q + h];
#pragma unroll
            for (int k = 0; k < Q; ++k) x[q * P + P - 1 - (h * Q + k)] = v[k];
          } else {
            *reinterpret_cast<float4*>(v) = reinterpret_cast<const float4*>(row)[q * (P / Q) + h];
#pragma unroll
            for (int k = 0; k < Q; ++k) x[q * P + h * Q + k] = v[k];
          }
        }
      };
      auto incl_group = [&](int q) {
#pragma unroll
        for (int k = 0; k < P; ++k) {
          const int e = q * P + k;
          y = (SEG && ((hw >> e) & 1u)) ? x[e] : y + x[e];
          x[e] = y;
          if (e == want) tv = y;
        }
      };
      if constexpr (!EXCL) {
#pragma unroll
        for (int q = 0; q < E / P; ++q) {
#pragma unroll
          for (int k = 0; k < P; ++k) {
            const int e = q * P + k;
            y = (SEG && ((hw >> e) & 1u)) ? x[e] : y + x[e];
            x[e] = y;
            if (e == want) tv = y;
          }
          {
            T o[P];
#pragma unroll
            for (int k = 0; k < P; ++k) o[k] = x[q * P + k];
            store_group(q, o);
          }
          promote_group(q);
        }
      } else {
        // exclusive output e is the inclusive value e - 1 (+0.0 at a head):
        // group q >= 1 goes out as soon as it is computed; group 0 needs the
        // previous lane's (or warp's) last inclusive value, known after a barrier
        T prev_last = absent<T>();
        const auto ex = [&](int e, T v) -> T { return (SEG && ((hw >> e) & 1u)) ? T(0.0) : v; };
#pragma unroll
        for (int q = 0; q < E / P; ++q) {
          incl_group(q);
          if (q > 0) {
            T o[P];
            o[0] = ex(q * P, prev_last);
#pragma unroll
            for (int k = 1; k < P; ++k) o[k] = ex(q * P + k, x[q * P + k - 1]);
            store_group(q, o);
          }
          prev_last = x[q * P + P - 1];
          if (q > 0) promote_group(q);
        }
        if (tid == 1023 && c + 1 < a.nchunks) publish<T>(a.tails + c, prev_last);
        if (lane == 31) sm.last[w] = prev_last;
        T pl = __shfl_up_sync(0xffffffffu, prev_last, 1);
        __syncthreads();
        if (lane == 0) pl = (w > 0) ? sm.last[w - 1] : T(0.0);   // chunk start: written later
        {
          T o[P];
          o[0] = ex(0, pl);
#pragma unroll
          for (int k = 1; k < P; ++k) o[k] = ex(k, x[k - 1]);
          store_group(0, o);
        }
        promote_group(0);
        if (tid == 0) {
          // the chunk's first element is the previous chunk's last inclusive
          // value: resolve the one deferred from the chunk before this one,
          // then defer this one (its predecessor may still be writing)
          if (pend_pos >= 0) {
            T v;
            wait_value<T>(a.tails + (pend_chunk - 1), v, a.status, a.timeout_ns);
            a.y[pend_pos] = v;
          }
          pend_pos = -1;
          if (c > 0 && !(SEG && head_of(hb, 0))) {
            pend_pos = gidx(c, 0);
            pend_chunk = c;
          }
        }
      }
      if (has_total) *a.total_out = tv;
      if (!have_next) break;
      if (!next_staged) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const long long t = (long long)cn * C + t0 + e;
          x[e] = t < a.n ? a.x[gidx(cn, t0 + e)] : absent<T>();
        }
      }
      __syncthreads();   // this chunk's shared data and the stage no longer read
      c = cn;
      hb ^= 1;
      set ^= 1;
      lx = lxn;
      lxf = lxfn;
      cn = c + stride;
      next_staged = cn < a.nchunks && can_prefetch(cn);
      if (next_staged) prefetch(cn, hb ^ 1, 0);
      continue;
    }
    {
      bool f1, f2;
      T y;
      segop<T, SEG>(SEG && sm.exclf, sm.excl, SEG && ((sm.wxf[set] >> w) & 1u), sm.wx[set][w], f1, y);
      segop<T, SEG>(f1, y, lxf, lx, f2, y);
      const unsigned hw = lane_heads(hb);
      if (SEG && (sizeof(T) == 8 || __any_sync(0xffffffffu, hw != 0u))) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          y = ((hw >> e) & 1u) ? x[e] : y + x[e];
          x[e] = y;
        }
      } else {   // no head in the warp's lanes (f32): plain additions
#pragma unroll
        for (int e = 0; e < E; ++e) {
          y = y + x[e];
          x[e] = y;
        }
      }
    }
    if (EXCL && tid == 1023 && c + 1 < a.nchunks) publish<T>(a.tails + c, x[E - 1]);
    if (a.total_out && base + t0 <= a.n - 1 && a.n - 1 < base + t0 + E) {
      // static indices only: a dynamic index would move x[] to local memory
      const long long want = a.n - 1 - base - t0;
      T tv = x[0];
#pragma unroll
      for (int e = 1; e < E; ++e)
        if (e == want) tv = x[e];
      *a.total_out = tv;
    }
    const bool full = nvalid == C;
    if (EXCL) {
      // previous inclusive value for this lane's first element
      if (lane == 31) sm.last[w] = x[E - 1];
      T pl = __shfl_up_sync(0xffffffffu, x[E - 1], 1);
      __syncthreads();
      if (lane == 0) pl = (w > 0) ? sm.last[w - 1] : T(0.0);   // chunk start: written later
      const unsigned hw = lane_heads(hb);
#pragma unroll
      for (int e = E - 1; e > 0; --e) x[e] = (SEG && ((hw >> e) & 1u)) ? T(0.0) : x[e - 1];
      x[0] = (SEG && (hw & 1u)) ? T(0.0) : pl;
    }
    {
      // forward f32 scans store through the warp's buffer (coalesced); the
      // others lane by lane, a full 32-byte sector per store (measured faster
      // for them: f64 scans are bound by the FP64 add rate)
      constexpr bool kStaged = sizeof(T) == 4 && !REV;
      const long long g0 = REV ? a.n - base - t0 - E : base + t0;
      const long long wlo = REV ? a.n - base - (long long)(w + 1) * 32 * E : base + (long long)w * 32 * E;
      if (kStaged && full && (reinterpret_cast<uintptr_t>(a.y + wlo) & 15) == 0) {
        warp_store_staged<T, E, REV>(obuf, x, a.y + wlo, lane);
      } else if (!kStaged && full && (reinterpret_cast<uintptr_t>(a.y + g0) & 31) == 0) {
        regs_to_global_256<T, E, REV>(a.y + g0, x);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e)
          if (t0 + e < nvalid) a.y[gidx(c, t0 + e)] = x[e];
      }
    }
    if (EXCL && tid == 0) {
      // the chunk's first element is the previous chunk's last inclusive
      // value: resolve the one deferred from the chunk before this one, then
      // defer this one (its predecessor may still be writing)
      if (pend_pos >= 0) {
        T v;
        wait_value<T>(a.tails + (pend_chunk - 1), v, a.status, a.timeout_ns);
        a.y[pend_pos] = v;
      }
      pend_pos = -1;
      if (c > 0 && !(SEG && head_of(hb, 0))) {
        pend_pos = gidx(c, 0);
        pend_chunk = c;
      }
    }

    if (!have_next) break;
    __syncthreads();   // this chunk's shared data is no longer read
    // ---- promote the next chunk to registers; prefetch the one after
    if (next_staged) {
      row_to_regs<T, E, REV>(stage + tid * ROW, x);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const long long t = (long long)cn * C + t0 + e;
        x[e] = t < a.n ? a.x[gidx(cn, t0 + e)] : absent<T>();
      }
    }
    __syncthreads();   // stage free
    c = cn;
    hb ^= 1;
    set ^= 1;
    lx = lxn;
    lxf = lxfn;
    cn = c + stride;
    next_staged = cn < a.nchunks && can_prefetch(cn);
    if (next_staged) prefetch(cn, hb ^ 1, 0);
  }
  if (EXCL && tid == 0 && pend_pos >= 0) {
    T v;
    wait_value<T>(a.tails + (pend_chunk - 1), v, a.status, a.timeout_ns);
    a.y[pend_pos] = v;
  }
}

// Per-segment restart: every segment is scanned as det_scan of the segment
// alone.  One CTA of 4 warps takes a segment and walks its chunks in order;
// per chunk the 32 virtual warps of 32 lanes x E elements are handled four at
// a time, the look-back reads the aggregates of the segment's previous chunks
// and its interval anchor from shared memory (this CTA computed them), so the
// association is exactly that of the chunked scan of the segment on its own.
// A virtual warp's 32 x E elements move between global and shared memory by
// coalesced warp accesses (any alignment) and reach their lanes from padded
// rows.
template <typename T, bool REV, bool EXCL>
__global__ void __launch_bounds__(128, 6)   // at most 64 (f32) / 72 (f64) registers: 6+ CTAs per SM
restart_kernel(const T* x, T* y, long long n, const long long* __restrict__ off, long long S,
               unsigned int* __restrict__ status) {
  using G = ScanGeom<T>;
  constexpr int E = G::E, C = G::C, NVW = 32, RS = E + 1;   // RS: padded row stride (conflict-free)
  __shared__ T stage[4][32 * RS];   // one staging buffer per warp: 32 rows (virtual lanes) of E
  __shared__ T lx[NVW][32];         // exclusive lane prefixes of the chunk
  __shared__ T wt[NVW];             // virtual-warp totals
  __shared__ T wx[NVW];             // exclusive virtual-warp prefixes
  __shared__ T hist[32];            // aggregates of the segment's last 32 chunks (ring)
  __shared__ T lastv[NVW];          // exclusive scans: last inclusive value of each virtual warp
  __shared__ T anchor, excl_s, carry;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  T* st = stage[w];
  if (blockIdx.x == 0 && tid == 0 && (off[0] != 0 || off[S] != n)) set_status(status, DET_ERR_INVALID_ARG);
  for (long long sg = blockIdx.x; sg < S; sg += gridDim.x) {
    const long long o0 = off[sg], o1 = off[sg + 1];
    if (o1 <= o0) {
      if (o1 < o0 && tid == 0) set_status(status, DET_ERR_INVALID_ARG);
      continue;
    }
    if (o0 < 0 || o1 > n) {   // invalid offsets: reported, the segment is left alone
      if (tid == 0) set_status(status, DET_ERR_INVALID_ARG);
      continue;
    }
    const long long len = o1 - o0, nch = (len + C - 1) / C;
    auto at = [&](long long t) -> long long { return REV ? o1 - 1 - t : o0 + t; };   // scan order -> array index
    // this warp's virtual warp starting at scan position b: lane l's E elements into v
    auto load_vw = [&](long long b, T (&v)[E]) {
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const int idx = i * 32 + lane;   // consecutive lanes on consecutive elements
        const long long t = b + idx;
        st[(idx / E) * RS + idx % E] = t < len ? x[at(t)] : absent<T>();
      }
      __syncwarp();
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = st[lane * RS + e];
      __syncwarp();
    };
    auto store_vw = [&](long long b, const T (&v)[E]) {
#pragma unroll
      for (int e = 0; e < E; ++e) st[lane * RS + e] = v[e];
      __syncwarp();
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const int idx = i * 32 + lane;
        const long long t = b + idx;
        if (t < len) y[at(t)] = st[(idx / E) * RS + idx % E];
      }
      __syncwarp();
    };
    for (long long k = 0; k < nch; ++k) {
      // virtual warps of this chunk that hold elements; the others are all
      // absent, so their totals are -0.0 and change nothing
      const int nvw = (int)min((long long)NVW, (len - k * C + 32LL * E - 1) / (32LL * E));
      // ---- phase 1: lane folds, Kogge-Stone over lanes, virtual-warp totals
      for (int vw = w; vw < nvw; vw += 4) {
        T v[E];
        load_vw(k * C + (long long)vw * 32 * E, v);
        T acc = v[0];
#pragma unroll
        for (int e = 1; e < E; ++e) acc = acc + v[e];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const T o = __shfl_up_sync(0xffffffffu, acc, d);
          if (lane >= d) acc = o + acc;
        }
        const T ex = __shfl_up_sync(0xffffffffu, acc, 1);
        lx[vw][lane] = lane == 0 ? absent<T>() : ex;
        if (lane == 31) wt[vw] = acc;
      }
      __syncthreads();
      // ---- warp 0: Kogge-Stone over the virtual warps, Agg(k), Excl(k), anchor
      if (w == 0) {
        T a = lane < nvw ? wt[lane] : absent<T>();
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const T o = __shfl_up_sync(0xffffffffu, a, d);
          if (lane >= d) a = o + a;
        }
        const T ex = __shfl_up_sync(0xffffffffu, a, 1);
        wx[lane] = lane == 0 ? absent<T>() : ex;
        const T agg = __shfl_sync(0xffffffffu, a, 31);
        const long long K = k / 32;
        const int j = (int)(k % 32);
        T v = absent<T>();
        if (lane < j)
          v = hist[(k - 1 - lane) & 31];
        else if (lane == j && K > 0)
          v = anchor;
#pragma unroll
        for (int s2 = 1; s2 < 32; s2 <<= 1) {
          const T o = __shfl_xor_sync(0xffffffffu, v, s2);
          v = (lane & s2) ? v + o : o + v;
        }
        __syncwarp();   // every lane has read hist and anchor
        if (lane == 0) {
          excl_s = v;
          if (j == 31) anchor = v + agg;   // A(K) = Excl(32K+31) + Agg(32K+31)
          hist[k & 31] = agg;
        }
      }
      __syncthreads();
      const T excl = excl_s;
      // ---- exclusive scans: the last inclusive value of every virtual warp
      if (EXCL) {
        for (int vw = w; vw < nvw; vw += 4) {
          T v[E];
          load_vw(k * C + (long long)vw * 32 * E, v);
          if (lane == 31) {
            T yv = (excl + wx[vw]) + lx[vw][31];
#pragma unroll
            for (int e = 0; e < E; ++e) yv = yv + v[e];
            lastv[vw] = yv;
          }
        }
        __syncthreads();
      }
      // ---- phase 2: element values (the chunk is read again, from L2)
      for (int vw = w; vw < nvw; vw += 4) {
        const long long b = k * C + (long long)vw * 32 * E;
        T v[E];
        load_vw(b, v);
        T yv = (excl + wx[vw]) + lx[vw][lane];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          yv = yv + v[e];
          v[e] = yv;
        }
        if (EXCL) {
          T first = __shfl_up_sync(0xffffffffu, v[E - 1], 1);
          if (lane == 0) first = vw > 0 ? lastv[vw - 1] : (k > 0 ? carry : T(0.0));
#pragma unroll
          for (int e = E - 1; e > 0; --e) v[e] = v[e - 1];
          v[0] = first;
        }
        store_vw(b, v);
      }
      __syncthreads();   // shared state is rewritten by the next chunk
      if (EXCL && tid == 0) carry = lastv[nvw - 1];   // a chunk followed by another is full
      __syncthreads();
    }
  }
}

// Segment heads in scan order: a bitmap over positions and a per-chunk flag.
template <int C, bool REV>
__global__ void seg_heads_kernel(const long long* __restrict__ off, long long nseg, long long n,
                                 unsigned int* __restrict__ bits, unsigned char* __restrict__ has_head,
                                 unsigned int* __restrict__ status) {
  const long long s = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= nseg) return;
  const long long lo = off[s], hi = off[s + 1];
  if (lo < 0 || hi > n || hi < lo) {
    set_status(status, DET_ERR_INVALID_ARG);
    return;
  }
  if (s == 0 && lo != 0) set_status(status, DET_ERR_INVALID_ARG);
  if (s == nseg - 1 && hi != n) set_status(status, DET_ERR_INVALID_ARG);
  if (lo == hi) return;
  const long long h = REV ? n - hi : lo;
  atomicOr(bits + (h >> 5), 1u << (h & 31));
  has_head[h / C] = 1;
}

}  // namespace

// Test hook state (det_test_hooks.h): host-side, read when a call is enqueued.
static long long g_scan_withhold = -1;
static unsigned long long g_scan_wait_ns = kWaitNs;

template <typename T> struct ScanWs {
  size_t desc, anchors, tails, bits, has_head, total;
};

template <typename T>
static ScanWs<T> scan_ws_layout(long long n, bool seg) {
  using U = typename Bits<T>::U;
  const long long C = ScanGeom<T>::C;
  const long long nch = (n + C - 1) / C;
  ScanWs<T> w;
  size_t off = kHeaderBytes;
  w.desc = off;
  off = align_up(off + (size_t)(nch + 1) * sizeof(U), 256);
  w.anchors = off;
  off = align_up(off + (size_t)(nch / 32 + 2) * sizeof(U), 256);
  w.tails = off;
  off = align_up(off + (size_t)(nch + 1) * sizeof(U), 256);
  w.bits = off;
  if (seg) off = align_up(off + (size_t)((n + 31) / 32 + 1) * 4, 256);
  w.has_head = off;
  if (seg) off = align_up(off + (size_t)nch + 1, 256);
  w.total = off;
  return w;
}

template <typename T, bool SEG, bool REV, bool EXCL>
static cudaError_t launch_scan(const ScanArgs<T>& a, int threads, cudaStream_t s) {
  if (threads == 1024) {
    // persistent: one CTA per SM (cooperative launch), chunks assigned round-robin
    const size_t smem =
        ScanGeom<T>::kStageBytes + align_up(sizeof(KeepSmem<T>), 16) + (sizeof(T) == 4 && !REV ? 32 * 2048 : 0);
    auto kern = scan_keep_kernel<T, SEG, REV, EXCL>;
    cudaError_t e = ensure_dyn_smem((const void*)kern, smem);
    if (e != cudaSuccess) return e;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorUnknown;
    const int per_sm = kernel_occupancy((const void*)kern, 1024, smem);
    if (per_sm < 0) return cudaErrorUnknown;
    const long long grid = min((long long)sms * per_sm, a.nchunks + 1);
    if (grid >= 2) {
      void* args[] = {const_cast<ScanArgs<T>*>(&a)};
      launch_begin(SEG ? "det_segmented_scan" : "det_scan", s);
      e = cudaLaunchCooperativeKernel((const void*)kern, dim3((unsigned)grid), dim3(1024), args, smem, s);
      launch_end(s);
      return e;
    }
    // a grid of one CTA cannot hold a worker and the chain: use the
    // shared-memory kernel below
  }
  const size_t smem = ScanGeom<T>::kStageBytes + sizeof(ScanSmem<T>);
  auto kern = scan_kernel<T, SEG, REV, EXCL>;
  cudaError_t e = ensure_dyn_smem((const void*)kern, smem);
  if (e != cudaSuccess) return e;
  launch_begin(SEG ? "det_segmented_scan" : "det_scan", s);
  kern<<<(unsigned)(a.nchunks + 1), threads, smem, s>>>(a);
  launch_end(s);
  return cudaGetLastError();
}

// Launch the one-cluster scan (a CTA per chunk) when this device can host
// such a cluster: 1 launched, 0 not possible here, -1 a CUDA error.
template <typename T>
static int launch_scan_cluster(const ScanArgs<T>& a, bool rev, bool excl, cudaStream_t s) {
  void (*k)(const T*, T*, long long, T*, unsigned int*) =
      rev ? (excl ? scan_cluster_kernel<T, true, true> : scan_cluster_kernel<T, true, false>)
          : (excl ? scan_cluster_kernel<T, false, true> : scan_cluster_kernel<T, false, false>);
  const size_t smem = ScanGeom<T>::kStageBytes;
  const unsigned nc = (unsigned)a.nchunks;
  // can a cluster of nc such CTAs be resident?  (cached per kernel, device and size)
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, unsigned>, int> fits;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  const auto key = std::make_tuple((const void*)k, dev, nc);
  int ok = -1;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = fits.find(key);
    if (it != fits.end()) ok = it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nc);
  cfg.blockDim = dim3(1024);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (ok < 0) {
    ok = 0;
    if (ensure_dyn_smem((const void*)k, smem) == cudaSuccess &&
        (nc <= 8 || cudaFuncSetAttribute((const void*)k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                        cudaSuccess)) {
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, (const void*)k, &cfg) == cudaSuccess && clusters >= 1) ok = 1;
    }
    cudaGetLastError();   // a refused query leaves no error behind
    std::lock_guard<std::mutex> lock(mu);
    fits[key] = ok;
  }
  if (!ok) return 0;
  launch_begin("det_scan", s);
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, k, a.x, a.y, (long long)a.n, a.total_out, a.status);
  launch_end(s);
  return e == cudaSuccess ? 1 : -1;
}

template <typename T, bool SEG>
static int scan_impl(const T* x, T* y, long long n, const long long* seg_off, long long nseg, int flags,
                     T* total_out, void* ws, size_t ws_bytes, int bt, cudaStream_t s) {
  const ScanWs<T> L = scan_ws_layout<T>(n, SEG);
  if (ws_bytes < L.total) return DET_ERR_WORKSPACE;
  char* w = reinterpret_cast<char*>(ws);
  if (n == 0) {
    if (cudaMemsetAsync(w, 0, kHeaderBytes, s) != cudaSuccess) return DET_ERR_CUDA;
    if (total_out && cudaMemsetAsync(total_out, 0, sizeof(T), s) != cudaSuccess) return DET_ERR_CUDA;
    return DET_OK;
  }
  // f64 only: measured faster there (25.8 -> 22.6 us at 164,738 elements, a
  // chunk's FP64 adds dominate and the memset and look-back go away); for f32
  // the cluster launch cost more than it saved (14.3 -> 15.7 us)
  const bool cluster =
      sizeof(T) == 8 && !SEG && bt == 0 && (n + ScanGeom<T>::C - 1) / ScanGeom<T>::C <= kClusterChunks;
  // one clearing memset: the header, every published word ("unpublished"
  // is all-zero) and, for segmented scans, the head bitmap and chunk flags
  // (the one-cluster path for small inputs publishes nothing in global
  // memory and writes the status word itself)
  if (!cluster && cudaMemsetAsync(w, 0, SEG ? L.total : L.bits, s) != cudaSuccess) return DET_ERR_CUDA;
  WsHeader* h = reinterpret_cast<WsHeader*>(ws);
  ScanArgs<T> a;
  a.x = x;
  a.y = y;
  a.n = n;
  a.nchunks = (n + ScanGeom<T>::C - 1) / ScanGeom<T>::C;
  a.desc = reinterpret_cast<typename Bits<T>::U*>(w + L.desc);
  a.anchors = reinterpret_cast<typename Bits<T>::U*>(w + L.anchors);
  a.tails = reinterpret_cast<typename Bits<T>::U*>(w + L.tails);
  a.head_bits = nullptr;
  a.has_head = nullptr;
  a.ticket = &h->ticket;
  a.role = &h->ticket2;
  a.status = &h->status;
  a.total_out = total_out;
  a.timeout_ns = g_scan_wait_ns;
  a.withhold = g_scan_withhold;
  const bool rev = flags & DET_SCAN_REVERSE, excl = flags & DET_SCAN_EXCLUSIVE;
  if (SEG) {
    unsigned int* bits = reinterpret_cast<unsigned int*>(w + L.bits);
    unsigned char* hh = reinterpret_cast<unsigned char*>(w + L.has_head);
    a.head_bits = bits;
    a.has_head = hh;
    if (nseg > 0) {
      const unsigned blocks = (unsigned)((nseg + 255) / 256);
      launch_begin("det_seg_heads", s);
      if (rev)
        seg_heads_kernel<ScanGeom<T>::C, true><<<blocks, 256, 0, s>>>(seg_off, nseg, n, bits, hh, &h->status);
      else
        seg_heads_kernel<ScanGeom<T>::C, false><<<blocks, 256, 0, s>>>(seg_off, nseg, n, bits, hh, &h->status);
      launch_end(s);
      if (cudaGetLastError() != cudaSuccess) return DET_ERR_CUDA;
    }
  }
  const int threads = bt ? bt : 1024;
  cudaError_t e;
  if (cluster) {
    const int rc = launch_scan_cluster<T>(a, rev, excl, s);
    if (rc == 1) return DET_OK;     // launched
    if (rc < 0) return DET_ERR_CUDA;
    // rc == 0: this device cannot host the cluster: clear, then the general kernels below
    if (cudaMemsetAsync(w, 0, L.bits, s) != cudaSuccess) return DET_ERR_CUDA;
  }
  if (rev) {
    e = excl ? launch_scan<T, SEG, true, true>(a, threads, s) : launch_scan<T, SEG, true, false>(a, threads, s);
  } else {
    e = excl ? launch_scan<T, SEG, false, true>(a, threads, s) : launch_scan<T, SEG, false, false>(a, threads, s);
  }
  return e == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

}  // namespace det

using namespace det;

template <typename T>
static int restart_impl(const T* x, T* y, long long n, const long long* off, long long S, int flags, void* ws,
                        cudaStream_t s) {
  unsigned int* status = reinterpret_cast<unsigned int*>(ws);
  const bool rev = flags & DET_SCAN_REVERSE, excl = flags & DET_SCAN_EXCLUSIVE;
  void (*kern)(const T*, T*, long long, const long long*, long long, unsigned int*) =
      rev ? (excl ? restart_kernel<T, true, true> : restart_kernel<T, true, false>)
          : (excl ? restart_kernel<T, false, true> : restart_kernel<T, false, false>);
  // persistent: one wave of resident CTAs takes the segments in turn
  const int per_sm = std::max(1, kernel_occupancy((const void*)kern, 128, 0));
  const long long grid = std::max(1LL, std::min(S, (long long)per_sm * std::max(device_sm_count(), 1)));
  launch_begin("det_segmented_scan_restart", s);
  kern<<<(unsigned)grid, 128, 0, s>>>(x, y, n, off, S, status);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

extern "C" size_t det_scan_workspace_bytes(int64_t n, int dtype) {
  if (n < 0 || !valid_dtype(dtype)) return 0;
  return dtype == DET_F32 ? scan_ws_layout<float>(n, false).total : scan_ws_layout<double>(n, false).total;
}

extern "C" size_t det_segmented_scan_workspace_bytes(int64_t n, int64_t num_segments, int dtype) {
  if (n < 0 || num_segments < 0 || !valid_dtype(dtype)) return 0;
  return dtype == DET_F32 ? scan_ws_layout<float>(n, true).total : scan_ws_layout<double>(n, true).total;
}

extern "C" int det_scan(const void* x, void* y, int64_t n, int dtype, int flags, void* total_out,
                        void* workspace, size_t workspace_bytes, int block_threads, void* stream) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (n < 0 || !workspace || (n > 0 && (!x || !y)) || (flags & ~3) || !valid_block_threads(block_threads))
    return DET_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return DET_ERR_WORKSPACE;
  if (n > 0 && x != y) {
    const char *xb = (const char*)x, *yb = (const char*)y;
    const size_t bytes = (size_t)n * elem_size(dtype);
    if (xb < yb + bytes && yb < xb + bytes) return DET_ERR_INVALID_ARG;  // partial overlap
  }
  if (dtype == DET_F32)
    return scan_impl<float, false>((const float*)x, (float*)y, n, nullptr, 0, flags, (float*)total_out,
                                   workspace, workspace_bytes, block_threads, as_stream(stream));
  return scan_impl<double, false>((const double*)x, (double*)y, n, nullptr, 0, flags, (double*)total_out,
                                  workspace, workspace_bytes, block_threads, as_stream(stream));
}

extern "C" int det_segmented_scan(const void* x, void* y, int64_t n, const int64_t* seg_offsets,
                                  int64_t num_segments, int dtype, int flags, void* workspace,
                                  size_t workspace_bytes, int block_threads, void* stream) {
  if (!valid_dtype(dtype)) return DET_ERR_DTYPE;
  if (n < 0 || num_segments < 0 || !workspace || (flags & ~7) || !valid_block_threads(block_threads))
    return DET_ERR_INVALID_ARG;
  if (n > 0 && (!x || !y || !seg_offsets || num_segments < 1)) return DET_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return DET_ERR_WORKSPACE;
  if (n > 0 && x != y) {
    const char *xb = (const char*)x, *yb = (const char*)y;
    const size_t bytes = (size_t)n * elem_size(dtype);
    if (xb < yb + bytes && yb < xb + bytes) return DET_ERR_INVALID_ARG;
  }
  if (flags & DET_SCAN_SEGMENT_RESTART) {
    if (workspace_bytes < kHeaderBytes) return DET_ERR_WORKSPACE;
    const cudaStream_t s = as_stream(stream);
    if (cudaMemsetAsync(workspace, 0, kHeaderBytes, s) != cudaSuccess) return DET_ERR_CUDA;
    if (n == 0) return DET_OK;
    return dtype == DET_F32 ? restart_impl<float>((const float*)x, (float*)y, n, (const long long*)seg_offsets,
                                                  num_segments, flags, workspace, s)
                            : restart_impl<double>((const double*)x, (double*)y, n, (const long long*)seg_offsets,
                                                   num_segments, flags, workspace, s);
  }
  if (dtype == DET_F32)
    return scan_impl<float, true>((const float*)x, (float*)y, n, (const long long*)seg_offsets, num_segments,
                                  flags, nullptr, workspace, workspace_bytes, block_threads, as_stream(stream));
  return scan_impl<double, true>((const double*)x, (double*)y, n, (const long long*)seg_offsets, num_segments,
                                 flags, nullptr, workspace, workspace_bytes, block_threads, as_stream(stream));
}

extern "C" int det_test_scan_withhold(int64_t chunk, uint64_t timeout_ns) {
  if (chunk < 0) {
    g_scan_withhold = -1;
    g_scan_wait_ns = kWaitNs;
    return DET_OK;
  }
  if (timeout_ns == 0 || timeout_ns > kWaitNs) return DET_ERR_INVALID_ARG;
  g_scan_withhold = chunk;
  g_scan_wait_ns = timeout_ns;
  return DET_OK;
}
