// Stable LSD radix sort of (key, value, index) records with a validity
// filter, and the segmented pairwise tree over the sorted values.
//
//   hist      one read of the keys: per-pass digit histograms of the valid
//             keys (CTA-private shared counters, warp-aggregated with
//             match.any, then integer atomics: order-free) and the valid count
//   dstart    one CTA: exclusive scan of each pass's digit histogram
//   pass p    per tile of K = threads * 32 records, in ticket order:
//             warp multi-split ranks (match.any + popc) against per-warp
//             shared counters give each record its rank among earlier records
//             of its digit inside the warp; a cross-warp prefix per digit and
//             an integer decoupled look-back over tiles (integer addition is
//             associative, so whatever mix of partial and inclusive states a
//             tile observes, the offsets are the same) give the global
//             position digit_start + tile offset + warp offset + rank.
//             Records keep their input order inside a digit: the pass is
//             stable, so after the last pass each destination's records are
//             in ascending original index.
//   bounds    (more than one pass) segment starts from the sorted keys
//   tree      out[b] = out[b] + PT(group b): groups of at most 2048 records
//             are reduced by one warp; longer groups are cut into
//             rank-aligned 2048-blocks (subtrees of the group's tree),
//             reduced by one warp each, then a tree over the block nodes.
#include "det_sort.cuh"

namespace det {
namespace {

constexpr int kIPT = 32;                 // records per thread per tile
constexpr unsigned long long kAggFlag = 1ull << 62;
constexpr unsigned long long kInclFlag = 1ull << 63;
constexpr unsigned long long kCountMask = (1ull << 40) - 1;

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
sort_hist_kernel(const int32_t* __restrict__ keys, long long n, long long key_offset, long long m, int passes,
                 int D, unsigned int* __restrict__ hist, unsigned int* __restrict__ n_valid) {
  __shared__ unsigned int sh[4][1024];
  const int tid = threadIdx.x, lane = tid & 31;
  const int ndig = 1 << D;
  const unsigned mask = (unsigned)ndig - 1u;
  for (int i = tid; i < 4 * 1024; i += blockDim.x) (&sh[0][0])[i] = 0u;
  __syncthreads();
  const long long nwarps_total = (long long)gridDim.x * (blockDim.x >> 5);
  const long long gwarp = (long long)blockIdx.x * (blockDim.x >> 5) + (tid >> 5);
  unsigned int local_valid = 0;
  for (long long wb = gwarp * 32; wb < n; wb += nwarps_total * 32) {
    const long long i = wb + lane;
    const long long key = (i < n) ? (long long)keys[i] + key_offset : -1;
    const bool valid = key >= 0 && key < m;
    local_valid += valid;
    for (int p = 0; p < passes; ++p) {
      const unsigned d = ((unsigned)key >> (p * D)) & mask;
      const unsigned peers = __match_any_sync(0xffffffffu, valid ? d : (0x80000000u | (unsigned)lane));
      if (valid && lane == __ffs(peers) - 1) atomicAdd(&sh[p][d], (unsigned)__popc(peers));
    }
  }
  __syncthreads();
  for (int p = 0; p < passes; ++p)
    for (int d = tid; d < ndig; d += blockDim.x)
      if (sh[p][d]) atomicAdd(&hist[p * 1024 + d], sh[p][d]);
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) local_valid += __shfl_xor_sync(0xffffffffu, local_valid, s);
  if (lane == 0 && local_valid) atomicAdd(n_valid, local_valid);
}

// One CTA of 1024 threads: dstart[p][d] = sum of hist[p][d'] for d' < d.
__global__ void __launch_bounds__(1024)
sort_dstart_kernel(const unsigned int* __restrict__ hist, int passes, int D, unsigned int* __restrict__ dstart) {
  __shared__ unsigned int wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ndig = 1 << D;
  for (int p = 0; p < passes; ++p) {
    const unsigned v = tid < ndig ? hist[p * 1024 + tid] : 0u;
    unsigned x = v;
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
      wsum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const unsigned before = (warp ? wsum[warp - 1] : 0u) + x - v;
    if (tid < ndig) dstart[p * 1025 + tid] = before;
    if (tid == ndig - 1) dstart[p * 1025 + ndig] = before + v;
    __syncthreads();
  }
}

template <int VB> struct Payload;
template <> struct Payload<0> { using U = unsigned int; };
template <> struct Payload<4> { using U = unsigned int; };
template <> struct Payload<8> { using U = unsigned long long; };

struct PassArgs {
  const int32_t* keys_in;
  const void* vals_in;
  const int32_t* idx_in;
  int32_t* keys_out;
  void* vals_out;
  int32_t* idx_out;
  long long n;
  long long key_offset;
  long long m;
  int shift;
  int D;
  const unsigned int* dstart;
  unsigned long long* state;
  unsigned int* ticket;
  unsigned int* status;
  const unsigned int* n_valid;
  unsigned long long timeout_ns;
};

template <int VB, bool FIRST, bool IDX, bool KEYS_OUT>
__global__ void __launch_bounds__(1024) sort_pass_kernel(PassArgs a) {
  using U = typename Payload<VB>::U;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int ndig = 1 << a.D;
  const unsigned mask = (unsigned)ndig - 1u;
  unsigned short* wcnt = reinterpret_cast<unsigned short*>(smem_raw);                 // [nwarps][ndig]
  unsigned int* gbase = reinterpret_cast<unsigned int*>(smem_raw + (size_t)nwarps * ndig * 2);  // [ndig]
  __shared__ long long s_tile;

  if (tid == 0) s_tile = (long long)atomicAdd(a.ticket, 1u);
  __syncthreads();
  const long long tile = s_tile;
  const long long N = FIRST ? a.n : (long long)*a.n_valid;
  const long long K = (long long)blockDim.x * kIPT;
  const long long tile_base = tile * K;
  if (tile_base >= N) return;
  const long long wbase = tile_base + (long long)warp * 32 * kIPT;

  for (int d = lane; d < ndig; d += 32) wcnt[warp * ndig + d] = 0;
  __syncwarp();

  // ---- rank inside the warp, record order = (round, lane) = input order
  unsigned packed[kIPT];
#pragma unroll
  for (int r = 0; r < kIPT; ++r) {
    const long long i = wbase + (long long)r * 32 + lane;
    bool valid = i < N;
    unsigned key = 0;
    if (valid) {
      if (FIRST) {
        const long long k = (long long)a.keys_in[i] + a.key_offset;
        valid = k >= 0 && k < a.m;
        key = (unsigned)k;
      } else {
        key = (unsigned)a.keys_in[i];
      }
    }
    const unsigned d = (key >> a.shift) & mask;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? d : (0x80000000u | (unsigned)lane));
    unsigned base = 0;
    if (valid) base = wcnt[warp * ndig + d];
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) wcnt[warp * ndig + d] = (unsigned short)(base + __popc(peers));
    __syncwarp();
    packed[r] = valid ? ((d << 16) | (base + __popc(peers & ((1u << lane) - 1u)))) : 0xffffffffu;
  }
  __syncthreads();

  // ---- per digit: warp offsets, tile count, look-back over tiles
  for (int d = tid; d < ndig; d += blockDim.x) {
    unsigned run = 0;
    for (int w = 0; w < nwarps; ++w) {
      const unsigned c = wcnt[w * ndig + d];
      wcnt[w * ndig + d] = (unsigned short)run;
      run += c;
    }
    unsigned long long* st = a.state + tile * ndig + d;
    if (tile == 0) {
      st_relaxed_u64(st, kInclFlag | run);
      gbase[d] = a.dstart[d];
      continue;
    }
    st_relaxed_u64(st, kAggFlag | run);
    unsigned long long excl = 0;
    long long t = tile - 1;
    bool ok = true;
    while (t >= 0) {
      const unsigned long long* q = a.state + t * ndig + d;
      unsigned long long v = ld_relaxed_u64(q);
      if (v == 0) {
        const unsigned long long t0 = gtimer();
        unsigned polls = 0;
        while ((v = ld_relaxed_u64(q)) == 0) {
          if ((++polls & 63u) == 0) {
            if (*(volatile unsigned int*)a.status != 0u) { ok = false; break; }
            if (gtimer() - t0 > a.timeout_ns) {
              set_status(a.status, DET_ERR_LOOKBACK_TIMEOUT);
              ok = false;
              break;
            }
          }
        }
        if (!ok) break;
      }
      excl += v & kCountMask;
      if (v & kInclFlag) break;
      --t;
    }
    st_relaxed_u64(st, kInclFlag | (excl + run));
    gbase[d] = a.dstart[d] + (unsigned)excl;
  }
  __syncthreads();

  // ---- move the payload to its sorted position
  const U* vin = reinterpret_cast<const U*>(a.vals_in);
  U* vout = reinterpret_cast<U*>(a.vals_out);
#pragma unroll
  for (int r = 0; r < kIPT; ++r) {
    const unsigned pk = packed[r];
    if (pk == 0xffffffffu) continue;
    const long long i = wbase + (long long)r * 32 + lane;
    const unsigned d = pk >> 16;
    const long long pos = (long long)gbase[d] + wcnt[warp * ndig + d] + (pk & 0xffffu);
    if (pos < 0 || pos >= a.n) {   // cannot happen for a correct ranking; never write out of bounds
      set_status(a.status, DET_ERR_INVALID_ARG);
      continue;
    }
    if (VB) vout[pos] = vin[i];
    if (IDX) a.idx_out[pos] = FIRST ? (int32_t)i : a.idx_in[i];
    if (KEYS_OUT) a.keys_out[pos] = FIRST ? (int32_t)((long long)a.keys_in[i] + a.key_offset) : a.keys_in[i];
  }
}

// seg[b] = first sorted position with key >= b, for b = 0..m (keys sorted).
__global__ void sort_bounds_kernel(const int32_t* __restrict__ keys, const unsigned int* __restrict__ n_valid,
                                   long long m, int32_t* __restrict__ seg, long long n) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long N = *n_valid;
  if (i > N || i > n) return;
  const long long prev = (i == 0) ? -1 : max(-1LL, min((long long)keys[i - 1], m));
  const long long cur = (i == N) ? m : max(-1LL, min((long long)keys[i], m));
  for (long long b = prev + 1; b <= cur; ++b) seg[b] = (int32_t)i;
}

__global__ void copy_u32_kernel(const unsigned int* __restrict__ src, int32_t* __restrict__ dst, long long count) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < count) dst[i] = (int32_t)src[i];
}

// ---------------------------------------------------------------------------
// PT over p[0..len) by one warp: rounds of 256 (8 per lane, in-register tree,
// then five shuffle levels) combined by a binary counter (rounds are aligned
// 256-blocks, i.e. nodes of level 8), collapsed by a right fold at the end.
template <typename T>
__device__ T warp_pt_range(const T* __restrict__ p, long long len) {
  const int lane = threadIdx.x & 31;
  T stack[40];
  long long cnt = 0;
  const long long rounds = (len + 255) / 256;
  for (long long r = 0; r < rounds; ++r) {
    T v[8];
    const long long b = r * 256 + lane * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = (b + e < len) ? __ldg(p + b + e) : absent<T>();
    T node = warp_pt(thread_pt(v));
    int lvl = 0;
    long long c = cnt;
    while (c & 1) {
      node = stack[lvl] + node;
      c >>= 1;
      ++lvl;
    }
    stack[lvl] = node;
    ++cnt;
  }
  T res = absent<T>();
  bool have = false;
  for (int lvl = 0; lvl < 40; ++lvl) {
    if ((cnt >> lvl) & 1) {
      res = have ? stack[lvl] + res : stack[lvl];
      have = true;
    }
  }
  return res;
}

struct LongSeg {
  long long bin;
  long long base;
  long long nblk;
};

template <typename T>
__global__ void __launch_bounds__(256)
segtree_bins_kernel(const T* __restrict__ vals, const int32_t* __restrict__ seg, long long m, T* __restrict__ out,
                    long long* __restrict__ blocks, LongSeg* __restrict__ lsegs, unsigned int* __restrict__ nblocks,
                    unsigned int* __restrict__ nlsegs, const unsigned int* __restrict__ n_valid, long long max_blocks,
                    long long max_lsegs, unsigned int* __restrict__ status) {
  const long long b = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (b >= m) return;
  const long long N = *n_valid;
  const long long hi = min((long long)seg[b + 1], N), lo = max(0LL, min((long long)seg[b], hi));
  const long long len = hi - lo;
  if (len <= 0) return;
  if (len <= kSegBlock) {
    const T t = warp_pt_range(vals + lo, len);
    if (lane == 0) out[b] = out[b] + t;
    return;
  }
  const long long nblk = (len + kSegBlock - 1) / kSegBlock;
  long long base = 0;
  if (lane == 0) {
    base = atomicAdd(nblocks, (unsigned)nblk);
    const unsigned s = atomicAdd(nlsegs, 1u);
    if (s < max_lsegs && base + nblk <= max_blocks)
      lsegs[s] = LongSeg{b, base, nblk};
    else
      set_status(status, DET_ERR_INVALID_ARG);
  }
  base = __shfl_sync(0xffffffffu, base, 0);
  if (base + nblk > max_blocks) return;
  for (long long k = lane; k < nblk; k += 32) blocks[base + k] = (b << 24) | k;
}

template <typename T>
__global__ void __launch_bounds__(256)
segtree_blocks_kernel(const T* __restrict__ vals, const int32_t* __restrict__ seg, const long long* __restrict__ blocks,
                      const unsigned int* __restrict__ nblocks, T* __restrict__ nodes,
                      const unsigned int* __restrict__ n_valid, long long max_blocks) {
  const long long q = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (q >= (long long)*nblocks || q >= max_blocks) return;
  const long long e = blocks[q];
  const long long b = e >> 24, k = e & ((1 << 24) - 1);
  const long long N = *n_valid;
  const long long hi = min((long long)seg[b + 1], N);
  const long long lo = max(0LL, min((long long)seg[b] + k * kSegBlock, hi));
  const long long len = min((long long)kSegBlock, hi - lo);
  const T t = warp_pt_range(vals + lo, len);
  if (lane == 0) nodes[q] = t;
}

template <typename T>
__global__ void __launch_bounds__(256)
segtree_long_kernel(const LongSeg* __restrict__ lsegs, const unsigned int* __restrict__ nlsegs,
                    const T* __restrict__ nodes, T* __restrict__ out, long long max_lsegs) {
  const long long s = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (s >= (long long)*nlsegs || s >= max_lsegs) return;
  const LongSeg L = lsegs[s];
  const T t = warp_pt_range(nodes + L.base, L.nblk);
  if (lane == 0) out[L.bin] = out[L.bin] + t;
}

}  // namespace

// ---------------------------------------------------------------------------

SortPlan make_sort_plan(long long n, long long m, int value_bytes, bool need_idx, int block_threads) {
  SortPlan p;
  p.n = n;
  p.m = m;
  p.value_bytes = value_bytes;
  p.need_idx = need_idx;
  int B = 0;
  while ((1LL << B) < m) ++B;
  p.passes = B <= 10 ? 1 : (B + 9) / 10;
  p.digit_bits = B == 0 ? 1 : (B + p.passes - 1) / p.passes;
  p.threads = block_threads ? block_threads : 512;
  p.ipt = kIPT;
  const long long K = (long long)p.threads * kIPT;
  p.tiles = (n + K - 1) / K;
  const long long ndig = 1LL << p.digit_bits;
  size_t off = kHeaderBytes;
  p.hist = off;
  off = align_up(off + 4 * 1024 * 4, 256);
  p.dstart = off;
  off = align_up(off + 4 * 1025 * 4, 256);
  p.state = off;
  off = align_up(off + (size_t)(p.tiles + 1) * ndig * 8, 256);
  const int nb = p.passes > 1 ? 2 : 1;
  for (int b = 0; b < nb; ++b) {
    if (p.passes > 1) {
      p.keys[b] = off;
      off = align_up(off + (size_t)n * 4 + 4, 256);
    }
    if (value_bytes) {
      p.vals[b] = off;
      off = align_up(off + (size_t)n * value_bytes + 8, 256);
    }
    if (need_idx) {
      p.idx[b] = off;
      off = align_up(off + (size_t)n * 4 + 4, 256);
    }
  }
  p.seg = off;
  off = align_up(off + (size_t)(m + 1) * 4, 256);
  p.max_blocks = 2 * (n / kSegBlock) + 2;
  p.max_lsegs = n / kSegBlock + 2;
  p.blocks = off;
  off = align_up(off + (size_t)p.max_blocks * 8, 256);
  p.lsegs = off;
  off = align_up(off + (size_t)p.max_lsegs * sizeof(LongSeg), 256);
  p.nodes = off;
  off = align_up(off + (size_t)p.max_blocks * 8, 256);
  p.total = off;
  return p;
}

template <int VB>
static cudaError_t launch_pass(const PassArgs& a, bool first, bool idx, bool keys_out, int threads, long long tiles,
                               cudaStream_t s) {
  const int ndig = 1 << a.D;
  const size_t smem = (size_t)(threads / 32) * ndig * 2 + (size_t)ndig * 4;
  void (*k)(PassArgs) = nullptr;
#define DET_PICK(F, I, KO) \
  if (first == F && idx == I && keys_out == KO) k = sort_pass_kernel<VB, F, I, KO>;
  DET_PICK(true, true, true) DET_PICK(true, true, false) DET_PICK(true, false, true) DET_PICK(true, false, false)
  DET_PICK(false, true, true) DET_PICK(false, true, false) DET_PICK(false, false, true) DET_PICK(false, false, false)
#undef DET_PICK
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  launch_begin("det_sort_pass", s);
  k<<<(unsigned)tiles, threads, smem, s>>>(a);
  launch_end(s);
  return cudaGetLastError();
}

int enqueue_sort(const SortPlan& p, void* ws, const int32_t* keys, long long key_offset, const void* values,
                 int32_t* perm_out, cudaStream_t s, int* final_buf) {
  char* w = reinterpret_cast<char*>(ws);
  SortHdr* h = reinterpret_cast<SortHdr*>(ws);
  // header + histograms are contiguous: one memset
  if (cudaMemsetAsync(w, 0, p.dstart, s) != cudaSuccess) return DET_ERR_CUDA;
  *final_buf = (p.passes - 1) & 1;
  if (p.n == 0 || p.m == 0) {
    if (cudaMemsetAsync(w + p.seg, 0, (size_t)(p.m + 1) * 4, s) != cudaSuccess) return DET_ERR_CUDA;
    return DET_OK;
  }
  unsigned int* hist = reinterpret_cast<unsigned int*>(w + p.hist);
  unsigned int* dstart = reinterpret_cast<unsigned int*>(w + p.dstart);
  {
    long long blocks = min((long long)2 * 152, (p.n + 1023) / 1024);
    if (blocks < 1) blocks = 1;
    launch_begin("det_sort_hist", s);
    sort_hist_kernel<<<(unsigned)blocks, 1024, 0, s>>>(keys, p.n, key_offset, p.m, p.passes, p.digit_bits, hist,
                                                      &h->n_valid);
    launch_end(s);
    if (cudaGetLastError() != cudaSuccess) return DET_ERR_CUDA;
    launch_begin("det_sort_dstart", s);
    sort_dstart_kernel<<<1, 1024, 0, s>>>(hist, p.passes, p.digit_bits, dstart);
    launch_end(s);
    if (cudaGetLastError() != cudaSuccess) return DET_ERR_CUDA;
  }
  const long long ndig = 1LL << p.digit_bits;
  for (int pass = 0; pass < p.passes; ++pass) {
    const bool first = pass == 0, last = pass == p.passes - 1;
    const int out = pass & 1, in = (pass - 1) & 1;
    if (cudaMemsetAsync(w + p.state, 0, (size_t)p.tiles * ndig * 8, s) != cudaSuccess) return DET_ERR_CUDA;
    PassArgs a;
    a.keys_in = first ? keys : reinterpret_cast<const int32_t*>(w + p.keys[in]);
    a.vals_in = first ? values : (p.value_bytes ? w + p.vals[in] : nullptr);
    a.idx_in = (first || !p.need_idx) ? nullptr : reinterpret_cast<const int32_t*>(w + p.idx[in]);
    a.keys_out = p.passes > 1 ? reinterpret_cast<int32_t*>(w + p.keys[out]) : nullptr;
    a.vals_out = p.value_bytes ? w + p.vals[out] : nullptr;
    a.idx_out = p.need_idx ? ((last && perm_out) ? perm_out : reinterpret_cast<int32_t*>(w + p.idx[out])) : nullptr;
    a.n = p.n;
    a.key_offset = key_offset;
    a.m = p.m;
    a.shift = pass * p.digit_bits;
    a.D = p.digit_bits;
    a.dstart = dstart + pass * 1025;
    a.state = reinterpret_cast<unsigned long long*>(w + p.state);
    a.ticket = &h->tickets[pass];
    a.status = &h->status;
    a.n_valid = &h->n_valid;
    a.timeout_ns = 2000000000ull;
    const bool keys_out = p.passes > 1;
    cudaError_t e;
    if (p.value_bytes == 8)
      e = launch_pass<8>(a, first, p.need_idx, keys_out, p.threads, p.tiles, s);
    else if (p.value_bytes == 4)
      e = launch_pass<4>(a, first, p.need_idx, keys_out, p.threads, p.tiles, s);
    else
      e = launch_pass<0>(a, first, p.need_idx, keys_out, p.threads, p.tiles, s);
    if (e != cudaSuccess) return DET_ERR_CUDA;
  }
  int32_t* seg = reinterpret_cast<int32_t*>(w + p.seg);
  if (p.passes == 1) {
    launch_begin("det_sort_seg_copy", s);
    copy_u32_kernel<<<(unsigned)((p.m + 1 + 255) / 256), 256, 0, s>>>(dstart, seg, p.m + 1);
    launch_end(s);
  } else {
    launch_begin("det_sort_bounds", s);
    sort_bounds_kernel<<<(unsigned)((p.n + 1 + 255) / 256), 256, 0, s>>>(
        reinterpret_cast<const int32_t*>(w + p.keys[*final_buf]), &h->n_valid, p.m, seg, p.n);
    launch_end(s);
  }
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

template <typename T>
int enqueue_segmented_tree(const SortPlan& p, void* ws, const T* sorted_vals, T* out, cudaStream_t s) {
  if (p.n == 0 || p.m == 0) return DET_OK;
  char* w = reinterpret_cast<char*>(ws);
  SortHdr* h = reinterpret_cast<SortHdr*>(ws);
  const int32_t* seg = reinterpret_cast<const int32_t*>(w + p.seg);
  long long* blocks = reinterpret_cast<long long*>(w + p.blocks);
  LongSeg* lsegs = reinterpret_cast<LongSeg*>(w + p.lsegs);
  T* nodes = reinterpret_cast<T*>(w + p.nodes);
  launch_begin("det_segtree_bins", s);
  segtree_bins_kernel<T><<<(unsigned)((p.m * 32 + 255) / 256), 256, 0, s>>>(
      sorted_vals, seg, p.m, out, blocks, lsegs, &h->long_blocks, &h->long_segs, &h->n_valid, p.max_blocks,
      p.max_lsegs, &h->status);
  launch_end(s);
  launch_begin("det_segtree_blocks", s);
  segtree_blocks_kernel<T><<<(unsigned)((p.max_blocks * 32 + 255) / 256), 256, 0, s>>>(
      sorted_vals, seg, blocks, &h->long_blocks, nodes, &h->n_valid, p.max_blocks);
  launch_end(s);
  launch_begin("det_segtree_long", s);
  segtree_long_kernel<T><<<(unsigned)((p.max_lsegs * 32 + 255) / 256), 256, 0, s>>>(lsegs, &h->long_segs, nodes, out,
                                                                                    p.max_lsegs);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}

template int enqueue_segmented_tree<float>(const SortPlan&, void*, const float*, float*, cudaStream_t);
template int enqueue_segmented_tree<double>(const SortPlan&, void*, const double*, double*, cudaStream_t);

}  // namespace det
