// Stable LSD radix sort of (key, value, index) records with a validity
// filter, and the segmented pairwise tree over the sorted values.
//
//   count p   per tile of K = threads * 32 records: digit counts of the
//             valid records (shared integer atomics: order-free)
//   colscan p per digit: exclusive prefix of the counts over tiles, and the
//             digit totals (pass 0 also sums them into the valid count)
//   pass p    per tile, independently: digit starts from the totals; a warp
//             multi-split (peer masks OR-ed into per-warp shared words) and
//             per-warp shared counters give each record its rank among
//             earlier records of its digit inside the warp; position = digit
//             start + tile prefix + warp prefix + rank.
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
// ---------------------------------------------------------------------------
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
  long long tiles;
  long long K;                 // records per tile
  unsigned int* counts;        // [tiles][ndig]: tile counts, then exclusive column prefixes
  unsigned int* totals;        // [ndig] column totals
  unsigned int* status;
  unsigned int* n_valid;
  int32_t* seg_out;            // one-pass sorts: segment starts (m + 1), written by CTA 0 of the pass
  int32_t* rank_out;           // one-pass sorts: sorted position of every valid record, in input order
};

// Digit of record i of a pass, or 0xffffffff if it is past the end or
// (first pass) its destination is outside [0, m).
// The count kernel reads the keys with a normal cached load so that the
// pass kernel, which reads them last, mostly finds them in L2.
template <bool FIRST>
__device__ __forceinline__ unsigned digit_of(const PassArgs& a, int32_t raw, unsigned mask) {
  if (FIRST) {
    if (a.key_offset == 0) return (unsigned)raw < (unsigned long long)a.m ? ((unsigned)raw >> a.shift) & mask : 0xffffffffu;
    const long long k = (long long)raw + a.key_offset;
    return (k >= 0 && k < a.m) ? ((unsigned)k >> a.shift) & mask : 0xffffffffu;
  }
  return ((unsigned)raw >> a.shift) & mask;
}
template <bool FIRST, bool LAST_USE>
__device__ __forceinline__ unsigned record_digit(const PassArgs& a, long long i, long long N, unsigned mask) {
  if (i >= N) return 0xffffffffu;
  return digit_of<FIRST>(a, LAST_USE ? __ldcs(a.keys_in + i) : __ldg(a.keys_in + i), mask);
}

// counts[tile][d] = records of the tile with digit d.  The tile is the
// scatter pass's tile (K = pass_threads * kIPT records); counting is
// order-free, so here each thread simply streams its share of the tile with
// 16-byte loads, several in flight, and keeps a run of equal digits in
// registers, adding it by one shared atomic when the digit changes (a hot
// digit costs almost no atomics).
template <bool FIRST>
__global__ void __launch_bounds__(256, 8) sort_count_kernel(PassArgs a, long long K) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned int* cnt = reinterpret_cast<unsigned int*>(smem_raw);   // [ndig]
  const int tid = threadIdx.x, lane = tid & 31;
  const int ndig = 1 << a.D;
  const unsigned mask = (unsigned)ndig - 1u;
  const long long tile = blockIdx.x;
  const long long N = FIRST ? a.n : (long long)*a.n_valid;
  for (int d = tid; d < ndig; d += blockDim.x) cnt[d] = 0u;
  __syncthreads();
  const long long t0 = tile * K, t1 = min(N, t0 + K);
  // a run of equal digits is kept in registers and added by one atomic when
  // the digit changes (records are counted in any order)
  unsigned rd = 0xffffffffu, rc = 0;
  auto count = [&](int k, bool in) {
    unsigned d = 0xffffffffu;
    if (in) {
      if (FIRST) {
        if (a.key_offset == 0) {
          if ((unsigned)k < (unsigned long long)a.m) d = ((unsigned)k >> a.shift) & mask;
        } else {
          const long long kk = (long long)k + a.key_offset;
          if (kk >= 0 && kk < a.m) d = ((unsigned)kk >> a.shift) & mask;
        }
      } else {
        d = ((unsigned)k >> a.shift) & mask;
      }
    }
    if (d == 0xffffffffu) return;
    if (d != rd) {
      if (rc) atomicAdd(&cnt[rd], rc);
      rd = d;
      rc = 0;
    }
    ++rc;
  };
  if (t0 < t1) {
    const bool vec = (reinterpret_cast<uintptr_t>(a.keys_in + t0) & 15) == 0;
    constexpr int U = 4;   // 16-byte loads in flight per thread per step
    long long i = t0;
    if (vec) {
      const long long span = (long long)blockDim.x * 4 * U;
      for (; i + span <= t1; i += span) {
        int4 q[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
          q[u] = __ldg(reinterpret_cast<const int4*>(a.keys_in + i + (long long)u * blockDim.x * 4) + tid);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          count(q[u].x, true);
          count(q[u].y, true);
          count(q[u].z, true);
          count(q[u].w, true);
        }
      }
    }
    // remainder: whole warps step together, lanes past the end count nothing
    for (long long b = i + (long long)(tid & ~31); b < t1; b += blockDim.x) {
      const long long j = b + lane;
      count(j < t1 ? __ldg(a.keys_in + j) : 0, j < t1);
    }
  }
  if (rc) atomicAdd(&cnt[rd], rc);
  __syncthreads();
  for (int d = tid; d < ndig; d += blockDim.x) a.counts[tile * ndig + d] = cnt[d];
}

// For each digit column: exclusive prefix over tiles (in place) and the
// column total.  CTA of 1024 threads = 8 digit lanes x 128 tile groups (a
// warp reads 8 consecutive digits of 4 tiles: whole 32-byte sectors).
constexpr int kColDigits = 8, kColGroups = 128;
__global__ void __launch_bounds__(1024) sort_colscan_kernel(PassArgs a, int count_valid) {
  __shared__ unsigned int part[kColGroups][kColDigits + 1];
  const int dl = threadIdx.x % kColDigits, g = threadIdx.x / kColDigits;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ndig = 1 << a.D;
  const int d = blockIdx.x * kColDigits + dl;
  const long long T = a.tiles;
  const long long TG = (T + kColGroups - 1) / kColGroups;
  const long long t0 = g * TG, t1 = min(T, t0 + TG);
  unsigned sum = 0;
  if (d < ndig)
    for (long long t = t0; t < t1; ++t) sum += a.counts[t * ndig + d];
  part[g][dl] = sum;
  __syncthreads();
  if (warp < kColDigits) {
    // exclusive scan over the 128 groups of digit column `warp`: 4 groups per lane
    const int c = warp;
    unsigned v[kColGroups / 32], loc = 0;
#pragma unroll
    for (int k = 0; k < kColGroups / 32; ++k) {
      v[k] = part[lane * (kColGroups / 32) + k][c];
      loc += v[k];
    }
    unsigned x = loc;
#pragma unroll
    for (int s2 = 1; s2 < 32; s2 <<= 1) {
      const unsigned o = __shfl_up_sync(0xffffffffu, x, s2);
      if (lane >= s2) x += o;
    }
    unsigned run = x - loc;
#pragma unroll
    for (int k = 0; k < kColGroups / 32; ++k) {
      part[lane * (kColGroups / 32) + k][c] = run;
      run += v[k];
    }
    const unsigned total = __shfl_sync(0xffffffffu, x, 31);
    const int dc = blockIdx.x * kColDigits + c;
    if (lane == 0 && dc < ndig) {
      a.totals[dc] = total;
      if (count_valid && total) atomicAdd(a.n_valid, total);
    }
  }
  __syncthreads();
  unsigned run = part[g][dl];
  if (d < ndig)
    for (long long t = t0; t < t1; ++t) {
      const unsigned v = a.counts[t * ndig + d];
      a.counts[t * ndig + d] = run;
      run += v;
    }
}

// Exclusive block scan of the digit totals into base[0..ndig]; 1024 threads.
__device__ __forceinline__ void digit_starts(const unsigned int* totals, int ndig, unsigned int* base,
                                             unsigned int* wsum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int per = (ndig + blockDim.x - 1) / blockDim.x;   // digits per thread (contiguous)
  unsigned loc = 0;
  for (int k = 0; k < per; ++k) {
    const int d = tid * per + k;
    if (d < ndig) loc += totals[d];
  }
  unsigned x = loc;
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
    const unsigned o = __shfl_up_sync(0xffffffffu, x, s);
    if (lane >= s) x += o;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned wv = lane < nw ? wsum[lane] : 0u;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const unsigned o = __shfl_up_sync(0xffffffffu, wv, s);
      if (lane >= s) wv += o;
    }
    wsum[lane] = wv;
  }
  __syncthreads();
  unsigned run = (warp ? wsum[warp - 1] : 0u) + x - loc;
  for (int k = 0; k < per; ++k) {
    const int d = tid * per + k;
    if (d < ndig) {
      base[d] = run;
      run += totals[d];
    }
  }
  if (tid == blockDim.x - 1) base[ndig] = run;
  __syncthreads();
}

// 4- or 8-byte asynchronous copy global -> shared (both naturally aligned).
template <int BYTES>
__device__ __forceinline__ void cp_async_small(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(sa), "l"(gmem), "n"(BYTES) : "memory");
}
__device__ __forceinline__ void cp_async_commit_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}

template <int VB> struct Payload;
template <> struct Payload<0> { using U = unsigned int; };
template <> struct Payload<4> { using U = unsigned int; };
template <> struct Payload<8> { using U = unsigned long long; };

// Shared bytes of the staging area of a pass (records in tile-sorted order).
__host__ __device__ inline size_t pass_staging_bytes(long long K, int vb, bool idx, bool keys_out) {
  return (size_t)K * (vb + (idx ? 4 : 0) + (keys_out ? 4 : 0) + 2);
}
__host__ __device__ inline size_t pass_front_bytes(int nwarps, int ndig, long long K, int vb, bool idx, bool keys_out,
                                                   bool stage) {
  const size_t ranking = (size_t)nwarps * ndig * 6;
  const size_t staging = stage ? pass_staging_bytes(K, vb, idx, keys_out) : 0;
  return align_up(ranking > staging ? ranking : staging, 16);
}

template <int VB, bool FIRST, bool IDX, bool KEYS_OUT, bool STAGE>
__global__ void __launch_bounds__(256, 3) sort_pass_kernel(PassArgs a) {
  using U = typename Payload<VB>::U;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int ndig = 1 << a.D;
  const unsigned mask = (unsigned)ndig - 1u;
  unsigned int* pmask = reinterpret_cast<unsigned int*>(smem_raw);                           // [nwarps][ndig]
  unsigned short* wcnt = reinterpret_cast<unsigned short*>(smem_raw + (size_t)nwarps * ndig * 4); // [nwarps][ndig]
  unsigned int* gbase = reinterpret_cast<unsigned int*>(
      smem_raw + pass_front_bytes(nwarps, ndig, a.K, VB, IDX, KEYS_OUT, STAGE));   // [ndig + 1]
  __shared__ unsigned int wsum[32];
  __shared__ unsigned int n_digits;   // distinct digits of the tile

  const long long tile = blockIdx.x;
  const long long N = FIRST ? a.n : (long long)*a.n_valid;
  const long long K = (long long)blockDim.x * kIPT;
  const long long tile_base = tile * K;
  if (tile_base >= N) return;
  const long long wbase = tile_base + (long long)warp * 32 * kIPT;
  {
    // the payloads are read after the ranking: start moving them into L2 now
    const long long cnt = min(K, N - tile_base);
    if (VB) prefetch_l2(reinterpret_cast<const unsigned char*>(a.vals_in) + tile_base * VB, (size_t)cnt * VB, tid, 32);
    if (IDX && !FIRST) prefetch_l2(a.idx_in + tile_base, (size_t)cnt * 4, tid, 32);
  }

  // ---- this tile's digits; record order = (round, lane) = input order.
  // A full, aligned tile comes in by one bulk copy into the front of shared
  // memory (the ranking arrays, zeroed only after the digit-start scan's
  // barriers): 4-byte loads from every thread cannot keep enough requests in
  // flight.  Other tiles use plain loads.
  unsigned packed[kIPT];
  __shared__ __align__(8) unsigned long long keys_bar;
  const bool bulk = (N - tile_base) >= K &&
                    (size_t)K * 4 <= pass_front_bytes(nwarps, ndig, a.K, VB, IDX, KEYS_OUT, STAGE) &&
                    (reinterpret_cast<uintptr_t>(a.keys_in + tile_base) & 15) == 0;
  if (bulk) {
    if (tid == 0) {
      mbar_init(&keys_bar, 1);
      mbar_arrive_expect_tx(&keys_bar, (unsigned)(K * 4));
      bulk_copy_g2s(smem_raw, a.keys_in + tile_base, (unsigned)(K * 4), &keys_bar);
    }
    __syncthreads();   // the barrier is initialised before anyone waits on it
    const bool ok = mbar_wait(&keys_bar, 0, kWaitNs);
    if (__syncthreads_or(!ok)) {
      // the copy did not complete: record it, give it (bounded) time to land, leave
      if (tid == 0) {
        set_status(a.status, DET_ERR_COPY_TIMEOUT);
        mbar_wait(&keys_bar, 0, kWaitNs);
      }
      __syncthreads();
      return;
    }
    const int32_t* sk = reinterpret_cast<const int32_t*>(smem_raw) + warp * 32 * kIPT;
#pragma unroll
    for (int r = 0; r < kIPT; ++r) packed[r] = digit_of<FIRST>(a, sk[r * 32 + lane], mask);
  } else {
#pragma unroll
    for (int r = 0; r < kIPT; ++r) packed[r] = record_digit<FIRST, true>(a, wbase + (long long)r * 32 + lane, N, mask);
  }

  // digit starts (from the column totals) plus this tile's column prefixes
  if (tid == 0) n_digits = 0u;
  digit_starts(a.totals, ndig, gbase, wsum);
  if (tile == 0 && a.seg_out)   // digit = destination: the digit starts are the segment starts
    for (long long b = tid; b <= a.m; b += blockDim.x) a.seg_out[b] = (int32_t)gbase[b];
  for (int d = tid; d < ndig; d += blockDim.x) gbase[d] += a.counts[tile * ndig + d];
  for (int d = lane; d < ndig; d += 32) {
    wcnt[warp * ndig + d] = 0;
    pmask[warp * ndig + d] = 0u;
  }
  __syncwarp();

  // ---- rank inside the warp
  // The lanes of a round that share a digit ("peers") are found without a
  // warp vote per digit bit: lanes with lane 0's digit by one ballot, the
  // others by OR-ing their lane bit into a per-warp mask word of their digit
  // (OR is order-free, so the mask -- and the rank -- are deterministic).
  unsigned* pm = pmask + warp * ndig;
  unsigned short* wc = wcnt + warp * ndig;
#pragma unroll
  for (int r = 0; r < kIPT; ++r) {
    const unsigned d = packed[r];
    const bool valid = d != 0xffffffffu;
    const unsigned d0 = __shfl_sync(0xffffffffu, d, 0);
    const bool in0 = valid && d == d0;
    const unsigned same0 = __ballot_sync(0xffffffffu, in0);
    if (valid && !in0) atomicOr(pm + d, 1u << lane);
    __syncwarp();
    const unsigned peers = in0 ? same0 : (valid ? pm[d] : 0u);
    const unsigned base = valid ? wc[d] : 0u;
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) {
      wc[d] = (unsigned short)(base + __popc(peers));
      if (!in0) pm[d] = 0u;
    }
    __syncwarp();
    packed[r] = valid ? ((d << 16) | (base + __popc(peers & ((1u << lane) - 1u)))) : 0xffffffffu;
  }
  __syncthreads();

  if (!STAGE) {
    // ---- direct scatter (payloads too large to stage): warp prefixes, then
    // each record goes straight to its global position
    for (int d = tid; d < ndig; d += blockDim.x) {
      unsigned run = 0;
      for (int w = 0; w < nwarps; ++w) {
        const unsigned c = wcnt[w * ndig + d];
        wcnt[w * ndig + d] = (unsigned short)run;
        run += c;
      }
    }
    __syncthreads();
    const U* __restrict__ vin = reinterpret_cast<const U*>(a.vals_in);
    U* __restrict__ vout = reinterpret_cast<U*>(a.vals_out);
    const int32_t* __restrict__ iin = a.idx_in;
    int32_t* __restrict__ iout = a.idx_out;
    const int32_t* __restrict__ kin = a.keys_in;
    int32_t* __restrict__ kout = a.keys_out;
    const unsigned short* __restrict__ wc_tile = wcnt + warp * ndig;
    constexpr int B = 4;
#pragma unroll
    for (int r0 = 0; r0 < kIPT; r0 += B) {
      U vv[B];
      int32_t ii[B], kk[B];
#pragma unroll
      for (int e = 0; e < B; ++e) {
        const long long i = wbase + (long long)(r0 + e) * 32 + lane;
        const bool ok = packed[r0 + e] != 0xffffffffu;
        if (VB) vv[e] = ok ? __ldg(vin + i) : U(0);
        if (IDX) ii[e] = ok ? (FIRST ? (int32_t)i : __ldg(iin + i)) : 0;
        if (KEYS_OUT) kk[e] = ok ? (FIRST ? (int32_t)((long long)__ldg(kin + i) + a.key_offset) : __ldg(kin + i)) : 0;
      }
#pragma unroll
      for (int e = 0; e < B; ++e) {
        const unsigned pk = packed[r0 + e];
        if (pk == 0xffffffffu) continue;
        const unsigned d = pk >> 16;
        const long long pos = (long long)gbase[d] + wc_tile[d] + (pk & 0xffffu);
        if (pos < 0 || pos >= a.n) {
          set_status(a.status, DET_ERR_INVALID_ARG);
          continue;
        }
        if (VB) vout[pos] = vv[e];
        if (IDX) iout[pos] = ii[e];
        if (KEYS_OUT) kout[pos] = kk[e];
      }
    }
    return;
  }

  // ---- per digit: exclusive prefix over the warps of this tile, and the
  // tile's digit counts
  unsigned int* lstart = gbase + (ndig + 1);   // [ndig + 1] tile-local digit starts
  {
    unsigned nz = 0;
    for (int d = tid; d < ndig; d += blockDim.x) {
      unsigned run = 0;
      for (int w = 0; w < nwarps; ++w) {
        const unsigned c = wcnt[w * ndig + d];
        wcnt[w * ndig + d] = (unsigned short)run;
        run += c;
      }
      lstart[d] = run;   // count for now; turned into starts below
      nz += run != 0;
    }
    if (nz) atomicAdd(&n_digits, nz);
  }
  __syncthreads();
  {
    // exclusive scan of the tile's digit counts (reuses the digit-start scan)
    unsigned int* tmp = gbase + 2 * (ndig + 1);   // [ndig + 1]
    digit_starts(lstart, ndig, tmp, wsum);
    for (int d = tid; d <= ndig; d += blockDim.x) lstart[d] = tmp[d];
  }
  __syncthreads();
  // tile-local sorted position of each record (digit-major, stable)
#pragma unroll
  for (int r = 0; r < kIPT; ++r) {
    const unsigned pk = packed[r];
    if (pk == 0xffffffffu) continue;
    const unsigned d = pk >> 16;
    packed[r] = (d << 16) | (lstart[d] + wcnt[warp * ndig + d] + (pk & 0xffffu));
  }
  if (a.rank_out) {
    // only each record's sorted position is wanted: write it in input order
    // (coalesced) and move nothing
#pragma unroll
    for (int r = 0; r < kIPT; ++r) {
      const unsigned pk = packed[r];
      if (pk == 0xffffffffu) continue;
      const unsigned d = pk >> 16;
      a.rank_out[wbase + (long long)r * 32 + lane] = (int32_t)(gbase[d] - lstart[d] + (pk & 0xffffu));
    }
    return;
  }
  __syncthreads();   // the peer-mask and counter words are free from here on

  // ---- one-pass sorts of full, aligned tiles whose digit runs are long (16
  // records or more on average, so that a warp's stores mostly fall in one
  // run): the tile's values come in by one bulk copy (input order) into the
  // freed front of shared memory, and each thread stores its records' values
  // straight to their global places.  Short runs go through the staging below.
  const size_t front_bytes = pass_front_bytes(nwarps, ndig, a.K, VB, IDX, KEYS_OUT, STAGE);
  if (VB > 0 && !KEYS_OUT && (!IDX || FIRST) && (N - tile_base) >= K && (size_t)K * VB <= front_bytes &&
      lstart[ndig] >= 16u * n_digits &&
      (reinterpret_cast<uintptr_t>(reinterpret_cast<const unsigned char*>(a.vals_in) + tile_base * VB) & 15) == 0) {
    __shared__ __align__(8) unsigned long long vals_bar;
    if (tid == 0) {
      // the front was last written by ordinary stores: order them before the copy engine's writes
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_init(&vals_bar, 1);
      mbar_arrive_expect_tx(&vals_bar, (unsigned)(K * VB));
      bulk_copy_g2s(smem_raw, reinterpret_cast<const unsigned char*>(a.vals_in) + tile_base * VB, (unsigned)(K * VB),
                    &vals_bar);
    }
    // global position of each record: local position + (global - local digit start)
#pragma unroll
    for (int r = 0; r < kIPT; ++r) {
      const unsigned pk = packed[r];
      if (pk == 0xffffffffu) continue;
      const unsigned d = pk >> 16;
      packed[r] = gbase[d] - lstart[d] + (pk & 0xffffu);
    }
    __syncthreads();   // the barrier is initialised before anyone waits on it
    const bool ok = mbar_wait(&vals_bar, 0, kWaitNs);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        set_status(a.status, DET_ERR_COPY_TIMEOUT);
        mbar_wait(&vals_bar, 0, kWaitNs);
      }
      __syncthreads();
      return;
    }
    const U* sv = reinterpret_cast<const U*>(smem_raw) + warp * 32 * kIPT;
    U* __restrict__ vout = reinterpret_cast<U*>(a.vals_out);
#pragma unroll
    for (int r = 0; r < kIPT; ++r) {
      const unsigned pos = packed[r];
      if (pos == 0xffffffffu) continue;
      if ((long long)pos >= a.n) {   // cannot happen for a correct ranking; never write out of bounds
        set_status(a.status, DET_ERR_INVALID_ARG);
        continue;
      }
      vout[pos] = sv[r * 32 + lane];
      if (IDX) a.idx_out[pos] = (int32_t)(wbase + (long long)r * 32 + lane);
    }
    return;
  }

  // ---- stage the records in shared memory in tile-sorted order, then write
  // each digit's run to its global place with consecutive threads on
  // consecutive positions (coalesced runs instead of one sector per record)
  const long long nvalid_tile = lstart[ndig];
  unsigned char* stage = smem_raw;   // overlaps pmask / wcnt
  U* s_val = reinterpret_cast<U*>(stage);
  int32_t* s_idx = reinterpret_cast<int32_t*>(stage + (size_t)VB * a.K);
  int32_t* s_key = reinterpret_cast<int32_t*>(stage + (size_t)(VB + (IDX ? 4 : 0)) * a.K);
  unsigned short* s_dig =
      reinterpret_cast<unsigned short*>(stage + (size_t)(VB + (IDX ? 4 : 0) + (KEYS_OUT ? 4 : 0)) * a.K);
  const U* __restrict__ vin = reinterpret_cast<const U*>(a.vals_in);
  U* __restrict__ vout = reinterpret_cast<U*>(a.vals_out);
  const int32_t* __restrict__ iin = a.idx_in;
  int32_t* __restrict__ iout = a.idx_out;
  const int32_t* __restrict__ kin = a.keys_in;
  int32_t* __restrict__ kout = a.keys_out;
  // payloads go from global memory (L2, prefetched above) straight to their
  // sorted slot by asynchronous copies: no registers, one round trip
#pragma unroll
  for (int r = 0; r < kIPT; ++r) {
    const unsigned pk = packed[r];
    if (pk == 0xffffffffu) continue;
    const long long i = wbase + (long long)r * 32 + lane;
    const unsigned lp = pk & 0xffffu;
    if (VB) cp_async_small<VB>(s_val + lp, vin + i);
    if (IDX) {
      if (FIRST)
        s_idx[lp] = (int32_t)i;
      else
        cp_async_small<4>(s_idx + lp, iin + i);
    }
    if (KEYS_OUT) cp_async_small<4>(s_key + lp, kin + i);   // raw key; the offset is added on the way out
    s_dig[lp] = (unsigned short)(pk >> 16);
  }
  // global position = local position + (global digit start - local digit start)
  for (int d = tid; d < ndig; d += blockDim.x) gbase[d] -= lstart[d];
  cp_async_commit_wait_all();
  __syncthreads();
#pragma unroll 4
  for (long long i = tid; i < nvalid_tile; i += blockDim.x) {
    const unsigned d = s_dig[i];
    const long long pos = (long long)gbase[d] + i;
    if (pos < 0 || pos >= a.n) {   // cannot happen for a correct ranking; never write out of bounds
      set_status(a.status, DET_ERR_INVALID_ARG);
      continue;
    }
    if (VB) vout[pos] = s_val[i];
    if (IDX) iout[pos] = s_idx[i];
    if (KEYS_OUT) kout[pos] = FIRST ? (int32_t)((long long)s_key[i] + a.key_offset) : s_key[i];
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


// ---------------------------------------------------------------------------
// PT over p[0..len) by one warp: rounds of 256 (8 per lane, in-register tree,
// then five shuffle levels) combined by a binary counter (rounds are aligned
// 256-blocks, i.e. nodes of level 8), collapsed by a right fold at the end.
// COHERENT: read through L2 only (values written by other CTAs of the same launch).
// NEG: the leaves are the negated values (absent padding stays -0.0).
template <typename T, bool COHERENT = false, bool NEG = false>
__device__ T warp_pt_range(const T* __restrict__ p, long long len) {
  const int lane = threadIdx.x & 31;
  NodeCounter<T, 8> nc;
  const long long rounds = (len + 255) / 256;
  if (!COHERENT && rounds > 1) prefetch_l2(p, (size_t)len * sizeof(T), lane, 32);   // later rounds then come from L2
  for (long long r = 0; r < rounds; ++r) {
    T v[8];
    const long long b = r * 256 + lane * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (b + e < len) {
        const T x = COHERENT ? __ldcg(p + b + e) : __ldg(p + b + e);
        v[e] = NEG ? -x : x;
      } else {
        v[e] = absent<T>();
      }
    }
    nc.push(warp_pt(thread_pt(v)));   // node of the aligned 256-block r (level 8)
  }
  return nc.result();
}

struct LongSeg {
  long long bin;
  long long base;
  long long nblk;
};

// NEG: the tree is over the negated values (scatter-sub).  The leaves are
// negated, not the result: an exact zero from cancellation is +0.0 either
// way, so -PT(v) and PT(-v) can differ in the sign of a zero.
template <typename T, bool NEG>
__global__ void __launch_bounds__(256)
segtree_bins_kernel(const T* __restrict__ vals, const int32_t* __restrict__ seg, long long m, T* __restrict__ out,
                    long long* __restrict__ blocks, LongSeg* __restrict__ lsegs, unsigned int* __restrict__ ldone,
                    unsigned int* __restrict__ nblocks, unsigned int* __restrict__ nlsegs,
                    const unsigned int* __restrict__ n_valid, long long max_blocks, long long max_lsegs,
                    unsigned int* __restrict__ status, long long ostride) {
  const long long b = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (b >= m) return;
  const long long N = *n_valid;
  const long long hi = min((long long)seg[b + 1], N), lo = max(0LL, min((long long)seg[b], hi));
  const long long len = hi - lo;
  if (len <= 0) return;
  if (len <= kSegBlock) {
    const T t = warp_pt_range<T, false, NEG>(vals + lo, len);
    if (lane == 0) out[b * ostride] = out[b * ostride] + t;
    return;
  }
  const long long nblk = (len + kSegBlock - 1) / kSegBlock;
  long long base = 0, sidx = 0;
  if (lane == 0) {
    base = atomicAdd(nblocks, (unsigned)nblk);
    sidx = atomicAdd(nlsegs, 1u);
    if (sidx < max_lsegs && base + nblk <= max_blocks) {
      lsegs[sidx] = LongSeg{b, base, nblk};
      ldone[sidx] = 0u;
    } else {
      set_status(status, DET_ERR_INVALID_ARG);
    }
  }
  base = __shfl_sync(0xffffffffu, base, 0);
  sidx = __shfl_sync(0xffffffffu, sidx, 0);
  if (sidx >= max_lsegs || base + nblk > max_blocks) return;
  for (long long k = lane; k < nblk; k += 32) blocks[base + k] = (sidx << 24) | k;
}

// One CTA of 256 threads per rank-aligned 2048-record block of a long bin.
// All leaves are read in one coalesced round into shared memory; thread t
// then takes leaves [8t, 8t+8) (a level-3 node), the warp's butterfly gives
// the level-8 node and the tree over the 8 warps the level-11 node -- the
// same node as any other aligned decomposition of the block.  The CTA that
// completes a bin's last block (a per-bin counter) forms the PT over the
// bin's block nodes and adds it to out[bin]: who does it varies, the tree
// does not.
template <typename T, bool NEG>
__global__ void __launch_bounds__(256)
segtree_blocks_kernel(const T* __restrict__ vals, const int32_t* __restrict__ seg, const long long* __restrict__ blocks,
                      const unsigned int* __restrict__ nblocks, const LongSeg* __restrict__ lsegs,
                      unsigned int* __restrict__ ldone, T* nodes, T* __restrict__ out,
                      const unsigned int* __restrict__ n_valid, long long max_blocks, long long max_lsegs,
                      long long ostride) {
  static_assert(kSegBlock == 256 * 8, "one CTA of 256 threads x 8 leaves per block");
  __shared__ __align__(16) T buf[kSegBlock];
  __shared__ T wnode[8];
  __shared__ int last;
  const long long q = blockIdx.x;
  if (q >= (long long)*nblocks || q >= max_blocks) return;
  const int tid = threadIdx.x;
  const long long e = blocks[q];
  const long long sidx = e >> 24, k = e & ((1 << 24) - 1);
  if (sidx >= max_lsegs) return;
  const LongSeg L = lsegs[sidx];
  const long long N = *n_valid;
  const long long hi = min((long long)seg[L.bin + 1], N);
  const long long lo = max(0LL, min((long long)seg[L.bin] + k * kSegBlock, hi));
  const long long len = min((long long)kSegBlock, hi - lo);
#pragma unroll
  for (int i = 0; i < kSegBlock / 256; ++i) {
    const int j = i * 256 + tid;
    buf[j] = j < len ? (NEG ? -__ldg(vals + lo + j) : __ldg(vals + lo + j)) : absent<T>();
  }
  __syncthreads();
  constexpr int NQ = 8 * (int)sizeof(T) / 16;
  float4 q4[NQ];
#pragma unroll
  for (int i = 0; i < NQ; ++i) q4[i] = reinterpret_cast<const float4*>(buf + tid * 8)[i];
  T v[8];
  memcpy(v, q4, sizeof(v));
  const T node = warp_pt(thread_pt(v));
  if ((tid & 31) == 0) wnode[tid >> 5] = node;
  __syncthreads();
  if (tid == 0) {
    const T a01 = wnode[0] + wnode[1], a23 = wnode[2] + wnode[3];
    const T a45 = wnode[4] + wnode[5], a67 = wnode[6] + wnode[7];
    nodes[q] = (a01 + a23) + (a45 + a67);
    __threadfence();
    last = atomicAdd(&ldone[sidx], 1u) == (unsigned)(L.nblk - 1);
  }
  __syncthreads();
  if (last && tid < 32) {
    __threadfence();
    const T t = warp_pt_range<T, true>(nodes + L.base, L.nblk);   // nodes already hold the negated leaves
    if (tid == 0) out[L.bin * ostride] = out[L.bin * ostride] + t;
  }
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
  // The sort's tile is threads x kIPT records.  block_threads = 128 gives
  // 4,096-record tiles; every other choice the 8,192-record tiles of 256
  // threads (the ranking's per-warp digit arrays make larger CTAs pointless),
  // except that by default sorts of at most 2^22 records take the smaller
  // tiles, so that they still spread over every SM.  Tiling never changes
  // the bits: the sort is stable.
  p.threads = (block_threads == 128 || (block_threads == 0 && n <= (1LL << 22))) ? 128 : 256;
  p.ipt = kIPT;
  const long long K = (long long)p.threads * kIPT;
  p.tiles = (n + K - 1) / K;
  const long long ndig = 1LL << p.digit_bits;
  size_t off = kHeaderBytes;
  p.totals = off;
  off = align_up(off + 1025 * 4, 256);
  p.counts = off;
  off = align_up(off + (size_t)(p.tiles + 1) * ndig * 4, 256);
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
  // blocks of long bins: ceil(len / 2048) <= len / 2048 + 1 each, and at most
  // min(m, n / 2048) bins are long (each holds more than 2048 records)
  p.max_blocks = n / kSegBlock + std::min(m, n / kSegBlock) + 2;
  p.max_lsegs = n / kSegBlock + 2;
  p.blocks = off;
  off = align_up(off + (size_t)p.max_blocks * 8, 256);
  p.lsegs = off;
  off = align_up(off + (size_t)p.max_lsegs * sizeof(LongSeg), 256);
  p.ldone = off;
  off = align_up(off + (size_t)p.max_lsegs * 4, 256);
  p.nodes = off;
  off = align_up(off + (size_t)p.max_blocks * 8, 256);
  p.total = off;
  return p;
}

template <int VB>
static cudaError_t launch_pass(const PassArgs& a, bool first, bool idx, bool keys_out, int threads, long long tiles,
                               cudaStream_t s) {
  const int ndig = 1 << a.D;
  const int max_smem = device_max_smem_optin();
  const size_t tail = (size_t)3 * (ndig + 1) * 4;
  const bool stage = pass_front_bytes(threads / 32, ndig, a.K, VB, idx, keys_out, true) + tail <= (size_t)max_smem;
  const size_t smem = pass_front_bytes(threads / 32, ndig, a.K, VB, idx, keys_out, stage) + tail;
  void (*k)(PassArgs) = nullptr;
#define DET_PICK(F, I, KO)                                                            \
  if (first == F && idx == I && keys_out == KO)                                       \
    k = stage ? sort_pass_kernel<VB, F, I, KO, true> : sort_pass_kernel<VB, F, I, KO, false>;
  DET_PICK(true, true, true) DET_PICK(true, true, false) DET_PICK(true, false, true) DET_PICK(true, false, false)
  DET_PICK(false, true, true) DET_PICK(false, true, false) DET_PICK(false, false, true) DET_PICK(false, false, false)
#undef DET_PICK
  cudaError_t e = ensure_dyn_smem((const void*)k, smem);
  if (e != cudaSuccess) return e;
  launch_begin("det_sort_pass", s);
  k<<<(unsigned)tiles, threads, smem, s>>>(a);
  launch_end(s);
  return cudaGetLastError();
}

int enqueue_sort(const SortPlan& p, void* ws, const int32_t* keys, long long key_offset, const void* values,
                 int32_t* perm_out, cudaStream_t s, int* final_buf, int32_t* rank_out) {
  char* w = reinterpret_cast<char*>(ws);
  SortHdr* h = reinterpret_cast<SortHdr*>(ws);
  if (cudaMemsetAsync(w, 0, kHeaderBytes, s) != cudaSuccess) return DET_ERR_CUDA;
  *final_buf = (p.passes - 1) & 1;
  int32_t* seg = reinterpret_cast<int32_t*>(w + p.seg);
  if (p.n == 0 || p.m == 0) {
    if (cudaMemsetAsync(seg, 0, (size_t)(p.m + 1) * 4, s) != cudaSuccess) return DET_ERR_CUDA;
    return DET_OK;
  }
  const int ndig = 1 << p.digit_bits;
  unsigned int* totals = reinterpret_cast<unsigned int*>(w + p.totals);
  unsigned int* counts = reinterpret_cast<unsigned int*>(w + p.counts);
  for (int pass = 0; pass < p.passes; ++pass) {
    const bool first = pass == 0, last = pass == p.passes - 1;
    const int out = pass & 1, in = (pass - 1) & 1;
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
    a.tiles = p.tiles;
    a.K = (long long)p.threads * kIPT;
    a.counts = counts;
    a.totals = totals;
    a.status = &h->status;
    a.n_valid = &h->n_valid;
    a.seg_out = p.passes == 1 ? seg : nullptr;
    a.rank_out = p.passes == 1 ? rank_out : nullptr;
    const size_t csmem = (size_t)ndig * 4;
    const long long K = (long long)p.threads * kIPT;
    launch_begin("det_sort_count", s);
    if (first)
      sort_count_kernel<true><<<(unsigned)p.tiles, 256, csmem, s>>>(a, K);
    else
      sort_count_kernel<false><<<(unsigned)p.tiles, 256, csmem, s>>>(a, K);
    launch_end(s);
    launch_begin("det_sort_colscan", s);
    sort_colscan_kernel<<<(unsigned)((ndig + kColDigits - 1) / kColDigits), 1024, 0, s>>>(a, first ? 1 : 0);
    launch_end(s);
    const int rc = check_launch("sort: digit counts");
    if (rc != DET_OK) return rc;
    const bool keys_out = p.passes > 1;
    cudaError_t e;
    if (p.value_bytes == 8)
      e = launch_pass<8>(a, first, p.need_idx, keys_out, p.threads, p.tiles, s);
    else if (p.value_bytes == 4)
      e = launch_pass<4>(a, first, p.need_idx, keys_out, p.threads, p.tiles, s);
    else
      e = launch_pass<0>(a, first, p.need_idx, keys_out, p.threads, p.tiles, s);
    if (e != cudaSuccess) return cuda_fail(e, "sort: pass");
  }
  if (p.passes > 1) {   // one-pass sorts got their segment starts from the pass
    launch_begin("det_sort_bounds", s);
    sort_bounds_kernel<<<(unsigned)((p.n + 1 + 255) / 256), 256, 0, s>>>(
        reinterpret_cast<const int32_t*>(w + p.keys[*final_buf]), &h->n_valid, p.m, seg, p.n);
    launch_end(s);
  }
  return check_launch("sort: segment starts");
}

template <typename T>
int enqueue_segmented_tree(const SortPlan& p, void* ws, const T* sorted_vals, T* out, cudaStream_t s, bool negate,
                           long long ostride, bool reset_counters) {
  if (p.n == 0 || p.m == 0) return DET_OK;
  char* w = reinterpret_cast<char*>(ws);
  SortHdr* h = reinterpret_cast<SortHdr*>(ws);
  const int32_t* seg = reinterpret_cast<const int32_t*>(w + p.seg);
  long long* blocks = reinterpret_cast<long long*>(w + p.blocks);
  LongSeg* lsegs = reinterpret_cast<LongSeg*>(w + p.lsegs);
  T* nodes = reinterpret_cast<T*>(w + p.nodes);
  unsigned int* ldone = reinterpret_cast<unsigned int*>(w + p.ldone);
  if (reset_counters && cudaMemsetAsync(&h->long_blocks, 0, 2 * sizeof(unsigned int), s) != cudaSuccess)
    return DET_ERR_CUDA;
  launch_begin("det_segtree_bins", s);
  auto* kb = negate ? segtree_bins_kernel<T, true> : segtree_bins_kernel<T, false>;
  kb<<<(unsigned)((p.m * 32 + 255) / 256), 256, 0, s>>>(sorted_vals, seg, p.m, out, blocks, lsegs, ldone,
                                                         &h->long_blocks, &h->long_segs, &h->n_valid, p.max_blocks,
                                                         p.max_lsegs, &h->status, ostride);
  launch_end(s);
  const int rc = check_launch("segmented tree: bins");
  if (rc != DET_OK) return rc;
  launch_begin("det_segtree_blocks", s);
  auto* kk = negate ? segtree_blocks_kernel<T, true> : segtree_blocks_kernel<T, false>;
  kk<<<(unsigned)p.max_blocks, 256, 0, s>>>(sorted_vals, seg, blocks, &h->long_blocks, lsegs, ldone, nodes, out,
                                            &h->n_valid, p.max_blocks, p.max_lsegs, ostride);
  launch_end(s);
  return check_launch("segmented tree: blocks");
}

template int enqueue_segmented_tree<float>(const SortPlan&, void*, const float*, float*, cudaStream_t, bool, long long,
                                           bool);
template int enqueue_segmented_tree<double>(const SortPlan&, void*, const double*, double*, cudaStream_t, bool,
                                            long long, bool);

}  // namespace det
