// Stable LSD radix sort of (key, value, index) records with a validity
// filter, and the segmented pairwise tree over the sorted values.
//
//   count p   per tile of K = threads * 16 records: digit counts of the
//             valid records (shared integer atomics: order-free)
//   colscan p per digit: exclusive prefix of the counts over tiles, and the
//             digit totals (pass 0 also sums them into the valid count)
//   pass p    per tile, independently: a stable sort of the tile's records
//             by digit in shared memory (one or two counting sub-passes of
//             32 buckets), then record p of that order goes to
//             digit start + tile prefix + (p - tile-local digit start).
//             Records keep their input order inside a digit: the pass is
//             stable, so after the last pass each destination's records are
//             in ascending original index.
//   bounds    (more than one pass) segment starts from the sorted keys
//   tree      out[b] = out[b] + PT(group b): groups of at most 1024 records
//             by one thread; longer groups are cut into rank-aligned
//             4096-blocks (subtrees of the group's tree), reduced by one CTA
//             each, then a tree over the block nodes.
#include "det_sort.cuh"

namespace det {
namespace {

constexpr int kIPT = 16;                 // records per thread of a pass
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
  int width;                   // wide records: components per record (input row-major, output one
  long long comp_stride;       // array per component, comp_stride elements apart)
};

// counts[tile][d] = records of the tile with digit d.  The tile is the
// scatter pass's tile (K = pass_threads * kIPT records).  A full, aligned
// tile's keys come in by one bulk copy into shared memory (32 KB in flight
// per CTA); counting is order-free, so each thread then adds its keys by
// shared atomics (dropped keys into a spare slot).  A group of four keys
// that is one digit across the whole warp is added by lane 0 alone: a hot
// digit would otherwise serialise the warp's atomics on one address.
// OFFSET (first pass only): keys are shifted by key_offset before the range
// test.  The first pass takes the lowest digit, so it never shifts.
template <bool FIRST, bool OFFSET>
__global__ void __launch_bounds__(256) sort_count_kernel(PassArgs a, long long K) {
  dep_wait();   // launched early (programmatic dependent launch): wait for the previous kernel
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ __align__(8) unsigned long long keys_bar;
  const int ndig = 1 << a.D;
  unsigned int* cnt = reinterpret_cast<unsigned int*>(smem_raw);   // [ndig + 1]; ndig = dropped
  int32_t* skeys = reinterpret_cast<int32_t*>(smem_raw + align_up((size_t)(ndig + 1) * 4, 16));   // [K]
  const int tid = threadIdx.x, lane = tid & 31;
  const unsigned mask = (unsigned)ndig - 1u;
  const long long tile = blockIdx.x;
  const long long N = FIRST ? a.n : (long long)*a.n_valid;
  const long long t0 = tile * K, t1 = min(N, t0 + K);
  const bool bulk = t1 - t0 == K && (reinterpret_cast<uintptr_t>(a.keys_in + t0) & 15) == 0;
  if (bulk && tid == 0) {
    mbar_init(&keys_bar, 1);
    mbar_arrive_expect_tx(&keys_bar, (unsigned)(K * 4));
    bulk_copy_g2s(skeys, a.keys_in + t0, (unsigned)(K * 4), &keys_bar);
  }
  for (int d = tid; d <= ndig; d += blockDim.x) cnt[d] = 0u;
  __syncthreads();
  const unsigned m32 = (unsigned)min(a.m, (long long)0x80000000LL);   // keys are int32
  const int shift = a.shift;
  auto digit = [&](int k) -> unsigned {
    if (FIRST && !OFFSET) return (unsigned)k < m32 ? (unsigned)k & mask : (unsigned)ndig;
    if (FIRST) {
      const long long kk = (long long)k + a.key_offset;
      return (kk >= 0 && kk < a.m) ? (unsigned)kk & mask : (unsigned)ndig;
    }
    return ((unsigned)k >> shift) & mask;
  };
  if (bulk) {
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
    const int4* k4 = reinterpret_cast<const int4*>(skeys);
#pragma unroll 4
    for (int g = tid; g < (int)(K / 4); g += blockDim.x) {
      const int4 q = k4[g];
      const unsigned d0 = digit(q.x), d1 = digit(q.y), d2 = digit(q.z), d3 = digit(q.w);
      const unsigned w0 = __shfl_sync(0xffffffffu, d0, 0);
      if (__all_sync(0xffffffffu, d0 == w0 && d1 == w0 && d2 == w0 && d3 == w0)) {
        if (lane == 0) atomicAdd(&cnt[w0], 128u);
      } else {
        atomicAdd(&cnt[d0], 1u);
        atomicAdd(&cnt[d1], 1u);
        atomicAdd(&cnt[d2], 1u);
        atomicAdd(&cnt[d3], 1u);
      }
    }
  } else {
    for (long long j = t0 + tid; j < t1; j += blockDim.x) atomicAdd(&cnt[digit(__ldg(a.keys_in + j))], 1u);
  }
  __syncthreads();
  for (int d = tid; d < ndig; d += blockDim.x) a.counts[tile * ndig + d] = cnt[d];
}

// For each digit column: exclusive prefix over tiles (in place) and the
// column total.  CTA of 1024 threads = 8 digit lanes x 128 tile groups (a
// warp reads 8 consecutive digits of 4 tiles: whole 32-byte sectors).
constexpr int kColDigits = 8, kColGroups = 128;
__global__ void __launch_bounds__(1024) sort_colscan_kernel(PassArgs a, int count_valid) {
  dep_wait();   // launched early (programmatic dependent launch): wait for the previous kernel
  __shared__ unsigned int part[kColGroups][kColDigits + 1];
  const int dl = threadIdx.x % kColDigits, g = threadIdx.x / kColDigits;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ndig = 1 << a.D;
  const int d = blockIdx.x * kColDigits + dl;
  const long long T = a.tiles;
  const long long TG = (T + kColGroups - 1) / kColGroups;
  const long long t0 = g * TG, t1 = min(T, t0 + TG);
  // a group of at most kR tiles is read once, all loads in flight, and kept
  // in registers for the rewrite; longer groups are read eight at a time,
  // twice
  constexpr int kR = 16, kU = 8;
  const bool regs = TG <= kR;
  unsigned r[kR];
  unsigned sum = 0;
  if (d < ndig && regs) {
#pragma unroll
    for (int k = 0; k < kR; ++k) r[k] = t0 + k < t1 ? a.counts[(t0 + k) * ndig + d] : 0u;
#pragma unroll
    for (int k = 0; k < kR; ++k) sum += r[k];
  } else if (d < ndig)
    for (long long t = t0; t < t1; t += kU) {
      unsigned v[kU];
#pragma unroll
      for (int k = 0; k < kU; ++k) v[k] = t + k < t1 ? a.counts[(t + k) * ndig + d] : 0u;
#pragma unroll
      for (int k = 0; k < kU; ++k) sum += v[k];
    }
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
      a.counts[T * ndig + dc] = total;   // row `tiles`: the pass takes a tile's counts as E[t + 1] - E[t]
      if (count_valid && total) atomicAdd(a.n_valid, total);
    }
  }
  __syncthreads();
  unsigned run = part[g][dl];
  if (d < ndig && regs) {
#pragma unroll
    for (int k = 0; k < kR; ++k) {
      if (t0 + k < t1) a.counts[(t0 + k) * ndig + d] = run;
      run += r[k];
    }
  } else if (d < ndig)
    for (long long t = t0; t < t1; t += kU) {
      unsigned v[kU];
#pragma unroll
      for (int k = 0; k < kU; ++k) v[k] = t + k < t1 ? a.counts[(t + k) * ndig + d] : 0u;
#pragma unroll
      for (int k = 0; k < kU; ++k) {
        if (t + k < t1) a.counts[(t + k) * ndig + d] = run;
        run += v[k];
      }
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

// ---------------------------------------------------------------------------
// The scatter pass.  Inside a tile the records are ranked by a stable sort in
// shared memory; record p of the tile's sorted order then goes to
//   digit start + earlier tiles' records of its digit + (p - the tile-local
//   start of its digit)
// and consecutive p of one digit land on consecutive positions.
//
// The tile's valid records are sorted by digit with one or two stable
// counting sub-passes of 32 buckets (the low 5 bits, then the rest; one
// sub-pass for digits of at most 5 bits).  In a sub-pass thread t holds the
// 16 consecutive records [16t, 16t + 16) of the current order:
//   walk 1  count its records per bucket in its own counter column
//   scan    exclusive scan of all counters, bucket-major, thread-minor
//   walk 2  rank = its scanned counter, post-incremented, in record order
// so equal buckets keep thread order and, inside a thread, record order: the
// sub-pass is stable, and so is the sort.  Dropped records (past the end,
// or a destination outside [0, m)) carry a flag; the last sub-pass neither
// counts nor places them, so the valid records take ranks [0, valid count).
// Counters are the 16-bit halves of 32-bit words: word (row r, thread t) at
// r * T + t (swizzled like the records) counts bucket r (low half) and
// bucket r + 16 (high half), so a warp's counter accesses never share a
// bank.
// Records live in shared memory as 32-bit words (flag << 31 | digit << 13 |
// tile-local index) under an XOR swizzle of the 16-byte chunks in each
// 128-byte line, so that the per-thread row reads are conflict-free.
constexpr int kIdxBits = 13;          // tile-local record index (tiles of at most 8,192 records)
constexpr unsigned kDropped = 1u << 31;

template <int VB> struct Payload;
template <> struct Payload<0> { using U = unsigned int; };
template <> struct Payload<4> { using U = unsigned int; };
template <> struct Payload<8> { using U = unsigned long long; };

// Physical word of logical record position p.  With kSwizzle the 16-byte
// chunks of each 128-byte line are XOR-permuted by the line index (an
// involution), which makes the per-thread row reads conflict-free; without
// it those reads take four wavefronts per phase (measured slower overall).
constexpr bool kSwizzle = true;
__device__ __forceinline__ unsigned swz(unsigned p) { return kSwizzle ? p ^ (((p >> 5) & 7u) << 2) : p; }

// Shared-memory layout of a pass (bytes; every part 16-byte aligned).
struct PassSmem {
  size_t recs, rkeys, vals, idx, cnt, off, total;
};
__host__ __device__ inline PassSmem pass_smem(int T, int ndig, int vb, bool idx_in, bool keys_out) {
  const size_t K = (size_t)T * kIPT;
  PassSmem s;
  size_t o = 0;
  s.recs = o;
  o += K * 4;
  s.rkeys = o;   // raw keys, kept apart from the records only when they are written out
  o += keys_out ? K * 4 : 0;
  s.vals = o;
  o += K * (size_t)vb;
  s.idx = o;
  o += idx_in ? K * 4 : 0;
  s.cnt = o;
  o += (size_t)17 * T * 4;   // 16 counter rows and a spare row for dropped records
  s.off = o;
  o += align_up((size_t)(ndig + 1) * 4, 16);
  s.total = o;
  return s;
}

// Exclusive scan of one value per thread over the CTA in thread order;
// *total receives the sum.  wsum: 32 words of shared memory.  Ends with a
// barrier, so wsum can be reused at once.
__device__ __forceinline__ unsigned block_excl_scan(unsigned v, unsigned* wsum, unsigned* total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  unsigned x = v;
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
  const unsigned pre = (warp ? wsum[warp - 1] : 0u) + x - v;
  *total = wsum[nw - 1];
  __syncthreads();
  return pre;
}

// This thread's row of records: logical positions [16t, 16t + 16).
__device__ __forceinline__ void load_row(unsigned (&rec)[kIPT], const unsigned* recs) {
  const int tid = threadIdx.x;
  const uint4* q4 = reinterpret_cast<const uint4*>(recs);
  const unsigned g0 = 4u * tid, x = kSwizzle ? (g0 >> 3) & 7u : 0u;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 q = q4[(g0 + c) ^ x];
    rec[4 * c] = q.x;
    rec[4 * c + 1] = q.y;
    rec[4 * c + 2] = q.z;
    rec[4 * c + 3] = q.w;
  }
}

// One stable counting sub-pass by bucket (rec >> S) & 31.  LAST: dropped
// records are left out -- counted in a spare row 16 that the scan skips,
// and "placed" on that row's word, so every record takes the same
// branch-free steps.  The ranked records are written to `recs` in the new
// order; unless LAST, rec[] then holds this thread's row of it.
template <int S, bool LAST>
__device__ __forceinline__ void rank_subpass(unsigned (&rec)[kIPT], unsigned* __restrict__ recs,
                                             unsigned* __restrict__ cnt, unsigned* wsum) {
  const int T = blockDim.x, tid = threadIdx.x;
  // counter words take the records' swizzle: with T a multiple of 256,
  // swz(r * T + t) = r * T + swz(t), so a thread's column stays one
  // per-thread offset, and the scan's 16-word runs become conflict-free
  unsigned* col = cnt + swz(tid);
  unsigned* spare = col + 16 * T;
#pragma unroll
  for (int r = 0; r < 16; ++r) col[r * T] = 0u;
#pragma unroll
  for (int j = 0; j < kIPT; ++j) {
    const unsigned b = (rec[j] >> S) & 31u;
    unsigned* w = col + (b & 15u) * T;
    if (LAST) w = (rec[j] & kDropped) ? spare : w;
    *w += 1u << (b & 16u);
  }
  __syncthreads();
  // scan: thread t takes the words [16t, 16t + 16) of the row-major counter
  // matrix; the low halves (buckets < 16) all come before the high halves
  uint4* run = reinterpret_cast<uint4*>(cnt);
  const unsigned g0 = 4u * tid, gx = kSwizzle ? (g0 >> 3) & 7u : 0u;
  uint4 v[4];
  unsigned sum = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    v[c] = run[(g0 + c) ^ gx];
    sum += v[c].x + v[c].y + v[c].z + v[c].w;
  }
  unsigned tot;
  unsigned pre = block_excl_scan(sum, wsum, &tot);
  pre += (tot & 0xffffu) << 16;   // halves never carry: every count is at most 8,192
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 o;
    o.x = pre;
    pre += v[c].x;
    o.y = pre;
    pre += v[c].y;
    o.z = pre;
    pre += v[c].z;
    o.w = pre;
    pre += v[c].w;
    run[(g0 + c) ^ gx] = o;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kIPT; ++j) {
    const unsigned b = (rec[j] >> S) & 31u;
    const bool drop = LAST && (rec[j] & kDropped);
    unsigned* w = drop ? spare : col + (b & 15u) * T;
    const unsigned x = *w;
    *w = x + (1u << (b & 16u));
    unsigned* dst = recs + swz((x >> (b & 16u)) & 0xffffu);
    *(drop ? spare : dst) = rec[j];
  }
  __syncthreads();
  if (!LAST) load_row(rec, recs);
}

// WIDE (one-pass sorts only): each record carries `width` components of VB
// bytes, read as a row-major record array; the write-out puts component c of
// sorted record p at vals_out[c * comp_stride + position], so each
// component's groups come out contiguous for the segmented tree.
template <int VB, bool FIRST, bool IDX, bool KEYS_OUT, bool WIDE = false>
__global__ void __launch_bounds__(512, 2) sort_pass_kernel(PassArgs a) {
  dep_wait();   // launched early (programmatic dependent launch): wait for the previous kernel
  using U = typename Payload<VB>::U;
  constexpr bool IDX_IN = IDX && !FIRST;                // input indices carried from the previous pass
  constexpr bool RANK = VB == 0 && !IDX && !KEYS_OUT;   // only each record's sorted position is wanted
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ unsigned int wsum[32];
  __shared__ __align__(8) unsigned long long pay_bar;
  const int T = blockDim.x, tid = threadIdx.x;
  const int ndig = 1 << a.D;
  const unsigned mask = (unsigned)ndig - 1u;
  const int W = WIDE ? a.width : 1;   // components per record
  const PassSmem L = pass_smem(T, ndig, VB * W, IDX_IN, KEYS_OUT);
  unsigned* recs = reinterpret_cast<unsigned*>(smem_raw + L.recs);
  unsigned* rkeys = KEYS_OUT ? reinterpret_cast<unsigned*>(smem_raw + L.rkeys) : recs;
  U* sval = reinterpret_cast<U*>(smem_raw + L.vals);
  int32_t* sidx = reinterpret_cast<int32_t*>(smem_raw + L.idx);
  unsigned* cnt = reinterpret_cast<unsigned*>(smem_raw + L.cnt);
  unsigned* off = reinterpret_cast<unsigned*>(smem_raw + L.off);

  const long long tile = blockIdx.x;
  const long long N = FIRST ? a.n : (long long)*a.n_valid;
  const long long K = (long long)T * kIPT;
  const long long tile_base = tile * K;
  if (tile_base >= N) return;
  const int cn = (int)min(K, N - tile_base);   // records of this tile

  // ---- payloads (values, carried indices): one bulk copy each for a full,
  // aligned tile, landing while the keys are ranked; plain loads otherwise
  constexpr bool PAYLOAD = VB > 0 || IDX_IN;
  const unsigned char* vsrc = reinterpret_cast<const unsigned char*>(a.vals_in) + tile_base * VB * W;
  const int32_t* isrc = IDX_IN ? a.idx_in + tile_base : nullptr;
  const bool bulk = PAYLOAD && cn == K && (VB == 0 || (reinterpret_cast<uintptr_t>(vsrc) & 15) == 0) &&
                    (!IDX_IN || (reinterpret_cast<uintptr_t>(isrc) & 15) == 0);
  if (bulk && tid == 0) {
    mbar_init(&pay_bar, 1);
    mbar_arrive_expect_tx(&pay_bar, (unsigned)(K * VB * W + (IDX_IN ? K * 4 : 0)));
    // read for the last time: leave L2 to the sorted output, which the trees read next
    const unsigned long long pol = l2_evict_first();
    if (VB) bulk_copy_g2s_hint(sval, vsrc, (unsigned)(K * VB * W), &pay_bar, pol);
    if (IDX_IN) bulk_copy_g2s_hint(sidx, isrc, (unsigned)(K * 4), &pay_bar, pol);
  }
  if (PAYLOAD && !bulk) {
    for (int p = tid; p < cn * W; p += T)
      if (VB) sval[p] = __ldg(reinterpret_cast<const U*>(vsrc) + p);
    if (IDX_IN)
      for (int p = tid; p < cn; p += T) sidx[p] = __ldg(isrc + p);
  }

  // ---- raw keys into the swizzled record array: 16-byte asynchronous
  // copies for a full, aligned tile (32 KB in flight per CTA), completed
  // after the digit offsets below
  const int32_t* ksrc = a.keys_in + tile_base;
  const bool kasync = cn == K && (reinterpret_cast<uintptr_t>(ksrc) & 15) == 0;
  if (kasync) {
    const unsigned long long kpol = l2_evict_first();   // the keys' last read
    for (int g = tid; g < (int)(K / 4); g += T)
      asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(rkeys + swz(4u * g))),
                   "l"(ksrc + 4 * g), "l"(kpol)
                   : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
  } else {
    for (int p = tid; p < (int)K; p += T) rkeys[swz(p)] = p < cn ? (unsigned)__ldg(ksrc + p) : 0u;
  }

  // ---- per digit d: global position of the tile's first record of d, less
  // d's tile-local start.  With E the column prefixes (row `tiles` holds the
  // totals) and c = E[tile + 1] - E[tile] the tile's own counts:
  //   off[d] = (sum_{d' < d} total[d'] + E[tile][d]) - sum_{d' < d} c[d']
  if (tile == 0 && a.seg_out) {   // digit = destination: the digit starts are the segment starts
    digit_starts(a.totals, ndig, off, wsum);
    for (long long b = tid; b <= a.m; b += T) a.seg_out[b] = (int32_t)off[b];
    __syncthreads();
  }
  unsigned nvalid_tile;
  {
    constexpr int kMaxPer = 1024 / 256;   // digits per thread at most
    const int per = (ndig + T - 1) / T;
    const unsigned* e0 = a.counts + tile * ndig;
    const unsigned* e1 = e0 + ndig;
    unsigned x[kMaxPer], b0[kMaxPer], loc = 0;
#pragma unroll
    for (int k = 0; k < kMaxPer; ++k) {
      const int d = tid * per + k;
      x[k] = 0u;
      b0[k] = 0u;
      if (k < per && d < ndig) {
        b0[k] = e0[d];
        x[k] = a.totals[d] - (e1[d] - b0[k]);
        loc += x[k];
      }
    }
    unsigned tot;
    unsigned run = block_excl_scan(loc, wsum, &tot);
#pragma unroll
    for (int k = 0; k < kMaxPer; ++k) {
      const int d = tid * per + k;
      if (k < per && d < ndig) off[d] = b0[k] + run;
      run += x[k];
    }
    nvalid_tile = *a.n_valid - tot;   // sum of the tile's counts
    if (nvalid_tile > (unsigned)cn) {   // cannot happen with consistent counts
      if (tid == 0) set_status(a.status, DET_ERR_INVALID_ARG);
      nvalid_tile = 0u;
    }
  }

  if (kasync) asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  // ---- this thread's records: digit and tile-local index, or the dropped flag
  unsigned rec[kIPT];
  load_row(rec, rkeys);
  {
    const unsigned m32 = (unsigned)min(a.m, (long long)0x80000000LL);   // keys are int32
    const bool plain = !FIRST || a.key_offset == 0;
#pragma unroll
    for (int j = 0; j < kIPT; ++j) {
      const unsigned li = (unsigned)(tid * kIPT + j);
      const unsigned k = rec[j];
      bool ok = li < (unsigned)cn;
      unsigned kk = k;
      if (FIRST) {
        if (plain) {
          ok = ok && k < m32;
        } else {
          const long long o = (long long)(int32_t)k + a.key_offset;
          ok = ok && o >= 0 && o < a.m;
          kk = (unsigned)o;
        }
      }
      const unsigned d = (FIRST ? kk : kk >> a.shift) & mask;   // the first pass takes the lowest digit
      rec[j] = ok ? (d << kIdxBits) | li : kDropped | li;
    }
  }

  // ---- stable ranking inside the tile
  if (ndig <= 32) {
    rank_subpass<kIdxBits, true>(rec, recs, cnt, wsum);
  } else {
    rank_subpass<kIdxBits, false>(rec, recs, cnt, wsum);
    rank_subpass<kIdxBits + 5, true>(rec, recs, cnt, wsum);
  }

  if (bulk) {
    const bool ok = mbar_wait(&pay_bar, 0, kWaitNs);
    if (__syncthreads_or(!ok)) {
      // the copy did not complete: record it, give it (bounded) time to land, leave
      if (tid == 0) {
        set_status(a.status, DET_ERR_COPY_TIMEOUT);
        mbar_wait(&pay_bar, 0, kWaitNs);
      }
      __syncthreads();
      return;
    }
  }

  // ---- write out in sorted order: runs of one digit are consecutive
  // positions, so consecutive threads store to consecutive addresses
  U* __restrict__ vout = reinterpret_cast<U*>(a.vals_out);
  const unsigned n32 = (unsigned)a.n;   // sort sizes are below 2^31
  bool bad = false;
  // p = tid + kT with T a multiple of 256: swz(p) = p ^ xw for this thread
  const unsigned xw = kSwizzle ? ((unsigned)(tid >> 5) & 7u) << 2 : 0u;
#pragma unroll 4
  for (unsigned p = tid; p < nvalid_tile; p += T) {
    const unsigned r = recs[p ^ xw];
    const unsigned d = r >> kIdxBits, li = r & ((1u << kIdxBits) - 1u);
    const unsigned pos = off[d & mask] + p;
    // cannot fail for a correct ranking; never write out of bounds
    const bool ok = d < (unsigned)ndig && pos < n32;
    bad |= !ok;
    if (ok) {
      if (RANK) a.rank_out[tile_base + li] = (int32_t)pos;
      if (WIDE) {
        for (int c = 0; c < W; ++c) vout[c * a.comp_stride + pos] = sval[li * W + c];
      } else if (VB) {
        vout[pos] = sval[li];
      }
      if (IDX) a.idx_out[pos] = IDX_IN ? sidx[li] : (int32_t)(tile_base + li);
      if (KEYS_OUT) {
        const int32_t k = (int32_t)rkeys[swz(li)];
        a.keys_out[pos] = FIRST ? (int32_t)((long long)k + a.key_offset) : k;
      }
    }
  }
  if (bad) set_status(a.status, DET_ERR_INVALID_ARG);
}

// seg[b] = first sorted position with key >= b, for b = 0..m (keys sorted).
// Thread t covers positions [P t, P t + P) -- P keys by 16-byte loads, all
// in flight (P = 16 for large sorts, 4 for smaller ones, which need the
// threads) -- and, for the thread that reaches it, position N (the valid
// count), where every remaining bin starts.
template <int kBoundsPer>
__global__ void sort_bounds_kernel(const int32_t* __restrict__ keys, const unsigned int* __restrict__ n_valid,
                                   long long m, int32_t* __restrict__ seg, long long n) {
  dep_wait();   // launched early (programmatic dependent launch): wait for the previous kernel
  // sort sizes, positions and keys are below 2^31: 32-bit arithmetic throughout
  // (64-bit compares and clamps made this kernel bound by its integer pipe)
  // (positions as unsigned: i0 + e stays below 2^32 for every sort size)
  const int m32 = (int)m;
  const long long i0l = (long long)kBoundsPer * ((long long)blockIdx.x * blockDim.x + threadIdx.x);
  const unsigned N = (unsigned)min((long long)*n_valid, n);
  if (i0l > (long long)N) return;
  const unsigned i0 = (unsigned)i0l;
  auto clampk = [&](int32_t k) { return max(-1, min(k, m32)); };
  int32_t kr[kBoundsPer];   // the keys at i0 + e (m from N on)
  const int before = i0 == 0 ? -1 : clampk(__ldg(keys + i0 - 1));
  if (i0 + kBoundsPer <= N && (reinterpret_cast<uintptr_t>(keys + i0) & 15) == 0) {
#pragma unroll
    for (int q = 0; q < kBoundsPer / 4; ++q) {
      const int4 v = __ldg(reinterpret_cast<const int4*>(keys + i0) + q);
      kr[4 * q] = v.x;
      kr[4 * q + 1] = v.y;
      kr[4 * q + 2] = v.z;
      kr[4 * q + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < kBoundsPer; ++e) kr[e] = i0 + e < N ? __ldg(keys + i0 + e) : 0;
  }
  int prev = before;
#pragma unroll
  for (int e = 0; e < kBoundsPer; ++e) {
    if (i0 + e > N) break;
    const int cur = i0 + e < N ? clampk(kr[e]) : m32;
    for (int b = prev + 1; b <= cur; ++b) seg[b] = (int32_t)(i0 + e);
    prev = cur;
  }
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

// One rank-aligned block of a long bin: its leaves are vals[lo, lo + len).
struct BlockDesc {
  long long lo;
  unsigned int len;
  unsigned int sidx;   // the bin's entry in the long-segment list
};

constexpr int kMediumGroup = 1024;   // groups up to this size are reduced by one thread; longer ones by blocks

// Leaves [0, W) of a short group by one thread: the group's len <= W values
// (negated for NEG) padded with absent terms, then the in-register tree --
// PT padded to W, which is PT of the group.
template <typename T, bool NEG, int W>
__device__ __forceinline__ T thread_group_pt(const T* __restrict__ p, int len) {
  T v[W];
#pragma unroll
  for (int e = 0; e < W; ++e) {
    if (e < len) {
      const T x = __ldg(p + e);
      v[e] = NEG ? -x : x;
    } else {
      v[e] = absent<T>();
    }
  }
  return thread_pt(v);
}

// One thread per bin b: out[b] = out[b] + PT(group b).
//   up to kMediumGroup records: the thread's own in-register trees over
//     128-byte chunks of leaves, merged by a counter
//   longer groups: cut into rank-aligned 4096-blocks (subtrees of the
//     group's tree) for the block kernel; the warp writes their list
// NEG: the tree is over the negated values (scatter-sub).  The leaves are
// negated, not the result: an exact zero from cancellation is +0.0 either
// way, so -PT(v) and PT(-v) can differ in the sign of a zero.
template <typename T, bool NEG>
__global__ void __launch_bounds__(256)
segtree_bins_kernel(const T* __restrict__ vals, const int32_t* __restrict__ seg, long long m, T* __restrict__ out,
                    BlockDesc* __restrict__ blocks, LongSeg* __restrict__ lsegs,
                    unsigned int* __restrict__ nblocks, unsigned int* __restrict__ nlsegs,
                    const unsigned int* __restrict__ n_valid, long long max_blocks, long long max_lsegs,
                    unsigned int* __restrict__ status, long long ostride) {
  dep_wait();   // launched early (programmatic dependent launch): wait for the previous kernel
  const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const long long N = *n_valid;
  long long lo = 0, len = 0;
  if (b < m) {
    const long long hi = min((long long)seg[b + 1], N);
    lo = max(0LL, min((long long)seg[b], hi));
    len = hi - lo;
  }
  // groups of at most one 128-byte chunk: PT over the group padded to W, the
  // warp's largest such group rounded up to a power of two (padding beyond
  // the group is absent, so any W >= len gives the same bits; a small W keeps
  // warps of tiny groups from issuing adds on padding alone -- every FP64 add
  // instruction costs the whole warp's width)
  constexpr int CW = 128 / (int)sizeof(T);
  const bool in_chunk = len > 0 && len <= CW;
  const unsigned wmax = __reduce_max_sync(0xffffffffu, in_chunk ? (unsigned)len : 0u);
  if (wmax > 0) {
    T t = absent<T>();
    const T* g = vals + lo;
    const int gl = in_chunk ? (int)len : 0;
    if (wmax <= 1)
      t = thread_group_pt<T, NEG, 1>(g, gl);
    else if (wmax <= 2)
      t = thread_group_pt<T, NEG, 2>(g, gl);
    else if (wmax <= 4)
      t = thread_group_pt<T, NEG, 4>(g, gl);
    else if (wmax <= 8)
      t = thread_group_pt<T, NEG, 8>(g, gl);
    else if (wmax <= 16)
      t = thread_group_pt<T, NEG, 16>(g, gl);
    else
      t = thread_group_pt<T, NEG, CW>(g, gl);
    if (in_chunk) out[b * ostride] = out[b * ostride] + t;
  }
  if (len > CW && len <= kMediumGroup) {
    // rank-aligned chunks of 128 bytes of leaves (level-5 nodes for f32,
    // level-4 for f64; absent terms past the group) merged by a binary
    // counter.  Neighbouring bins have similar sizes in practice, so the
    // lanes of a warp mostly run the same number of chunks.
    NodeCounter<T, 6> nc;
    const T* g = vals + lo;
    const int l32 = (int)len;   // at most kMediumGroup: 32-bit loop arithmetic
    for (int c = 0; c < l32; c += CW) nc.push(thread_group_pt<T, NEG, CW>(g + c, l32 - c));
    out[b * ostride] = out[b * ostride] + nc.result();
  }
  // long groups: their blocks are reserved (the reservation order does not
  // matter: a group's tree reads only its own nodes) and listed
  const bool is_long = len > kMediumGroup;
  const long long nblk = is_long ? (len + kSegBlock - 1) / kSegBlock : 0;
  // one reservation per warp: exclusive prefixes of the block counts and of
  // the long groups over the lanes, lane 31 adding the warp's totals
  long long pre = nblk;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const long long o = __shfl_up_sync(0xffffffffu, pre, d);
    if (lane >= d) pre += o;
  }
  const unsigned longs = __ballot_sync(0xffffffffu, is_long);
  long long wbase = 0, wsidx = 0;
  if (lane == 31 && longs) {
    wbase = atomicAdd(nblocks, (unsigned)pre);
    wsidx = atomicAdd(nlsegs, (unsigned)__popc(longs));
  }
  wbase = __shfl_sync(0xffffffffu, wbase, 31);
  wsidx = __shfl_sync(0xffffffffu, wsidx, 31);
  const long long base = wbase + pre - nblk;
  const long long sidx = wsidx + __popc(longs & ((1u << lane) - 1u));
  bool reg = false;
  if (is_long) {
    reg = sidx < max_lsegs && base + nblk <= max_blocks;
    if (reg) {
      lsegs[sidx] = LongSeg{b, base, nblk};
    } else {
      set_status(status, DET_ERR_INVALID_ARG);
    }
  }
  // a group of at most 32 blocks writes its own list; the warp writes the
  // lists of longer groups together, one group at a time
  if (reg && nblk <= 32)
    for (long long k = 0; k < nblk; ++k)
      blocks[base + k] = BlockDesc{lo + k * kSegBlock, (unsigned)min((long long)kSegBlock, len - k * kSegBlock),
                                   (unsigned)sidx};
  unsigned lng = __ballot_sync(0xffffffffu, reg && nblk > 32);
  while (lng) {
    const int src = __ffs(lng) - 1;
    lng &= lng - 1;
    const long long glo = __shfl_sync(0xffffffffu, lo, src), glen = __shfl_sync(0xffffffffu, len, src);
    const long long gbase = __shfl_sync(0xffffffffu, base, src), gn = __shfl_sync(0xffffffffu, nblk, src);
    const unsigned gs = (unsigned)__shfl_sync(0xffffffffu, sidx, src);
    for (long long k = lane; k < gn; k += 32)
      blocks[gbase + k] =
          BlockDesc{glo + k * kSegBlock, (unsigned)min((long long)kSegBlock, glen - k * kSegBlock), gs};
  }
}

// A CTA of 256 threads per rank-aligned 4096-record block of a long bin, a
// block at a time (persistent CTAs: the largest possible block count is far
// above the real one, which only the device knows).  All leaves are read in one coalesced round (16 loads per thread in
// flight) into shared memory; thread t then reduces leaves [16t, 16t+16) in
// registers (a level-4 node), and warp 0 takes the 256 thread nodes eight
// per lane (level-7 nodes) and finishes with the shuffle levels (the
// level-12 node) -- the same node as any other aligned decomposition of the
// block.  Only the last eight levels run in one warp, so nearly every add
// the SM issues is one of the tree's own (GB300's FP64 rate counts whole
// warp instructions).  A second launch forms the PT over each bin's block
// nodes and adds it to out[bin].
template <typename T, bool NEG>
__global__ void __launch_bounds__(256, sizeof(T) == 8 ? 5 : 6)
segtree_blocks_kernel(const T* __restrict__ vals, const BlockDesc* __restrict__ blocks,
                      const unsigned int* __restrict__ nblocks, T* __restrict__ nodes, long long max_blocks,
                      long long max_lsegs) {
  dep_wait();   // launched early (programmatic dependent launch): wait for the previous kernel
  static_assert(kSegBlock == 256 * 16, "one CTA of 256 threads x 16 leaves");
  __shared__ __align__(16) T buf[kSegBlock];
  __shared__ T tnode[8 * 33];   // thread t's node at (t % 8) * 33 + t / 8: warp 0 reads it conflict-free
  const int tid = threadIdx.x;
  // block counts and record positions are below 2^31 (sort sizes are)
  const unsigned nb = (unsigned)min((long long)*nblocks, max_blocks);
  // persistent: the launch is sized by the SMs, not by the largest possible
  // block count (only known on the device)
  for (unsigned q = blockIdx.x; q < nb; q += gridDim.x) {
  const BlockDesc B = blocks[q];
  if (B.sidx >= max_lsegs) continue;
  const T* __restrict__ leaves = vals + B.lo;
  const int len = (int)min((unsigned)kSegBlock, B.len);
  // leaves sit in shared memory with the 16-byte chunks of each 128-byte
  // line XOR-permuted by the line index, so that the per-thread reads of 16
  // consecutive leaves are conflict-free
  constexpr int EPC = 16 / (int)sizeof(T);   // leaves per 16-byte chunk
  auto pchunk = [](int c) { return c ^ ((c >> 3) & 7); };
#pragma unroll
  for (int i = 0; i < kSegBlock / 256; ++i) {
    const int j = i * 256 + tid;
    buf[pchunk(j / EPC) * EPC + j % EPC] = j < len ? (NEG ? -__ldg(leaves + j) : __ldg(leaves + j)) : absent<T>();
  }
  __syncthreads();
  {
    constexpr int NQ = 16 * (int)sizeof(T) / 16;
    float4 q4[NQ];
    const int c0 = tid * 16 / EPC;
#pragma unroll
    for (int i = 0; i < NQ; ++i) q4[i] = reinterpret_cast<const float4*>(buf)[pchunk(c0 + i)];
    T v[16];
    memcpy(v, q4, sizeof(v));
    tnode[(tid & 7) * 33 + (tid >> 3)] = thread_pt(v);
  }
  __syncthreads();
  if (tid < 32) {
    T v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = tnode[i * 33 + tid];   // thread node 8 * tid + i
    const T node = warp_pt(thread_pt(v));
    if (tid == 0) nodes[q] = node;
  }
  __syncthreads();   // buf and tnode are reused by the next block
  }
}

// One warp per long bin: the PT over the bin's block nodes (in block order,
// absent padding), added to out[bin].  The block nodes come from the
// previous launch.
template <typename T>
__global__ void __launch_bounds__(256)
segtree_finish_kernel(const LongSeg* __restrict__ lsegs, const unsigned int* __restrict__ nlsegs,
                      const T* __restrict__ nodes, T* __restrict__ out, long long max_lsegs, long long ostride) {
  dep_wait();   // launched early (programmatic dependent launch): wait for the previous kernel
  const long long ns = min((long long)*nlsegs, max_lsegs);
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long sidx = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; sidx < ns; sidx += nwarps) {
    const LongSeg L = lsegs[sidx];
    const T t = warp_pt_range<T>(nodes + L.base, L.nblk);   // nodes already hold the negated leaves
    if ((threadIdx.x & 31) == 0) out[L.bin * ostride] = out[L.bin * ostride] + t;
  }
}

}  // namespace

// ---------------------------------------------------------------------------

// Warps of the passes that stay resident on one SM with CTAs of T threads:
// 228 KB of shared memory per SM, 1 KB of it reserved per CTA; registers
// (at most 64 per thread) allow two CTAs of 512 threads or four of 256.
static int resident_pass_warps(const SortPlan& p, int T) {
  size_t worst = 0;
  for (int pass = 0; pass < p.passes; ++pass)
    worst = std::max(worst, pass_smem(T, 1 << p.digit_bits, p.value_bytes, p.need_idx && pass > 0, p.passes > 1).total);
  const long long ctas = std::min<long long>(233472 / (long long)(worst + 1024 + 256), T == 512 ? 2 : 4);
  return (int)ctas * (T / 32);
}

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
  // The sort's tile is threads x kIPT records: 4,096 (CTAs of 256 threads)
  // for block_threads = 128, 8,192 (512 threads) for 256, 512 or 1024.  By
  // default sorts of at most 2^22 records take the smaller tiles, so that
  // they still spread over every SM; larger ones take whichever size keeps
  // more warps resident under the passes' shared memory.  Tiling never
  // changes the bits: the sort is stable.
  if (block_threads == 128 || block_threads == 256 || block_threads == 512 || block_threads == 1024) {
    p.threads = block_threads == 128 ? 256 : 512;
  } else if (n <= (1LL << 22)) {
    p.threads = 256;
  } else {
    p.threads = resident_pass_warps(p, 512) >= resident_pass_warps(p, 256) ? 512 : 256;
  }
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
  // blocks of long bins: ceil(len / B) <= len / B + 1 each (B = kSegBlock), and
  // at most min(m, n / kMediumGroup) bins are long (each holds more than
  // kMediumGroup records)
  p.max_blocks = n / kSegBlock + std::min(m, n / kMediumGroup) + 2;
  p.max_lsegs = std::min(m, n / kMediumGroup) + 2;
  p.blocks = off;
  off = align_up(off + (size_t)p.max_blocks * sizeof(BlockDesc), 256);
  p.lsegs = off;
  off = align_up(off + (size_t)p.max_lsegs * sizeof(LongSeg), 256);
  p.nodes = off;
  off = align_up(off + (size_t)p.max_blocks * 8, 256);
  p.total = off;
  return p;
}

template <int VB>
static cudaError_t launch_pass(const PassArgs& a, bool first, bool idx, bool keys_out, int threads, long long tiles,
                               cudaStream_t s, bool wide = false) {
  const int ndig = 1 << a.D;
  const size_t smem = pass_smem(threads, ndig, VB * (wide ? a.width : 1), idx && !first, keys_out).total;
  void (*k)(PassArgs) = nullptr;
  if (wide) k = sort_pass_kernel<VB, true, false, false, true>;
#define DET_PICK(F, I, KO) \
  if (!wide && first == F && idx == I && keys_out == KO) k = sort_pass_kernel<VB, F, I, KO>;
  DET_PICK(true, true, true) DET_PICK(true, true, false) DET_PICK(true, false, true) DET_PICK(true, false, false)
  DET_PICK(false, true, true) DET_PICK(false, true, false) DET_PICK(false, false, true) DET_PICK(false, false, false)
#undef DET_PICK
  cudaError_t e = ensure_dyn_smem((const void*)k, smem);
  if (e != cudaSuccess) return e;
  launch_begin("det_sort_pass", s);
  const cudaError_t le = launch_dep(k, dim3((unsigned)tiles), dim3(threads), smem, s, a);
  launch_end(s);
  return le;
}

int enqueue_sort(const SortPlan& p, void* ws, const int32_t* keys, long long key_offset, const void* values,
                 int32_t* perm_out, cudaStream_t s, int* final_buf, int32_t* rank_out, void* comp_out) {
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
    a.width = 1;
    a.comp_stride = 0;
    if (p.wide) {   // one-pass plans only: whole records into one array per component
      a.vals_out = comp_out;
      a.width = p.wide;
      a.comp_stride = p.n;
    }
    const size_t csmem = align_up((size_t)(ndig + 1) * 4, 16) + (size_t)p.threads * kIPT * 4;
    const long long K = (long long)p.threads * kIPT;
    void (*ck)(PassArgs, long long) = !first            ? sort_count_kernel<false, false>
                                      : key_offset == 0 ? sort_count_kernel<true, false>
                                                        : sort_count_kernel<true, true>;
    const cudaError_t ce = ensure_dyn_smem((const void*)ck, csmem);
    if (ce != cudaSuccess) return cuda_fail(ce, "sort: digit counts");
    launch_begin("det_sort_count", s);
    const cudaError_t e1 = launch_dep(ck, dim3((unsigned)p.tiles), dim3(256), csmem, s, a, K);
    launch_end(s);
    if (e1 != cudaSuccess) return cuda_fail(e1, "sort: digit counts");
    launch_begin("det_sort_colscan", s);
    const cudaError_t e2 = launch_dep(sort_colscan_kernel, dim3((unsigned)((ndig + kColDigits - 1) / kColDigits)),
                                      dim3(1024), 0, s, a, first ? 1 : 0);
    launch_end(s);
    if (e2 != cudaSuccess) return cuda_fail(e2, "sort: column scan");
    const bool keys_out = p.passes > 1;
    cudaError_t e;
    if (p.wide)
      e = p.wide_elem == 8 ? launch_pass<8>(a, true, false, false, p.threads, p.tiles, s, true)
                           : launch_pass<4>(a, true, false, false, p.threads, p.tiles, s, true);
    else if (p.value_bytes == 8)
      e = launch_pass<8>(a, first, p.need_idx, keys_out, p.threads, p.tiles, s);
    else if (p.value_bytes == 4)
      e = launch_pass<4>(a, first, p.need_idx, keys_out, p.threads, p.tiles, s);
    else
      e = launch_pass<0>(a, first, p.need_idx, keys_out, p.threads, p.tiles, s);
    if (e != cudaSuccess) return cuda_fail(e, "sort: pass");
  }
  if (p.passes > 1) {   // one-pass sorts got their segment starts from the pass
    launch_begin("det_sort_bounds", s);
    const int32_t* fkeys = reinterpret_cast<const int32_t*>(w + p.keys[*final_buf]);
    const unsigned int* nv = &h->n_valid;
    const cudaError_t e3 =
        p.n > (1LL << 24)
            ? launch_dep(sort_bounds_kernel<16>, dim3((unsigned)((p.n + 1 + 4095) / 4096)), dim3(256), 0, s, fkeys, nv,
                         p.m, seg, p.n)
            : launch_dep(sort_bounds_kernel<4>, dim3((unsigned)((p.n + 1 + 1023) / 1024)), dim3(256), 0, s, fkeys, nv,
                         p.m, seg, p.n);
    launch_end(s);
    if (e3 != cudaSuccess) return cuda_fail(e3, "sort: segment starts");
  }
  return DET_OK;
}

template <typename T>
int enqueue_segmented_tree(const SortPlan& p, void* ws, const T* sorted_vals, T* out, cudaStream_t s, bool negate,
                           long long ostride, bool reset_counters) {
  if (p.n == 0 || p.m == 0) return DET_OK;
  char* w = reinterpret_cast<char*>(ws);
  SortHdr* h = reinterpret_cast<SortHdr*>(ws);
  const int32_t* seg = reinterpret_cast<const int32_t*>(w + p.seg);
  BlockDesc* blocks = reinterpret_cast<BlockDesc*>(w + p.blocks);
  LongSeg* lsegs = reinterpret_cast<LongSeg*>(w + p.lsegs);
  T* nodes = reinterpret_cast<T*>(w + p.nodes);
  if (reset_counters && cudaMemsetAsync(&h->long_blocks, 0, 2 * sizeof(unsigned int), s) != cudaSuccess)
    return DET_ERR_CUDA;
  launch_begin("det_segtree_bins", s);
  auto* kb = negate ? segtree_bins_kernel<T, true> : segtree_bins_kernel<T, false>;
  const cudaError_t eb =
      launch_dep(kb, dim3((unsigned)((p.m + 255) / 256)), dim3(256), 0, s, sorted_vals, seg, p.m, out, blocks, lsegs,
                 &h->long_blocks, &h->long_segs, (const unsigned int*)&h->n_valid, p.max_blocks, p.max_lsegs,
                 &h->status, ostride);
  launch_end(s);
  if (eb != cudaSuccess) return cuda_fail(eb, "segmented tree: bins");
  launch_begin("det_segtree_blocks", s);
  auto* kk = negate ? segtree_blocks_kernel<T, true> : segtree_blocks_kernel<T, false>;
  const long long sms = std::max(device_sm_count(), 1);
  const cudaError_t ek = launch_dep(kk, dim3((unsigned)std::min(p.max_blocks, sms * 32)), dim3(256), 0, s,
                                    sorted_vals, (const BlockDesc*)blocks, (const unsigned int*)&h->long_blocks,
                                    nodes, p.max_blocks, p.max_lsegs);
  launch_end(s);
  if (ek != cudaSuccess) return cuda_fail(ek, "segmented tree: blocks");
  launch_begin("det_segtree_finish", s);
  const cudaError_t ef =
      launch_dep(segtree_finish_kernel<T>, dim3((unsigned)std::min((p.max_lsegs * 32 + 255) / 256, sms * 32)),
                 dim3(256), 0, s, (const LongSeg*)lsegs, (const unsigned int*)&h->long_segs, (const T*)nodes, out,
                 p.max_lsegs, ostride);
  launch_end(s);
  return ef == cudaSuccess ? DET_OK : cuda_fail(ef, "segmented tree: finish");
}

template int enqueue_segmented_tree<float>(const SortPlan&, void*, const float*, float*, cudaStream_t, bool, long long,
                                           bool);
template int enqueue_segmented_tree<double>(const SortPlan&, void*, const double*, double*, cudaStream_t, bool,
                                            long long, bool);

}  // namespace det
