// det_slot_alloc: the deterministic form of
//     slot = wp.atomic_add(counter, index[i], count[i])
// over threads i = 0 .. n-1 (Warp user guide "Deterministic Execution",
// "Pattern 2: Slot Allocation"): the reservations are sorted stably by
// counter element (thread order inside one element), an exclusive int32 scan
// of the requested counts gives every reservation's place in its group, and
// the slot is the counter's value before the launch plus that place; then
// each counter advances by its group's total ("Counter arrays are allocation
// counters": pre-existing values and append-style launches work).  int32
// arithmetic wraps modulo 2^32 as an int32 atomic add does.
#include "det_iscan.cuh"
#include "det_sort.cuh"

#include <algorithm>

namespace det {
namespace {

constexpr long long kSmemSeg = 8192;   // segment starts kept in shared memory up to this many entries

// slot_out[perm[p]] = counter[b] + (requests before p in counter b's group).
template <bool COUNTS, bool SMEM>
__global__ void __launch_bounds__(256)
slot_kernel(const int32_t* __restrict__ seg, long long C, const int32_t* __restrict__ perm,
            const unsigned* __restrict__ excl, const int32_t* __restrict__ counter,
            const unsigned int* __restrict__ n_valid, long long n, int32_t* __restrict__ slot_out,
            unsigned int* __restrict__ status) {
  extern __shared__ int32_t sseg[];
  if (SMEM) {
    for (long long i = threadIdx.x; i <= C; i += blockDim.x) sseg[i] = seg[i];
    __syncthreads();
  }
  const int32_t* sg = SMEM ? sseg : seg;
  const long long N = min((long long)*n_valid, n);
  for (long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x; p < N; p += (long long)gridDim.x * blockDim.x) {
    // the counter whose group holds p: sg[b] <= p < sg[b + 1] (sg[0] = 0, sg[C] = N)
    long long lo = 0, hi = C;
    while (hi - lo > 1) {
      const long long mid = (lo + hi) >> 1;
      if (sg[mid] <= p)
        lo = mid;
      else
        hi = mid;
    }
    const unsigned before = COUNTS ? excl[p] - excl[sg[lo]] : (unsigned)(p - sg[lo]);
    const long long r = perm[p];
    if (r < 0 || r >= n) {   // cannot happen for a correct sort; never write out of bounds
      set_status(status, DET_ERR_INVALID_ARG);
      continue;
    }
    slot_out[r] = (int32_t)((unsigned)counter[lo] + before);
  }
}

// counter[b] += its group's total (after every slot has read the old value).
template <bool COUNTS>
__global__ void counter_kernel(const int32_t* __restrict__ seg, long long C, const unsigned* __restrict__ excl,
                               int32_t* __restrict__ counter) {
  const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= C) return;
  const int32_t s0 = seg[b], s1 = seg[b + 1];
  if (s1 <= s0) return;
  const unsigned add = COUNTS ? excl[s1] - excl[s0] : (unsigned)(s1 - s0);
  counter[b] = (int32_t)((unsigned)counter[b] + add);
}

// One counter element: no sort is needed -- in thread order, every record's
// slot is the counter plus the requests of the records before it.
struct RequestSrc {
  const int32_t* index;
  const int32_t* count;
  long long off;
  __device__ __forceinline__ void load(long long i0, long long n, unsigned (&v)[kIScanPer]) const {
    int32_t ix[kIScanPer], cn[kIScanPer];
    const bool vec = i0 + kIScanPer <= n && (reinterpret_cast<uintptr_t>(index + i0) & 15) == 0 &&
                     (!count || (reinterpret_cast<uintptr_t>(count + i0) & 15) == 0);
    if (vec) {
#pragma unroll
      for (int q = 0; q < kIScanPer / 4; ++q) {
        const int4 w = __ldg(reinterpret_cast<const int4*>(index + i0) + q);
        ix[4 * q] = w.x, ix[4 * q + 1] = w.y, ix[4 * q + 2] = w.z, ix[4 * q + 3] = w.w;
        if (count) {
          const int4 c = __ldg(reinterpret_cast<const int4*>(count + i0) + q);
          cn[4 * q] = c.x, cn[4 * q + 1] = c.y, cn[4 * q + 2] = c.z, cn[4 * q + 3] = c.w;
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < kIScanPer; ++e) {
        const bool in = i0 + e < n;
        ix[e] = in ? __ldg(index + i0 + e) : -1;
        cn[e] = (in && count) ? __ldg(count + i0 + e) : 0;
      }
    }
#pragma unroll
    for (int e = 0; e < kIScanPer; ++e) {
      const bool valid = i0 + e < n && (long long)ix[e] + off == 0;
      v[e] = valid ? (count ? (unsigned)cn[e] : 1u) : 0u;
    }
  }
};

struct SlotDst {
  const int32_t* index;
  long long off;
  const int32_t* counter;
  int32_t* slot_out;
  __device__ __forceinline__ void store(long long i0, long long n, const unsigned (&ex)[kIScanPer],
                                        const unsigned (&)[kIScanPer]) const {
    const unsigned c0 = (unsigned)*counter;   // advanced only by a later kernel
#pragma unroll
    for (int e = 0; e < kIScanPer; ++e) {
      const long long i = i0 + e;
      if (i >= n) break;
      const bool valid = (long long)__ldg(index + i) + off == 0;
      slot_out[i] = valid ? (int32_t)(c0 + ex[e]) : -1;
    }
  }
};

__global__ void advance_counter_kernel(int32_t* __restrict__ counter, const int32_t* __restrict__ total) {
  *counter = (int32_t)((unsigned)*counter + (unsigned)*total);
}

// One slot each and a one-pass sort: in input order, slot_out[i] =
// counter[b] + (sorted position of i - start of b's group), b = index[i] +
// offset; the sort wrote the positions in input order.
template <bool SMEM>
__global__ void __launch_bounds__(256)
slot_rank_kernel(const int32_t* __restrict__ seg, long long C, const int32_t* __restrict__ index, long long off,
                 const int32_t* __restrict__ rank, const int32_t* __restrict__ counter, long long n,
                 int32_t* __restrict__ slot_out) {
  extern __shared__ int32_t sseg[];
  if (SMEM) {
    for (long long i = threadIdx.x; i <= C; i += blockDim.x) sseg[i] = seg[i];
    __syncthreads();
  }
  const int32_t* sg = SMEM ? sseg : seg;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long b = (long long)__ldg(index + i) + off;
    int32_t slot = -1;
    if (b >= 0 && b < C) slot = (int32_t)((unsigned)counter[b] + (unsigned)(__ldg(rank + i) - sg[b]));
    slot_out[i] = slot;
  }
}

struct SlotLayout {
  SortPlan plan;
  size_t excl = 0, iscan = 0, total = 0;
};

SlotLayout slot_layout(long long n, long long C, bool counts, int bt) {
  SlotLayout L;
  L.plan = make_sort_plan(n, C, counts ? 4 : 0, true, bt);
  size_t off = align_up(L.plan.total, 256);
  L.excl = off;
  off = align_up(off + (size_t)(n + 1) * 4, 256);
  L.iscan = off;
  off += iscan_ws_bytes(n + 1);
  L.total = align_up(off, 256);
  return L;
}

}  // namespace
}  // namespace det

using namespace det;

extern "C" size_t det_slot_alloc_workspace_bytes(int64_t n, int64_t num_counters) {
  if (n < 0 || num_counters < 0) return 0;
  // the largest layout: smallest sort tiles (128 threads) and a count payload
  return slot_layout(n, num_counters, true, 128).total;
}

extern "C" int det_slot_alloc(int32_t* counter, int64_t num_counters, const int32_t* index, int64_t index_offset,
                              const int32_t* count, int64_t n, int32_t* slot_out, void* workspace,
                              size_t workspace_bytes, int block_threads, void* stream) {
  if (n < 0 || num_counters < 0 || !workspace || !valid_block_threads(block_threads)) return DET_ERR_INVALID_ARG;
  if (n > DET_MAX_RECORDS || num_counters > 2147483647LL) return DET_ERR_TOO_LARGE;
  if ((num_counters > 0 && !counter) || (n > 0 && (!index || !slot_out))) return DET_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return DET_ERR_WORKSPACE;
  const cudaStream_t s = as_stream(stream);
  const long long C = num_counters;
  const SlotLayout L = slot_layout(n, C, count != nullptr, block_threads);
  if (workspace_bytes < L.total) return DET_ERR_WORKSPACE;
  char* w = reinterpret_cast<char*>(workspace);
  if (C == 1 && n > 0) {
    // one counter element: an exclusive scan of the requests, no sort
    if (cudaMemsetAsync(workspace, 0, kHeaderBytes, s) != cudaSuccess) return DET_ERR_CUDA;
    int32_t* total = reinterpret_cast<int32_t*>(w + L.excl);
    unsigned* tsum = reinterpret_cast<unsigned*>(w + L.iscan);
    int rc = enqueue_iscan(RequestSrc{index, count, index_offset}, SlotDst{index, index_offset, counter, slot_out},
                           n, total, tsum, s);
    if (rc != DET_OK) return rc;
    launch_begin("det_slot_counters", s);
    advance_counter_kernel<<<1, 1, 0, s>>>(counter, total);
    launch_end(s);
    return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
  }
  const int sms = device_sm_count();
  const long long grid = std::max(1LL, std::min((long long)((n + 255) / 256), 8LL * std::max(sms, 1)));
  const bool smem = C + 1 <= kSmemSeg;
  const size_t sb = smem ? (size_t)(C + 1) * 4 : 0;
  if (!count && n > 0 && C > 0) {
    const SortPlan rp = make_sort_plan(n, C, 0, false, block_threads);
    if (rp.passes == 1 && rp.total <= L.excl) {
      // one slot each, one sort pass: the pass writes every record's sorted
      // position in input order, and the slots follow in input order too
      int32_t* rank = reinterpret_cast<int32_t*>(w + L.excl);
      int fb = 0;
      int rc = enqueue_sort(rp, workspace, index, index_offset, nullptr, nullptr, s, &fb, rank);
      if (rc != DET_OK) return rc;
      const int32_t* seg = reinterpret_cast<const int32_t*>(w + rp.seg);
      launch_begin("det_slot_alloc", s);
      if (smem)
        slot_rank_kernel<true><<<(unsigned)grid, 256, sb, s>>>(seg, C, index, index_offset, rank, counter, n, slot_out);
      else
        slot_rank_kernel<false><<<(unsigned)grid, 256, 0, s>>>(seg, C, index, index_offset, rank, counter, n,
                                                               slot_out);
      launch_end(s);
      launch_begin("det_slot_counters", s);
      counter_kernel<false><<<(unsigned)((C + 255) / 256), 256, 0, s>>>(seg, C, nullptr, counter);
      launch_end(s);
      return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
    }
  }
  // skipped records keep slot -1
  if (n > 0 && cudaMemsetAsync(slot_out, 0xff, (size_t)n * 4, s) != cudaSuccess) return DET_ERR_CUDA;
  if (n == 0 || C == 0) return cudaMemsetAsync(workspace, 0, kHeaderBytes, s) == cudaSuccess ? DET_OK : DET_ERR_CUDA;
  const SortPlan& p = L.plan;
  int fb = 0;
  int rc = enqueue_sort(p, workspace, index, index_offset, count, nullptr, s, &fb);
  if (rc != DET_OK) return rc;
  SortHdr* h = reinterpret_cast<SortHdr*>(workspace);
  const int32_t* seg = reinterpret_cast<const int32_t*>(w + p.seg);
  const int32_t* perm = reinterpret_cast<const int32_t*>(w + p.idx[fb]);
  unsigned* excl = reinterpret_cast<unsigned*>(w + L.excl);
  if (count) {
    // excl[p] = requests of sorted records [0, p); excl[n] = all of them
    const int32_t* sorted_counts = reinterpret_cast<const int32_t*>(w + p.vals[fb]);
    rc = enqueue_scan_i32(sorted_counts, reinterpret_cast<int32_t*>(excl), n, true,
                          reinterpret_cast<int32_t*>(excl + n), w + L.iscan, s);
    if (rc != DET_OK) return rc;
  }
  launch_begin("det_slot_alloc", s);
  if (count) {
    if (smem)
      slot_kernel<true, true><<<(unsigned)grid, 256, sb, s>>>(seg, C, perm, excl, counter, &h->n_valid, n, slot_out,
                                                               &h->status);
    else
      slot_kernel<true, false><<<(unsigned)grid, 256, 0, s>>>(seg, C, perm, excl, counter, &h->n_valid, n, slot_out,
                                                               &h->status);
  } else {
    if (smem)
      slot_kernel<false, true><<<(unsigned)grid, 256, sb, s>>>(seg, C, perm, excl, counter, &h->n_valid, n, slot_out,
                                                                &h->status);
    else
      slot_kernel<false, false><<<(unsigned)grid, 256, 0, s>>>(seg, C, perm, excl, counter, &h->n_valid, n,
                                                                slot_out, &h->status);
  }
  launch_end(s);
  launch_begin("det_slot_counters", s);
  if (count)
    counter_kernel<true><<<(unsigned)((C + 255) / 256), 256, 0, s>>>(seg, C, excl, counter);
  else
    counter_kernel<false><<<(unsigned)((C + 255) / 256), 256, 0, s>>>(seg, C, excl, counter);
  launch_end(s);
  return cudaGetLastError() == cudaSuccess ? DET_OK : DET_ERR_CUDA;
}
