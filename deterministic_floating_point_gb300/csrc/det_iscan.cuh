// int32 prefix sums (modular, so every order of the additions gives the same
// bits): the count -> exclusive scan -> write step of deterministic slot
// allocation (Warp user guide "Deterministic Execution", "Pattern 2: Slot
// Allocation" and "Picking the Right Mode").
#pragma once
#include "det_common.cuh"

namespace det {

constexpr long long kIScanTile = 4096;   // elements per CTA of 256 threads (16 each)

// Workspace bytes of enqueue_scan_i32 for n elements (no header).
size_t iscan_ws_bytes(long long n);

// y[i] = x[0] + ... + x[i] (inclusive) or x[0] + ... + x[i-1] (exclusive),
// modulo 2^32; *total (device, may be null) = the sum of all n values.
// x may equal y.  ws: iscan_ws_bytes(n) bytes, 256-byte aligned.
int enqueue_scan_i32(const int32_t* x, int32_t* y, long long n, bool exclusive, int32_t* total, void* ws,
                     cudaStream_t s);

}  // namespace det
