/*
 * det_profile.h -- measurement hooks of libdet.so.  Not part of any
 * computation: they let a benchmark time each kernel the library launches
 * with CUDA events on the launching stream, and count the launches.
 * The pages have no counterpart; these exist so that a measurement of the
 * library can name its dominant kernel and its share of a call.
 *
 * Host-side state, one per process, not thread-safe: set it, make the calls
 * to be timed from one host thread, read it, clear it.
 */
#ifndef DET_PROFILE_H
#define DET_PROFILE_H

#ifdef __cplusplus
extern "C" {
#endif

/* events: an array of 2*capacity cudaEvent_t (passed as void*), created by
 * the caller.  While set, kernel launch i of the library records events[2i]
 * before and events[2i+1] after the launch, on the launch's stream, until
 * capacity launches have been recorded.  NULL (or capacity 0) switches the
 * recording off.  Returns 0. */
int det_profile_set_events(void* const* events, int capacity);

/* Launches recorded since the last det_profile_set_events(). */
int det_profile_event_count(void);

/* Name of the kernel of recorded launch i (static string), or NULL. */
const char* det_profile_event_name(int i);

/* Kernel launches made by this library since the process started. */
unsigned long long det_launch_count(void);

/* det_profile_add_rate_probe -- enqueue on `stream` one launch that only adds:
 * every thread of (SMs x 8) CTAs of 256 threads runs 8 independent chains of
 * `iters` dependent additions in `dtype` (DET_F32 or DET_F64), registers
 * only.  Timed with CUDA events by the caller, *adds_out / time is the
 * device's add rate for that type (the bound of the f64 sum and scan when
 * FP64 arithmetic, not HBM, limits them).
 *   sink      device, one element of dtype (never written in practice)
 *   adds_out  host: the number of additions the launch performs
 * Returns DET_OK, DET_ERR_DTYPE, DET_ERR_INVALID_ARG (iters <= 0, null
 * pointer) or DET_ERR_CUDA. */
int det_profile_add_rate_probe(int dtype, int iters, void* sink, void* stream,
                               unsigned long long* adds_out);

#ifdef __cplusplus
}
#endif

#endif /* DET_PROFILE_H */
