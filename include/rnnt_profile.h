/*
 * rnnt_profile.h -- per-kernel timing of librnnt_gb300, for measurement tools.
 *
 * Not part of the method (the pages define no instrumentation): while a
 * profiling session is open, every step of the path that rnnt_fwd / rnnt_bwd
 * run is bracketed by a pair of CUDA events recorded on the step's own
 * stream, so the device time of each step can be summed by name after the
 * fact.  A bracket holds one kernel launch, except the encoder-gradient
 * steps (tc_enc_prep, tc_enc_grads), which hold up to four and five.  Recording an event is asynchronous; nothing is
 * synchronized until rnnt_profile_stop.  Sessions are process-wide: library
 * calls from several host threads may record into an open session (each
 * bracket takes its own slot), but rnnt_profile_start and rnnt_profile_stop
 * must not run while a library call is in progress.  Events are created by rnnt_profile_start (no device memory
 * is allocated for them) and destroyed by rnnt_profile_stop.
 */
#ifndef RNNT_GB300_PROFILE_H
#define RNNT_GB300_PROFILE_H

#include "rnnt.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Open a session able to record `capacity` brackets (further ones are not
 * recorded).  RNNT_ERR_INVALID_ARG if capacity < 1 or a session
 * is already open; RNNT_ERR_CUDA if the events cannot be created. */
rnnt_status rnnt_profile_start(int capacity);

/* Close the session: synchronize on the recorded events, sum the elapsed
 * times per kernel name.  Returns the number of distinct kernel names (>= 0),
 * or -1 if no session was open or the events could not be read. */
int rnnt_profile_stop(void);

/* Entry i (0 <= i < the count rnnt_profile_stop returned) of the last
 * closed session: step name (static string), total milliseconds and the
 * number of kernel launches its brackets held.  RNNT_ERR_INVALID_ARG if i is out of range. */
rnnt_status rnnt_profile_entry(int i, const char** name, double* total_ms, int* launches);

#ifdef __cplusplus
}
#endif
#endif /* RNNT_GB300_PROFILE_H */
