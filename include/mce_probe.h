/*
 * mce_probe.h -- measurement helpers of libmce_probe.so (roofline denominators).
 *
 * These entry points are not part of the method: "Parallelizing Maximal Clique Enumeration on
 * GPUs" has no counterpart.  They time, on the current CUDA device, the integer operation that
 * dominates the search -- scoring one 32-bit bitset word of a candidate row against the current
 * P set: AND, population count, accumulate (Section 2.3's pivot rule evaluated bit-parallel) --
 * so that a measured rate of the search can be set against what the SMs can sustain.
 */
#ifndef MCE_PROBE_H
#define MCE_PROBE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Runs a register-only kernel on every SM at full occupancy in which each thread repeats
 * "acc += popc(a & (b ^ acc))" (one logic op, one popcount, one add) on 8 independent register
 * words `iters` times, and reports the best of `reps` timings.
 *   words_per_s  receives the sustained rate in 32-bit words per second (host pointer).
 *   ms           receives the best kernel time in milliseconds (host pointer, may be NULL).
 * Returns 0 on success, 1 for invalid arguments, 9 for a CUDA error.  Synchronises the device.
 */
int mce_probe_word_rate(int iters, int reps, double *words_per_s, float *ms);

#ifdef __cplusplus
}
#endif

#endif /* MCE_PROBE_H */
