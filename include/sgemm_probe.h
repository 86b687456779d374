/*
 * sgemm_probe.h -- measurement probes shipped in the same library, used by
 * the benchmark to measure the roofline denominators in the same process and
 * run as the GEMM.
 *
 * - "Optimizing CUDA matmul, steps 4 to 6" (opening section): the FMA peak of
 *   the card is measured in the same run as the kernels it judges.
 * - "Optimizing Matrix Multiply on CUDA, Part 2", section "Power Throttling":
 *   under a sustained load the clock, and with it the peak, drops; the probe
 *   is therefore run for as long as the GEMM it is compared with.
 *
 * Each call queues one kernel on `stream` (a cudaStream_t, NULL = legacy
 * default stream) and return at once; the caller times them with events.
 */
#ifndef GB300_SGEMM_PROBE_H
#define GB300_SGEMM_PROBE_H

#include <stdint.h>

#include "sgemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * sgemm_probe_ffma -- `blocks` CTAs of 512 threads; each thread runs `iters`
 * iterations of 128 independent FP32 multiply-adds (16 chains x 8), as
 * scalar FFMA (paired == 0) or as 64 packed two-wide FFMA (paired != 0).
 * FLOPs per launch = blocks * 512 * iters * 128 * 2.  sink: device buffer of
 * at least `blocks` floats (written only in a case that does not occur, so
 * the compiler keeps the chains).  Returns SGEMM_ERR_INVALID_ARG for
 * iters < 1, blocks < 1 or sink == NULL.
 */
SGEMM_API sgemm_status_t sgemm_probe_ffma(int paired, int64_t iters, int blocks, float *sink, void *stream);

/*
 * sgemm_probe_read -- grid-stride streaming read (128-bit, evict-first) of
 * n_floats floats at device pointer buf (16-byte aligned, n_floats a multiple
 * of 4).  Bytes per launch = 4 * n_floats.  sink as above (>= blocks floats).
 */
SGEMM_API sgemm_status_t sgemm_probe_read(const float *buf, int64_t n_floats, float *sink, int blocks,
                                void *stream);

/*
 * sgemm_probe_tf32 -- the tensor pipe's TF32 dense rate, against which the
 * 3xTF32 entry point is judged: `blocks` CTAs (one per SM: launch as many as
 * the GPU has SMs) each issue iters * 4 back-to-back tcgen05.mma kind::tf32
 * of M 128, N 256, K 8 into tensor memory, from zeroed shared-memory
 * operands.  FLOPs per launch = blocks * iters * 4 * 2 * 128 * 256 * 8.  The
 * final wait for the MMAs is bounded; if it gives up, sgemm_device_status()
 * reports SGEMM_ERR_DEVICE_TIMEOUT.  Returns SGEMM_ERR_INVALID_ARG for
 * iters < 1, iters > 2^18 (a launch stays near 80 ms or less) or blocks < 1,
 * SGEMM_ERR_NO_DEVICE without an sm_103 device.
 */
SGEMM_API sgemm_status_t sgemm_probe_tf32(int64_t iters, int blocks, void *stream);

/*
 * sgemm_probe_hold -- one thread that sleeps on the GPU global timer for `ns`
 * nanoseconds and does nothing else.  A benchmark queues it ahead of a batch
 * of timed launches so that the host has queued the whole batch before the
 * device reaches it: the device then never idles waiting for the host, and
 * an event pair around one launch times that launch alone.  Returns
 * SGEMM_ERR_INVALID_ARG unless 0 < ns <= 10^9 (one second).
 */
SGEMM_API sgemm_status_t sgemm_probe_hold(int64_t ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_SGEMM_PROBE_H */
