/*
 * rs_peaks.h -- throughput microbenchmarks of the instructions the compositing kernels of rs.h are
 * bound by, for the roofline's compute denominators: measured on the device at the clock it runs
 * at, instead of the nominal SMs x lanes x maximum clock.  The pages have no counterpart (they
 * quote no roofline); these calls exist for the benchmark.
 *
 * Each call launches one kernel of `blocks` blocks of 256 threads on `stream` and returns at once;
 * time it with events recorded on the same stream.  The work it represents is written to the
 * host double behind the last pointer.  Errors: RS_ERR_INVALID_ARG (checked before the launch),
 * RS_ERR_CUDA.
 */
#ifndef RS_PEAKS_H
#define RS_PEAKS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Single-precision fused multiply-adds: 8 independent chains per thread, `iters` x 32 steps each.
 * *lane_ops = blocks x 256 x iters x 256 (one FMA of one lane = one op).  d_sink: device float
 * [blocks x 256], never written in practice (it keeps the chains from being optimised away). */
int rs_peak_ffma(int32_t blocks, int32_t iters, float* d_sink, double* lane_ops, void* stream);

/* The multi-function unit's base-2 exponential (ex2.approx.ftz.f32, as the rasterisers use it):
 * 8 chains x -> 2^-x per thread, `iters` x 32 steps each.  *lane_ops = blocks x 256 x iters x 256. */
int rs_peak_ex2(int32_t blocks, int32_t iters, float* d_sink, double* lane_ops, void* stream);

/* Float atomic adds whose result is unused (red.global.add.f32) to scattered words of d_target
 * [n_targets] (1 <= n_targets <= 2^30; a buffer that fits in L2 measures the L2's atomic rate, as
 * the compositing backward's per-Gaussian sums see it): each thread adds 1.0 `iters` times, the 32
 * lanes of a warp to 32 different 128-byte lines.  *red_ops = blocks x 256 x iters. */
int rs_peak_red(int32_t blocks, int32_t iters, float* d_target, uint32_t n_targets, double* red_ops,
                void* stream);

/* Streaming multiprocessors of the current device (cudaDevAttrMultiProcessorCount). */
int rs_device_sm_count(int32_t* sms);

#ifdef __cplusplus
}
#endif
#endif /* RS_PEAKS_H */
