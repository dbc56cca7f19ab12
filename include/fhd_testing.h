/*
 * fhd_testing.h - test-only entry points of the fhd library.
 *
 * Not part of the operator API in fhd.h; they exist so the test-suite can
 * exercise the bounded-wait failure path without faulting or hanging a GPU,
 * force or inspect the gather path, replay the schedule on the host, check
 * pointers without launching, check the per-pair phasor on its own, and
 * measure the device's packed FP32 rate.
 * The library has no counterpart of these on the pages it implements.
 */
#ifndef FHD_TESTING_H
#define FHD_TESTING_H

#include "fhd.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fhd_compute (same arguments, layout and validation), except that the
 * producer warp of the gather kernel never issues the shared-memory copy of
 * work item `skip_tile` (a (target block, source tile) index in the kernel's
 * schedule; -1 skips nothing).  The consumers waiting for that tile then hit
 * their bounded-wait limit (about one second), set the timeout bit in the
 * workspace status word and leave; the producer drains its other copies and
 * leaves.  fhd_workspace_status() then returns FHD_ERR_TIMEOUT and the CUDA
 * context stays usable.  Output contents are unspecified after a timeout.
 */
FHD_API fhd_status fhd_test_compute_skip_tile(int64_t M, const float *kx, const float *ky, const float *kz,
                                      const float *Dr, const float *Di,
                                      int64_t N, const float *x, const float *y, const float *z,
                                      float *rho_r, float *rho_i, fhd_mode mode,
                                      void *workspace, size_t workspace_bytes, fhd_stream_t stream,
                                      int64_t skip_tile);

/*
 * Selects the gather path of every later call in this process, for tests that
 * must exercise one path on inputs the automatic choice would send to the
 * other: 0 automatic (the default), 1 always the persistent tiled gather,
 * 2 always the split gather that fhd_compute uses for small problems (one
 * target per thread, sources split into slices across CTAs).  Results agree
 * within the tolerance of the mode, not bit for bit, between the two paths.
 * Returns the previous setting, or -1 (setting unchanged) for any other
 * value.  Process-wide and not ordered with calls running in other threads.
 * Makes no CUDA call.
 */
FHD_API int fhd_test_set_path(int path);

/*
 * Turns the adjoint gather's step records on (1, the default) or off (0) for
 * every later call in this process.  The records hold, per sample, the step
 * phasor exp(i 2 pi k.d) and the chain coefficients of the target-side
 * recurrence for the launch's common voxel spacing d, evaluated once in
 * double precision; without them every thread evaluates its own.  Results
 * agree within the tolerance of the mode, not bit for bit.  Returns the
 * previous setting, or -1 (setting unchanged) for any other value.
 * Process-wide and not ordered with calls running in other threads.  Makes
 * no CUDA call.
 */
FHD_API int fhd_test_set_step_records(int enable);

/*
 * The packed FP32 rate this device reaches in practice, in FP32 lane
 * operations per second (an FMA counts as one per lane, a packed FMA as two):
 * one CTA of 256 threads per SM, each stepping 16 independent chains of
 * packed f32x2 FMAs (x = x * m + a) in registers, timed with CUDA events on
 * the legacy default stream of `device` after one warm-up launch (a few
 * milliseconds in all).  The gather kernels' bound counts FP32 lane
 * operations against the nominal 128 per SM per clock; this is the same unit
 * as the hardware delivers it to a kernel that does nothing else.
 * Synchronises the device's legacy default stream.  Returns FHD_ERR_CUDA on
 * any CUDA error (and *lane_ops_per_s = 0).
 */
FHD_API fhd_status fhd_test_fma2_rate(int device, double *lane_ops_per_s);

/*
 * The automatic path choice and split-gather shape for one gather of
 * n_targets targets and n_sources sources (both >= 1) on a device with `sms`
 * SMs running `ctas_max` persistent CTAs, with partial_bytes of partial rows
 * in the workspace.  Returns 1 when the split gather is chosen, 0 when the
 * persistent gather is, -1 for invalid arguments; *n_slices and *slice_len
 * (either may be NULL) receive the split shape.  Makes no CUDA call.
 */
FHD_API int fhd_test_split_shape(int64_t n_targets, int64_t n_sources, int sms, int ctas_max,
                                 size_t partial_bytes, int *n_slices, int64_t *slice_len);

/*
 * Host-side replay of the gather schedule for n_targets targets, n_sources
 * sources and `ctas` persistent CTAs (capped at the number of work items),
 * using the same schedule functions as the kernels.  Returns 0 when every CTA
 * owns at least one work item, every target block is finished exactly once
 * (written whole by one CTA, or summed by exactly one fix-up owner), and each
 * fix-up's contributors cover the block's source tiles once, in order;
 * otherwise a positive code naming the first violated property.  Makes no
 * CUDA call.
 */
FHD_API int fhd_test_schedule(int64_t n_targets, int64_t n_sources, int ctas);

/*
 * The per-array check every operator applies before launching: `p` must be
 * non-NULL, 4-byte aligned, device (or managed) memory of `device`, and
 * [p, p + bytes) must lie inside p's allocation.  Returns FHD_OK,
 * FHD_ERR_INVALID_VALUE, FHD_ERR_MISALIGNED or FHD_ERR_RANGE; launches
 * nothing, so a rejected pointer is never dereferenced.
 */
FHD_API fhd_status fhd_test_check_array(const void *p, size_t bytes, int device);

/*
 * The per-pair phasor of the sums, evaluated on its own: for i < n, the
 * phase p_i = ax_i bx_i + ay_i by_i + az_i bz_i (in cycles) and
 * s_i, c_i ~= sin(2 pi p_i), cos(2 pi p_i) by the method `which` selects:
 *   0  accurate mode: the compensated reduced phase (each product reduced on
 *      its own) and the accurate FMA-pipe polynomial, as every accurate path
 *      evaluates a pair;
 *   1  fast mode, hardware sin/cos: p as one float32 FMA chain, reduced to
 *      t = p - rint(p), sin/cos of 2 pi t on the MUFU pipe;
 *   2  fast mode, FMA-pipe share: the same p, the fast polynomial;
 *   3  CUDA's sincospif(2 t) of the t of method 1 (a reference for 4);
 *   4  the accurate polynomial of the t of method 1.
 * All arrays are float32 device arrays of n elements (inputs ax..bz, outputs
 * s, c), 4-byte aligned; the call validates them as the operators do and
 * returns FHD_ERR_INVALID_VALUE for an unknown `which` or n < 0.  Enqueued on
 * `stream`, asynchronous.
 */
FHD_API fhd_status fhd_test_phasor(int which, int64_t n, const float *ax, const float *ay, const float *az,
                                   const float *bx, const float *by, const float *bz, float *s, float *c,
                                   fhd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FHD_TESTING_H */
