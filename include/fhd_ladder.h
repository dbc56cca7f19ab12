/*
 * fhd_ladder.h - comparison kernels: the optimisation ladder of "Case study -
 * iterative MRI reconstruction" (sections 17.3.1-17.3.6 and the speed-up table
 * of section 17.3.6), and the scatter formulation that section 17.3.1
 * rejects.  Each variant computes F^H D, rho_n = sum_m D_m exp(+i 2 pi k_m.x_n),
 * with the technique of one step, so the steps can be measured side by side
 * on this GPU.  They are not the library's fast path (fhd_compute is).
 *
 * Arguments, layout, units and ownership as fhd_compute (include/fhd.h); N and
 * M must be below 2^31 (the page's kernels use 32-bit indices).  Outputs are
 * overwritten.  Accuracy: the L0-L3 variants use libm cosf/sinf on the
 * unreduced phase 2 pi k.x in fp32, L4, L5 and SCATTER the hardware
 * approximations; the phase rounding makes their error grow with |k.x|.
 * SCATTER adds with atomicAdd, so its fp32 summation order (and its last bits)
 * vary from run to run.  The CONSTANT, INTRINSICS and UNROLL variants stage
 * samples through one __constant__ array of the library: calls of those
 * variants must not overlap on the GPU.
 */
#ifndef FHD_LADDER_H
#define FHD_LADDER_H

#include "fhd.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FHD_VARIANT_NAIVE = 0,      /* L0: gather, global accumulation inside the loop, cosf/sinf */
    FHD_VARIANT_FISSION = 1,    /* L1: + 2 pi k precomputed by a separate kernel */
    FHD_VARIANT_PRIVATE = 2,    /* L2: + accumulators in registers */
    FHD_VARIANT_CONSTANT = 3,   /* L3: + 64 KB __constant__ chunks of AoS records */
    FHD_VARIANT_INTRINSICS = 4, /* L4: + __sincosf */
    FHD_VARIANT_UNROLL = 5,     /* L5: + unrolling by 4 */
    FHD_VARIANT_SCATTER = 6     /* one thread per sample, atomicAdd into every voxel */
} fhd_variant;

/* Workspace bytes of variant v (never 0 for a valid variant); 0 if invalid. */
FHD_API size_t fhd_variant_workspace_bytes(fhd_variant v, int64_t N, int64_t M);

/* F^H D with the technique of variant v.  Errors as fhd_compute. */
FHD_API fhd_status fhd_compute_variant(fhd_variant v, int64_t M, const float *kx, const float *ky, const float *kz,
                                       const float *Dr, const float *Di,
                                       int64_t N, const float *x, const float *y, const float *z,
                                       float *rho_r, float *rho_i, void *workspace, size_t workspace_bytes,
                                       fhd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FHD_LADDER_H */
