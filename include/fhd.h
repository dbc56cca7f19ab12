/*
 * fhd.h - C ABI of the GB300 library for the non-uniform Fourier sums of
 * iterative non-Cartesian MRI reconstruction.
 *
 * Source of the operations: "Case study - iterative MRI reconstruction"
 * (PMPP chapter 17 study notes):
 *   - section 17.2: the reconstruction minimises ||F rho - D||^2 + lambda R(rho)
 *     by conjugate gradients, whose inner loop applies F^H D and F^H F rho;
 *   - section 17.3: rho_n = sum_m D_m exp(i 2 pi k_m . x_n), with the complex
 *     multiply-accumulate of the gather kernel in 17.3.1
 *     (re += Dr cos - Di sin, im += Dr sin + Di cos);
 *   - section 17.3.2: loop fission - per-sample quantities are prepared in a
 *     separate pass, and F^H F rho runs as two kernels
 *     (image -> k-space, then k-space -> image).
 * and "Chapter 17: MRI Reconstruction" (mtuann PMPP notes), step 1 (gather
 * instead of scatter) and step 4 (samples as an array of structures).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Units      voxel coordinates x, y, z in field-of-view units; sample
 *            coordinates kx, ky, kz in cycles per field of view; the phase of
 *            a (voxel, sample) pair is 2 pi (kx x + ky y + kz z) radians.
 *            There is no normalisation, density compensation or coil weight.
 * Layout     every array is a contiguous float32 device array (structure of
 *            arrays); complex values are split into separate real and
 *            imaginary arrays.  Element i of each array belongs to voxel i
 *            (length N) or sample i (length M).
 * Alignment  every array pointer must be 4-byte aligned; the workspace must be
 *            256-byte aligned.
 * Ownership  all pointers are owned by the caller and must be device memory
 *            of the current CUDA device (cudaMalloc'd or managed).  The
 *            library allocates no memory and keeps no pointer after a call
 *            returns.  Its only process-wide state: a cache of each device's
 *            resident gather CTA count (filled on first use), the static
 *            scratch array of fhd_compute_noalloc (described there) and the
 *            path setting of the test hook fhd_test_set_path.
 * Outputs    are overwritten, never accumulated into.  Outputs must not
 *            overlap any input, each other, or the workspace.
 * Async      a call validates its arguments on the host, enqueues its kernels
 *            on `stream` and returns without synchronising.  Results (and the
 *            workspace status word) are valid once the stream has completed.
 *            NULL is the legacy default stream.
 * Errors     returned as an fhd_status, never thrown.  Argument errors are
 *            detected on the host before anything is launched, and then
 *            nothing is written.  A CUDA error raised while enqueueing returns
 *            FHD_ERR_CUDA.  A kernel whose internal pipeline wait exceeded its
 *            time limit (about one second) records FHD_ERR_TIMEOUT in the
 *            workspace status word and exits early; read it with
 *            fhd_workspace_status() after synchronising.
 * Modes      Phases are in cycles, and every sin/cos follows the range
 *            reduction t = k.x - rint(k.x).
 *            FHD_MODE_ACCURATE forms each pair's reduced phase from the
 *            three products k_j x_j reduced one by one (error below 2e-7
 *            cycles for any |k.x| < 2^21) and evaluates sin/cos with an
 *            FMA-pipe minimax polynomial (error below 2.4e-7).  The step
 *            phasors of the equal-spacing recurrences come, on an image grid
 *            (voxels with one common spacing), from per-sample step records
 *            evaluated in double precision (both modes), else from sincospif
 *            per thread.
 *            Relative L2 error against an fp64 evaluation: below 2e-6 on
 *            the benchmark workloads, and within 1e-5 up to |k| = 4096
 *            cycles/FOV on a unit FOV (tested).
 *            FHD_MODE_FAST forms the phase as one float32 FMA chain, whose
 *            rounding grows with |k.x| (relative L2 error about
 *            6.5e-8 * max|k| for k uniform in a cube on a unit FOV: 3e-4 at
 *            |k| = 4096, below 2e-5 on the benchmark workloads), and uses
 *            the hardware sin/cos approximations on 2 pi t in [-pi, pi],
 *            partly replaced by an FMA-pipe polynomial.  Relative L2 error
 *            3.3e-4 measured at |k| = 4096 (|k.x| up to 3500 cycles); it grows
 *            in proportion to |k.x| and reaches 1e-3 near 1e4 cycles.
 *            Either may be OR-ed with FHD_MODE_DIRECT, see below.
 * Spacing    where a thread's 32 consecutive targets (voxels for F^H D,
 *            samples for F rho) are exactly equally spaced, as the voxels of a
 *            regular image grid are, the kernel evaluates one phasor per
 *            (thread, source), two where the thread's spacing is not the one
 *            the per-sample step records hold, and reaches the other targets
 *            by the recurrence
 *            exp(i 2 pi k.(x0 + v d)) = exp(i 2 pi k.x0) exp(i 2 pi k.d)^v,
 *            an exact identity evaluated in fp32 (same tolerances).  Other
 *            targets are evaluated pair by pair.  Likewise, where runs of
 *            consecutive sources are exactly equally spaced (32 voxels of a
 *            grid row as sources of F rho; 16 or 32 samples along a straight
 *            line as sources of F^H D), each target evaluates one phasor per
 *            run (two when the run's step changes) and reaches the rest by
 *            powers of the step phasor: in F rho Clenshaw's recurrence
 *            (fast mode; its rounding grows with the run where k.d is near
 *            an integer or half-integer, within the fast tolerance) or
 *            Horner's rule (accurate mode), the same recurrence in F^H D.  FHD_MODE_DIRECT forces the pair-by-pair
 *            evaluation everywhere.
 * Small      problems too small to occupy the persistent kernel (a few blocks
 *            of 8192 targets times a few tiles of 256 sources) are evaluated
 *            pair by pair with one target per thread and the sources split
 *            into slices across CTAs; the slices are added in a fixed order.
 * Results are bit-identical from run to run on the same device: the sample
 * dimension is split among CTAs in a fixed way and the partial sums are
 * added in a fixed order, without atomics.
 */
#ifndef FHD_H
#define FHD_H

#include <stddef.h>
#include <stdint.h>

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define FHD_API __attribute__((visibility("default")))
#else
#define FHD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *fhd_stream_t;

typedef enum {
    FHD_OK = 0,
    FHD_ERR_INVALID_VALUE = 1, /* negative size, NULL pointer, unknown mode/op, or not device memory */
    FHD_ERR_MISALIGNED = 2,    /* array not 4-byte aligned, or workspace not 256-byte aligned */
    FHD_ERR_ALIAS = 3,         /* an output overlaps an input, another output or the workspace */
    FHD_ERR_WORKSPACE = 4,     /* workspace smaller than fhd_workspace_bytes() */
    FHD_ERR_CUDA = 5,          /* a CUDA runtime call failed (see cudaGetLastError) */
    FHD_ERR_TIMEOUT = 6,       /* a kernel's bounded pipeline wait expired (status word) */
    FHD_ERR_RANGE = 7,         /* an array extends past the end of its device allocation */
    FHD_ERR_TOO_LARGE = 8      /* fhd_compute_noalloc: problem exceeds its static scratch */
} fhd_status;

typedef enum {
    FHD_MODE_ACCURATE = 0,
    FHD_MODE_FAST = 1,
    FHD_MODE_DIRECT = 2,          /* flag: no equal-spacing recurrence */
    FHD_MODE_ACCURATE_DIRECT = 2,
    FHD_MODE_FAST_DIRECT = 3
} fhd_mode;

typedef enum {
    FHD_OP_FHD = 0, /* fhd_compute  */
    FHD_OP_FWD = 1, /* fwd_compute  */
    FHD_OP_FHF = 2  /* fhfrho_apply */
} fhd_op;

/*
 * Workspace size in bytes that `op` needs for N voxels and M samples on CUDA
 * device `device` (it depends on the device's SM count).  Returns 0 for an
 * invalid op, negative sizes or an unknown device.  The same workspace may be
 * reused by later calls on the same stream; calls that may run at the same
 * time (on different streams) need separate workspaces.
 */
FHD_API size_t fhd_workspace_bytes(fhd_op op, int64_t N, int64_t M, int device);

/*
 * Adjoint non-uniform Fourier sum F^H D (section 17.3, the rho_n equation):
 *
 *     rho_n = sum_{m=0}^{M-1} D_m exp(+i 2 pi (kx_m x_n + ky_m y_n + kz_m z_n))
 *
 * for n = 0..N-1.  Inputs: M samples kx, ky, kz, Dr, Di (length M each) and N
 * voxels x, y, z (length N each).  Outputs: rho_r, rho_i (length N).
 * M == 0 writes zeros; N == 0 does nothing (pointers may then be NULL).
 */
FHD_API fhd_status fhd_compute(int64_t M, const float *kx, const float *ky, const float *kz,
                       const float *Dr, const float *Di,
                       int64_t N, const float *x, const float *y, const float *z,
                       float *rho_r, float *rho_i, fhd_mode mode,
                       void *workspace, size_t workspace_bytes, fhd_stream_t stream);

/* Same type as cudaEvent_t. */
typedef struct CUevent_st *fhd_event_t;

/*
 * fhd_compute, additionally recording `gather_start` on `stream` just before
 * the gather kernel is launched and `gather_stop` just after its fix-up kernel
 * (the sample-pack kernel runs before `gather_start`).  Either event may be
 * NULL.  Used to time the dominant kernel inside a larger timed region.
 */
FHD_API fhd_status fhd_compute_profiled(int64_t M, const float *kx, const float *ky, const float *kz,
                                const float *Dr, const float *Di,
                                int64_t N, const float *x, const float *y, const float *z,
                                float *rho_r, float *rho_i, fhd_mode mode,
                                void *workspace, size_t workspace_bytes, fhd_stream_t stream,
                                fhd_event_t gather_start, fhd_event_t gather_stop);

/*
 * Forward non-uniform Fourier sum F rho (the image -> k-space operator of
 * section 17.2; its kernel is the conjugate of the adjoint's):
 *
 *     D_m = sum_{n=0}^{N-1} rho_n exp(-i 2 pi (kx_m x_n + ky_m y_n + kz_m z_n))
 *
 * for m = 0..M-1, gathered per sample.  Inputs: N voxels x, y, z, rho_r, rho_i
 * and M sample coordinates kx, ky, kz.  Outputs: Dr, Di (length M).
 * N == 0 writes zeros; M == 0 does nothing.
 */
FHD_API fhd_status fwd_compute(int64_t N, const float *x, const float *y, const float *z,
                       const float *rho_r, const float *rho_i,
                       int64_t M, const float *kx, const float *ky, const float *kz,
                       float *Dr, float *Di, fhd_mode mode,
                       void *workspace, size_t workspace_bytes, fhd_stream_t stream);

/*
 * Normal operator of the conjugate-gradient loop, out = F^H F rho
 * (section 17.2; section 17.3.2 splits it into the forward pass and the
 * adjoint pass as two kernels).  F rho is held in the workspace as float32.
 * Inputs: N voxels x, y, z, rho_r, rho_i and M sample coordinates.
 * Outputs: out_r, out_i (length N).  M == 0 writes zeros; N == 0 does nothing.
 */
FHD_API fhd_status fhfrho_apply(int64_t N, const float *x, const float *y, const float *z,
                        const float *rho_r, const float *rho_i,
                        int64_t M, const float *kx, const float *ky, const float *kz,
                        float *out_r, float *out_i, fhd_mode mode,
                        void *workspace, size_t workspace_bytes, fhd_stream_t stream);

/*
 * Status word of the last call that used `workspace`: synchronises `stream`,
 * reads the word and returns FHD_OK or FHD_ERR_TIMEOUT (FHD_ERR_CUDA if the
 * read fails, FHD_ERR_INVALID_VALUE for a NULL workspace).
 */
FHD_API fhd_status fhd_workspace_status(const void *workspace, fhd_stream_t stream);

/* Static, NUL-terminated description of a status code. */
FHD_API const char *fhd_status_string(fhd_status status);

/*
 * Launch shape the sums use on `device`: CTAs per launch (one persistent CTA
 * per resident slot), consumer threads per CTA, targets per thread, sources
 * per staged tile and pipeline stages.  Any pointer may be NULL.  Returns
 * FHD_ERR_INVALID_VALUE for an unknown device.
 */
FHD_API fhd_status fhd_launch_shape(int device, fhd_mode mode, int *ctas, int *threads,
                            int *targets_per_thread, int *tile_sources, int *stages);

/*
 * F^H D without any allocation, for callers that cannot allocate device
 * memory.  The operation, argument meaning, layout, validation and results
 * are those of fhd_compute, but there is no workspace argument: the scratch
 * space (packed sample records and step records, per-CTA partial sums,
 * status word) is a
 * file-scope static device array of FHD_NOALLOC_SCRATCH_BYTES inside the
 * library.  The pages this library implements have no counterpart of this
 * entry point; it exists for deployment.
 *
 * Who needs it: callers that must not allocate device memory after start-up,
 * for example a scanner's real-time reconstruction loop running under a
 * device-memory budget fixed at start-up (cudaMalloc can synchronise the
 * device and can fail under memory pressure), or a host application that
 * hands this library its data buffers but owns no allocator it may call.
 *
 * Limits: M <= FHD_NOALLOC_MAX_SAMPLES samples, and a device with at most
 * FHD_NOALLOC_MAX_CTAS resident gather CTAs (a GB300 uses 152).  Larger
 * problems return FHD_ERR_TOO_LARGE before anything is launched; N is not
 * limited.
 *
 * Memory: every GPU that loads the library holds the array (about 26 MiB)
 * until the process exits.  The first call on a device, with that device
 * current, looks up the array's device address (cudaGetSymbolAddress) and
 * caches it; make that first call before any stream capture begins.
 *
 * Sharing: all calls on a device use the same array, which keeps the last
 * call's contents.  Everything a call reads from it is written earlier in
 * the same call (the status word is cleared first), so stale contents do
 * not leak into results, but calls whose kernels overlap on the GPU (other
 * streams, other host threads) race on the array: serialise them, e.g. on one
 * stream.  fhd_workspace_status() does not apply to this entry point.
 */
#define FHD_NOALLOC_MAX_SAMPLES 131072
#define FHD_NOALLOC_MAX_CTAS 160
#define FHD_NOALLOC_SCRATCH_BYTES (1024 + (size_t)FHD_NOALLOC_MAX_SAMPLES * 49 + \
                                   (size_t)FHD_NOALLOC_MAX_CTAS * 2 * 2 * 8192 * 4)
FHD_API fhd_status fhd_compute_noalloc(int64_t M, const float *kx, const float *ky, const float *kz,
                               const float *Dr, const float *Di,
                               int64_t N, const float *x, const float *y, const float *z,
                               float *rho_r, float *rho_i, fhd_mode mode, fhd_stream_t stream);

/*
 * Conjugate-gradient reconstruction: solves (F^H F + lambda I) rho = F^H D for
 * rho, starting from rho = 0, with the loop of the host skeleton in section
 * 17.3.6 of the case study:
 *
 *     b = F^H D;  r = p = b;  rs_old = <r, r>
 *     repeat max_iter times:
 *         Ap = (F^H F + lambda I) p;  alpha = rs_old / <p, Ap>
 *         rho += alpha p;  r -= alpha Ap;  rs_new = <r, r>
 *         stop if rs_new < tol;  p = r + (rs_new / rs_old) p;  rs_old = rs_new
 *
 * lambda >= 0 adds the Tikhonov term lambda I (the plainest reading of the
 * regulariser R(rho) of section 17.2; lambda = 0 is the page's loop).  tol is
 * compared with rs_new = ||r||^2, as on the page (absolute, squared).
 * <a, b> = sum conj(a) b, accumulated in fp64 in a fixed order.
 *
 * Inputs and outputs as fhd_compute (M samples kx, ky, kz, Dr, Di; N voxels
 * x, y, z; result rho_r, rho_i, overwritten).  The workspace (size from
 * fhd_cg_workspace_bytes) holds r, p, A p, F p and the scalars.  Every
 * iteration is enqueued on `stream` without a host synchronisation: the
 * scalars stay on the device, and once rs_new < tol every later kernel of
 * the call returns immediately.  fhd_cg_info() reports the outcome.
 * Errors as for fhd_compute; also FHD_ERR_INVALID_VALUE for lambda < 0,
 * max_iter < 0 or tol < 0.
 */
FHD_API size_t fhd_cg_workspace_bytes(int64_t N, int64_t M, int device);
FHD_API fhd_status fhd_cg_solve(int64_t M, const float *kx, const float *ky, const float *kz,
                                const float *Dr, const float *Di,
                                int64_t N, const float *x, const float *y, const float *z,
                                float lambda, int max_iter, double tol,
                                float *rho_r, float *rho_i, fhd_mode mode,
                                void *workspace, size_t workspace_bytes, fhd_stream_t stream);

/*
 * Outcome of the last fhd_cg_solve on `workspace`: synchronises `stream`, then
 * reports the completed iterations, the last rs_new = ||r||^2 and whether the
 * loop stopped early (1: rs_new < tol, 0: ran max_iter iterations, -1: stopped
 * because <p, A p> was not positive).  Any output pointer may be NULL.
 * Returns FHD_ERR_TIMEOUT if a kernel's bounded wait expired during the call.
 */
FHD_API fhd_status fhd_cg_info(const void *workspace, fhd_stream_t stream, int *iterations, double *residual,
                               int *stopped);

/* Library version as major*10000 + minor*100 + patch. */
FHD_API int fhd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FHD_H */
