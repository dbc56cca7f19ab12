/*
 * fhd_oracle.c - plain fp64 CPU oracle for the non-uniform Fourier sums.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference for the
 * CUDA library.  Only the test-suite, the smoke check and the benchmark's CPU
 * baseline may load it; the library never links, calls or falls back to it.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (definitions written out, no blocking, no reordering):
 *
 *   Adjoint  F^H D  ("Case study - iterative MRI reconstruction", section 17.3,
 *   the rho_n equation, and the complex multiply-accumulate of the naive
 *   gather kernel in 17.3.1):
 *
 *       rho_n = sum_{m=0}^{M-1} D_m * exp(+i 2 pi (k_m . x_n))
 *       re += Dr*cos - Di*sin ;  im += Dr*sin + Di*cos
 *
 *   Forward  F rho  (section 17.2 defines F as the image -> k-space operator of
 *   the least-squares objective; as the adjoint of the sum above its kernel is
 *   exp(-i 2 pi k.x)):
 *
 *       (F rho)_m = sum_{n=0}^{N-1} rho_n * exp(-i 2 pi (k_m . x_n))
 *       re += rr*cos + ri*sin ;  im += ri*cos - rr*sin
 *
 * Arithmetic: every input arrives as double (the Python wrapper promotes the
 * float32 arrays exactly).  The phase p = kx*x + ky*y + kz*z is formed in
 * double; because exp(i 2 pi p) has period 1 in p, t = p - nearbyint(p) is
 * used as the libm argument (exact in double, it only keeps the argument of
 * sin/cos within [-pi, pi]).  sin and cos are glibc's double routines.  Each
 * output is a plain sequential double sum in ascending index order.
 *
 * Parallelism: one OpenMP "parallel for" over the independent outputs; the
 * order of every individual sum is unchanged.
 *
 * Planted mistakes: building with -DORACLE_MUTANT=k (k >= 1) deliberately
 * breaks one step (see the MUTANT blocks).  The test-suite compiles these
 * variants to prove that its pins catch each kind of mistake; the normal
 * build never defines the macro.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

static const double TWO_PI = 2.0 * 3.14159265358979323846;

/* exp(+i 2 pi p) as (c, s), with the period-1 reduction described above. */
static void unit_phasor(double p, double *c, double *s)
{
    double t = p - nearbyint(p);
    double a = TWO_PI * t;
#if ORACLE_MUTANT == 6
    a = 0.5 * TWO_PI * t; /* mistake: pi instead of 2 pi */
#endif
    *c = cos(a);
    *s = sin(a);
}

static double phase(double kx, double ky, double kz, double x, double y, double z)
{
#if ORACLE_MUTANT == 2
    (void)kz; (void)z;
    return kx * x + ky * y; /* mistake: dropped kz*z term */
#elif ORACLE_MUTANT == 5
    (void)x;
    return kx * y + ky * y + kz * z; /* mistake: wrong coordinate index */
#else
    return kx * x + ky * y + kz * z;
#endif
}

/* rho_n = sum_m D_m exp(+i 2 pi k_m.x_n), n = 0..N-1. */
void oracle_adjoint(int64_t M, const double *kx, const double *ky, const double *kz,
                    const double *Dr, const double *Di,
                    int64_t N, const double *x, const double *y, const double *z,
                    double *rho_r, double *rho_i)
{
    int64_t n;
#pragma omp parallel for schedule(static)
    for (n = 0; n < N; ++n) {
        double re = 0.0, im = 0.0;
        int64_t m = 0;
#if ORACLE_MUTANT == 7
        m = 1; /* mistake: first sample skipped */
#endif
        for (; m < M; ++m) {
            double c, s;
            unit_phasor(phase(kx[m], ky[m], kz[m], x[n], y[n], z[n]), &c, &s);
#if ORACLE_MUTANT == 1
            s = -s; /* mistake: exponent sign flipped */
#endif
#if ORACLE_MUTANT == 3
            re += Di[m] * c - Dr[m] * s; /* mistake: Dr and Di transposed */
            im += Di[m] * s + Dr[m] * c;
#elif ORACLE_MUTANT == 4
            re += Dr[m] * c + Di[m] * s; /* mistake: wrong sign in the real part */
            im += Dr[m] * s + Di[m] * c;
#else
            re += Dr[m] * c - Di[m] * s;
            im += Dr[m] * s + Di[m] * c;
#endif
        }
        rho_r[n] = re;
        rho_i[n] = im;
    }
}

/* (F rho)_m = sum_n rho_n exp(-i 2 pi k_m.x_n), m = 0..M-1. */
void oracle_forward(int64_t N, const double *x, const double *y, const double *z,
                    const double *rr, const double *ri,
                    int64_t M, const double *kx, const double *ky, const double *kz,
                    double *out_r, double *out_i)
{
    int64_t m;
#pragma omp parallel for schedule(static)
    for (m = 0; m < M; ++m) {
        double re = 0.0, im = 0.0;
        int64_t n;
        for (n = 0; n < N; ++n) {
            double c, s;
            unit_phasor(phase(kx[m], ky[m], kz[m], x[n], y[n], z[n]), &c, &s);
#if ORACLE_MUTANT == 8
            s = -s; /* mistake: forward uses the adjoint's sign */
#endif
            re += rr[n] * c + ri[n] * s;
            im += ri[n] * c - rr[n] * s;
        }
        out_r[m] = re;
        out_i[m] = im;
    }
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_threads(void)
{
#ifdef _OPENMP
    int t = 1;
#pragma omp parallel
    {
#pragma omp single
        t = omp_get_num_threads();
    }
    return t;
#else
    return 1;
#endif
}

/* Sets the OpenMP thread count of later calls (no effect without OpenMP);
 * the benchmark uses it to time the oracle on one core as well as on all.
 * Returns the previous count. */
int oracle_set_threads(int n)
{
#ifdef _OPENMP
    const int prev = omp_get_max_threads();
    if (n > 0) omp_set_num_threads(n);
    return prev;
#else
    (void)n;
    return 1;
#endif
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }
