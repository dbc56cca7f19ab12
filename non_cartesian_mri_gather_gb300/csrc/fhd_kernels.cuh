// fhd_kernels.cuh - sm_103a kernels for the non-uniform Fourier sums.
//
// One gather kernel serves both directions.  For the adjoint F^H D
// ("Case study - iterative MRI reconstruction", section 17.3, rho_n equation)
// the targets are voxels and the sources are samples {k, D}:
//
//     out_t = sum_s w_s exp(+i 2 pi (a_s . b_t))
//
// with b_t = x_n, a_s = k_m, w_s = D_m.  The forward sum F rho has the kernel
// exp(-i 2 pi k.x) = exp(+i 2 pi k.(-x)), so it is the same gather with the
// samples as targets and the voxels, coordinates negated (exact in fp32), as
// sources.  That is the loop fission of section 17.3.2: F^H F rho runs as a
// forward gather followed by an adjoint gather, each its own kernel.
//
// Pipeline of one call:
//   1. pack_sources   - loop fission / per-source precompute (section 17.3.2):
//                       SoA source arrays -> 32-byte AoS records
//                       {A.x, A.x, A.y, A.y, A.z, A.z, w.re, w.im} (A the
//                       source coordinates, negated for the forward sum),
//                       padded with zero-weight
//                       records to a whole number of tiles.  The
//                       array-of-structures record follows the mtuann notes'
//                       step 4 and the SampleChunk struct of section 17.3.4.
//                       For the adjoint sum it also writes one step record
//                       per source: the step phasor and chain coefficients of
//                       the target-side recurrence for the voxels' common
//                       spacing, in double.
//   2. gather_kernel  - persistent CTAs; each owns an equal contiguous range
//                       of (target block, source tile) work items.  A
//                       producer warp streams source tiles into a shared-
//                       memory ring with non-multicast bulk async copies
//                       completing on mbarriers; consumer warps read each
//                       record as a broadcast (the role the constant cache
//                       plays in section 17.3.4), keep per-tile accumulators
//                       of kV consecutive targets in registers (privatisation,
//                       section 17.3.3) and write every output once.  Per warp
//                       and tile one of three paths: equally spaced targets
//                       take a recurrence instead of a sin/cos per pair
//                       (accumulate_tile_pre with the staged step records
//                       where the warp's spacing is the launch's common one,
//                       accumulate_tile_strided otherwise); otherwise tiles
//                       of equally spaced source segments (described by
//                       describe_segments) a source-side evaluation
//                       (source_tile: Clenshaw's recurrence in fast mode and
//                       Horner's rule in accurate mode in the forward gather,
//                       a recurrence in the adjoint gather); otherwise pair
//                       by pair (direct_tile).  Instantiated per mode, source
//                       segment length and weight form: the adjoint gathers
//                       (polar weights) and the forward gathers (Cartesian
//                       weights) of each mode.
//   3. fixup_kernel   - target blocks whose source range was split between
//                       CTAs are summed from per-CTA partials in a fixed
//                       order (no atomics, bit-reproducible).
//   Small problems, which would leave most of the persistent CTAs or threads
//   idle, take split_gather_kernel (one target per thread, the sources split
//   into slices across CTAs) and split_reduce_kernel instead of 2 and 3.
//
// Every pipeline wait is bounded by a time limit; on expiry the waiting
// thread records an error bit in the status word and its CTA leaves early
// after the producer has drained its own copies in flight.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "sincos_poly.cuh"

namespace fhd {

// ---------------------------------------------------------------- shape
// Compile-time launch shape (overridable with -D for tuning builds).
#ifndef FHD_THREADS
#define FHD_THREADS 256
#endif
#ifndef FHD_V
#define FHD_V 32
#endif
#ifndef FHD_TILE
#define FHD_TILE 256
#endif
#ifndef FHD_STAGES
#define FHD_STAGES 5
#endif
#ifndef FHD_MIN_CTAS_PER_SM
#define FHD_MIN_CTAS_PER_SM 1
#endif
#ifndef FHD_FAST_POLY_SLOTS
#define FHD_FAST_POLY_SLOTS 2
#endif
#ifndef FHD_UNROLL
#define FHD_UNROLL 4
#endif
#ifndef FHD_POLAR_WEIGHTS
#define FHD_POLAR_WEIGHTS 1
#endif
#ifndef FHD_HORNER_GROUP
#define FHD_HORNER_GROUP 8
#endif
#ifndef FHD_UNROLL_PRE
#define FHD_UNROLL_PRE 3
#endif
#ifndef FHD_GOERTZEL
#define FHD_GOERTZEL 1
#endif
#ifndef FHD_GOERTZEL_GROUP
#define FHD_GOERTZEL_GROUP 8
#endif
#ifndef FHD_UNROLL_PRE_ACCURATE
#define FHD_UNROLL_PRE_ACCURATE 4
#endif

constexpr int kThreads = FHD_THREADS;    // consumer threads per CTA
constexpr int kWarps = kThreads / 32;    // consumer warps
constexpr int kV = FHD_V;                // targets per consumer thread
constexpr int kTargetsPerBlock = kThreads * kV;
constexpr int kTile = FHD_TILE;          // sources per staged tile
constexpr int kStages = FHD_STAGES;      // shared-memory ring depth
constexpr int kRecordBytes = 32;         // one packed source
constexpr int kTileBytes = kTile * kRecordBytes;
constexpr int kStepBytes = kTile * 16;   // one step record (float4) per source
// Source segments: kSegment consecutive packed sources (fast mode; accurate
// mode's length is set below) whose coordinates are exactly equally spaced
// take the source-side path; one 16-byte descriptor {step.x, step.y,
// step.z, flag} per segment, at most kDescBytes per tile.
constexpr int kSegment = 16;
constexpr int kSegmentsPerTile = kTile / kSegment;
constexpr int kDescBytes = kSegmentsPerTile * 16;
static_assert(kTile % kSegment == 0, "tiles hold whole segments");
constexpr int kCtaThreads = kThreads + 32;  // + one producer warp
constexpr int kMinCtasPerSm = FHD_MIN_CTAS_PER_SM;
constexpr int kUnroll = FHD_UNROLL;      // sources per unrolled inner-loop step
constexpr int kUnrollSharedU = 12;       // the same in the accurate warp-shared-phasor loop (measured best)
// and in the target-side recurrence's sample loop (measured best): two
// chains (the fast adjoint and the accurate kernels), one chain (the fast
// forward kernel)
constexpr int kUnrollTwoChains = 6;
constexpr int kUnrollOneChain = 3;
// the same with the staged step records (accumulate_tile_pre), per mode
// (measured best: 3 of 1-8 in fast mode, 4 of 2-8 in accurate mode)
constexpr int kUnrollPreFast = FHD_UNROLL_PRE;
constexpr int kUnrollPreAccurate = FHD_UNROLL_PRE_ACCURATE;
// The adjoint gathers store each weight in polar form, {|w|, arg(w) / 2 pi}
// (see pack_sources); the forward gathers, whose voxel weights Horner's rule
// adds as complex numbers, keep {w.re, w.im}.
constexpr bool kPolarAdjoint = FHD_POLAR_WEIGHTS != 0;
static_assert(kThreads % 32 == 0 && kTile % 2 == 0 && kStages >= 2, "bad launch shape");

// status word bits
constexpr uint32_t kStatusConsumerTimeout = 1u;
constexpr uint32_t kStatusProducerTimeout = 2u;
constexpr uint32_t kStatusDrainTimeout = 4u;

enum Mode : int { kAccurate = 0, kFast = 1 };
// Source segments are kSegment sources long in the fast adjoint gather and
// kSegmentAccurate elsewhere, where the longer segment halves the
// per-(target, segment) sin/cos cost of the source side (the recurrence's
// three-term error bound, eps * s^2 / 2, stays below 3e-5 over 32 sources;
// Horner's rule grows only linearly); the descriptor array is sized for
// kSegment.
constexpr int kSegmentAccurate = 32;
static_assert(kTile % kSegmentAccurate == 0, "tiles hold whole segments");
// Segment length of the adjoint gather in each mode; the forward gather
// (voxel sources) takes kSegmentAccurate in both modes, in a kernel
// instantiation of its own.
template <int MODE>
__host__ __device__ constexpr int segment_len() {
    return MODE == kAccurate ? kSegmentAccurate : kSegment;
}
// The pair-by-pair path walks a thread's kV targets in groups (coordinates and
// per-tile sums of one group in registers at a time): 8 in fast mode and 4 in
// accurate mode, whose compensated phase and polynomial hold more values per
// target (measured best with the packed path: fast 16 and 4 were 11 % and
// 12 % slower, accurate 8 and 16 7 % and 11 %).
#ifndef FHD_DIRECT_GROUP
#define FHD_DIRECT_GROUP 8
#endif
#ifndef FHD_DIRECT_GROUP_ACCURATE
#define FHD_DIRECT_GROUP_ACCURATE 4
#endif
template <int MODE>
__host__ __device__ constexpr int direct_group() {
    return (MODE == kAccurate ? FHD_DIRECT_GROUP_ACCURATE : FHD_DIRECT_GROUP) < kV
               ? (MODE == kAccurate ? FHD_DIRECT_GROUP_ACCURATE : FHD_DIRECT_GROUP)
               : kV;
}
static_assert(kV % direct_group<kFast>() == 0 && kV % direct_group<kAccurate>() == 0,
              "kV must be a multiple of the direct-path groups");
// Of a fast pair-by-pair group of 8 targets, how many take the FMA-pipe
// polynomial instead of the hardware sin/cos: 2 (one packed pair) balances
// the FP32 pipe (11 lane operations per pair) against the 16-lane sin/cos
// pipe (1.5 per pair); measured 9 % faster than 1.
constexpr int kFastPolySlots = FHD_FAST_POLY_SLOTS;
static_assert(kFastPolySlots >= 0 && kFastPolySlots <= direct_group<kFast>(), "bad polynomial split");
// The source-side recurrence (adjoint gathers) walks a thread's targets in
// groups of kSourceGroup; Horner's rule (forward gathers) in groups of
// kHornerGroup (below).
#ifndef FHD_SOURCE_GROUP
#define FHD_SOURCE_GROUP 8
#endif
constexpr int kSourceGroup = kV < FHD_SOURCE_GROUP ? kV : FHD_SOURCE_GROUP;
static_assert(kV % kSourceGroup == 0, "kV must be a multiple of the source-recurrence group");


// Static schedule shared by the gather and fix-up kernels (and by the
// host-side schedule check).  The work items (target block b, source tile j)
// are numbered w = b * n_tiles + j and CTA c owns [start(c), start(c+1)).
// The part of CTA c's range inside block b is a "segment"; a segment that
// covers all of block b's tiles is written straight to the output, any other
// segment goes to a partial slot of CTA c: slot 2c for its first block, 2c+1
// for its last (only the first and the last segment of a range can be
// partial).  A block is split exactly when some boundary start(c), c >= 1,
// lies strictly inside it; the lowest such boundary owns the block's fix-up,
// whose contributors are CTAs c-1 .. last_contributor().
struct Schedule {
    int64_t n_targets;   // targets (voxels for F^H D, samples for F rho)
    int64_t n_tiles;     // source tiles per target block
    int64_t n_blocks;    // target blocks of kTargetsPerBlock
    int64_t work;        // n_blocks * n_tiles
    int ctas;            // persistent CTAs in the launch

    __host__ __device__ int64_t start(int64_t c) const { return (c * work) / ctas; }
    __host__ __device__ int64_t first_block(int64_t c) const { return start(c) / n_tiles; }
    __host__ __device__ int64_t slot(int64_t c, int64_t b) const { return 2 * c + (b == first_block(c) ? 0 : 1); }
    // Block whose fix-up boundary c (1 <= c < ctas) owns, or -1.
    __host__ __device__ int64_t fixup_block(int64_t c) const {
        if (c < 1 || c >= ctas) return -1;
        const int64_t s = start(c);
        if (s % n_tiles == 0) return -1;
        const int64_t b = s / n_tiles;
        if (c >= 2 && start(c - 1) > b * n_tiles) return -1;  // an earlier boundary owns block b
        return b;
    }
    // Last CTA whose range intersects block b, scanning up from CTA c.
    __host__ __device__ int64_t last_contributor(int64_t c, int64_t b) const {
        while (c + 1 < ctas && start(c + 1) < (b + 1) * n_tiles) ++c;
        return c;
    }
};

struct GatherArgs {
    Schedule sch;
    const float* __restrict__ tx;   // target coordinates
    const float* __restrict__ ty;
    const float* __restrict__ tz;
    const float4* __restrict__ packed;  // n_tiles * kTile records of 2 float4
    const float4* __restrict__ desc;    // n_tiles * (kTile / SEG) segment descriptors
    const float4* __restrict__ steps;   // n_tiles * kTile step records, or nullptr (see pack_sources)
    float* __restrict__ out_r;
    float* __restrict__ out_i;
    float* __restrict__ partial;    // [2*ctas slots][2][kTargetsPerBlock]
    uint32_t* status;
    uint64_t wait_limit_ns;          // bounded-wait time limit
    int64_t skip_tile;               // test hook: work item whose copy is never issued (-1: none)
    int allow_strided;               // 1: use the equal-spacing recurrence where it applies
    const uint32_t* skip;            // optional device word: non-zero at launch -> do nothing
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with parity `parity` to complete, for at most
// `limit_ns` (plus an iteration cap in case the timer does not advance).
// On expiry sets `code` in the status word and returns false.
__device__ __noinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* status,
                                               uint32_t code, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1; it < (1u << 26); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0 && global_timer_ns() - t0 > limit_ns) break;
    }
    atomicOr(status, code);
    return false;
}

// Bulk async copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, size a multiple of 16 (kTileBytes is).
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// ---------------------------------------------------------------- per-pair math
// Phases are in cycles in both modes: the packed source coordinates are the
// caller's, unscaled (k in cycles per FOV, or -x for the forward sum), and the
// phasor of a pair is exp(i 2 pi p) with p = a.b.  Every sin/cos follows the
// range reduction t = p - rint(p) ("Case study - iterative MRI
// reconstruction", section 17.3.5: the hardware sin/cos lose accuracy once
// 2 pi has been multiplied into a large argument), so the hardware
// approximations only ever see 2 pi t in [-pi, pi], the interval on which
// they are specified.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr float kTwoPi = 6.28318530717958647692f;

// rint(v) on the FMA pipe: for |v| < 2^22, (v + 1.5*2^23) - 1.5*2^23 == rint(v)
// in round-to-nearest-even (the sum's ulp is 1).  rintf() itself issues on
// the 16-lane/SM/clock pipe of the hardware sin/cos approximations, so it is
// used only where that pipe has room: the recurrences (4 sin/cos per 32
// pairs) and the accurate mode (no hardware sin/cos at all).
__device__ __forceinline__ float rint_fma(float v) { return (v + kRoundMagic) - kRoundMagic; }

// Fast mode, MUFU pipe: t = p - rint(p) in [-1/2, 1/2] (exact in float32 for
// |p| < 2^22), then the hardware sin/cos of 2 pi t.
__device__ __forceinline__ void phasor_mufu(float p, float& s, float& c) {
    const float th = kTwoPi * (p - rint_fma(p));
    s = __sinf(th);
    c = __cosf(th);
}

// sin(2 pi t), cos(2 pi t) on the FMA pipe, for |t| < 2^21: the half-period
// reduction n = rint(2t), u = t - n/2 in [-1/4, 1/4] (exact), the minimax
// polynomials of sincos_poly.cuh in u, and the sign (-1)^n on both results (a
// shift by half a period flips both).  The parity of n is the low mantissa bit
// of 2t + 1.5*2^23, whose ulp is 1.  ACC selects the accurate coefficient set
// (max error 2.4e-7) or the fast one (7.6e-7).
template <bool ACC>
__device__ __forceinline__ void sincos2pi_poly(float t, float& s, float& c) {
    const float q = fmaf(t, 2.0f, kRoundMagic);
    const float u = fmaf(q - kRoundMagic, -0.5f, t);
    const uint32_t flip = __float_as_uint(q) << 31;
    const float w = u * u;
    float sn, pc;
    if constexpr (ACC) {
        float ps = poly::kAccurateSin[poly::kAccurateSinTerms - 1];
#pragma unroll
        for (int i = poly::kAccurateSinTerms - 2; i >= 1; --i) ps = fmaf(ps, w, poly::kAccurateSin[i]);
        sn = fmaf(poly::kAccurateSin[0], u, (u * w) * ps);  // the leading term's product exact in the FMA
        pc = poly::kAccurateCos[poly::kAccurateCosTerms - 1];
#pragma unroll
        for (int i = poly::kAccurateCosTerms - 2; i >= 0; --i) pc = fmaf(pc, w, poly::kAccurateCos[i]);
    } else {
        float ps = poly::kFastSin[poly::kFastSinTerms - 1];
#pragma unroll
        for (int i = poly::kFastSinTerms - 2; i >= 0; --i) ps = fmaf(ps, w, poly::kFastSin[i]);
        sn = ps * u;
        pc = poly::kFastCos[poly::kFastCosTerms - 1];
#pragma unroll
        for (int i = poly::kFastCosTerms - 2; i >= 0; --i) pc = fmaf(pc, w, poly::kFastCos[i]);
    }
    s = __uint_as_float(__float_as_uint(sn) ^ flip);
    c = __uint_as_float(__float_as_uint(pc) ^ flip);
}

// Accurate mode: the reduced phase of a pair, compensated.  A phase formed as
// one float32 dot product carries a rounding error that grows with |a.b|
// (about 2^-24 |a.b| cycles: 6e-6 cycles at |a.b| = 100, the dominant error
// of the sum on large grids).  Here each product is reduced on its own,
// frac(a b) = a b - rint(fl(a b)) in one FMA: the product is exact inside the
// FMA and only a result of magnitude at most 1/2 + ulp(a b)/2 is rounded,
// within 2^-25 of the exact fraction.  Their sum t (|t| < 2) is within
// 3e-7 cycles of a.b - rint(a.b) + an integer for any |a.b| < 2^22.
__device__ __forceinline__ float frac_mul(float a, float b) { return fmaf(a, b, -rintf(a * b)); }

__device__ __forceinline__ float phase_accurate(float ax, float ay, float az, float bx, float by, float bz) {
    return (frac_mul(ax, bx) + frac_mul(ay, by)) + frac_mul(az, bz);
}

// Accurate mode: sin, cos of 2 pi a.b for the pair (a, b).
__device__ __forceinline__ void phasor_accurate(float ax, float ay, float az, float bx, float by, float bz,
                                                float& s, float& c) {
    sincos2pi_poly<true>(phase_accurate(ax, ay, az, bx, by, bz), s, c);
}

// The same for 2 pi (a.b + phi), |phi| <= 1/2: the phase of a polar weight
// (see pack_sources) added to the reduced phase, one more rounding of a value
// below 2.5.
__device__ __forceinline__ void phasor_accurate_off(float phi, float ax, float ay, float az, float bx, float by,
                                                    float bz, float& s, float& c) {
    sincos2pi_poly<true>(phase_accurate(ax, ay, az, bx, by, bz) + phi, s, c);
}

// Accurate mode, the step phasor of a recurrence: sin, cos of 2 pi a.b with
// sincospif on the compensated phase.  A recurrence rotates by the step's
// angle once per target, so a relative error of that angle grows with the
// target's position (31 steps), where an error of the anchor phasor only
// scales every term alike: the step needs sin and cos correct to about an
// ulp, which the polynomial (absolute error 2.4e-7, its slope at 0 off by
// 1e-7 relative) does not give.  A step phasor is evaluated once per 32
// pairs or fewer.
__device__ __forceinline__ void phasor_step_accurate(float ax, float ay, float az, float bx, float by, float bz,
                                                     float& s, float& c) {
    sincospif(2.0f * phase_accurate(ax, ay, az, bx, by, bz), &s, &c);
}

// 2 cos(2 theta) from s = sin(theta), c = cos(theta), in the form that keeps
// the precision of the inputs where the recurrence needs it: 2 - 4 s^2 where
// 2 theta is near a multiple of 2 pi (the coefficient near 2), 4 c^2 - 2
// where it is near an odd multiple of pi (near -2).  Near those ends the
// angle a three-term recurrence turns by is most sensitive to its
// coefficient, and the other form would carry 8 times the error of its
// input there.
__device__ __forceinline__ float two_cos_double(float s, float c) {
    return fabsf(s) < fabsf(c) ? fmaf(-4.0f * s, s, 2.0f) : fmaf(4.0f * c, c, -2.0f);
}

// ---------------------------------------------------------------- pack
// The launch's common target spacing along one axis: the float32 value of
// t[1] - t[0], the difference formed in double exactly as the gather's
// per-thread spacing check (equally_spaced) forms it, so the two agree bit
// for bit; 0 with fewer than two targets.
__device__ __forceinline__ float launch_step(const float* __restrict__ t, int64_t n) {
    return n >= 2 ? (float)((double)t[1] - (double)t[0]) : 0.f;
}

// Source records {A.x, A.x, A.y, A.y, A.z, A.z, w.re, w.im} with A = sign*a
// (exact; sign is -1 for the forward sum, whose sources are the voxels, and +1
// for the adjoint sum; phases are in cycles in both modes): each coordinate
// twice, so one 16-byte load gives (A.x, A.x, A.y, A.y) as the packed pairs
// the recurrence multiplies by (x0, dx) and (y0, dy).  With `polar` the
// weight is stored as {|w|, phi}, phi = arg(w) / 2 pi in [-1/2, 1/2] cycles
// (both from double precision, each rounded once): w exp(i 2 pi a.b) =
// |w| exp(i 2 pi (a.b + phi)), so phi joins the phase (the first product of
// the phase becomes an FMA) and the complex multiply-accumulate of a pair
// becomes two real ones.
// Records n..n_padded-1 are zero (weight 0, so they add exactly 0).
//
// With `steps`, the kernel also writes one step record per source for the
// launch's common target spacing d (launch_step): {cos theta, sin theta,
// 2 cos theta, 2 cos 2 theta} with theta = 2 pi A.d, each evaluated in double
// (the three products of float32 values are exact there, the phase is
// reduced by its nearest integer before sincospi, and 2 cos 2 theta =
// 2 (cos theta - sin theta)(cos theta + sin theta)) and rounded once.  These
// are the step phasor u and the two chain coefficients of the target-side
// recurrence; on an image grid every thread's spacing is d, so the gather
// reads them instead of evaluating them per thread.  Padding records are zero.
//
// With `reset_status`, block 0 thread 0 also clears the status word (stream
// order puts this before the gather kernel); the second pass of F^H F rho
// keeps the word so a timeout of the first pass stays visible.
__global__ void pack_sources(const float* __restrict__ ax, const float* __restrict__ ay,
                             const float* __restrict__ az, const float* __restrict__ wr,
                             const float* __restrict__ wi, float sign, int polar, int64_t n, int64_t n_padded,
                             float4* __restrict__ out, const float* __restrict__ tx, const float* __restrict__ ty,
                             const float* __restrict__ tz, int64_t n_targets, float4* __restrict__ steps,
                             uint32_t* status, int reset_status, const uint32_t* skip) {
    if (skip != nullptr && *skip != 0u) return;
    if (reset_status && blockIdx.x == 0 && threadIdx.x == 0) *status = 0u;
    double dx = 0.0, dy = 0.0, dz = 0.0;
    if (steps != nullptr) {
        dx = launch_step(tx, n_targets);
        dy = launch_step(ty, n_targets);
        dz = launch_step(tz, n_targets);
    }
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_padded;
         i += (int64_t)gridDim.x * blockDim.x) {
        float4 r0 = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 r1 = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < n) {
            const float X = sign * ax[i], Y = sign * ay[i], Z = sign * az[i];
            r0 = make_float4(X, X, Y, Y);
            if (polar) {
                const double re = wr[i], im = wi[i];
                r1 = make_float4(Z, Z, (float)hypot(re, im), (float)(atan2(im, re) * 0.15915494309189533577));
            } else {
                r1 = make_float4(Z, Z, wr[i], wi[i]);
            }
            if (steps != nullptr) {
                const double p = (double)X * dx + (double)Y * dy + (double)Z * dz;
                const double t = p - rint(p);
                double su, cu;
                sincospi(2.0 * t, &su, &cu);
                q = make_float4((float)cu, (float)su, (float)(2.0 * cu), (float)(2.0 * (cu - su) * (cu + su)));
            }
        }
        out[2 * i] = r0;
        out[2 * i + 1] = r1;
        if (steps != nullptr) steps[i] = q;
    }
}

// Segment descriptors: one thread per SEG sources.  A segment is flagged
// when its real sources (index < n) have coordinates a_s = a_0 + (s - s0) * D
// exactly, with the step D itself a float32 value (checked in double on the
// caller's coordinates, where these products and sums are exact); the
// descriptor holds sign * D.  Sources at index >= n are zero-weight padding.
template <int SEG>
__global__ void describe_segments(const float* __restrict__ ax, const float* __restrict__ ay,
                                  const float* __restrict__ az, float sign, int64_t n, int64_t n_segments,
                                  float4* __restrict__ desc, const uint32_t* skip) {
    if (skip != nullptr && *skip != 0u) return;
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < n_segments;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t s0 = g * SEG;
        const int64_t real = n - s0 < SEG ? (n - s0 > 0 ? n - s0 : 0) : SEG;
        float4 out = make_float4(0.f, 0.f, 0.f, 1.f);
        if (real >= 2) {
            const double x0 = ax[s0], y0 = ay[s0], z0 = az[s0];
            const double dx = (double)ax[s0 + 1] - x0, dy = (double)ay[s0 + 1] - y0, dz = (double)az[s0 + 1] - z0;
            bool ok = (double)(float)dx == dx && (double)(float)dy == dy && (double)(float)dz == dz;
            for (int64_t s = 2; s < real && ok; ++s)
                ok = (double)ax[s0 + s] == x0 + (double)s * dx && (double)ay[s0 + s] == y0 + (double)s * dy &&
                     (double)az[s0 + s] == z0 + (double)s * dz;
            out = make_float4(sign * (float)dx, sign * (float)dy, sign * (float)dz, ok ? 1.f : 0.f);
        }
        desc[g] = out;
    }
}

// ---------------------------------------------------------------- gather
struct __align__(16) GatherSmem {
    float4 ring[kStages][kTile * 2];
    float4 desc[kStages][kSegmentsPerTile];
    // The tile's step records (pack_sources), staged with it when the launch
    // has them.
    float4 step[kStages][kTile];
    // Running sums of the current segment, one private column per consumer
    // thread (rows: kV real parts, then kV imaginary parts).  They are touched
    // once per tile, so keeping them here instead of in registers frees
    // 2*kV registers per thread for more resident warps.
    float run[2 * kV][kThreads];
    // Target coordinates of the current segment, one private column per
    // consumer thread (rows: x, y, z of each of the kV targets).  The
    // pair-by-pair path re-reads one group of targets' coordinates per tile;
    // the recurrence needs only b_0 and d, which stay in registers.
    float coord[3 * kV][kThreads];
    uint64_t full[kStages];
    uint64_t empty[kStages];
};

// Sum of one staged tile over the thread's kV targets, pair by pair, on
// records with Cartesian weights (the forward gather; polar records take
// accumulate_tile_packed): every record is read by all lanes at once
// (broadcast).  Targets go in groups of direct_group<MODE>() with fresh
// per-tile accumulators; each group's tile sums are folded into the thread's
// running sums in shared memory.  In fast mode the last NPOLY slots of a
// group take the FMA-pipe polynomial, the others the MUFU pipe; accurate mode
// takes the compensated phase and the accurate polynomial on every pair.
template <int MODE, int NPOLY>
__device__ __forceinline__ void accumulate_tile(const float4* __restrict__ rec, const float (*coord)[kThreads],
                                                float (*run)[kThreads], int tid) {
    constexpr int kDirectGroup = direct_group<MODE>();
#pragma unroll 1
    for (int g = 0; g < kV; g += kDirectGroup) {
        float bx[kDirectGroup], by[kDirectGroup], bz[kDirectGroup];
#pragma unroll
        for (int v = 0; v < kDirectGroup; ++v) {
            bx[v] = coord[g + v][tid];
            by[v] = coord[kV + g + v][tid];
            bz[v] = coord[2 * kV + g + v][tid];
        }
        float gr[kDirectGroup], gi[kDirectGroup];
#pragma unroll
        for (int v = 0; v < kDirectGroup; ++v) {
            gr[v] = 0.f;
            gi[v] = 0.f;
        }
#pragma unroll kUnroll
        for (int s = 0; s < kTile; ++s) {
            const float4 r0 = rec[2 * s];      // A.x A.x A.y A.y
            const float4 r1 = rec[2 * s + 1];  // A.z A.z w.re w.im
#pragma unroll
            for (int v = 0; v < kDirectGroup; ++v) {
                float sn, cs;
                if constexpr (MODE == kAccurate) {
                    phasor_accurate(r0.x, r0.z, r1.x, bx[v], by[v], bz[v], sn, cs);
                } else {
                    const float p = fmaf(r1.x, bz[v], fmaf(r0.z, by[v], r0.x * bx[v]));
                    if (v >= kDirectGroup - NPOLY)
                        sincos2pi_poly<false>(p, sn, cs);
                    else
                        phasor_mufu(p, sn, cs);
                }
                gr[v] = fmaf(r1.z, cs, gr[v]);
                gr[v] = fmaf(-r1.w, sn, gr[v]);
                gi[v] = fmaf(r1.z, sn, gi[v]);
                gi[v] = fmaf(r1.w, cs, gi[v]);
            }
        }
#pragma unroll
        for (int v = 0; v < kDirectGroup; ++v) {
            run[g + v][tid] += gr[v];
            run[kV + g + v][tid] += gi[v];
        }
    }
}

// Packed pairs of float32 (low = first, high = second) for the sm_100-family
// f32x2 instructions: one instruction does two fp32 operations, so the
// recurrence below spends one issue slot per target per operation.
typedef unsigned long long f2_t;

__device__ __forceinline__ f2_t f2_pack(float lo, float hi) {
    f2_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(f2_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
    f2_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2_t f2_mul(f2_t a, f2_t b) {
    f2_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2_t f2_add(f2_t a, f2_t b) {
    f2_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2_t f2_sub(f2_t a, f2_t b) {
    f2_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// (hi, lo) of (lo, hi)
__device__ __forceinline__ f2_t f2_swap(f2_t v) {
    float lo, hi;
    f2_unpack(v, lo, hi);
    return f2_pack(hi, lo);
}

// ---------------------------------------------------------------- packed pair-by-pair path
// Accurate mode, two targets at once: frac(a b) for the packed pair b (see
// frac_mul), the rounding of each half on the 16-lane pipe.
__device__ __forceinline__ f2_t frac_mul2(f2_t a, f2_t b) {
    float h0, h1;
    f2_unpack(f2_mul(a, b), h0, h1);
    return f2_fma(a, b, f2_pack(-rintf(h0), -rintf(h1)));
}

// sincos2pi_poly<ACC> on a packed pair t: s, c without the sign (-1)^n of
// the half-period reduction, which is applied to the pair of weights m
// instead (flipping the weight flips both of its products).
template <bool ACC>
__device__ __forceinline__ void sincos2pi_poly2(f2_t t, f2_t& s, f2_t& c, f2_t& m) {
    const f2_t q = f2_fma(t, f2_pack(2.0f, 2.0f), f2_pack(kRoundMagic, kRoundMagic));
    const f2_t u = f2_fma(f2_add(q, f2_pack(-kRoundMagic, -kRoundMagic)), f2_pack(-0.5f, -0.5f), t);
    float q0, q1, m0, m1;
    f2_unpack(q, q0, q1);
    f2_unpack(m, m0, m1);
    m = f2_pack(__uint_as_float(__float_as_uint(m0) ^ (__float_as_uint(q0) << 31)),
                __uint_as_float(__float_as_uint(m1) ^ (__float_as_uint(q1) << 31)));
    const f2_t w = f2_mul(u, u);
    if constexpr (ACC) {
        f2_t ps = f2_pack(poly::kAccurateSin[poly::kAccurateSinTerms - 1],
                          poly::kAccurateSin[poly::kAccurateSinTerms - 1]);
#pragma unroll
        for (int i = poly::kAccurateSinTerms - 2; i >= 1; --i)
            ps = f2_fma(ps, w, f2_pack(poly::kAccurateSin[i], poly::kAccurateSin[i]));
        s = f2_fma(f2_pack(poly::kAccurateSin[0], poly::kAccurateSin[0]), u, f2_mul(f2_mul(u, w), ps));
        f2_t pc = f2_pack(poly::kAccurateCos[poly::kAccurateCosTerms - 1],
                          poly::kAccurateCos[poly::kAccurateCosTerms - 1]);
#pragma unroll
        for (int i = poly::kAccurateCosTerms - 2; i >= 0; --i)
            pc = f2_fma(pc, w, f2_pack(poly::kAccurateCos[i], poly::kAccurateCos[i]));
        c = pc;
    } else {
        f2_t ps = f2_pack(poly::kFastSin[poly::kFastSinTerms - 1], poly::kFastSin[poly::kFastSinTerms - 1]);
#pragma unroll
        for (int i = poly::kFastSinTerms - 2; i >= 0; --i)
            ps = f2_fma(ps, w, f2_pack(poly::kFastSin[i], poly::kFastSin[i]));
        s = f2_mul(ps, u);
        f2_t pc = f2_pack(poly::kFastCos[poly::kFastCosTerms - 1], poly::kFastCos[poly::kFastCosTerms - 1]);
#pragma unroll
        for (int i = poly::kFastCosTerms - 2; i >= 0; --i)
            pc = f2_fma(pc, w, f2_pack(poly::kFastCos[i], poly::kFastCos[i]));
        c = pc;
    }
}

// The pair-by-pair path on polar records (the adjoint gather) with targets
// v and v+1 of a group in one packed f32x2 pair: the phase with the weight's
// phase, its reduction and the two real multiply-accumulates of both targets
// run as one instruction each (the record holds every coordinate twice, so
// (A.x, A.x) multiplies (x_v, x_{v+1}) as it stands).  The operations per
// target are those of accumulate_tile, in about half the issue slots for
// the FP32 work; the sin/cos stay per target.  In fast mode the last NPOLY
// (0, 1 or 2) targets of a group take the fast polynomial (with 2, both
// halves of the last pair, in packed arithmetic).
template <int MODE, int NPOLY>
__device__ __forceinline__ void accumulate_tile_packed(const float4* __restrict__ rec,
                                                       const float (*coord)[kThreads], float (*run)[kThreads],
                                                       int tid) {
    constexpr int kG = direct_group<MODE>();
    constexpr int kH = kG / 2;
    static_assert(kG % 2 == 0 && NPOLY <= 2, "the packed path pairs the targets of a group");
    const f2_t magic = f2_pack(kRoundMagic, kRoundMagic), nmagic = f2_pack(-kRoundMagic, -kRoundMagic);
    const f2_t neg1 = f2_pack(-1.0f, -1.0f), two_pi = f2_pack(kTwoPi, kTwoPi);
#pragma unroll 1
    for (int g = 0; g < kV; g += kG) {
        f2_t bx[kH], by[kH], bz[kH], ar[kH], ai[kH];
#pragma unroll
        for (int h = 0; h < kH; ++h) {
            bx[h] = f2_pack(coord[g + 2 * h][tid], coord[g + 2 * h + 1][tid]);
            by[h] = f2_pack(coord[kV + g + 2 * h][tid], coord[kV + g + 2 * h + 1][tid]);
            bz[h] = f2_pack(coord[2 * kV + g + 2 * h][tid], coord[2 * kV + g + 2 * h + 1][tid]);
            ar[h] = 0ull;  // +0.0f in both halves
            ai[h] = 0ull;
        }
#pragma unroll kUnroll
        for (int s = 0; s < kTile; ++s) {
            const float4 r0 = rec[2 * s];      // A.x A.x A.y A.y
            const float4 r1 = rec[2 * s + 1];  // A.z A.z |w| phi
            const f2_t ax = f2_pack(r0.x, r0.y), ay = f2_pack(r0.z, r0.w), az = f2_pack(r1.x, r1.y);
            const f2_t phi = f2_pack(r1.w, r1.w);
#pragma unroll
            for (int h = 0; h < kH; ++h) {
                f2_t sn, cs, m = f2_pack(r1.z, r1.z);
                if constexpr (MODE == kAccurate) {
                    const f2_t t = f2_add(f2_add(f2_add(frac_mul2(ax, bx[h]), frac_mul2(ay, by[h])),
                                                 frac_mul2(az, bz[h])), phi);
                    sincos2pi_poly2<true>(t, sn, cs, m);
                } else if (NPOLY == 2 && h == kH - 1) {  // both targets of the last pair on the polynomial
                    const f2_t p = f2_fma(az, bz[h], f2_fma(ay, by[h], f2_fma(ax, bx[h], phi)));
                    sincos2pi_poly2<false>(p, sn, cs, m);
                } else {
                    const f2_t p = f2_fma(az, bz[h], f2_fma(ay, by[h], f2_fma(ax, bx[h], phi)));
                    float s0, c0, s1, c1;
                    if (NPOLY == 1 && h == kH - 1) {
                        float p0, p1;
                        f2_unpack(p, p0, p1);
                        phasor_mufu(p0, s0, c0);
                        sincos2pi_poly<false>(p1, s1, c1);
                    } else {
                        // t = p - rint(p) (FMA-pipe rounding), 2 pi t, both halves at once
                        const f2_t th = f2_mul(f2_fma(f2_add(f2_add(p, magic), nmagic), neg1, p), two_pi);
                        float t0, t1;
                        f2_unpack(th, t0, t1);
                        s0 = __sinf(t0);
                        c0 = __cosf(t0);
                        s1 = __sinf(t1);
                        c1 = __cosf(t1);
                    }
                    sn = f2_pack(s0, s1);
                    cs = f2_pack(c0, c1);
                }
                ar[h] = f2_fma(m, cs, ar[h]);
                ai[h] = f2_fma(m, sn, ai[h]);
            }
        }
#pragma unroll
        for (int h = 0; h < kH; ++h) {
            float a0, a1, b0, b1;
            f2_unpack(ar[h], a0, a1);
            f2_unpack(ai[h], b0, b1);
            run[g + 2 * h][tid] += a0;
            run[g + 2 * h + 1][tid] += a1;
            run[kV + g + 2 * h][tid] += b0;
            run[kV + g + 2 * h + 1][tid] += b1;
        }
    }
}

// The pair-by-pair path of a gather instantiation: packed pairs of targets on
// polar records, one target at a time on Cartesian ones.
template <int MODE, int NPOLY, bool POLAR>
__device__ __forceinline__ void direct_tile(const float4* __restrict__ rec, const float (*coord)[kThreads],
                                            float (*run)[kThreads], int tid) {
    if constexpr (POLAR)
        accumulate_tile_packed<MODE, NPOLY>(rec, coord, run, tid);
    else
        accumulate_tile<MODE, NPOLY>(rec, coord, run, tid);
}

// Sign of the stored accumulator of target v in the recurrence below.
__host__ __device__ constexpr bool strided_negated(int v) { return (v & 2) != 0; }
// Sign of the stored accumulator of target v with the two-chain recurrence:
// targets 2j and 2j+1 carry the sign s_j = (+, -, -, +, ...) of their chains.
__host__ __device__ constexpr bool two_chain_negated(int v) { return ((v >> 1) & 3) == 1 || ((v >> 1) & 3) == 2; }

// Equal-spacing recurrence.  When a thread's kV consecutive targets satisfy
// b_v = b_0 + v*d exactly, exp(i 2 pi a.b_v) = exp(i 2 pi a.b_0) * u^v with
// u = exp(i 2 pi a.d).  Per source the thread evaluates two phasors (b_0 and
// d; in fast mode the phases are formed and reduced as packed pairs, in
// accurate mode each by the compensated reduction) and g_0 = w_s exp(i 2 pi
// a.b_0), g_1 = g_0 u.  The real and imaginary parts of g_v = g_0 u^v each
// follow g_{v+1} = 2 cos(theta_d) g_v - g_{v-1} (u + 1/u = 2 cos theta_d for
// |u| = 1); its fp32 error grows at most like eps * v^2 / 2.  The two-chain
// form steps by 2 cos(2 theta_d) (see two_cos_double for accurate mode).
// With the signs
// s_v = (+, +, -, -, ...) the scaled terms e_v = s_v g_v obey
// e_{v+1} = -+2 cos(theta_d) e_v + e_{v-1} (the coefficient alternating,
// -2 cos first), so each target costs one packed FMA for the step and one
// packed add into its accumulator, which holds s_v times the sum.  Voxels of a
// regular image grid, and samples along a radial spoke, are equally spaced.
template <int MODE, bool TWO, bool POLAR>
__device__ __forceinline__ void accumulate_tile_strided(const float4* __restrict__ rec, float x0, float y0,
                                                        float z0, float dx, float dy, float dz, f2_t (&acc)[kV]) {
#pragma unroll
    for (int v = 0; v < kV; ++v) acc[v] = 0ull;  // +0.0f in both halves
    const f2_t bx = f2_pack(x0, dx), by = f2_pack(y0, dy), bz = f2_pack(z0, dz);
    const f2_t two_pi = f2_pack(kTwoPi, kTwoPi);
    constexpr int kU = TWO ? kUnrollTwoChains : kUnrollOneChain;
#pragma unroll kU
    for (int s = 0; s < kTile; ++s) {
        const float4 r0 = rec[2 * s];      // A.x A.x A.y A.y
        const float4 r1 = rec[2 * s + 1];  // A.z A.z w.re w.im
        float s0, c0, sw, cw;
        if constexpr (MODE == kAccurate) {
            if constexpr (POLAR)
                phasor_accurate_off(r1.w, r0.x, r0.z, r1.x, x0, y0, z0, s0, c0);
            else
                phasor_accurate(r0.x, r0.z, r1.x, x0, y0, z0, s0, c0);
            phasor_step_accurate(r0.y, r0.w, r1.y, dx, dy, dz, sw, cw);
        } else {
            // (p0, pd) = A.b_0, A.d as one packed pair, reduced to
            // 2 pi (p - rint(p)) (the rounding on the XU pipe, which has room
            // here: 4 sin/cos per 32 pairs; reducing each half on its own
            // before the packed multiply measured fastest)
            const f2_t ph = f2_fma(f2_pack(r1.x, r1.y), bz,
                                   f2_fma(f2_pack(r0.z, r0.w), by, f2_mul(f2_pack(r0.x, r0.y), bx)));
            float p0, pd;
            f2_unpack(ph, p0, pd);
            if constexpr (POLAR) p0 += r1.w;  // the weight's phase (measured faster than in the packed FMA)
            const f2_t th = f2_mul(f2_pack(p0 - rintf(p0), pd - rintf(pd)), two_pi);
            float th0, thd;
            f2_unpack(th, th0, thd);
            s0 = __sinf(th0);
            c0 = __cosf(th0);
            sw = __sinf(thd);
            cw = __cosf(thd);
        }
        // g_0 = w_s * exp(i 2 pi a.b_0)
        const float fr = POLAR ? r1.z * c0 : fmaf(r1.z, c0, -r1.w * s0);
        const float fi = POLAR ? r1.z * s0 : fmaf(r1.z, s0, r1.w * c0);
        const float gr = fmaf(fr, cw, -fi * sw);      // g_1 = g_0 u
        const float gi = fmaf(fr, sw, fi * cw);
        if constexpr (TWO) {
            const float c2 = cw + cw;
            const f2_t kpos = f2_pack(c2, c2);
            const f2_t e0 = f2_pack(fr, fi), e1 = f2_pack(gr, gi);
            const f2_t e2n = f2_fma(f2_pack(-c2, -c2), e1, e0);  // -e_2
            const f2_t e3n = f2_fma(kpos, e2n, e1);              // -e_3
            // 2 cos(2 theta_d): accurate mode by two_cos_double; fast mode as
            // (2 cos theta_d)^2 - 2, one operation (its error, 8 times that of
            // the hardware cosine, stays two orders below the fast tolerance;
            // the precise forms measured 3 % slower here)
            const float cc = MODE == kAccurate ? two_cos_double(sw, cw) : fmaf(c2, c2, -2.0f);
            const f2_t kposC = f2_pack(cc, cc), knegC = f2_pack(-cc, -cc);
            f2_t amA = e0, aA = e2n, amB = e1, aB = e3n;           // chains over even and odd targets
            acc[0] = f2_add(acc[0], e0);
            acc[1] = f2_add(acc[1], e1);
            acc[2] = f2_add(acc[2], e2n);
            acc[3] = f2_add(acc[3], e3n);
#pragma unroll
            for (int j = 1; 2 * j + 3 < kV; ++j) {
                const f2_t nA = f2_fma((j & 1) ? kposC : knegC, aA, amA);  // s_{j+1} a_{j+1}
                const f2_t nB = f2_fma((j & 1) ? kposC : knegC, aB, amB);
                amA = aA;
                aA = nA;
                amB = aB;
                aB = nB;
                acc[2 * j + 2] = f2_add(acc[2 * j + 2], aA);
                acc[2 * j + 3] = f2_add(acc[2 * j + 3], aB);
            }
        } else {
            const float c2 = cw + cw;
            const f2_t kpos = f2_pack(c2, c2), kneg = f2_pack(-c2, -c2);
            f2_t em = f2_pack(fr, fi);  // e_{v-1}
            f2_t e = f2_pack(gr, gi);   // e_v
            acc[0] = f2_add(acc[0], em);
            acc[1] = f2_add(acc[1], e);
#pragma unroll
            for (int v = 1; v + 1 < kV; ++v) {
                const f2_t en = f2_fma((v & 1) ? kneg : kpos, e, em);  // e_{v+1}
                em = e;
                e = en;
                acc[v + 1] = f2_add(acc[v + 1], e);
            }
        }
    }
}

// Accurate mode, every lane of the warp with the same target spacing d (every
// warp of an image grid): the step phasor u_s = exp(i 2 pi a_s.d) and the
// chain coefficient 2 cos(2 theta_d) are the same for all lanes, so lane l
// evaluates them for sources 32k + l only and the others read them by
// shuffle.  Phases, sin/cos and coefficients are those of
// accumulate_tile_strided (the same operations in the same order), so the
// sums are bit-identical to it, with 1/32 of the sincospif evaluations of
// the step and of the coefficient's selection.  (Fast mode keeps the
// per-lane form: its step phasor is cheap, and the shuffles on the chain's
// critical path measured 1-7 % slower for every unroll factor tried.)
template <int MODE, bool POLAR>
__device__ __forceinline__ void accumulate_tile_strided_shared_u(const float4* __restrict__ rec, float x0,
                                                                 float y0, float z0, float dx, float dy, float dz,
                                                                 int lane, f2_t (&acc)[kV]) {
    static_assert(kTile % 32 == 0, "tiles hold whole warps of sources");
    static_assert(MODE == kAccurate, "the fast kernel evaluates the step phasor per lane");
#pragma unroll
    for (int v = 0; v < kV; ++v) acc[v] = 0ull;  // +0.0f in both halves
#pragma unroll 1
    for (int s32 = 0; s32 < kTile; s32 += 32) {
        float su_l, cu_l, cc_l;
        {
            const float4 r0 = rec[2 * (s32 + lane)];
            const float4 r1 = rec[2 * (s32 + lane) + 1];
            phasor_step_accurate(r0.y, r0.w, r1.y, dx, dy, dz, su_l, cu_l);
            cc_l = two_cos_double(su_l, cu_l);
        }
#pragma unroll kUnrollSharedU
        for (int q = 0; q < 32; ++q) {
            const float4 r0 = rec[2 * (s32 + q)];      // A.x A.x A.y A.y
            const float4 r1 = rec[2 * (s32 + q) + 1];  // A.z A.z w
            float s0, c0;
            if constexpr (POLAR)
                phasor_accurate_off(r1.w, r0.x, r0.z, r1.x, x0, y0, z0, s0, c0);
            else
                phasor_accurate(r0.x, r0.z, r1.x, x0, y0, z0, s0, c0);
            const float sw = __shfl_sync(0xffffffffu, su_l, q);
            const float cw = __shfl_sync(0xffffffffu, cu_l, q);
            const float cc = __shfl_sync(0xffffffffu, cc_l, q);  // 2 cos(2 theta_d)
            // g_0 = w_s * exp(i 2 pi a.b_0)
            const float fr = POLAR ? r1.z * c0 : fmaf(r1.z, c0, -r1.w * s0);
            const float fi = POLAR ? r1.z * s0 : fmaf(r1.z, s0, r1.w * c0);
            const float gr = fmaf(fr, cw, -fi * sw);      // g_1 = g_0 u
            const float gi = fmaf(fr, sw, fi * cw);
            const float c2 = cw + cw;
            const f2_t kpos = f2_pack(c2, c2);
            const f2_t e0 = f2_pack(fr, fi), e1 = f2_pack(gr, gi);
            const f2_t e2n = f2_fma(f2_pack(-c2, -c2), e1, e0);  // -e_2
            const f2_t e3n = f2_fma(kpos, e2n, e1);              // -e_3
            const f2_t kposC = f2_pack(cc, cc), knegC = f2_pack(-cc, -cc);
            f2_t amA = e0, aA = e2n, amB = e1, aB = e3n;           // chains over even and odd targets
            acc[0] = f2_add(acc[0], e0);
            acc[1] = f2_add(acc[1], e1);
            acc[2] = f2_add(acc[2], e2n);
            acc[3] = f2_add(acc[3], e3n);
#pragma unroll
            for (int j = 1; 2 * j + 3 < kV; ++j) {
                const f2_t nA = f2_fma((j & 1) ? kposC : knegC, aA, amA);  // s_{j+1} a_{j+1}
                const f2_t nB = f2_fma((j & 1) ? kposC : knegC, aB, amB);
                amA = aA;
                aA = nA;
                amB = aB;
                aB = nB;
                acc[2 * j + 2] = f2_add(acc[2 * j + 2], aA);
                acc[2 * j + 3] = f2_add(acc[2 * j + 3], aB);
            }
        }
    }
}

// Every thread of the warp with the launch's common target spacing d, and the
// tile's step records staged beside it (pack_sources: u = exp(i 2 pi a_s.d)
// and the chain coefficients 2 cos theta_d, 2 cos 2 theta_d, each from
// double precision): the thread evaluates only its anchor phasor per source,
// then the two chains of accumulate_tile_strided.  Polar records only (the
// adjoint gathers).
//
// The anchor phasor exp(i 2 pi (a_s.b_0 + phi_s)) of source s.
template <int MODE>
__device__ __forceinline__ void pre_anchor(const float4* __restrict__ rec, int s, float x0, float y0, float z0,
                                           float& s0, float& c0) {
    const float4 r0 = rec[2 * s];      // A.x A.x A.y A.y
    const float4 r1 = rec[2 * s + 1];  // A.z A.z |w| phi
    if constexpr (MODE == kAccurate) {
        phasor_accurate_off(r1.w, r0.x, r0.z, r1.x, x0, y0, z0, s0, c0);
    } else {
        // phase in cycles, the weight's phase first, reduced to
        // 2 pi (p - rint(p)) for the hardware sin/cos
        const float p0 = fmaf(r1.x, z0, fmaf(r0.z, y0, fmaf(r0.x, x0, r1.w)));
        const float th0 = (p0 - rintf(p0)) * kTwoPi;
        s0 = __sinf(th0);
        c0 = __cosf(th0);
    }
}

// Source s's terms for the thread's kV targets, from its anchor phasor
// (c0, s0) and its step record, added into acc.
__device__ __forceinline__ void pre_chains(const float4* __restrict__ rec, const float4* __restrict__ step, int s,
                                           float s0, float c0, f2_t (&acc)[kV]) {
    const float w = rec[2 * s + 1].z;  // |w|
    const float4 q = step[s];          // cos theta_d, sin theta_d, 2 cos theta_d, 2 cos 2 theta_d
    const float fr = w * c0;           // g_0 = |w| exp(i 2 pi (a.b_0 + phi))
    const float fi = w * s0;
    const float gr = fmaf(fr, q.x, -fi * q.y);  // g_1 = g_0 u
    const float gi = fmaf(fr, q.y, fi * q.x);
    const f2_t e0 = f2_pack(fr, fi), e1 = f2_pack(gr, gi);
    const f2_t e2n = f2_fma(f2_pack(-q.z, -q.z), e1, e0);  // -e_2
    const f2_t e3n = f2_fma(f2_pack(q.z, q.z), e2n, e1);   // -e_3
    const f2_t kposC = f2_pack(q.w, q.w), knegC = f2_pack(-q.w, -q.w);
    f2_t amA = e0, aA = e2n, amB = e1, aB = e3n;  // chains over even and odd targets
    acc[0] = f2_add(acc[0], e0);
    acc[1] = f2_add(acc[1], e1);
    acc[2] = f2_add(acc[2], e2n);
    acc[3] = f2_add(acc[3], e3n);
#pragma unroll
    for (int j = 1; 2 * j + 3 < kV; ++j) {
        const f2_t nA = f2_fma((j & 1) ? kposC : knegC, aA, amA);  // s_{j+1} a_{j+1}
        const f2_t nB = f2_fma((j & 1) ? kposC : knegC, aB, amB);
        amA = aA;
        aA = nA;
        amB = aB;
        aB = nB;
        acc[2 * j + 2] = f2_add(acc[2 * j + 2], aA);
        acc[2 * j + 3] = f2_add(acc[2 * j + 3], aB);
    }
}

template <int MODE>
__device__ __forceinline__ void accumulate_tile_pre(const float4* __restrict__ rec, const float4* __restrict__ step,
                                                    float x0, float y0, float z0, f2_t (&acc)[kV]) {
#pragma unroll
    for (int v = 0; v < kV; ++v) acc[v] = 0ull;  // +0.0f in both halves
    constexpr int kU = MODE == kAccurate ? kUnrollPreAccurate : kUnrollPreFast;
#pragma unroll kU
    for (int s = 0; s < kTile; ++s) {
        float s0, c0;
        pre_anchor<MODE>(rec, s, x0, y0, z0, s0, c0);
        pre_chains(rec, step, s, s0, c0, acc);
    }
}

// One staged tile on the target-side recurrence, folded into the thread's
// running sums (the signs of the stored terms undone here).  `step`: the
// tile's step records when the warp takes accumulate_tile_pre, else nullptr.
template <int MODE, bool TWO, bool POLAR>
__device__ __forceinline__ void strided_tile(const float4* __restrict__ rec, float x0, float y0, float z0,
                                             float dx, float dy, float dz, int lane, bool shared_u,
                                             const float4* __restrict__ step, float (*run)[kThreads], int tid) {
    static_assert(TWO || !POLAR, "the adjoint gathers run two chains");
    f2_t acc[kV];
    if (POLAR && step != nullptr) {
        if constexpr (POLAR) accumulate_tile_pre<MODE>(rec, step, x0, y0, z0, acc);
    } else if constexpr (MODE == kAccurate) {
        if (shared_u)
            accumulate_tile_strided_shared_u<MODE, POLAR>(rec, x0, y0, z0, dx, dy, dz, lane, acc);
        else
            accumulate_tile_strided<MODE, TWO, POLAR>(rec, x0, y0, z0, dx, dy, dz, acc);
    } else {
        accumulate_tile_strided<MODE, TWO, POLAR>(rec, x0, y0, z0, dx, dy, dz, acc);
    }
#pragma unroll
    for (int v = 0; v < kV; ++v) {
        float re, im;
        f2_unpack(acc[v], re, im);
        if (TWO ? two_chain_negated(v) : strided_negated(v)) {
            run[v][tid] -= re;
            run[kV + v][tid] -= im;
        } else {
            run[v][tid] += re;
            run[kV + v][tid] += im;
        }
    }
}

// True when c[v] == c[0] + v*d exactly for the first n entries, with d the
// float32 value c[1] - c[0] (checked in double, where these sums are exact).
__device__ __forceinline__ bool equally_spaced(const float (&c)[kV], int n, float& d) {
    if (n < 2) {
        d = 0.f;
        return true;
    }
    if (c[1] == c[0]) {
        // spacing 0 (a coordinate that is constant along a grid row): the
        // condition is c[v] == c[0], exact in float32 (and this GPU's double
        // rate is a small fraction of its float rate)
        d = 0.f;
        bool ok = true;
#pragma unroll
        for (int v = 2; v < kV; ++v)
            if (v < n) ok = ok && c[v] == c[0];
        return ok;
    }
    const double c0 = c[0];
    const double dd = (double)c[1] - c0;
    d = (float)dd;
    bool ok = (double)d == dd;
#pragma unroll
    for (int v = 2; v < kV; ++v)
        if (v < n) ok = ok && ((double)c[v] == c0 + (double)v * dd);
    return ok;
}

// Source-side recurrence, for tiles whose every segment of kSegment sources
// is equally spaced (a row of an image grid when the voxels are the sources,
// as in the forward sum F rho).  For target b and segment sources
// A_s = A_0 + s d: exp(i 2 pi A_s.b) = e_0 u^s with e_0 = exp(i 2 pi A_0.b)
// and u = exp(i 2 pi d.b).  Per (target, segment) one phasor, e_0, and per (target,
// run of segments with the same step) one more, u; the real and imaginary
// parts of e_s follow e_{s+1} = 2 cos(d.b) e_s - e_{s-1} (error growth at most
// eps * s^2 / 2 over the kSegment sources).  As in the target-side
// recurrence the stored terms are f_s = s_s e_s with s_s = (+, +, -, -, ...),
// so one packed FMA steps f (coefficient -+2 cos(d.b), then + f_{s-1}).  The
// weight is complex, so instead of a complex multiply per pair the thread
// keeps two packed sums per target, P = sum w.re e_s and Q = sum w.im e_s
// (the sign s_s moved onto the weights, shared by the group's targets), and
// sum w_s e_s = (P.re - Q.im) + i (P.im + Q.re) at the end: per pair three
// packed FMAs.  Targets go in groups of kSourceGroup; each group's tile sums
// are folded straight into the thread's running sums.
// A record's weight {w.re, w.im}; from polar records {|w|, phi}, |w| times
// (cos, sin)(2 pi phi), |phi| <= 1/2 (fast mode: the hardware sin/cos of
// 2 pi phi in [-pi, pi]; accurate mode: the accurate polynomial).
template <int MODE, bool POLAR>
__device__ __forceinline__ float2 record_weight(float a, float b) {
    if constexpr (!POLAR) {
        return make_float2(a, b);
    } else {
        float sn, cs;
        if constexpr (MODE == kAccurate) {
            sincos2pi_poly<true>(b, sn, cs);
        } else {
            const float th = kTwoPi * b;
            sn = __sinf(th);
            cs = __cosf(th);
        }
        return make_float2(a * cs, a * sn);
    }
}

template <int MODE, int SEG, bool POLAR>
__device__ __forceinline__ void accumulate_tile_src_strided(const float4* __restrict__ rec,
                                                            const float4* __restrict__ desc,
                                                            const float (*coord)[kThreads], float (*run)[kThreads],
                                                            int tid) {
    constexpr int kSeg = SEG;
#pragma unroll 1
    for (int g = 0; g < kV; g += kSourceGroup) {
        float bx[kSourceGroup], by[kSourceGroup], bz[kSourceGroup];
        f2_t P[kSourceGroup], Q[kSourceGroup];
#pragma unroll
        for (int v = 0; v < kSourceGroup; ++v) {
            bx[v] = coord[g + v][tid];
            by[v] = coord[kV + g + v][tid];
            bz[v] = coord[2 * kV + g + v][tid];
            P[v] = 0ull;  // +0.0f in both halves
            Q[v] = 0ull;
        }
        // u = exp(i d.b) is evaluated only when a segment's step d differs
        // from the previous segment's (on an image grid, once per tile), from
        // the phasor of half the step h: sin = 2 sin(h) cos(h), and
        // cos = 1 - 2 sin^2(h) near d.b = 0 (fast mode: always), 2 cos^2(h) - 1
        // near d.b = pi (accurate mode), which keeps the chain coefficient
        // 2 cos(d.b) precise where the chain is most sensitive to it, as in
        // the target-side recurrence; accurate mode takes the step from
        // sincospif (see phasor_step_accurate)
        float cu[kSourceGroup], su[kSourceGroup];
        float4 d_prev = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int j = 0; j < kTile / kSeg; ++j) {
            const float4 b0 = rec[2 * j * kSeg];      // A_0.x A_0.x A_0.y A_0.y
            const float4 b1 = rec[2 * j * kSeg + 1];  // A_0.z A_0.z w.re w.im
            const float4 d = desc[j];
            if (j == 0 || d.x != d_prev.x || d.y != d_prev.y || d.z != d_prev.z) {  // uniform over the CTA
                const float hx = 0.5f * d.x, hy = 0.5f * d.y, hz = 0.5f * d.z;
#pragma unroll
                for (int v = 0; v < kSourceGroup; ++v) {
                    float sh, ch;
                    if constexpr (MODE == kAccurate) {
                        phasor_step_accurate(hx, hy, hz, bx[v], by[v], bz[v], sh, ch);
                        cu[v] = fabsf(sh) < fabsf(ch) ? fmaf(-2.0f * sh, sh, 1.0f) : fmaf(2.0f * ch, ch, -1.0f);
                    } else {
                        phasor_mufu(fmaf(hz, bz[v], fmaf(hy, by[v], hx * bx[v])), sh, ch);
                        cu[v] = fmaf(-2.0f * sh, sh, 1.0f);
                    }
                    su[v] = (sh + sh) * ch;
                }
                d_prev = d;
            }
            f2_t fm[kSourceGroup], f[kSourceGroup], kpos[kSourceGroup], kneg[kSourceGroup];
#pragma unroll
            for (int v = 0; v < kSourceGroup; ++v) {
                float s0, c0;
                if constexpr (MODE == kAccurate)
                    phasor_accurate(b0.x, b0.z, b1.x, bx[v], by[v], bz[v], s0, c0);
                else
                    phasor_mufu(fmaf(b1.x, bz[v], fmaf(b0.z, by[v], b0.x * bx[v])), s0, c0);
                fm[v] = f2_pack(c0, s0);  // f_0 = e_0
                f[v] = f2_pack(fmaf(c0, cu[v], -s0 * su[v]), fmaf(c0, su[v], s0 * cu[v]));  // f_1 = e_0 u
                const float c2 = cu[v] + cu[v];
                kpos[v] = f2_pack(c2, c2);
                kneg[v] = f2_pack(-c2, -c2);
            }
            {  // source 0 (sign +) takes f_0
                const float2 w0 = record_weight<MODE, POLAR>(b1.z, b1.w);
                const f2_t wr = f2_pack(w0.x, w0.x), wi = f2_pack(w0.y, w0.y);
#pragma unroll
                for (int v = 0; v < kSourceGroup; ++v) {
                    P[v] = f2_fma(wr, fm[v], P[v]);
                    Q[v] = f2_fma(wi, fm[v], Q[v]);
                }
            }
#pragma unroll
            for (int s = 1; s < kSeg; ++s) {
                const float4 r = rec[2 * (j * kSeg + s) + 1];  // the weight in .z, .w
                const float2 w = record_weight<MODE, POLAR>(r.z, r.w);
                const float sg = strided_negated(s) ? -1.f : 1.f;   // s_s, folded into the weight
                const f2_t wr = f2_pack(sg * w.x, sg * w.x), wi = f2_pack(sg * w.y, sg * w.y);
#pragma unroll
                for (int v = 0; v < kSourceGroup; ++v) {
                    P[v] = f2_fma(wr, f[v], P[v]);
                    Q[v] = f2_fma(wi, f[v], Q[v]);
                    if (s + 1 < kSeg) {
                        const f2_t fn = f2_fma((s & 1) ? kneg[v] : kpos[v], f[v], fm[v]);  // f_{s+1}
                        fm[v] = f[v];
                        f[v] = fn;
                    }
                }
            }
        }
#pragma unroll
        for (int v = 0; v < kSourceGroup; ++v) {
            float pr, pi, qr, qi;
            f2_unpack(P[v], pr, pi);
            f2_unpack(Q[v], qr, qi);
            run[g + v][tid] += pr - qi;
            run[kV + g + v][tid] += pi + qr;
        }
    }
}

// Source-side sums by Horner's rule, the alternative to the recurrence
// above for the same tiles.  For target b and segment sources A_s = A_0 + s d
// (s = 0..S-1): sum_s w_s exp(i 2 pi A_s.b) = e_0 sum_s w_s z^s, with
// e_0 = exp(i 2 pi A_0.b) and z = exp(i 2 pi d.b).  The polynomial in z is
// evaluated by Horner's rule from the segment's last source, acc = acc z + w_s
// (one complex multiply-add per pair, its rounding growing linearly along
// the segment), then multiplied by e_0 once per (target, segment).  Two
// targets share every packed f32x2 pair, their real parts in one pair and
// their imaginary parts in another, so a pair costs two packed FMAs for the
// real parts and two for the imaginary parts of two targets: 4 FP32 lane
// operations in 2 instructions (the recurrence takes 6 in 3).  z is
// evaluated only when a segment's step differs from the previous one's (on
// an image grid, once per tile), from the phasor of half the step, as there.
constexpr int kHornerGroup = kV < FHD_HORNER_GROUP ? kV : FHD_HORNER_GROUP;
static_assert(kV % kHornerGroup == 0 && kHornerGroup % 2 == 0, "Horner's rule pairs the targets of a group");

template <int MODE, int SEG, bool POLAR>
__device__ __forceinline__ void accumulate_tile_src_horner(const float4* __restrict__ rec,
                                                           const float4* __restrict__ desc,
                                                           const float (*coord)[kThreads], float (*run)[kThreads],
                                                           int tid) {
    constexpr int kSourceGroup = kHornerGroup;  // targets per group, in kH packed pairs
    constexpr int kH = kSourceGroup / 2;
#pragma unroll 1
    for (int g = 0; g < kV; g += kSourceGroup) {
        float bx[kSourceGroup], by[kSourceGroup], bz[kSourceGroup];
#pragma unroll
        for (int v = 0; v < kSourceGroup; ++v) {
            bx[v] = coord[g + v][tid];
            by[v] = coord[kV + g + v][tid];
            bz[v] = coord[2 * kV + g + v][tid];
        }
        f2_t sr[kH], si[kH];  // tile sums: real, imaginary parts of targets 2h, 2h+1
        f2_t zr[kH], zi[kH], nzi[kH];
#pragma unroll
        for (int h = 0; h < kH; ++h) {
            sr[h] = 0ull;  // +0.0f in both halves
            si[h] = 0ull;
        }
        float4 d_prev = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int j = 0; j < kTile / SEG; ++j) {
            const float4 d = desc[j];
            if (j == 0 || d.x != d_prev.x || d.y != d_prev.y || d.z != d_prev.z) {  // uniform over the CTA
                const float hx = 0.5f * d.x, hy = 0.5f * d.y, hz = 0.5f * d.z;
                float cu[kSourceGroup], su[kSourceGroup];
#pragma unroll
                for (int v = 0; v < kSourceGroup; ++v) {
                    float sh, ch;
                    if constexpr (MODE == kAccurate) {
                        phasor_step_accurate(hx, hy, hz, bx[v], by[v], bz[v], sh, ch);
                        cu[v] = fabsf(sh) < fabsf(ch) ? fmaf(-2.0f * sh, sh, 1.0f) : fmaf(2.0f * ch, ch, -1.0f);
                    } else {
                        phasor_mufu(fmaf(hz, bz[v], fmaf(hy, by[v], hx * bx[v])), sh, ch);
                        cu[v] = fmaf(-2.0f * sh, sh, 1.0f);
                    }
                    su[v] = (sh + sh) * ch;
                }
#pragma unroll
                for (int h = 0; h < kH; ++h) {
                    zr[h] = f2_pack(cu[2 * h], cu[2 * h + 1]);
                    zi[h] = f2_pack(su[2 * h], su[2 * h + 1]);
                    nzi[h] = f2_pack(-su[2 * h], -su[2 * h + 1]);
                }
                d_prev = d;
            }
            f2_t ar[kH], ai[kH];
            {  // Horner's rule starts from the segment's last weight
                const float4 r = rec[2 * (j * SEG + SEG - 1) + 1];
                const float2 w = record_weight<MODE, POLAR>(r.z, r.w);
#pragma unroll
                for (int h = 0; h < kH; ++h) {
                    ar[h] = f2_pack(w.x, w.x);
                    ai[h] = f2_pack(w.y, w.y);
                }
            }
#pragma unroll
            for (int s = SEG - 2; s >= 0; --s) {
                const float4 r = rec[2 * (j * SEG + s) + 1];  // the weight in .z, .w
                const float2 w = record_weight<MODE, POLAR>(r.z, r.w);
                const f2_t wr = f2_pack(w.x, w.x), wi = f2_pack(w.y, w.y);
#pragma unroll
                for (int h = 0; h < kH; ++h) {
                    const f2_t nr = f2_fma(zr[h], ar[h], f2_fma(nzi[h], ai[h], wr));  // (acc z + w).re
                    const f2_t ni = f2_fma(zr[h], ai[h], f2_fma(zi[h], ar[h], wi));   // (acc z + w).im
                    ar[h] = nr;
                    ai[h] = ni;
                }
            }
            // times e_0 = exp(i 2 pi A_0.b), into the tile sums
            const float4 b0 = rec[2 * j * SEG];      // A_0.x A_0.x A_0.y A_0.y
            const float4 b1 = rec[2 * j * SEG + 1];  // A_0.z A_0.z w
            float c0[kSourceGroup], s0[kSourceGroup];
#pragma unroll
            for (int v = 0; v < kSourceGroup; ++v) {
                if constexpr (MODE == kAccurate)
                    phasor_accurate(b0.x, b0.z, b1.x, bx[v], by[v], bz[v], s0[v], c0[v]);
                else
                    phasor_mufu(fmaf(b1.x, bz[v], fmaf(b0.z, by[v], b0.x * bx[v])), s0[v], c0[v]);
            }
#pragma unroll
            for (int h = 0; h < kH; ++h) {
                const f2_t c = f2_pack(c0[2 * h], c0[2 * h + 1]);
                const f2_t sn = f2_pack(s0[2 * h], s0[2 * h + 1]), nsn = f2_pack(-s0[2 * h], -s0[2 * h + 1]);
                sr[h] = f2_fma(c, ar[h], f2_fma(nsn, ai[h], sr[h]));
                si[h] = f2_fma(c, ai[h], f2_fma(sn, ar[h], si[h]));
            }
        }
#pragma unroll
        for (int h = 0; h < kH; ++h) {
            float r0v, r1v, i0v, i1v;
            f2_unpack(sr[h], r0v, r1v);
            f2_unpack(si[h], i0v, i1v);
            run[g + 2 * h][tid] += r0v;
            run[g + 2 * h + 1][tid] += r1v;
            run[kV + g + 2 * h][tid] += i0v;
            run[kV + g + 2 * h + 1][tid] += i1v;
        }
    }
}

// Fast mode's source side in the forward gathers: the segment polynomial
// P = sum_s w_s z^s of accumulate_tile_src_horner by Clenshaw's recurrence
// for the basis z^s (z^{s+1} = c z^s - z^{s-1}, c = z + 1/z = 2 cos theta
// real on the unit circle; Goertzel's algorithm): from the last source down,
// y_s = w_s + c y_{s+1} - y_{s+2} (y_S = y_{S+1} = 0), then
// P = y_0 + (z - c) y_1 = y_0 - y_1 / z.  Each target keeps its (re, im)
// pair packed; with the signs sigma_s = (+, +, -, -, ...) folded into the
// stored u_s = sigma_s y_s the step is
// u_s = (sigma_s sigma_{s+1}) c u_{s+1} + (u_{s+2} + sigma_s w_s): one packed
// add or subtract and one packed FMA per (target, source), the 4 lane
// operations of Horner's rule, of which half are adds (a packed-add stream
// keeps the FP32 pipe busier than an FMA-only one).  Clenshaw's recurrence
// loses accuracy where theta is near 0 or pi (rounding grows like eps S^2
// there, 1e-4 relative at S = 32); fast mode only, accurate mode keeps
// Horner's rule.  Per (target, segment): e_0, P from (u_0, u_1) and e_0 P
// into the tile sums.
constexpr int kGoertzelGroup = kV < FHD_GOERTZEL_GROUP ? kV : FHD_GOERTZEL_GROUP;
static_assert(kV % kGoertzelGroup == 0, "Goertzel groups tile the thread's targets");

template <int SEG>
__device__ __forceinline__ void accumulate_tile_src_goertzel(const float4* __restrict__ rec,
                                                             const float4* __restrict__ desc,
                                                             const float (*coord)[kThreads],
                                                             float (*run)[kThreads], int tid) {
    constexpr int G = kGoertzelGroup;
#pragma unroll 1
    for (int g = 0; g < kV; g += G) {
        float bx[G], by[G], bz[G];
#pragma unroll
        for (int v = 0; v < G; ++v) {
            bx[v] = coord[g + v][tid];
            by[v] = coord[kV + g + v][tid];
            bz[v] = coord[2 * kV + g + v][tid];
        }
        f2_t acc[G];                // tile sums (re, im) of each target
        f2_t kp[G], kn[G];          // (c, c) and (-c, -c), c = 2 cos theta
        float zr[G], zi[G];         // z = exp(i theta)
#pragma unroll
        for (int v = 0; v < G; ++v) acc[v] = 0ull;  // +0.0f in both halves
        float4 d_prev = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int j = 0; j < kTile / SEG; ++j) {
            const float4 d = desc[j];
            if (j == 0 || d.x != d_prev.x || d.y != d_prev.y || d.z != d_prev.z) {  // uniform over the CTA
                // z from the phasor of half the step, as in Horner's rule
                const float hx = 0.5f * d.x, hy = 0.5f * d.y, hz = 0.5f * d.z;
#pragma unroll
                for (int v = 0; v < G; ++v) {
                    float sh, ch;
                    phasor_mufu(fmaf(hz, bz[v], fmaf(hy, by[v], hx * bx[v])), sh, ch);
                    zr[v] = fmaf(-2.0f * sh, sh, 1.0f);
                    zi[v] = (sh + sh) * ch;
                    const float c = zr[v] + zr[v];
                    kp[v] = f2_pack(c, c);
                    kn[v] = f2_pack(-c, -c);
                }
                d_prev = d;
            }
            f2_t u1[G], u2[G];  // u_{s+1}, u_{s+2}
#pragma unroll
            for (int v = 0; v < G; ++v) {
                u1[v] = 0ull;
                u2[v] = 0ull;
            }
#pragma unroll
            for (int s = SEG - 1; s >= 0; --s) {
                const float4 r = rec[2 * (j * SEG + s) + 1];  // the weight in .z, .w
                const f2_t w = f2_pack(r.z, r.w);
#pragma unroll
                for (int v = 0; v < G; ++v) {
                    const f2_t t = (s & 2) ? f2_sub(u2[v], w) : f2_add(u2[v], w);  // u_{s+2} + sigma_s w_s
                    const f2_t u = f2_fma((s & 1) ? kn[v] : kp[v], u1[v], t);        // sigma_s sigma_{s+1} = +-1
                    u2[v] = u1[v];
                    u1[v] = u;
                }
            }
            // u1 = u_0 = y_0, u2 = u_1 = y_1 (sigma_0 = sigma_1 = +1)
            const float4 b0 = rec[2 * j * SEG];      // A_0.x A_0.x A_0.y A_0.y
            const float4 b1 = rec[2 * j * SEG + 1];  // A_0.z A_0.z w
#pragma unroll
            for (int v = 0; v < G; ++v) {
                float s0, c0;
                phasor_mufu(fmaf(b1.x, bz[v], fmaf(b0.z, by[v], b0.x * bx[v])), s0, c0);
                // P = y_0 - y_1 / z = y_0 - conj(z) y_1
                const f2_t t = f2_fma(f2_pack(-zr[v], -zr[v]), u2[v], u1[v]);
                const f2_t P = f2_fma(f2_pack(-zi[v], zi[v]), f2_swap(u2[v]), t);
                // acc += e_0 P
                acc[v] = f2_fma(f2_pack(c0, c0), P, f2_fma(f2_pack(-s0, s0), f2_swap(P), acc[v]));
            }
        }
#pragma unroll
        for (int v = 0; v < G; ++v) {
            float re, im;
            f2_unpack(acc[v], re, im);
            run[g + v][tid] += re;
            run[kV + g + v][tid] += im;
        }
    }
}

// The source-side path of a gather instantiation: in the forward gathers
// (Cartesian records), whose tiles take this path, Clenshaw's recurrence in
// fast mode and Horner's rule in accurate mode; the recurrence in the
// adjoint gathers, where it is rare and where the recurrence measured faster
// for the kernel as a whole (the fast adjoint kernel inlines this path next
// to its hot target-side loop).
template <int MODE, int SEG, bool POLAR>
__device__ __forceinline__ void source_tile(const float4* __restrict__ rec, const float4* __restrict__ desc,
                                            const float (*coord)[kThreads], float (*run)[kThreads], int tid) {
    if constexpr (!POLAR) {
        if constexpr (MODE == kFast && FHD_GOERTZEL)
            accumulate_tile_src_goertzel<SEG>(rec, desc, coord, run, tid);
        else
            accumulate_tile_src_horner<MODE, SEG, POLAR>(rec, desc, coord, run, tid);
    } else {
        accumulate_tile_src_strided<MODE, SEG, POLAR>(rec, desc, coord, run, tid);
    }
}

// Out-of-line entry points of the pair-by-pair and source-side paths.  The
// gather kernel is one function holding all three paths, and the register
// allocation and scheduling of its hot loop depend on what else is inlined
// into it: measured on the 256^3 x 100000 grid, the accurate kernel runs its
// recurrence fastest with these two paths called out of line, the fast kernel
// with everything inlined.
template <int MODE, int NPOLY, bool POLAR>
__device__ __noinline__ void accumulate_tile_ool(const float4* __restrict__ rec, const float (*coord)[kThreads],
                                                 float (*run)[kThreads], int tid) {
    direct_tile<MODE, NPOLY, POLAR>(rec, coord, run, tid);
}
template <int MODE, int SEG, bool POLAR>
__device__ __noinline__ void accumulate_tile_src_strided_ool(const float4* __restrict__ rec,
                                                             const float4* __restrict__ desc,
                                                             const float (*coord)[kThreads],
                                                             float (*run)[kThreads], int tid) {
    source_tile<MODE, SEG, POLAR>(rec, desc, coord, run, tid);
}

// MODE: kAccurate or kFast.  NPOLY (fast mode only): how many of the kV
// register slots evaluate sin/cos with the FMA-pipe polynomial instead of the
// MUFU pipe; it sets the split between the two pipes.  SEG: the source segment
// length of the descriptors (segment_len<MODE>() for the adjoint gather,
// kSegmentAccurate for the forward gather).  POLAR: the records hold polar
// weights (the adjoint gather; see pack_sources).  Each combination in use is
// its own instantiation.
// FHD_GATHER_MAXNREG, when defined, sets the kernel's register cap directly
// (a 288-thread CTA fits up to 224 registers a thread); by default the launch
// bounds set it.
#ifdef FHD_GATHER_MAXNREG
#define FHD_GATHER_BOUNDS __maxnreg__(FHD_GATHER_MAXNREG)
#else
#define FHD_GATHER_BOUNDS __launch_bounds__(kCtaThreads, kMinCtasPerSm)
#endif
template <int MODE, int NPOLY, int SEG, bool POLAR>
__global__ void FHD_GATHER_BOUNDS gather_kernel(const GatherArgs args) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // The target-side recurrence runs as two chains (even and odd targets),
    // except in the fast forward gather, where a single chain measured faster
    // (its targets, the samples, rarely take the recurrence at all).
    constexpr bool kTwoChains = !(MODE == kFast && SEG == kSegmentAccurate);
    static_assert(MODE == kFast || kTwoChains, "the accurate kernel's fold assumes two chains");
    GatherSmem& sm = *reinterpret_cast<GatherSmem*>(smem_raw);

    // A set skip word (written by an earlier kernel on the stream, never while
    // this one runs) makes every thread return before any barrier or wait.
    if (args.skip != nullptr && *args.skip != 0u) return;
    const Schedule& sch = args.sch;
    const int c = blockIdx.x;
    const int64_t w_begin = sch.start(c);
    const int64_t w_end = sch.start(c + 1);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // step records: only the adjoint gathers' target-side recurrence uses them
    const bool with_steps = POLAR && args.steps != nullptr;

    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) {
            mbar_init(&sm.full[st], 1);
            mbar_init(&sm.empty[st], kWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();  // the only CTA-wide barrier: before any bounded wait

    if (warp == kWarps) {
        // ------------------------------------------------ producer warp
        if (lane != 0) return;
        int64_t issued = 0;
        bool ok = true;
        for (int64_t w = w_begin; w < w_end && ok; ++w, ++issued) {
            const int st = (int)(issued % kStages);
            if (issued >= kStages) {
                const uint32_t par = (uint32_t)(((issued / kStages) - 1) & 1);
                ok = mbar_wait_bounded(&sm.empty[st], par, args.status, kStatusProducerTimeout,
                                       args.wait_limit_ns);
                if (!ok) break;
            }
            if (w == args.skip_tile) continue;  // test hook: this copy never arrives
            const int64_t j = w % sch.n_tiles;
            constexpr int kTileDescBytes = kTile / SEG * 16;
            mbar_arrive_expect_tx(&sm.full[st], kTileBytes + kTileDescBytes + (with_steps ? kStepBytes : 0));
            bulk_copy_g2s(&sm.ring[st][0], args.packed + j * (kTile * 2), kTileBytes, &sm.full[st]);
            bulk_copy_g2s(&sm.desc[st][0], args.desc + j * (kTile / SEG), kTileDescBytes, &sm.full[st]);
            if (with_steps) bulk_copy_g2s(&sm.step[st][0], args.steps + j * kTile, kStepBytes, &sm.full[st]);
        }
        // Drain: the last copy issued into each stage must have landed before
        // this CTA's shared memory can be released.
        for (int st = 0; st < kStages; ++st) {
            // last index < issued that maps to stage st
            if (issued <= st) continue;
            const int64_t last = st + ((issued - 1 - st) / kStages) * kStages;
            if (w_begin + last == args.skip_tile) continue;
            mbar_wait_bounded(&sm.full[st], (uint32_t)((last / kStages) & 1), args.status, kStatusDrainTimeout,
                              args.wait_limit_ns);
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    // Thread tid owns the kV consecutive targets b*kTargetsPerBlock + tid*kV + v.
    float x0 = 0.f, y0 = 0.f, z0 = 0.f;  // first target of the thread (strided path)
    float sx = 0.f, sy = 0.f, sz = 0.f;  // target spacing of the strided path
    bool strided = false;                // warp-uniform
    bool shared_u = false;               // strided, and every lane has the same spacing
    bool pre = false;                    // strided, and every lane has the launch's common spacing
    const int tid = threadIdx.x;
    int64_t seg_first_tile = 0;  // first tile index of the current segment
    int64_t consumed = 0;

    for (int64_t w = w_begin; w < w_end; ++w, ++consumed) {
        const int64_t b = w / sch.n_tiles;
        const int64_t j = w % sch.n_tiles;
        if (w == w_begin || j == 0) {
            // new segment: this CTA's range enters target block b
            seg_first_tile = j;
            const int64_t base = b * kTargetsPerBlock + (int64_t)tid * kV;
            float bx[kV], by[kV], bz[kV];
#pragma unroll
            for (int v = 0; v < kV; ++v) {
                const int64_t t = base + v;
                const bool in = t < sch.n_targets;
                bx[v] = in ? args.tx[t] : 0.f;
                by[v] = in ? args.ty[t] : 0.f;
                bz[v] = in ? args.tz[t] : 0.f;
                sm.coord[v][tid] = bx[v];
                sm.coord[kV + v][tid] = by[v];
                sm.coord[2 * kV + v][tid] = bz[v];
                sm.run[v][tid] = 0.f;
                sm.run[kV + v][tid] = 0.f;
            }
            x0 = bx[0];
            y0 = by[0];
            z0 = bz[0];
            const int n_in = (int)(sch.n_targets - base < kV ? (sch.n_targets - base > 0 ? sch.n_targets - base : 0)
                                                             : kV);
            const bool spaced = equally_spaced(bx, n_in, sx) && equally_spaced(by, n_in, sy) &&
                                equally_spaced(bz, n_in, sz);
            // every lane executes every shuffle and vote (no short-circuit
            // around a full-mask warp primitive)
            const bool all_spaced = __all_sync(0xffffffffu, spaced);
            const float sx0 = __shfl_sync(0xffffffffu, sx, 0);
            const float sy0 = __shfl_sync(0xffffffffu, sy, 0);
            const float sz0 = __shfl_sync(0xffffffffu, sz, 0);
            const bool same_step = __all_sync(0xffffffffu, sx == sx0 && sy == sy0 && sz == sz0);
            strided = args.allow_strided && all_spaced;
            shared_u = strided && same_step;
            // the spacing the step records were evaluated for (pack_sources);
            // a thread with fewer than two targets has any spacing
            const bool common = with_steps && (n_in < 2 || (sx == launch_step(args.tx, sch.n_targets) &&
                                                             sy == launch_step(args.ty, sch.n_targets) &&
                                                             sz == launch_step(args.tz, sch.n_targets)));
            pre = strided && __all_sync(0xffffffffu, common);
        }

        const int st = (int)(consumed % kStages);
        if (!mbar_wait_bounded(&sm.full[st], (uint32_t)((consumed / kStages) & 1), args.status,
                               kStatusConsumerTimeout, args.wait_limit_ns))
            return;

        // Two-level accumulation: a fresh accumulator per tile, folded into the
        // running sum once per tile, keeps fp32 rounding growth at
        // O(sqrt(kTile) + sqrt(M / kTile)) instead of O(sqrt(M)).
        const float4* rec = &sm.ring[st][0];
        if (strided) {
            if constexpr (MODE == kFast) {
                strided_tile<MODE, kTwoChains, POLAR>(rec, x0, y0, z0, sx, sy, sz, lane, shared_u,
                                                      pre ? &sm.step[st][0] : nullptr, sm.run, tid);
            } else {
                f2_t acc[kV];
                if (POLAR && pre) {
                    if constexpr (POLAR) accumulate_tile_pre<MODE>(rec, &sm.step[st][0], x0, y0, z0, acc);
                } else if (shared_u)
                    accumulate_tile_strided_shared_u<MODE, POLAR>(rec, x0, y0, z0, sx, sy, sz, lane, acc);
                else
                    accumulate_tile_strided<MODE, kTwoChains, POLAR>(rec, x0, y0, z0, sx, sy, sz, acc);
#pragma unroll
                for (int v = 0; v < kV; ++v) {
                    float re, im;
                    f2_unpack(acc[v], re, im);
                    if (two_chain_negated(v)) {  // the accurate kernel always uses two chains
                        sm.run[v][tid] -= re;
                        sm.run[kV + v][tid] -= im;
                    } else {
                        sm.run[v][tid] += re;
                        sm.run[kV + v][tid] += im;
                    }
                }
            }
        } else {
            bool src_strided = args.allow_strided != 0;
#pragma unroll
            for (int q = 0; q < kTile / SEG; ++q)
                src_strided = src_strided && sm.desc[st][q].w != 0.f;
            if (src_strided) {
                if constexpr (MODE == kFast)
                    source_tile<MODE, SEG, POLAR>(rec, &sm.desc[st][0], sm.coord, sm.run, tid);
                else
                    accumulate_tile_src_strided_ool<MODE, SEG, POLAR>(rec, &sm.desc[st][0], sm.coord, sm.run, tid);
            } else {
                if constexpr (MODE == kFast)
                    direct_tile<MODE, NPOLY, POLAR>(rec, sm.coord, sm.run, tid);
                else
                    accumulate_tile_ool<MODE, NPOLY, POLAR>(rec, sm.coord, sm.run, tid);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[st]);

        if (w == w_end - 1 || j == sch.n_tiles - 1) {
            // end of segment: whole block -> output, else -> this CTA's partial slot
            const bool whole = (seg_first_tile == 0) && (j == sch.n_tiles - 1);
            const int64_t base = b * kTargetsPerBlock + (int64_t)tid * kV;
            if (whole) {
#pragma unroll
                for (int v = 0; v < kV; ++v) {
                    const int64_t t = base + v;
                    if (t < sch.n_targets) {
                        args.out_r[t] = sm.run[v][tid];
                        args.out_i[t] = sm.run[kV + v][tid];
                    }
                }
            } else {
                const int64_t slot = sch.slot(c, b);
                float* pr = args.partial + slot * (2 * kTargetsPerBlock);
                float* pi = pr + kTargetsPerBlock;
#pragma unroll
                for (int v = 0; v < kV; ++v) {
                    pr[tid * kV + v] = sm.run[v][tid];
                    pi[tid * kV + v] = sm.run[kV + v][tid];
                }
            }
        }
    }
}

// ---------------------------------------------------------------- fix-up
// kFixupSplit CTAs per CTA boundary c = 1..ctas-1, each summing one slice of
// kTargetsPerBlock / kFixupSplit targets.  A boundary strictly inside target
// block b means b was split; the lowest such boundary sums b's partial slots
// over the contributing CTAs c-1 .. c_hi in increasing order.
constexpr int kFixupSplit = 8;
constexpr int kFixupThreads = 256;
static_assert(kTargetsPerBlock % (4 * kFixupSplit) == 0, "fix-up slices are whole float4 groups");
__global__ void __launch_bounds__(kFixupThreads) fixup_kernel(const Schedule sch, const float* __restrict__ partial,
                                                              float* __restrict__ out_r, float* __restrict__ out_i,
                                                              const uint32_t* skip) {
    if (skip != nullptr && *skip != 0u) return;
    const int64_t c = (int64_t)blockIdx.x + 1;
    const int64_t b = sch.fixup_block(c);
    if (b < 0) return;
    const int64_t c_lo = c - 1;
    const int64_t c_hi = sch.last_contributor(c, b);
    constexpr int kSlice = kTargetsPerBlock / kFixupSplit;
    const int l_end = (int)(blockIdx.y + 1) * kSlice;
    for (int l = (int)blockIdx.y * kSlice + 4 * (int)threadIdx.x; l < l_end; l += 4 * kFixupThreads) {
        const int64_t t = b * kTargetsPerBlock + l;
        if (t >= sch.n_targets) break;
        // slot rows are whole blocks, so the float4 reads stay inside the slot
        float4 sr = make_float4(0.f, 0.f, 0.f, 0.f), si = sr;
        for (int64_t cc = c_lo; cc <= c_hi; ++cc) {
            const float* pr = partial + sch.slot(cc, b) * (2 * kTargetsPerBlock);
            const float4 a = *reinterpret_cast<const float4*>(pr + l);
            const float4 q = *reinterpret_cast<const float4*>(pr + kTargetsPerBlock + l);
            sr.x += a.x; sr.y += a.y; sr.z += a.z; sr.w += a.w;
            si.x += q.x; si.y += q.y; si.z += q.z; si.w += q.w;
        }
        const float vr[4] = {sr.x, sr.y, sr.z, sr.w}, vi[4] = {si.x, si.y, si.z, si.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (t + j < sch.n_targets) {
                out_r[t + j] = vr[j];
                out_i[t + j] = vi[j];
            }
    }
}

// ---------------------------------------------------------------- split gather
// Problems too small to occupy the persistent kernel (a few target blocks and
// source tiles, so most CTAs or most threads would idle) take this path: one
// target per thread, kSplitThreads targets per CTA along x, the sources split
// into n_slices equal slices along y.  Each CTA stages its slice through
// shared memory kSplitChunk sources at a time, read straight from the
// caller's arrays (no pack kernel on this path), and evaluates every pair
// directly (one phasor per pair, as on the pair-by-pair path); a slice's sums
// go to its own partial row, and split_reduce_kernel adds the rows in a fixed
// order (no atomics, bit-reproducible).  With one slice the CTA writes the
// output itself.
constexpr int kSplitThreads = 256;
constexpr int kSplitChunk = 256;

template <int MODE>
__global__ void __launch_bounds__(kSplitThreads) split_gather_kernel(
    const float* __restrict__ tx, const float* __restrict__ ty, const float* __restrict__ tz, int64_t n_targets,
    const float* __restrict__ ax, const float* __restrict__ ay, const float* __restrict__ az,
    const float* __restrict__ wr, const float* __restrict__ wi, float sign, int64_t n_sources, int64_t slice_len,
    float* __restrict__ partial, float* __restrict__ out_r, float* __restrict__ out_i, uint32_t* status,
    int reset_status, const uint32_t* skip) {
    if (skip != nullptr && *skip != 0u) return;
    if (reset_status && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *status = 0u;
    // a chunk of sources as (A.x, A.y, A.z) with A = sign * a, as
    // pack_sources stores them, and their weights
    __shared__ float4 rec[kSplitChunk];
    __shared__ float2 wrec[kSplitChunk];
    const int64_t t = (int64_t)blockIdx.x * kSplitThreads + threadIdx.x;
    const bool active = t < n_targets;
    const float bx = active ? tx[t] : 0.f, by = active ? ty[t] : 0.f, bz = active ? tz[t] : 0.f;
    const int64_t s0 = (int64_t)blockIdx.y * slice_len;
    const int64_t s1 = s0 + slice_len < n_sources ? s0 + slice_len : n_sources;
    float ar = 0.f, ai = 0.f;
    for (int64_t c0 = s0; c0 < s1; c0 += kSplitChunk) {
        const int n = (int)(s1 - c0 < kSplitChunk ? s1 - c0 : kSplitChunk);
        __syncthreads();  // the previous chunk is consumed
        for (int i = threadIdx.x; i < n; i += kSplitThreads) {
            const int64_t q = c0 + i;
            rec[i] = make_float4(sign * ax[q], sign * ay[q], sign * az[q], 0.f);
            wrec[i] = make_float2(wr[q], wi[q]);
        }
        __syncthreads();
#pragma unroll 4
        for (int s = 0; s < n; ++s) {
            const float4 r = rec[s];
            const float2 w = wrec[s];
            float sn, cs;
            if constexpr (MODE == kAccurate)
                phasor_accurate(r.x, r.y, r.z, bx, by, bz, sn, cs);
            else
                phasor_mufu(fmaf(r.z, bz, fmaf(r.y, by, r.x * bx)), sn, cs);
            ar = fmaf(w.x, cs, ar);
            ar = fmaf(-w.y, sn, ar);
            ai = fmaf(w.x, sn, ai);
            ai = fmaf(w.y, cs, ai);
        }
    }
    if (!active) return;
    if (gridDim.y == 1) {
        out_r[t] = ar;
        out_i[t] = ai;
    } else {
        partial[(2 * (int64_t)blockIdx.y) * n_targets + t] = ar;
        partial[(2 * (int64_t)blockIdx.y + 1) * n_targets + t] = ai;
    }
}

// out_t = sum over slices of partial row j, in a fixed order: 32 targets per
// CTA (one per lane); warp w adds slices w, w + kReduceWarps, ... in
// increasing order, then the kReduceWarps warp sums are added in warp order
// (no atomics, bit-reproducible).
constexpr int kReduceWarps = 8;
__global__ void __launch_bounds__(32 * kReduceWarps)
    split_reduce_kernel(const float* __restrict__ partial, int n_slices, int64_t n_targets,
                        float* __restrict__ out_r, float* __restrict__ out_i, const uint32_t* skip) {
    if (skip != nullptr && *skip != 0u) return;
    __shared__ float wr[kReduceWarps][32], wi[kReduceWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t = (int64_t)blockIdx.x * 32 + lane;
    float sr = 0.f, si = 0.f;
    if (t < n_targets) {
#pragma unroll 4
        for (int j = warp; j < n_slices; j += kReduceWarps) {
            sr += partial[(2 * (int64_t)j) * n_targets + t];
            si += partial[(2 * (int64_t)j + 1) * n_targets + t];
        }
    }
    wr[warp][lane] = sr;
    wi[warp][lane] = si;
    __syncthreads();
    if (warp == 0 && t < n_targets) {
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int w = 0; w < kReduceWarps; ++w) {
            a += wr[w][lane];
            b += wi[w][lane];
        }
        out_r[t] = a;
        out_i[t] = b;
    }
}

}  // namespace fhd
