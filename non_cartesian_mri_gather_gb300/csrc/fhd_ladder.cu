// fhd_ladder.cu - the optimisation ladder of the case study, for comparison.
//
// "Case study - iterative MRI reconstruction", sections 17.3.1-17.3.6, builds
// the F^H D gather up in steps and tabulates the speed of each (section
// 17.3.6); section 17.3.1 also describes, and rejects, the scatter form.  Each
// variant here computes the same sum as fhd_compute,
//
//     rho_n = sum_m D_m exp(+i 2 pi k_m . x_n),
//
// with that step's technique, written for this GPU only so the steps can be
// measured side by side.  They are comparison kernels, not the library's path:
//
//   L0  naive gather: one thread per voxel, samples read from global memory
//       (structure of arrays), phase 2 pi (k . x), libm cosf/sinf, and the sum
//       accumulated in rho in global memory inside the sample loop (the
//       global round trip per iteration that section 17.3.3 warns about)
//   L1  + loop fission / precompute (17.3.2): a separate kernel prepares
//       2 pi k, so the sample loop no longer multiplies by 2 pi
//   L2  + privatisation (17.3.3): accumulators in registers, rho written once
//   L3  + constant memory (17.3.4): samples as {kx, ky, kz, Dr, Di} records in
//       64 KB __constant__ chunks, one launch per chunk, read as broadcasts;
//       rho accumulates across chunks in global memory
//   L4  + __sincosf (17.3.5): hardware sin/cos approximations
//   L5  + unrolling by 4 (17.3.6, last row)
//   SC  scatter (17.3.1): one thread per sample adds its contribution to every
//       voxel with atomicAdd (order of the fp32 additions not fixed)
//
// L3 owns the library's one __constant__ array, so L3 calls must not overlap
// on the GPU.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/fhd.h"
#include "../../include/fhd_ladder.h"
#include "fhd_host.h"

namespace {

using namespace fhd::host;

constexpr float kTwoPi = 6.28318530717958647692f;
constexpr int kThreadsPerBlock = 256;

struct __align__(4) SampleRecord {
    float kx, ky, kz, dr, di;  // 20 bytes, as in the page's constant-memory record
};
constexpr int kChunk = 65536 / sizeof(SampleRecord);  // 3276 records in 64 KB
__constant__ SampleRecord c_samples[kChunk];

// L0 / L1: rho accumulated in global memory inside the loop.  `prescaled`
// selects whether k already carries the factor 2 pi (L1) or not (L0).
template <bool PRESCALED>
__global__ void ladder_global_acc(const float* kx, const float* ky, const float* kz, const float* dr,
                                  const float* di, const float* x, const float* y, const float* z, float* rho_r,
                                  float* rho_i, int m_count, int n_count) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= n_count) return;
    const float xn = x[n], yn = y[n], zn = z[n];
    rho_r[n] = 0.f;
    rho_i[n] = 0.f;
    for (int m = 0; m < m_count; ++m) {
        const float dot = kx[m] * xn + ky[m] * yn + kz[m] * zn;
        const float phi = PRESCALED ? dot : kTwoPi * dot;
        const float c = cosf(phi), s = sinf(phi);
        rho_r[n] += dr[m] * c - di[m] * s;  // may alias the inputs: a load and store per iteration
        rho_i[n] += dr[m] * s + di[m] * c;
    }
}

// L1 precompute pass: 2 pi k into separate arrays.
__global__ void ladder_prescale(const float* __restrict__ kx, const float* __restrict__ ky,
                                const float* __restrict__ kz, float* __restrict__ out, int m_count) {
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    if (m >= m_count) return;
    out[m] = kTwoPi * kx[m];
    out[m_count + m] = kTwoPi * ky[m];
    out[2 * m_count + m] = kTwoPi * kz[m];
}

// L2: privatised accumulators, prescaled k from the L1 pass.
__global__ void ladder_private(const float* __restrict__ kx2, const float* __restrict__ ky2,
                               const float* __restrict__ kz2, const float* __restrict__ dr,
                               const float* __restrict__ di, const float* __restrict__ x,
                               const float* __restrict__ y, const float* __restrict__ z, float* __restrict__ rho_r,
                               float* __restrict__ rho_i, int m_count, int n_count) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= n_count) return;
    const float xn = x[n], yn = y[n], zn = z[n];
    float ar = 0.f, ai = 0.f;
    for (int m = 0; m < m_count; ++m) {
        const float phi = kx2[m] * xn + ky2[m] * yn + kz2[m] * zn;
        const float c = cosf(phi), s = sinf(phi);
        ar += dr[m] * c - di[m] * s;
        ai += dr[m] * s + di[m] * c;
    }
    rho_r[n] = ar;
    rho_i[n] = ai;
}

// L3-L5: one constant-memory chunk of `count` records (2 pi already folded in);
// rho holds the sum over the earlier chunks.
template <bool INTRINSICS, int UNROLL>
__global__ void ladder_constant(const float* __restrict__ x, const float* __restrict__ y,
                                const float* __restrict__ z, float* __restrict__ rho_r, float* __restrict__ rho_i,
                                int count, int n_count, int first_chunk) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= n_count) return;
    const float xn = x[n], yn = y[n], zn = z[n];
    float ar = first_chunk ? 0.f : rho_r[n];
    float ai = first_chunk ? 0.f : rho_i[n];
#pragma unroll UNROLL
    for (int m = 0; m < count; ++m) {
        const SampleRecord r = c_samples[m];
        const float phi = r.kx * xn + r.ky * yn + r.kz * zn;
        float c, s;
        if (INTRINSICS) {
            __sincosf(phi, &s, &c);
        } else {
            c = cosf(phi);
            s = sinf(phi);
        }
        ar += r.dr * c - r.di * s;
        ai += r.dr * s + r.di * c;
    }
    rho_r[n] = ar;
    rho_i[n] = ai;
}

// Records for the constant-memory chunks: 2 pi k and D in AoS order.
__global__ void ladder_records(const float* __restrict__ kx, const float* __restrict__ ky,
                               const float* __restrict__ kz, const float* __restrict__ dr,
                               const float* __restrict__ di, SampleRecord* __restrict__ out, int m_count) {
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    if (m >= m_count) return;
    out[m] = SampleRecord{kTwoPi * kx[m], kTwoPi * ky[m], kTwoPi * kz[m], dr[m], di[m]};
}

__global__ void ladder_zero(float* __restrict__ a, float* __restrict__ b, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        a[i] = 0.f;
        b[i] = 0.f;
    }
}

// SC: one thread per sample, atomic adds into every voxel.
__global__ void ladder_scatter(const float* __restrict__ kx, const float* __restrict__ ky,
                               const float* __restrict__ kz, const float* __restrict__ dr,
                               const float* __restrict__ di, const float* __restrict__ x,
                               const float* __restrict__ y, const float* __restrict__ z, float* rho_r, float* rho_i,
                               int m_count, int n_count) {
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    if (m >= m_count) return;
    const float a = kTwoPi * kx[m], b = kTwoPi * ky[m], c = kTwoPi * kz[m], wr = dr[m], wi = di[m];
    for (int n = 0; n < n_count; ++n) {
        float s, co;
        __sincosf(a * x[n] + b * y[n] + c * z[n], &s, &co);
        atomicAdd(&rho_r[n], wr * co - wi * s);
        atomicAdd(&rho_i[n], wr * s + wi * co);
    }
}

int blocks_for(int64_t n) { return (int)((n + kThreadsPerBlock - 1) / kThreadsPerBlock); }

size_t variant_ws(fhd_variant v, int64_t M) {
    if (v == FHD_VARIANT_FISSION || v == FHD_VARIANT_PRIVATE) return align_up((size_t)3 * M * sizeof(float), 256);
    if (v == FHD_VARIANT_CONSTANT || v == FHD_VARIANT_INTRINSICS || v == FHD_VARIANT_UNROLL)
        return align_up((size_t)M * sizeof(SampleRecord), 256);
    return 0;
}

bool valid_variant(fhd_variant v) { return (int)v >= 0 && (int)v <= (int)FHD_VARIANT_SCATTER; }

}  // namespace

extern "C" {

size_t fhd_variant_workspace_bytes(fhd_variant v, int64_t N, int64_t M) {
    if (!valid_variant(v) || N < 0 || M < 0) return 0;
    const size_t b = variant_ws(v, M);
    return b ? b : 256;  // a non-empty size, so callers can always allocate it
}

fhd_status fhd_compute_variant(fhd_variant v, int64_t M, const float* kx, const float* ky, const float* kz,
                               const float* Dr, const float* Di, int64_t N, const float* x, const float* y,
                               const float* z, float* rho_r, float* rho_i, void* workspace, size_t workspace_bytes,
                               fhd_stream_t stream_) {
    if (!valid_variant(v) || N < 0 || M < 0) return FHD_ERR_INVALID_VALUE;
    if (N > INT32_MAX || M > INT32_MAX) return FHD_ERR_INVALID_VALUE;  // 32-bit indices, as on the page
    if (N == 0) return FHD_OK;
    const size_t mb = (size_t)M * 4, nb = (size_t)N * 4;
    const Buf ins[] = {{kx, mb}, {ky, mb}, {kz, mb}, {Dr, mb}, {Di, mb}, {x, nb}, {y, nb}, {z, nb}};
    const Buf outs[] = {{rho_r, nb}, {rho_i, nb}};
    const size_t need = variant_ws(v, M);
    if (need && (workspace == nullptr || workspace_bytes < need)) return FHD_ERR_WORKSPACE;
    const Buf wsb{workspace, need};
    for (int i = 0; i < 2; ++i) {
        for (const Buf& in : ins)
            if (overlaps(outs[i], in)) return FHD_ERR_ALIAS;
        if (overlaps(outs[i], wsb)) return FHD_ERR_ALIAS;
    }
    if (overlaps(outs[0], outs[1])) return FHD_ERR_ALIAS;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) {
        cudaGetLastError();
        return FHD_ERR_CUDA;
    }
    fhd_status s;
    for (const Buf& b : ins)
        if ((s = check_array(b.p, b.bytes, 4, device)) != FHD_OK) return s;
    for (const Buf& b : outs)
        if ((s = check_array(b.p, b.bytes, 4, device)) != FHD_OK) return s;
    if (need && (s = check_array(workspace, need, 256, device)) != FHD_OK) return s;

    cudaStream_t st = (cudaStream_t)stream_;
    const int n = (int)N, m = (int)M;
    const int gb = blocks_for(N);
    if (M == 0) {
        ladder_zero<<<gb, kThreadsPerBlock, 0, st>>>(rho_r, rho_i, n);
        return cuda_status(cudaGetLastError());
    }
    float* pre = reinterpret_cast<float*>(workspace);
    SampleRecord* rec = reinterpret_cast<SampleRecord*>(workspace);
    switch (v) {
        case FHD_VARIANT_NAIVE:
            ladder_global_acc<false><<<gb, kThreadsPerBlock, 0, st>>>(kx, ky, kz, Dr, Di, x, y, z, rho_r, rho_i, m, n);
            break;
        case FHD_VARIANT_FISSION:
            ladder_prescale<<<blocks_for(M), kThreadsPerBlock, 0, st>>>(kx, ky, kz, pre, m);
            ladder_global_acc<true><<<gb, kThreadsPerBlock, 0, st>>>(pre, pre + M, pre + 2 * M, Dr, Di, x, y, z,
                                                                     rho_r, rho_i, m, n);
            break;
        case FHD_VARIANT_PRIVATE:
            ladder_prescale<<<blocks_for(M), kThreadsPerBlock, 0, st>>>(kx, ky, kz, pre, m);
            ladder_private<<<gb, kThreadsPerBlock, 0, st>>>(pre, pre + M, pre + 2 * M, Dr, Di, x, y, z, rho_r,
                                                            rho_i, m, n);
            break;
        case FHD_VARIANT_CONSTANT:
        case FHD_VARIANT_INTRINSICS:
        case FHD_VARIANT_UNROLL: {
            ladder_records<<<blocks_for(M), kThreadsPerBlock, 0, st>>>(kx, ky, kz, Dr, Di, rec, m);
            for (int c0 = 0; c0 < m; c0 += kChunk) {
                const int cnt = (m - c0 < kChunk) ? (m - c0) : kChunk;
                cudaError_t e = cudaMemcpyToSymbolAsync(c_samples, rec + c0, (size_t)cnt * sizeof(SampleRecord), 0,
                                                        cudaMemcpyDeviceToDevice, st);
                if (e != cudaSuccess) return FHD_ERR_CUDA;
                const int first = c0 == 0;
                if (v == FHD_VARIANT_CONSTANT)
                    ladder_constant<false, 1><<<gb, kThreadsPerBlock, 0, st>>>(x, y, z, rho_r, rho_i, cnt, n, first);
                else if (v == FHD_VARIANT_INTRINSICS)
                    ladder_constant<true, 1><<<gb, kThreadsPerBlock, 0, st>>>(x, y, z, rho_r, rho_i, cnt, n, first);
                else
                    ladder_constant<true, 4><<<gb, kThreadsPerBlock, 0, st>>>(x, y, z, rho_r, rho_i, cnt, n, first);
            }
            break;
        }
        case FHD_VARIANT_SCATTER:
            ladder_zero<<<gb, kThreadsPerBlock, 0, st>>>(rho_r, rho_i, n);
            ladder_scatter<<<blocks_for(M), kThreadsPerBlock, 0, st>>>(kx, ky, kz, Dr, Di, x, y, z, rho_r, rho_i, m,
                                                                       n);
            break;
    }
    return cuda_status(cudaGetLastError());
}

}  // extern "C"
