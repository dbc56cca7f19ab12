// fhd_cg.cu - conjugate-gradient reconstruction on the device.
//
// Solves (F^H F + lambda I) rho = F^H D from rho = 0 with the loop of the host
// skeleton in "Case study - iterative MRI reconstruction", section 17.3.6
// (b = F^H D; r = p = b; per iteration Ap = F^H F p, alpha = rs_old / <p, Ap>,
// rho += alpha p, r -= alpha Ap, stop when rs_new < tol, p = r + beta p).  The
// Tikhonov term lambda I is the plainest reading of the regulariser R(rho) of
// section 17.2; lambda = 0 is the page's loop.
//
// Everything is enqueued on the caller's stream without a host round trip:
// the scalars (rs_old, <p, Ap>, alpha, beta) live in device memory, every dot
// product is a fixed-order two-pass fp64 reduction (bit-reproducible), and a
// device "done" word written when rs_new < tol makes every later kernel of the
// enqueued iterations (gathers included) return at once.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/fhd.h"
#include "fhd_host.h"

namespace {

using namespace fhd::host;

constexpr int kRedBlocks = 512;   // blocks of every reduction (fixed: fixed summation order)
constexpr int kRedThreads = 256;
constexpr size_t kStateOffset = 64;  // CgState inside the gather workspace header

struct CgState {
    double rs_old;
    double rs_new;
    double pap;
    double alpha;
    double beta;
    uint32_t done;        // 1 once the loop has stopped
    uint32_t iterations;  // completed iterations
    uint32_t breakdown;   // 1 if <p, Ap> was not positive and finite
    uint32_t pad;
};
static_assert(kStateOffset + sizeof(CgState) <= kHeaderBytes, "CG state must fit in the workspace header");

struct CgLayout {
    Layout gather;  // the F^H F workspace (header, records, partial slots, F rho)
    size_t r, p, ap, partial, total;
};

CgLayout cg_layout(int64_t N, int64_t M, int sms) {
    CgLayout L;
    L.gather = layout_for(FHD_OP_FHF, N, M, sms);
    const size_t vec = align_up((size_t)2 * (size_t)(N > 0 ? N : 1) * sizeof(float), kWsAlign);
    L.r = L.gather.total;
    L.p = L.r + vec;
    L.ap = L.p + vec;
    L.partial = L.ap + vec;
    L.total = L.partial + align_up(kRedBlocks * sizeof(double), kWsAlign);
    return L;
}

// Fixed-order block sum: each thread's grid-stride partial, then a shared
// memory tree; thread 0 returns the block's total.
__device__ double block_sum(double v) {
    __shared__ double red[kRedThreads];
    red[threadIdx.x] = v;
    __syncthreads();
    for (int s = kRedThreads / 2; s > 0; s >>= 1) {
        if ((int)threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
        __syncthreads();
    }
    return red[0];
}

__device__ double sum_partials(const double* partial) {
    double v = 0.0;
    for (int i = threadIdx.x; i < kRedBlocks; i += kRedThreads) v += partial[i];
    return block_sum(v);
}

// p = r (r already holds b = F^H D), rho = 0, partial sums of |r|^2.
__global__ void cg_start(int64_t n, const float* __restrict__ rr, const float* __restrict__ ri,
                         float* __restrict__ pr, float* __restrict__ pi, float* __restrict__ xr,
                         float* __restrict__ xi, double* __restrict__ partial) {
    double acc = 0.0;
    for (int64_t i = blockIdx.x * (int64_t)kRedThreads + threadIdx.x; i < n; i += (int64_t)kRedBlocks * kRedThreads) {
        const float a = rr[i], b = ri[i];
        pr[i] = a;
        pi[i] = b;
        xr[i] = 0.f;
        xi[i] = 0.f;
        acc += (double)a * a + (double)b * b;
    }
    const double s = block_sum(acc);
    if (threadIdx.x == 0) partial[blockIdx.x] = s;
}

__global__ void cg_start_finish(const double* __restrict__ partial, CgState* st) {
    const double rs = sum_partials(partial);
    if (threadIdx.x == 0) {
        st->rs_old = rs;
        st->rs_new = rs;
        st->pap = 0.0;
        st->alpha = 0.0;
        st->beta = 0.0;
        st->iterations = 0;
        st->breakdown = 0;
        st->done = (rs == 0.0) ? 1u : 0u;  // b = 0: rho = 0 is the solution
    }
}

// partial sums of Re <p, (A + lambda I) p> with A p in ap.
__global__ void cg_pap(int64_t n, const float* __restrict__ pr, const float* __restrict__ pi,
                       const float* __restrict__ ar, const float* __restrict__ ai, float lambda,
                       double* __restrict__ partial, const CgState* st) {
    if (st->done) return;
    double acc = 0.0;
    for (int64_t i = blockIdx.x * (int64_t)kRedThreads + threadIdx.x; i < n; i += (int64_t)kRedBlocks * kRedThreads) {
        const double a = pr[i], b = pi[i];
        acc += a * ((double)ar[i] + lambda * a) + b * ((double)ai[i] + lambda * b);
    }
    const double s = block_sum(acc);
    if (threadIdx.x == 0) partial[blockIdx.x] = s;
}

__global__ void cg_alpha(const double* __restrict__ partial, CgState* st) {
    if (st->done) return;
    const double pap = sum_partials(partial);
    if (threadIdx.x == 0) {
        st->pap = pap;
        if (!(pap > 0.0) || !isfinite(pap)) {
            st->breakdown = 1;
            st->done = 1;
        } else {
            st->alpha = st->rs_old / pap;
        }
    }
}

// rho += alpha p; r -= alpha (A p + lambda p); partial sums of |r|^2.
__global__ void cg_update(int64_t n, float* __restrict__ xr, float* __restrict__ xi, float* __restrict__ rr,
                          float* __restrict__ ri, const float* __restrict__ pr, const float* __restrict__ pi,
                          const float* __restrict__ ar, const float* __restrict__ ai, float lambda,
                          double* __restrict__ partial, const CgState* st) {
    if (st->done) return;
    const float alpha = (float)st->alpha;
    double acc = 0.0;
    for (int64_t i = blockIdx.x * (int64_t)kRedThreads + threadIdx.x; i < n; i += (int64_t)kRedBlocks * kRedThreads) {
        const float p0 = pr[i], p1 = pi[i];
        xr[i] = fmaf(alpha, p0, xr[i]);
        xi[i] = fmaf(alpha, p1, xi[i]);
        const float r0 = fmaf(-alpha, fmaf(lambda, p0, ar[i]), rr[i]);
        const float r1 = fmaf(-alpha, fmaf(lambda, p1, ai[i]), ri[i]);
        rr[i] = r0;
        ri[i] = r1;
        acc += (double)r0 * r0 + (double)r1 * r1;
    }
    const double s = block_sum(acc);
    if (threadIdx.x == 0) partial[blockIdx.x] = s;
}

__global__ void cg_beta(const double* __restrict__ partial, CgState* st, double tol) {
    if (st->done) return;
    const double rs = sum_partials(partial);
    if (threadIdx.x == 0) {
        st->rs_new = rs;
        st->iterations += 1;
        if (rs < tol) {
            st->done = 1;
        } else {
            st->beta = rs / st->rs_old;
            st->rs_old = rs;
        }
    }
}

// p = r + beta p.
__global__ void cg_direction(int64_t n, float* __restrict__ pr, float* __restrict__ pi, const float* __restrict__ rr,
                             const float* __restrict__ ri, const CgState* st) {
    if (st->done) return;
    const float beta = (float)st->beta;
    for (int64_t i = blockIdx.x * (int64_t)kRedThreads + threadIdx.x; i < n; i += (int64_t)kRedBlocks * kRedThreads) {
        pr[i] = fmaf(beta, pr[i], rr[i]);
        pi[i] = fmaf(beta, pi[i], ri[i]);
    }
}

}  // namespace

extern "C" {

size_t fhd_cg_workspace_bytes(int64_t N, int64_t M, int device) {
    if (N < 0 || M < 0) return 0;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return cg_layout(N, M, sms).total;
}

fhd_status fhd_cg_solve(int64_t M, const float* kx, const float* ky, const float* kz, const float* Dr,
                        const float* Di, int64_t N, const float* x, const float* y, const float* z, float lambda,
                        int max_iter, double tol, float* rho_r, float* rho_i, fhd_mode mode, void* workspace,
                        size_t workspace_bytes, fhd_stream_t stream_) {
    if (!(lambda >= 0.f) || !std::isfinite(lambda) || max_iter < 0 || !(tol >= 0.0)) return FHD_ERR_INVALID_VALUE;
    const size_t mb = (size_t)(N > 0 ? M : 0) * 4, nb = (size_t)N * 4;
    const Buf ins[] = {{kx, mb}, {ky, mb}, {kz, mb}, {Dr, mb}, {Di, mb}, {x, nb}, {y, nb}, {z, nb}};
    const Buf outs[] = {{rho_r, nb}, {rho_i, nb}};
    int device = -1;
    Layout gl;
    // validates sizes, pointers and aliasing against the F^H F part of the workspace
    fhd_status s = validate(FHD_OP_FHF, N, M, mode, ins, 8, outs, 2, workspace, workspace_bytes, &device, &gl);
    if (s != FHD_OK || device < 0) return s;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        cudaGetLastError();
        return FHD_ERR_CUDA;
    }
    const CgLayout L = cg_layout(N, M, sms);
    if (workspace_bytes < L.total) return FHD_ERR_WORKSPACE;
    const Buf wsb{workspace, L.total};
    for (const Buf& o : outs)
        if (overlaps(o, wsb)) return FHD_ERR_ALIAS;
    for (const Buf& i : ins)
        if (overlaps(i, wsb)) return FHD_ERR_ALIAS;
    if ((s = check_array(workspace, L.total, kWsAlign, device)) != FHD_OK) return s;

    cudaStream_t stream = (cudaStream_t)stream_;
    unsigned char* ws = (unsigned char*)workspace;
    CgState* st = reinterpret_cast<CgState*>(ws + kStateOffset);
    const uint32_t* done = &st->done;
    float* rr = reinterpret_cast<float*>(ws + L.r);
    float* ri = rr + N;
    float* pr = reinterpret_cast<float*>(ws + L.p);
    float* pi = pr + N;
    float* ar = reinterpret_cast<float*>(ws + L.ap);
    float* ai = ar + N;
    float* fr = reinterpret_cast<float*>(ws + gl.frho);
    float* fi = fr + (M > 0 ? M : 0);
    double* partial = reinterpret_cast<double*>(ws + L.partial);

    // b = F^H D into r
    GatherProblem adj_b{N, x, y, z, M, kx, ky, kz, Dr, Di, 1.0f, rr, ri};
    if ((s = run_gather(adj_b, mode, ws, gl, device, stream, nullptr, nullptr, -1, true, nullptr)) != FHD_OK)
        return s;
    cg_start<<<kRedBlocks, kRedThreads, 0, stream>>>(N, rr, ri, pr, pi, rho_r, rho_i, partial);
    cg_start_finish<<<1, kRedThreads, 0, stream>>>(partial, st);
    if (cudaGetLastError() != cudaSuccess) return FHD_ERR_CUDA;

    for (int it = 0; it < max_iter; ++it) {
        if (M > 0) {
            // Ap = F^H F p: forward gather into F rho, then the adjoint gather
            GatherProblem fwd{M, kx, ky, kz, N, x, y, z, pr, pi, -1.0f, fr, fi};
            if ((s = run_gather(fwd, mode, ws, gl, device, stream, nullptr, nullptr, -1, false, done)) != FHD_OK)
                return s;
            GatherProblem adj{N, x, y, z, M, kx, ky, kz, fr, fi, 1.0f, ar, ai};
            if ((s = run_gather(adj, mode, ws, gl, device, stream, nullptr, nullptr, -1, false, done)) != FHD_OK)
                return s;
        }
        cg_pap<<<kRedBlocks, kRedThreads, 0, stream>>>(N, pr, pi, ar, ai, lambda, partial, st);
        cg_alpha<<<1, kRedThreads, 0, stream>>>(partial, st);
        cg_update<<<kRedBlocks, kRedThreads, 0, stream>>>(N, rho_r, rho_i, rr, ri, pr, pi, ar, ai, lambda, partial,
                                                          st);
        cg_beta<<<1, kRedThreads, 0, stream>>>(partial, st, tol);
        cg_direction<<<kRedBlocks, kRedThreads, 0, stream>>>(N, pr, pi, rr, ri, st);
        if (cudaGetLastError() != cudaSuccess) return FHD_ERR_CUDA;
    }
    return FHD_OK;
}

fhd_status fhd_cg_info(const void* workspace, fhd_stream_t stream, int* iterations, double* residual,
                       int* stopped) {
    if (!workspace) return FHD_ERR_INVALID_VALUE;
    CgState st;
    uint32_t status = 0;
    cudaError_t e = cudaMemcpyAsync(&st, (const unsigned char*)workspace + kStateOffset, sizeof(st),
                                    cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&status, workspace, sizeof(status), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return FHD_ERR_CUDA;
    if (iterations) *iterations = (int)st.iterations;
    if (residual) *residual = st.rs_new;
    if (stopped) *stopped = st.breakdown ? -1 : (int)st.done;
    return status == 0 ? FHD_OK : FHD_ERR_TIMEOUT;
}

}  // extern "C"
