// fhd_api.cu - C ABI of the library: argument validation, workspace layout and
// kernel launches.  Declarations and the contract are in include/fhd.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/fhd.h"
#include "../../include/fhd_testing.h"
#include "fhd_host.h"
#include "fhd_kernels.cuh"

namespace fhd {
namespace host {

constexpr int kVersion = 100;  // 0.1.0

// Resident CTAs of the gather kernel on `device` (SMs x CTAs per SM), queried
// once per (device, mode) and cached: it depends only on the device and the
// compiled kernel.
constexpr int kCtaCacheDevices = 64;
std::atomic<int> g_ctas_cache[kCtaCacheDevices][2];  // 0: not yet queried

cudaError_t max_ctas(int device, fhd_mode mode, int* out) {
    const int fast = fast_mode(mode) ? 1 : 0;
    if (device >= 0 && device < kCtaCacheDevices) {
        const int cached = g_ctas_cache[device][fast].load(std::memory_order_relaxed);
        if (cached > 0) {
            *out = cached;
            return cudaSuccess;
        }
    }
    int sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    const size_t smem = sizeof(GatherSmem);
    if (fast)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, gather_kernel<kFast, kFastPolySlots, segment_len<kFast>(), kPolarAdjoint>, kCtaThreads, smem);
    else
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, gather_kernel<kAccurate, 0, segment_len<kAccurate>(), kPolarAdjoint>, kCtaThreads, smem);
    if (e != cudaSuccess) return e;
    per_sm = std::min(std::max(per_sm, 1), kMinCtasPerSm);
    *out = sms * per_sm;
    if (device >= 0 && device < kCtaCacheDevices) g_ctas_cache[device][fast].store(*out, std::memory_order_relaxed);
    return cudaSuccess;
}

// Workspace for a gather with up to `n_sources` sources, sized for the most
// CTAs any mode can launch on the device.
Layout layout_for(fhd_op op, int64_t N, int64_t M, int sms) {
    Layout L{};
    const int64_t max_sources = (op == FHD_OP_FHD) ? M : (op == FHD_OP_FWD) ? N : std::max(N, M);
    const int64_t padded = ceil_div(std::max<int64_t>(max_sources, 1), kTile) * kTile;
    const int64_t ctas = (int64_t)sms * kMinCtasPerSm;
    size_t off = kHeaderBytes;
    L.packed = off;
    off = align_up(off + (size_t)padded * kRecordBytes, kWsAlign);
    L.desc = off;
    off = align_up(off + (size_t)(padded / kSegment) * 16, kWsAlign);
    // step records of the adjoint gather, whose sources are the M samples
    L.steps = 0;
    if (op != FHD_OP_FWD) {
        L.steps = off;
        off = align_up(off + (size_t)(ceil_div(std::max<int64_t>(M, 1), kTile) * kTile) * 16, kWsAlign);
    }
    L.partial = off;
    off = align_up(off + (size_t)(2 * ctas) * 2 * kTargetsPerBlock * sizeof(float), kWsAlign);
    L.frho = off;
    if (op == FHD_OP_FHF) off = align_up(off + (size_t)2 * std::max<int64_t>(M, 1) * sizeof(float), kWsAlign);
    L.total = off;
    return L;
}

// ---------------------------------------------------------------- validation
typedef CUresult(CUDAAPI* PFN_range)(CUdeviceptr*, size_t*, CUdeviceptr);

bool overlaps(const Buf& a, const Buf& b) {
    if (a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

typedef CUresult(CUDAAPI* PFN_attrs)(unsigned int, CUpointer_attribute*, void**, CUdeviceptr);

// Device-memory, alignment and allocation-range checks for one array: one
// driver query (cuPointerGetAttributes) for the memory type, device,
// managed flag and the allocation's range; where that entry point cannot be
// resolved, the runtime's pointer attributes and cuMemGetAddressRange.
fhd_status check_array(const void* p, size_t bytes, size_t align, int device) {
    if (bytes == 0) return FHD_OK;
    if (p == nullptr) return FHD_ERR_INVALID_VALUE;
    if ((uintptr_t)p % align != 0) return FHD_ERR_MISALIGNED;
    // Driver entry point, resolved once per process (thread-safe static init).
    static const PFN_attrs attrs_fn = [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        const bool ok = cudaGetDriverEntryPointByVersion("cuPointerGetAttributes", &fn, 12000, cudaEnableDefault,
                                                         &q) == cudaSuccess &&
                        q == cudaDriverEntryPointSuccess;
        cudaGetLastError();
        return ok ? (PFN_attrs)fn : (PFN_attrs) nullptr;
    }();
    if (attrs_fn) {
        // each slot zeroed and wider than the value the driver writes into it
        unsigned long long memtype = 0, managed = 0, start = 0, size = 0;
        int ordinal = -1;
        CUpointer_attribute which[5] = {CU_POINTER_ATTRIBUTE_MEMORY_TYPE, CU_POINTER_ATTRIBUTE_DEVICE_ORDINAL,
                                        CU_POINTER_ATTRIBUTE_IS_MANAGED, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR,
                                        CU_POINTER_ATTRIBUTE_RANGE_SIZE};
        void* data[5] = {&memtype, &ordinal, &managed, &start, &size};
        // a pointer CUDA does not know gets zero attributes, not an error
        if (attrs_fn(5, which, data, (CUdeviceptr)(uintptr_t)p) != CUDA_SUCCESS) return FHD_ERR_INVALID_VALUE;
        if (managed == 0 && ((CUmemorytype)memtype != CU_MEMORYTYPE_DEVICE || ordinal != device))
            return FHD_ERR_INVALID_VALUE;
        if (size != 0 && (uintptr_t)p + bytes > (uintptr_t)start + size) return FHD_ERR_RANGE;
        return FHD_OK;
    }
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return FHD_ERR_INVALID_VALUE;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return FHD_ERR_INVALID_VALUE;
    if (attr.type == cudaMemoryTypeDevice && attr.device != device) return FHD_ERR_INVALID_VALUE;
    // Driver entry point, resolved once per process (thread-safe static init).
    static const PFN_range range_fn = [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        const bool ok = cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 12000, cudaEnableDefault,
                                                         &q) == cudaSuccess &&
                        q == cudaDriverEntryPointSuccess;
        cudaGetLastError();
        return ok ? (PFN_range)fn : (PFN_range) nullptr;
    }();
    if (range_fn) {
        CUdeviceptr base = 0;
        size_t size = 0;
        if (range_fn(&base, &size, (CUdeviceptr)(uintptr_t)p) == CUDA_SUCCESS) {
            if ((uintptr_t)p + bytes > (uintptr_t)base + size) return FHD_ERR_RANGE;
        }
    }
    return FHD_OK;
}

fhd_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FHD_OK : FHD_ERR_CUDA; }

// ---------------------------------------------------------------- launches
// Path override for the test-suite (fhd_test_set_path): 0 automatic,
// 1 always the persistent gather, 2 always the split gather.
std::atomic<int> g_test_path{0};
// Step records of the adjoint gather on (1) or off (fhd_test_set_step_records).
std::atomic<int> g_test_step_records{1};

// Shape of the split gather for n_targets x n_sources, and whether the
// persistent gather would leave more than half of the device's CTA thread
// slots idle (few work items, or target blocks mostly empty), in which case
// the split gather is used.  The slices fill about 8 CTAs of 256 threads per
// SM, hold at least kMinSliceSources sources each, and their partial rows fit
// the partial region of the workspace (partial_bytes).
SplitShape split_shape(int64_t n_targets, int64_t n_sources, int sms, int ctas_max, size_t partial_bytes) {
    constexpr int64_t kMinSliceSources = 32;
    SplitShape r{};
    const int64_t work = ceil_div(n_targets, kTargetsPerBlock) * ceil_div(n_sources, kTile);
    const int64_t busy_threads =
        std::min<int64_t>(work, ctas_max) *
        std::min<int64_t>(kThreads, ceil_div(std::min<int64_t>(n_targets, kTargetsPerBlock), kV));
    r.worth_it = 2 * busy_threads < (int64_t)ctas_max * kThreads;
    const int64_t chunks = ceil_div(n_targets, kSplitThreads);
    int64_t slices = ceil_div((int64_t)sms * 8, chunks);
    slices = std::min(slices, ceil_div(n_sources, kMinSliceSources));
    slices = std::min<int64_t>(slices, (int64_t)(partial_bytes / (2 * sizeof(float) * (size_t)n_targets)));
    slices = std::min<int64_t>(slices, 65535);
    if (slices < 2) slices = 1;
    r.slice_len = ceil_div(n_sources, slices);
    r.n_slices = (int)ceil_div(n_sources, r.slice_len);
    return r;
}

fhd_status run_gather(const GatherProblem& g, fhd_mode mode, unsigned char* ws, const Layout& L, int device,
                      cudaStream_t stream, cudaEvent_t ev_start, cudaEvent_t ev_stop, int64_t skip_tile,
                      bool first_pass, const uint32_t* skip) {
    if (g.n_targets == 0) return FHD_OK;
    if (g.n_sources == 0) {
        cudaError_t e = first_pass ? cudaMemsetAsync(ws, 0, sizeof(uint32_t), stream) : cudaSuccess;
        if (e == cudaSuccess) e = cudaMemsetAsync(g.out_r, 0, (size_t)g.n_targets * sizeof(float), stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(g.out_i, 0, (size_t)g.n_targets * sizeof(float), stream);
        return cuda_status(e);
    }
    int ctas_max = 0;
    cudaError_t e = max_ctas(device, mode, &ctas_max);
    if (e != cudaSuccess) return FHD_ERR_CUDA;

    Schedule sch;
    sch.n_targets = g.n_targets;
    sch.n_tiles = ceil_div(g.n_sources, kTile);
    sch.n_blocks = ceil_div(g.n_targets, kTargetsPerBlock);
    sch.work = sch.n_blocks * sch.n_tiles;
    sch.ctas = (int)std::min<int64_t>(ctas_max, sch.work);

    uint32_t* status = reinterpret_cast<uint32_t*>(ws);
    float4* packed = reinterpret_cast<float4*>(ws + L.packed);
    float* partial = reinterpret_cast<float*>(ws + L.partial);

    const int64_t padded = sch.n_tiles * kTile;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    const float sign = g.sign;  // phases in cycles in both modes

    const SplitShape split = split_shape(g.n_targets, g.n_sources, sms, ctas_max, L.frho - L.partial);
    bool use_split = split.worth_it;
    const int forced = g_test_path.load();
    if (forced == 1) use_split = false;
    if (forced == 2) use_split = true;
    if (skip_tile >= 0) use_split = false;  // the skipped tile belongs to the persistent schedule
    if (use_split) {
        // reads the caller's source arrays itself: no pack kernel
        if (ev_start && (e = cudaEventRecord(ev_start, stream)) != cudaSuccess) return FHD_ERR_CUDA;
        const dim3 grid((unsigned)ceil_div(g.n_targets, kSplitThreads), (unsigned)split.n_slices);
        if (fast_mode(mode))
            split_gather_kernel<kFast><<<grid, kSplitThreads, 0, stream>>>(
                g.tx, g.ty, g.tz, g.n_targets, g.sx, g.sy, g.sz, g.wr, g.wi, sign, g.n_sources, split.slice_len,
                partial, g.out_r, g.out_i, status, first_pass ? 1 : 0, skip);
        else
            split_gather_kernel<kAccurate><<<grid, kSplitThreads, 0, stream>>>(
                g.tx, g.ty, g.tz, g.n_targets, g.sx, g.sy, g.sz, g.wr, g.wi, sign, g.n_sources, split.slice_len,
                partial, g.out_r, g.out_i, status, first_pass ? 1 : 0, skip);
        if ((e = cudaGetLastError()) != cudaSuccess) return FHD_ERR_CUDA;
        if (split.n_slices > 1) {
            split_reduce_kernel<<<(unsigned)ceil_div(g.n_targets, 32), 32 * kReduceWarps, 0, stream>>>(
                partial, split.n_slices, g.n_targets, g.out_r, g.out_i, skip);
            if ((e = cudaGetLastError()) != cudaSuccess) return FHD_ERR_CUDA;
        }
        if (ev_stop && (e = cudaEventRecord(ev_stop, stream)) != cudaSuccess) return FHD_ERR_CUDA;
        return FHD_OK;
    }

    // polar weights in the adjoint gather (see pack_sources)
    const bool polar = kPolarAdjoint && g.sign > 0.f;
    const int pack_grid = (int)std::min<int64_t>(ceil_div(padded, 256), (int64_t)sms * 8);
    // step records for the target-side recurrence of the adjoint gather
    float4* steps = (polar && L.steps != 0 && g_test_step_records.load() != 0)
                        ? reinterpret_cast<float4*>(ws + L.steps)
                        : nullptr;
    pack_sources<<<pack_grid, 256, 0, stream>>>(g.sx, g.sy, g.sz, g.wr, g.wi, sign, polar ? 1 : 0, g.n_sources,
                                                padded, packed, g.tx, g.ty, g.tz, g.n_targets, steps, status,
                                                first_pass ? 1 : 0, skip);
    if ((e = cudaGetLastError()) != cudaSuccess) return FHD_ERR_CUDA;

    float4* desc = reinterpret_cast<float4*>(ws + L.desc);
    // The forward gather (voxel sources, sign -1) and accurate mode use
    // kSegmentAccurate-source segments, the fast adjoint gather kSegment.
    const bool long_segments = g.sign < 0.f || !fast_mode(mode);
    const int64_t n_segments = padded / (long_segments ? kSegmentAccurate : kSegment);
    const int desc_grid = (int)std::min<int64_t>(ceil_div(n_segments, 256), (int64_t)sms * 8);
    if (long_segments)
        describe_segments<kSegmentAccurate><<<desc_grid, 256, 0, stream>>>(g.sx, g.sy, g.sz, sign, g.n_sources,
                                                                           n_segments, desc, skip);
    else
        describe_segments<kSegment><<<desc_grid, 256, 0, stream>>>(g.sx, g.sy, g.sz, sign, g.n_sources, n_segments,
                                                                   desc, skip);
    if ((e = cudaGetLastError()) != cudaSuccess) return FHD_ERR_CUDA;

    GatherArgs a;
    a.sch = sch;
    a.tx = g.tx;
    a.ty = g.ty;
    a.tz = g.tz;
    a.packed = packed;
    a.desc = desc;
    a.steps = steps;
    a.out_r = g.out_r;
    a.out_i = g.out_i;
    a.partial = partial;
    a.status = status;
    a.wait_limit_ns = kWaitLimitNs;
    a.skip_tile = skip_tile;
    a.allow_strided = ((int)mode & FHD_MODE_DIRECT) ? 0 : 1;
    a.skip = skip;

    if (ev_start && (e = cudaEventRecord(ev_start, stream)) != cudaSuccess) return FHD_ERR_CUDA;
    const size_t smem = sizeof(GatherSmem);
    if (fast_mode(mode)) {
        if (g.sign < 0.f) {
            constexpr auto k = gather_kernel<kFast, kFastPolySlots, kSegmentAccurate, false>;
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            k<<<sch.ctas, kCtaThreads, smem, stream>>>(a);
        } else {
            constexpr auto k = gather_kernel<kFast, kFastPolySlots, kSegment, kPolarAdjoint>;
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            k<<<sch.ctas, kCtaThreads, smem, stream>>>(a);
        }
    } else {
        if (g.sign < 0.f) {
            constexpr auto k = gather_kernel<kAccurate, 0, kSegmentAccurate, false>;
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            k<<<sch.ctas, kCtaThreads, smem, stream>>>(a);
        } else {
            constexpr auto k = gather_kernel<kAccurate, 0, kSegmentAccurate, kPolarAdjoint>;
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            k<<<sch.ctas, kCtaThreads, smem, stream>>>(a);
        }
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return FHD_ERR_CUDA;
    if (sch.ctas > 1) {
        fixup_kernel<<<dim3(sch.ctas - 1, kFixupSplit), kFixupThreads, 0, stream>>>(sch, partial, g.out_r, g.out_i,
                                                                                     skip);
        if ((e = cudaGetLastError()) != cudaSuccess) return FHD_ERR_CUDA;
    }
    if (ev_stop && (e = cudaEventRecord(ev_stop, stream)) != cudaSuccess) return FHD_ERR_CUDA;
    return FHD_OK;
}



// Shared validation for the three operators.  `ins`/`outs` list every array.
fhd_status validate(fhd_op op, int64_t N, int64_t M, fhd_mode mode, const Buf* ins, int n_in, const Buf* outs,
                    int n_out, void* workspace, size_t workspace_bytes, int* device_out, Layout* L) {
    if (N < 0 || M < 0 || !valid_mode(mode)) return FHD_ERR_INVALID_VALUE;
    // int64 index arithmetic in the kernels stays far from overflow below 2^40 elements
    if (N > (int64_t(1) << 40) || M > (int64_t(1) << 40)) return FHD_ERR_INVALID_VALUE;
    // NULL checks first: they need no CUDA call
    for (int i = 0; i < n_in; ++i)
        if (ins[i].bytes && !ins[i].p) return FHD_ERR_INVALID_VALUE;
    for (int i = 0; i < n_out; ++i)
        if (outs[i].bytes && !outs[i].p) return FHD_ERR_INVALID_VALUE;
    for (int i = 0; i < n_in; ++i)
        if (ins[i].bytes && (uintptr_t)ins[i].p % 4) return FHD_ERR_MISALIGNED;
    for (int i = 0; i < n_out; ++i)
        if (outs[i].bytes && (uintptr_t)outs[i].p % 4) return FHD_ERR_MISALIGNED;
    const bool has_work = [&] {
        for (int i = 0; i < n_out; ++i)
            if (outs[i].bytes) return true;
        return false;
    }();
    if (has_work) {
        if (!workspace) return FHD_ERR_WORKSPACE;
        if ((uintptr_t)workspace % kWsAlign) return FHD_ERR_MISALIGNED;
    }
    for (int i = 0; i < n_out; ++i) {
        for (int j = 0; j < n_in; ++j)
            if (overlaps(outs[i], ins[j])) return FHD_ERR_ALIAS;
        for (int j = i + 1; j < n_out; ++j)
            if (overlaps(outs[i], outs[j])) return FHD_ERR_ALIAS;
    }
    if (!has_work) {
        *device_out = -1;
        return FHD_OK;
    }
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) {
        cudaGetLastError();
        return FHD_ERR_CUDA;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        cudaGetLastError();
        return FHD_ERR_CUDA;
    }
    *L = layout_for(op, N, M, sms);
    if (workspace_bytes < L->total) return FHD_ERR_WORKSPACE;
    const Buf wsb{workspace, L->total};
    for (int i = 0; i < n_out; ++i)
        if (overlaps(outs[i], wsb)) return FHD_ERR_ALIAS;
    for (int i = 0; i < n_in; ++i)
        if (overlaps(ins[i], wsb)) return FHD_ERR_ALIAS;
    fhd_status s;
    for (int i = 0; i < n_in; ++i)
        if ((s = check_array(ins[i].p, ins[i].bytes, 4, device)) != FHD_OK) return s;
    for (int i = 0; i < n_out; ++i)
        if ((s = check_array(outs[i].p, outs[i].bytes, 4, device)) != FHD_OK) return s;
    if ((s = check_array(workspace, L->total, kWsAlign, device)) != FHD_OK) return s;
    *device_out = device;
    return FHD_OK;
}

fhd_status fhd_compute_impl(int64_t M, const float* kx, const float* ky, const float* kz, const float* Dr,
                            const float* Di, int64_t N, const float* x, const float* y, const float* z,
                            float* rho_r, float* rho_i, fhd_mode mode, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1, int64_t skip_tile) {
    const size_t mb = (size_t)(N > 0 ? M : 0) * 4, nb = (size_t)N * 4;
    const Buf ins[] = {{kx, mb}, {ky, mb}, {kz, mb}, {Dr, mb}, {Di, mb}, {x, nb}, {y, nb}, {z, nb}};
    const Buf outs[] = {{rho_r, nb}, {rho_i, nb}};
    int device = -1;
    Layout L;
    fhd_status s = validate(FHD_OP_FHD, N, M, mode, ins, 8, outs, 2, workspace, workspace_bytes, &device, &L);
    if (s != FHD_OK || device < 0) return s;
    GatherProblem g{N, x, y, z, M, kx, ky, kz, Dr, Di, 1.0f, rho_r, rho_i};
    return run_gather(g, mode, (unsigned char*)workspace, L, device, stream, ev0, ev1, skip_tile);
}

}  // namespace host
}  // namespace fhd

using namespace fhd;
using namespace fhd::host;

extern "C" {

size_t fhd_workspace_bytes(fhd_op op, int64_t N, int64_t M, int device) {
    if (N < 0 || M < 0) return 0;
    if (op != FHD_OP_FHD && op != FHD_OP_FWD && op != FHD_OP_FHF) return 0;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return layout_for(op, N, M, sms).total;
}

fhd_status fhd_compute(int64_t M, const float* kx, const float* ky, const float* kz, const float* Dr,
                       const float* Di, int64_t N, const float* x, const float* y, const float* z, float* rho_r,
                       float* rho_i, fhd_mode mode, void* workspace, size_t workspace_bytes, fhd_stream_t stream) {
    return fhd_compute_impl(M, kx, ky, kz, Dr, Di, N, x, y, z, rho_r, rho_i, mode, workspace, workspace_bytes,
                            (cudaStream_t)stream, nullptr, nullptr, -1);
}

fhd_status fhd_compute_profiled(int64_t M, const float* kx, const float* ky, const float* kz, const float* Dr,
                                const float* Di, int64_t N, const float* x, const float* y, const float* z,
                                float* rho_r, float* rho_i, fhd_mode mode, void* workspace,
                                size_t workspace_bytes, fhd_stream_t stream, fhd_event_t gather_start,
                                fhd_event_t gather_stop) {
    return fhd_compute_impl(M, kx, ky, kz, Dr, Di, N, x, y, z, rho_r, rho_i, mode, workspace, workspace_bytes,
                            (cudaStream_t)stream, (cudaEvent_t)gather_start, (cudaEvent_t)gather_stop, -1);
}

fhd_status fwd_compute(int64_t N, const float* x, const float* y, const float* z, const float* rho_r,
                       const float* rho_i, int64_t M, const float* kx, const float* ky, const float* kz, float* Dr,
                       float* Di, fhd_mode mode, void* workspace, size_t workspace_bytes, fhd_stream_t stream) {
    const size_t nb = (size_t)(M > 0 ? N : 0) * 4, mb = (size_t)M * 4;
    const Buf ins[] = {{x, nb}, {y, nb}, {z, nb}, {rho_r, nb}, {rho_i, nb}, {kx, mb}, {ky, mb}, {kz, mb}};
    const Buf outs[] = {{Dr, mb}, {Di, mb}};
    int device = -1;
    Layout L;
    fhd_status s = validate(FHD_OP_FWD, N, M, mode, ins, 8, outs, 2, workspace, workspace_bytes, &device, &L);
    if (s != FHD_OK || device < 0) return s;
    GatherProblem g{M, kx, ky, kz, N, x, y, z, rho_r, rho_i, -1.0f, Dr, Di};
    return run_gather(g, mode, (unsigned char*)workspace, L, device, (cudaStream_t)stream, nullptr, nullptr, -1);
}

fhd_status fhfrho_apply(int64_t N, const float* x, const float* y, const float* z, const float* rho_r,
                        const float* rho_i, int64_t M, const float* kx, const float* ky, const float* kz,
                        float* out_r, float* out_i, fhd_mode mode, void* workspace, size_t workspace_bytes,
                        fhd_stream_t stream) {
    const size_t nb = (size_t)N * 4, mb = (size_t)(N > 0 ? M : 0) * 4;
    const Buf ins[] = {{x, nb}, {y, nb}, {z, nb}, {rho_r, nb}, {rho_i, nb}, {kx, mb}, {ky, mb}, {kz, mb}};
    const Buf outs[] = {{out_r, nb}, {out_i, nb}};
    int device = -1;
    Layout L;
    fhd_status s = validate(FHD_OP_FHF, N, M, mode, ins, 8, outs, 2, workspace, workspace_bytes, &device, &L);
    if (s != FHD_OK || device < 0) return s;
    unsigned char* ws = (unsigned char*)workspace;
    if (M == 0) {
        cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), (cudaStream_t)stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(out_r, 0, nb, (cudaStream_t)stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(out_i, 0, nb, (cudaStream_t)stream);
        return cuda_status(e);
    }
    float* fr = reinterpret_cast<float*>(ws + L.frho);
    float* fi = fr + M;
    // pass 1: F rho, gathered per sample (voxels are the sources, coordinates negated)
    GatherProblem g1{M, kx, ky, kz, N, x, y, z, rho_r, rho_i, -1.0f, fr, fi};
    s = run_gather(g1, mode, ws, L, device, (cudaStream_t)stream, nullptr, nullptr, -1);
    if (s != FHD_OK) return s;
    // pass 2: F^H (F rho), gathered per voxel
    GatherProblem g2{N, x, y, z, M, kx, ky, kz, fr, fi, 1.0f, out_r, out_i};
    return run_gather(g2, mode, ws, L, device, (cudaStream_t)stream, nullptr, nullptr, -1, false);
}

fhd_status fhd_workspace_status(const void* workspace, fhd_stream_t stream) {
    if (!workspace) return FHD_ERR_INVALID_VALUE;
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return FHD_ERR_CUDA;
    return word == 0 ? FHD_OK : FHD_ERR_TIMEOUT;
}

const char* fhd_status_string(fhd_status s) {
    switch (s) {
        case FHD_OK: return "ok";
        case FHD_ERR_INVALID_VALUE: return "invalid value (size, NULL pointer, mode, op or non-device memory)";
        case FHD_ERR_MISALIGNED: return "misaligned pointer (arrays need 4 bytes, workspace 256 bytes)";
        case FHD_ERR_ALIAS: return "an output overlaps an input, another output or the workspace";
        case FHD_ERR_WORKSPACE: return "workspace smaller than fhd_workspace_bytes()";
        case FHD_ERR_CUDA: return "CUDA runtime error";
        case FHD_ERR_TIMEOUT: return "kernel pipeline wait timed out";
        case FHD_ERR_RANGE: return "array extends past the end of its device allocation";
        case FHD_ERR_TOO_LARGE: return "problem exceeds the static scratch of fhd_compute_noalloc";
    }
    return "unknown status";
}

fhd_status fhd_launch_shape(int device, fhd_mode mode, int* ctas, int* threads, int* targets_per_thread,
                            int* tile_sources, int* stages) {
    if (!valid_mode(mode)) return FHD_ERR_INVALID_VALUE;
    int n = 0;
    if (max_ctas(device, mode, &n) != cudaSuccess) {
        cudaGetLastError();
        return FHD_ERR_INVALID_VALUE;
    }
    if (ctas) *ctas = n;
    if (threads) *threads = kThreads;
    if (targets_per_thread) *targets_per_thread = kV;
    if (tile_sources) *tile_sources = kTile;
    if (stages) *stages = kStages;
    return FHD_OK;
}

int fhd_version(void) { return kVersion; }

}  // extern "C"

// ---------------------------------------------------------------- no-allocation variant
// fhd_compute for callers that cannot allocate device memory (see include/fhd.h):
// the scratch that fhd_compute takes from the caller's workspace lives in this
// static device array instead.  Layout inside it is the same layout_for()
// layout fhd_compute uses, which fits because M and the resident CTA count are
// capped; everything the kernels read from it is written earlier in the same
// call (pack_sources, or on the small-problem path the split gather, clears
// the status word; pack_sources rewrites every record; each partial slot or
// row that a fix-up or reduction reads is written first by its CTA).
namespace {

// FHD_NOALLOC_SCRATCH_BYTES is the size for the default launch shape (8192
// targets per block); builds with other shape constants size the array for
// their own layout.
constexpr size_t kNoAllocLayoutBytes = kHeaderBytes + (size_t)FHD_NOALLOC_MAX_SAMPLES * kRecordBytes + kWsAlign +
                                       (size_t)FHD_NOALLOC_MAX_SAMPLES / kSegment * 16 + kWsAlign +
                                       (size_t)FHD_NOALLOC_MAX_SAMPLES * 16 + kWsAlign +
                                       (size_t)FHD_NOALLOC_MAX_CTAS * 2 * 2 * kTargetsPerBlock * sizeof(float);
constexpr size_t kNoAllocScratchBytes =
    FHD_NOALLOC_SCRATCH_BYTES > kNoAllocLayoutBytes ? FHD_NOALLOC_SCRATCH_BYTES : kNoAllocLayoutBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the static scratch on `device` (the current device):
// looked up once per device with cudaGetSymbolAddress, then cached.  In host
// code g_noalloc_scratch names a host-side stand-in, never the device array.
fhd_status noalloc_scratch(int device, void** out) {
    if (device < 0 || device >= kNoAllocMaxDevices) return FHD_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[device] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return FHD_ERR_CUDA;
        }
        g_noalloc_ptr[device] = p;
    }
    *out = g_noalloc_ptr[device];
    return FHD_OK;
}

}  // namespace

extern "C" {

fhd_status fhd_compute_noalloc(int64_t M, const float* kx, const float* ky, const float* kz, const float* Dr,
                               const float* Di, int64_t N, const float* x, const float* y, const float* z,
                               float* rho_r, float* rho_i, fhd_mode mode, fhd_stream_t stream) {
    if (N < 0 || M < 0 || !valid_mode(mode)) return FHD_ERR_INVALID_VALUE;
    if (M > FHD_NOALLOC_MAX_SAMPLES) return FHD_ERR_TOO_LARGE;
    if (N == 0) return FHD_OK;
    int device = 0, sms = 0;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        cudaGetLastError();
        return FHD_ERR_CUDA;
    }
    if ((int64_t)sms * kMinCtasPerSm > FHD_NOALLOC_MAX_CTAS) return FHD_ERR_TOO_LARGE;
    void* scratch = nullptr;
    const fhd_status s = noalloc_scratch(device, &scratch);
    if (s != FHD_OK) return s;
    return fhd_compute_impl(M, kx, ky, kz, Dr, Di, N, x, y, z, rho_r, rho_i, mode, scratch, kNoAllocScratchBytes,
                            (cudaStream_t)stream, nullptr, nullptr, -1);
}

}  // extern "C"

namespace fhd {
namespace {

// fhd_test_phasor: one thread per pair, the methods listed in fhd_testing.h.
__global__ void test_phasor_kernel(int which, int64_t n, const float* __restrict__ ax, const float* __restrict__ ay,
                                   const float* __restrict__ az, const float* __restrict__ bx,
                                   const float* __restrict__ by, const float* __restrict__ bz, float* __restrict__ s,
                                   float* __restrict__ c) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float sn = 0.f, cs = 0.f;
        const float p = fmaf(az[i], bz[i], fmaf(ay[i], by[i], ax[i] * bx[i]));
        const float t = p - rint_fma(p);
        switch (which) {
            case 0: phasor_accurate(ax[i], ay[i], az[i], bx[i], by[i], bz[i], sn, cs); break;
            case 1: phasor_mufu(p, sn, cs); break;
            case 2: sincos2pi_poly<false>(p, sn, cs); break;
            case 3: sincospif(2.0f * t, &sn, &cs); break;
            default: sincos2pi_poly<true>(t, sn, cs); break;
        }
        s[i] = sn;
        c[i] = cs;
    }
}

// fhd_test_fma2_rate: each thread steps kProbeChains independent packed
// chains x = x * m + a (fma.rn.f32x2) kProbeIters times, the work held in
// registers; 8 warps per CTA, two per scheduler as in the gather's consumers.
constexpr int kProbeThreads = 256;
constexpr int kProbeChains = 16;
constexpr int kProbeIters = 16384;
__device__ float g_probe_sink;

__global__ void __launch_bounds__(kProbeThreads, 1) fma2_probe_kernel(float m0) {
    f2_t x[kProbeChains];
    const f2_t m = f2_pack(m0, m0), a = f2_pack(1e-7f, 2e-7f);
#pragma unroll
    for (int k = 0; k < kProbeChains; ++k) x[k] = f2_pack(threadIdx.x * 1e-3f + k, 0.5f * k);
#pragma unroll 1
    for (int i = 0; i < kProbeIters; ++i) {
#pragma unroll
        for (int k = 0; k < kProbeChains; ++k) x[k] = f2_fma(x[k], m, a);
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kProbeChains; ++k) {
        float lo, hi;
        f2_unpack(x[k], lo, hi);
        s += lo + hi;
    }
    if (s == -1.0f) g_probe_sink = s;  // never true; keeps the chains live
}

}  // namespace
}  // namespace fhd

extern "C" {

// Declared in include/fhd_testing.h.
fhd_status fhd_test_fma2_rate(int device, double* lane_ops_per_s) {
    if (lane_ops_per_s == nullptr) return FHD_ERR_INVALID_VALUE;
    *lane_ops_per_s = 0.0;
    int prev = 0, sms = 0;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) return FHD_ERR_CUDA;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    float ms = 0.f;
    if (e == cudaSuccess) {
        fma2_probe_kernel<<<sms, kProbeThreads>>>(0.999f);  // warm-up
        cudaEventRecord(e0);
        fma2_probe_kernel<<<sms, kProbeThreads>>>(0.999f);
        cudaEventRecord(e1);
        e = cudaEventSynchronize(e1);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaSetDevice(prev);
    if (e != cudaSuccess || ms <= 0.f) return FHD_ERR_CUDA;
    *lane_ops_per_s = (double)sms * kProbeThreads * kProbeIters * kProbeChains * 2.0 / (ms * 1e-3);
    return FHD_OK;
}

// Declared in include/fhd_testing.h.
fhd_status fhd_test_phasor(int which, int64_t n, const float* ax, const float* ay, const float* az, const float* bx,
                           const float* by, const float* bz, float* s, float* c, fhd_stream_t stream) {
    if (which < 0 || which > 4 || n < 0) return FHD_ERR_INVALID_VALUE;
    if (n == 0) return FHD_OK;
    const size_t b = (size_t)n * sizeof(float);
    const Buf ins[] = {{ax, b}, {ay, b}, {az, b}, {bx, b}, {by, b}, {bz, b}};
    const Buf outs[] = {{s, b}, {c, b}};
    for (const Buf& o : outs)
        for (const Buf& in : ins)
            if (overlaps(o, in)) return FHD_ERR_ALIAS;
    if (overlaps(outs[0], outs[1])) return FHD_ERR_ALIAS;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) {
        cudaGetLastError();
        return FHD_ERR_CUDA;
    }
    fhd_status st;
    for (const Buf& a : ins)
        if ((st = check_array(a.p, a.bytes, 4, device)) != FHD_OK) return st;
    for (const Buf& a : outs)
        if ((st = check_array(a.p, a.bytes, 4, device)) != FHD_OK) return st;
    const int grid = (int)std::min<int64_t>(ceil_div(n, 256), 4096);
    test_phasor_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(which, n, ax, ay, az, bx, by, bz, s, c);
    return cuda_status(cudaGetLastError());
}

// Declared in include/fhd_testing.h.
fhd_status fhd_test_check_array(const void* p, size_t bytes, int device) {
    if (bytes == 0) return p ? check_array(p, 4, 4, device) : FHD_ERR_INVALID_VALUE;
    return check_array(p, bytes, 4, device);
}

// Declared in include/fhd_testing.h.
int fhd_test_set_path(int path) {
    if (path < 0 || path > 2) return -1;
    return g_test_path.exchange(path);
}

// Declared in include/fhd_testing.h.
int fhd_test_set_step_records(int enable) {
    if (enable != 0 && enable != 1) return -1;
    return g_test_step_records.exchange(enable);
}

// Declared in include/fhd_testing.h.
int fhd_test_split_shape(int64_t n_targets, int64_t n_sources, int sms, int ctas_max, size_t partial_bytes,
                         int* n_slices, int64_t* slice_len) {
    if (n_targets < 1 || n_sources < 1 || sms < 1 || ctas_max < 1) return -1;
    const SplitShape r = split_shape(n_targets, n_sources, sms, ctas_max, partial_bytes);
    if (n_slices) *n_slices = r.n_slices;
    if (slice_len) *slice_len = r.slice_len;
    return r.worth_it ? 1 : 0;
}

// Declared in include/fhd_testing.h.  Replays, on the host, the segment
// logic of gather_kernel and fixup_kernel over the Schedule methods they use.
int fhd_test_schedule(int64_t n_targets, int64_t n_sources, int ctas) {
    if (n_targets <= 0 || n_sources <= 0 || ctas <= 0) return 1;
    Schedule sch;
    sch.n_targets = n_targets;
    sch.n_tiles = ceil_div(n_sources, kTile);
    sch.n_blocks = ceil_div(n_targets, kTargetsPerBlock);
    sch.work = sch.n_blocks * sch.n_tiles;
    sch.ctas = (int)std::min<int64_t>(ctas, sch.work);
    if (sch.start(0) != 0 || sch.start(sch.ctas) != sch.work) return 2;
    std::vector<int> direct(sch.n_blocks, 0), fixed(sch.n_blocks, 0);
    // (cta, block) -> [first tile, last tile] of the partial segment in that slot
    std::vector<int64_t> slot_block(2 * (size_t)sch.ctas, -1), slot_lo(2 * (size_t)sch.ctas, -1),
        slot_hi(2 * (size_t)sch.ctas, -1);
    for (int64_t c = 0; c < sch.ctas; ++c) {
        const int64_t w0 = sch.start(c), w1 = sch.start(c + 1);
        if (w1 <= w0) return 3;  // every CTA owns at least one item
        int64_t seg_first = 0;
        for (int64_t w = w0; w < w1; ++w) {
            const int64_t b = w / sch.n_tiles, j = w % sch.n_tiles;
            if (w == w0 || j == 0) seg_first = j;
            if (w == w1 - 1 || j == sch.n_tiles - 1) {
                if (seg_first == 0 && j == sch.n_tiles - 1) {
                    direct[b]++;
                } else {
                    const int64_t sl = sch.slot(c, b);
                    if (sl < 2 * c || sl > 2 * c + 1) return 4;
                    if (slot_block[sl] != -1) return 5;  // slot written twice
                    slot_block[sl] = b;
                    slot_lo[sl] = seg_first;
                    slot_hi[sl] = j;
                }
            }
        }
    }
    for (int64_t c = 1; c < sch.ctas; ++c) {
        const int64_t b = sch.fixup_block(c);
        if (b < 0) continue;
        fixed[b]++;
        const int64_t hi = sch.last_contributor(c, b);
        int64_t next = 0;  // contributors' tile ranges must tile [0, n_tiles) in order
        for (int64_t cc = c - 1; cc <= hi; ++cc) {
            const int64_t sl = sch.slot(cc, b);
            if (slot_block[sl] != b) return 6;
            if (slot_lo[sl] != next) return 7;
            next = slot_hi[sl] + 1;
        }
        if (next != sch.n_tiles) return 8;
    }
    for (int64_t b = 0; b < sch.n_blocks; ++b)
        if (direct[b] + fixed[b] != 1) return 9;  // every block finished exactly once
    return 0;
}

fhd_status fhd_test_compute_skip_tile(int64_t M, const float* kx, const float* ky, const float* kz,
                                      const float* Dr, const float* Di, int64_t N, const float* x, const float* y,
                                      const float* z, float* rho_r, float* rho_i, fhd_mode mode, void* workspace,
                                      size_t workspace_bytes, fhd_stream_t stream, int64_t skip_tile) {
    return fhd_compute_impl(M, kx, ky, kz, Dr, Di, N, x, y, z, rho_r, rho_i, mode, workspace, workspace_bytes,
                            (cudaStream_t)stream, nullptr, nullptr, skip_tile);
}

}  // extern "C"
