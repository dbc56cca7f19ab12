// fhd_host.h - host-side helpers shared by the library's translation units:
// argument validation, workspace layout and the gather launch sequence.
// Internal: not part of the C ABI (include/fhd.h).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/fhd.h"

namespace fhd {
namespace host {

constexpr size_t kWsAlign = 256;
constexpr size_t kHeaderBytes = 256;              // status word + reserved
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per pipeline wait

constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Mode word: bit 0 selects fast sin/cos, bit 1 (FHD_MODE_DIRECT) disables the
// equal-spacing recurrence.
inline bool valid_mode(fhd_mode m) { return ((int)m & ~3) == 0; }
inline bool fast_mode(fhd_mode m) { return ((int)m & FHD_MODE_FAST) != 0; }

struct Layout {
    size_t packed;   // offset of packed source records
    size_t desc;     // offset of the per-segment descriptors of the packed records
    size_t steps;    // offset of the adjoint gather's step records (0: none, the forward-only layout)
    size_t partial;  // offset of per-CTA partial slots
    size_t frho;     // offset of F rho (fhfrho_apply only)
    size_t total;
};

struct Buf {
    const void* p;
    size_t bytes;
};

// One gather: out_t = sum_s w_s exp(+i 2 pi (sign * a_s) . b_t).
struct GatherProblem {
    int64_t n_targets;
    const float *tx, *ty, *tz;
    int64_t n_sources;
    const float *sx, *sy, *sz, *wr, *wi;
    float sign;  // +1: adjoint kernel; -1: forward (source coordinates negated)
    float *out_r, *out_i;
};

Layout layout_for(fhd_op op, int64_t N, int64_t M, int sms);

// Launch shape of the split gather (small problems).
struct SplitShape {
    bool worth_it;     // the persistent gather would leave most thread slots idle
    int n_slices;      // source slices (grid y); 1 writes the output directly
    int64_t slice_len; // sources per slice (the last may be shorter)
};
SplitShape split_shape(int64_t n_targets, int64_t n_sources, int sms, int ctas_max, size_t partial_bytes);
fhd_status cuda_status(cudaError_t e);
bool overlaps(const Buf& a, const Buf& b);
fhd_status check_array(const void* p, size_t bytes, size_t align, int device);

// Shared argument checks; on success *device_out is the current device, or -1
// when there is nothing to compute, and *L the workspace layout of `op`.
fhd_status validate(fhd_op op, int64_t N, int64_t M, fhd_mode mode, const Buf* ins, int n_in, const Buf* outs,
                    int n_out, void* workspace, size_t workspace_bytes, int* device_out, Layout* L);

// Enqueue one gather on `stream`: pack, describe, the persistent gather and
// its fix-up; or, for problems too small to fill the persistent CTAs (see
// split_shape), the split gather and its slice reduction.  `skip`, when
// not NULL, is a device word: if it is non-zero when the kernels start they
// return at once (used to stop a conjugate-gradient loop on the device).
fhd_status run_gather(const GatherProblem& g, fhd_mode mode, unsigned char* ws, const Layout& L, int device,
                      cudaStream_t stream, cudaEvent_t ev_start, cudaEvent_t ev_stop, int64_t skip_tile,
                      bool first_pass = true, const uint32_t* skip = nullptr);

}  // namespace host
}  // namespace fhd
