// Host-side declarations shared by the translation units of libwtconv (not part of the
// public C ABI; that lives in include/wtconv.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stddef.h>

#include "wtconv.h"

namespace wt {

// TMA element type of an I/O dtype.
template <typename T>
inline CUtensorMapDataType tma_dtype();
template <>
inline CUtensorMapDataType tma_dtype<float>() { return CU_TENSOR_MAP_DATA_TYPE_FLOAT32; }
template <>
inline CUtensorMapDataType tma_dtype<__nv_bfloat16>() { return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; }
template <>
inline CUtensorMapDataType tma_dtype<__half>() { return CU_TENSOR_MAP_DATA_TYPE_FLOAT16; }

// Calls f(T{}) with T the element type of the I/O dtype (float, bfloat16 or half).
template <typename F>
auto with_io_type(wt_dtype io, F&& f) {
    switch (io) {
        case WT_BF16: return f(__nv_bfloat16{});
        case WT_F16: return f(__half{});
        default: return f(float{});
    }
}

// A plane side padded with zeros up to a multiple of 2^L: the kernels run every level on
// the padded plane, which equals zero-padding each odd carrier by one row / column before
// its analysis and cropping each synthesis output (only the H x W outputs are stored).
inline int padded_side(int n, int levels) {
    const int m = 1 << levels;
    return (n + m - 1) / m * m;
}

// Bytes per element of an I/O dtype.
inline size_t io_bytes(wt_dtype io) { return io == WT_F32 ? 4 : 2; }

// The first 256 bytes of every workspace: one status word per kind of call (set by the
// plane kernel when one of its bounded waits timed out), each followed by that call's plane
// counter; a launch clears only its own pair, so wtconv_workspace_status can report the
// most recent call of each kind.
constexpr int kStatusForward = 0;         // words 0, 1
constexpr int kStatusBackwardData = 2;    // words 2, 3
constexpr int kStatusBackwardWeight = 4;  // words 4, 5
constexpr size_t kStatusBytes = 256;

// Limit of every bounded wait inside the kernels, in nanoseconds of %globaltimer (1 s
// unless a test shortened it with wtconv_testing_set_wait_limit_ns).
unsigned long long wait_limit_ns();

// sm_103a: 227 KB of shared memory per block (opt-in), 152 SMs.
constexpr size_t kMaxSmemPerBlock = 227 * 1024;
constexpr int kNumSMs = 152;

// forward (flip = 0) and backward-data (flip = 1, no bias): one persistent launch; the
// workspace holds one deep-level scratch slot per CTA (none when L < 2)
wt_status launch_forward(const wt_desc& d, const void* x, const float* w0f, const float* b0f,
                         const float* wlf, void* y, int flip, void* ws, size_t ws_bytes,
                         cudaStream_t stream, int* launches);
bool forward_sizes(const wt_desc& d, size_t* smem, size_t* ws);

// per-phase clocks of the two plane kernels (32 counters each; only in a library built with
// -DWT_PHASE_CLOCKS, else WT_ERR_UNSUPPORTED)
wt_status phase_clocks_forward(int reset, unsigned long long* out);
wt_status phase_clocks_backward_weight(int reset, unsigned long long* out);

// backward-weight: plane kernel + reduce/unfold kernel
wt_status launch_backward_weight(const wt_desc& d, const void* x, const void* dy,
                                 const float* w0, const float* b0, const float* s0,
                                 const float* wl, const float* sl, float* dw0, float* db0,
                                 float* ds0, float* dwl, float* dsl, void* ws, size_t ws_bytes,
                                 cudaStream_t stream, int* launches);
size_t backward_weight_ws_bytes(const wt_desc& d);
// pieces of the backward-weight path: the per-plane partial kernel alone (partials
// [C][d.n][KP] to `part`; its CTAs' level-2 scratch slots, backward_weight_slot_bytes each,
// in [slots, slots + slots_bytes), the grid shrinking to the slots that fit; err[0] is
// set on a timed-out wait and err[1] is the plane counter, zero before the launch; err may
// be null) and the reduce + unfold kernel alone over [C][groups][KP] (NaN gradients when
// err is non-null and *err != 0)
wt_status launch_dw_partials(const wt_desc& d, const void* x, const void* dy, float* part,
                             float* slots, size_t slots_bytes, int* err, cudaStream_t stream,
                             int* launches);
size_t backward_weight_slot_bytes(const wt_desc& d);
wt_status launch_dw_reduce(const wt_desc& d, const float* part, int groups, const float* w0,
                           const float* b0, const float* s0, const float* wl, const float* sl,
                           float* dw0, float* db0, float* ds0, float* dwl, float* dsl,
                           const int* err, cudaStream_t stream, int* launches);
size_t dw_partial_floats(const wt_desc& d);
size_t backward_weight_smem_bytes(const wt_desc& d);

// 3-D tiled TMA tensor map: dims {d0, d1, d2}, byte strides {s1, s2}, box {b0, b1, 1};
// reads outside the tensor return zeros. False when the driver cannot encode it.
bool encode_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, unsigned long long d0,
               unsigned long long d1, unsigned long long d2, unsigned long long s1_bytes,
               unsigned long long s2_bytes, unsigned b0, unsigned b1);

// number of kernel launches of the calling thread's last successful entry-point call
void set_last_launch_count(int launches);

// scale folding (Eq. 8): one launch
wt_status launch_fold(const wt_desc& d, const float* w0, const float* b0, const float* s0,
                      const float* wl, const float* sl, float* w0f, float* b0f, float* wlf,
                      cudaStream_t stream, int* launches);

}  // namespace wt
