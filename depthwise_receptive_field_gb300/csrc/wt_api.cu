// C ABI of libwtconv: argument validation, workspace sizing, the scale-folding kernel
// (§4.3 Eq. 8 of "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
// Reformulation") and dispatch to the forward / backward kernels.
#include <stdint.h>

#include <atomic>

#include "wt_common.cuh"
#include "wt_internal.h"
#include "wt_tma.cuh"
#include "wtconv_debug.h"
#include "wtconv_testing.h"

namespace wt {

namespace {

thread_local int g_last_launches = 0;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

wt_status check_desc(const wt_desc* d) {
    if (d == nullptr) return WT_ERR_INVALID_ARG;
    if (d->n < 1 || d->c < 1 || d->h < 1 || d->w < 1) return WT_ERR_INVALID_ARG;
    if (d->io != WT_F32 && d->io != WT_BF16 && d->io != WT_F16) return WT_ERR_INVALID_ARG;
    if (d->k < 1 || (d->k % 2) == 0) return WT_ERR_INVALID_ARG;
    if (d->levels < 0 || d->levels > kMaxLevels) return WT_ERR_INVALID_ARG;
    if ((size_t)d->n * d->c > 0x7fffffffull) return WT_ERR_INVALID_ARG;  // grid limit
    if (d->k > 7) return WT_ERR_UNSUPPORTED;
    return WT_OK;
}

wt_status check_io(const void* p) {
    if (p == nullptr || !aligned(p, 16)) return WT_ERR_INVALID_ARG;
    return WT_OK;
}

wt_status check_param(const void* p) {
    if (p == nullptr || !aligned(p, 4)) return WT_ERR_INVALID_ARG;
    return WT_OK;
}

}  // namespace

void set_last_launch_count(int launches) { g_last_launches = launches; }

namespace {
std::atomic<unsigned long long> g_wait_limit_ns{0};  // 0: the default
}  // namespace

unsigned long long wait_limit_ns() {
    const unsigned long long v = g_wait_limit_ns.load(std::memory_order_relaxed);
    return v == 0 ? kWaitLimitNs : v;
}

// §4.3 Eq. 8: one thread per folded weight (plus the bias fold).
__global__ void wt_fold_kernel(int C, int KK, int L, const float* w0, const float* b0,
                               const float* s0, const float* wl, const float* sl, float* w0f,
                               float* b0f, float* wlf) {
    const size_t n0 = (size_t)C * KK, nl = (size_t)L * C * 4 * KK;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n0 + nl + C;
         e += (size_t)gridDim.x * blockDim.x) {
        if (e < n0) {
            w0f[e] = s0[e / KK] * w0[e];
        } else if (e < n0 + nl) {
            const size_t q = e - n0;
            wlf[q] = sl[q / KK] * wl[q];
        } else if (b0f != nullptr) {
            const size_t c = e - n0 - nl;
            b0f[c] = b0 ? s0[c] * b0[c] : 0.f;
        }
    }
}

wt_status launch_fold(const wt_desc& d, const float* w0, const float* b0, const float* s0,
                      const float* wl, const float* sl, float* w0f, float* b0f, float* wlf,
                      cudaStream_t stream, int* launches) {
    const int KK = d.k * d.k;
    const size_t total = (size_t)d.c * KK + (size_t)d.levels * d.c * 4 * KK + d.c;
    const unsigned blocks = (unsigned)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    wt_fold_kernel<<<blocks, 256, 0, stream>>>(d.c, KK, d.levels, w0, b0, s0, wl, sl, w0f, b0f,
                                               wlf);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    ++*launches;
    return WT_OK;
}

}  // namespace wt

using namespace wt;

extern "C" {

wt_status wtconv_workspace_size(const wt_desc* desc, size_t* fwd, size_t* bwd_data,
                                size_t* bwd_weight) {
    wt_status st = check_desc(desc);
    if (st != WT_OK) return st;
    size_t fsmem = 0, fws = 0;
    if (!forward_sizes(*desc, &fsmem, &fws)) return WT_ERR_UNSUPPORTED;
    if (fsmem > kMaxSmemPerBlock) return WT_ERR_UNSUPPORTED;
    if (backward_weight_smem_bytes(*desc) > kMaxSmemPerBlock) return WT_ERR_UNSUPPORTED;
    if (fwd) *fwd = fws;
    if (bwd_data) *bwd_data = fws;
    if (bwd_weight) *bwd_weight = backward_weight_ws_bytes(*desc);
    return WT_OK;
}

wt_status wtconv_fold_scales(const wt_desc* desc, const float* w0, const float* b0,
                             const float* s0, const float* wl, const float* sl, float* w0f,
                             float* b0f, float* wlf, wt_stream_t stream) {
    wt_status st = check_desc(desc);
    if (st != WT_OK) return st;
    if (check_param(w0) || check_param(s0) || check_param(w0f)) return WT_ERR_INVALID_ARG;
    if (b0 && !aligned(b0, 4)) return WT_ERR_INVALID_ARG;
    if (b0f && !aligned(b0f, 4)) return WT_ERR_INVALID_ARG;
    if (desc->levels > 0 && (check_param(wl) || check_param(sl) || check_param(wlf)))
        return WT_ERR_INVALID_ARG;
    int launches = 0;
    st = launch_fold(*desc, w0, b0, s0, wl, sl, w0f, b0f, wlf,
                     reinterpret_cast<cudaStream_t>(stream), &launches);
    if (st == WT_OK) g_last_launches = launches;
    return st;
}

wt_status wtconv_forward(const wt_desc* desc, const void* x, const float* w0f,
                         const float* b0f, const float* wlf, void* y, void* ws,
                         size_t ws_bytes, wt_stream_t stream) {
    wt_status st = check_desc(desc);
    if (st != WT_OK) return st;
    if (check_io(x) || check_io(y) || check_param(w0f)) return WT_ERR_INVALID_ARG;
    if (ws && !aligned(ws, 256)) return WT_ERR_INVALID_ARG;
    if (b0f && !aligned(b0f, 4)) return WT_ERR_INVALID_ARG;
    if (desc->levels > 0 && check_param(wlf)) return WT_ERR_INVALID_ARG;
    int launches = 0;
    st = launch_forward(*desc, x, w0f, b0f, wlf, y, 0, ws, ws_bytes,
                        reinterpret_cast<cudaStream_t>(stream), &launches);
    if (st == WT_OK) g_last_launches = launches;
    return st;
}

wt_status wtconv_backward_data(const wt_desc* desc, const void* dy, const float* w0f,
                               const float* wlf, void* dx, void* ws, size_t ws_bytes,
                               wt_stream_t stream) {
    wt_status st = check_desc(desc);
    if (st != WT_OK) return st;
    if (check_io(dy) || check_io(dx) || check_param(w0f)) return WT_ERR_INVALID_ARG;
    if (ws && !aligned(ws, 256)) return WT_ERR_INVALID_ARG;
    if (desc->levels > 0 && check_param(wlf)) return WT_ERR_INVALID_ARG;
    int launches = 0;
    st = launch_forward(*desc, dy, w0f, nullptr, wlf, dx, 1, ws, ws_bytes,
                        reinterpret_cast<cudaStream_t>(stream), &launches);
    if (st == WT_OK) g_last_launches = launches;
    return st;
}

wt_status wtconv_backward_weight(const wt_desc* desc, const void* x, const void* dy,
                                 const float* w0, const float* b0, const float* s0,
                                 const float* wl, const float* sl, float* dw0, float* db0,
                                 float* ds0, float* dwl, float* dsl, void* ws,
                                 size_t ws_bytes, wt_stream_t stream) {
    wt_status st = check_desc(desc);
    if (st != WT_OK) return st;
    if (check_io(x) || check_io(dy)) return WT_ERR_INVALID_ARG;
    if (check_param(w0) || check_param(s0) || check_param(dw0) || check_param(ds0))
        return WT_ERR_INVALID_ARG;
    if ((b0 && !aligned(b0, 4)) || (db0 && !aligned(db0, 4))) return WT_ERR_INVALID_ARG;
    if (desc->levels > 0 &&
        (check_param(wl) || check_param(sl) || check_param(dwl) || check_param(dsl)))
        return WT_ERR_INVALID_ARG;
    if (ws && !aligned(ws, 256)) return WT_ERR_INVALID_ARG;
    if (ws_bytes < backward_weight_ws_bytes(*desc) || ws == nullptr) return WT_ERR_WORKSPACE;
    int launches = 0;
    st = launch_backward_weight(*desc, x, dy, w0, b0, s0, wl, sl, dw0, db0, ds0, dwl, dsl, ws,
                                ws_bytes, reinterpret_cast<cudaStream_t>(stream), &launches);
    if (st == WT_OK) g_last_launches = launches;
    return st;
}

wt_status wtconv_backward(const wt_desc* desc, const void* x, const void* dy,
                          const float* w0f, const float* wlf, const float* w0,
                          const float* b0, const float* s0, const float* wl, const float* sl,
                          void* dx, float* dw0, float* db0, float* ds0, float* dwl,
                          float* dsl, void* ws, size_t ws_bytes, wt_stream_t stream) {
    wt_status st = check_desc(desc);
    if (st != WT_OK) return st;
    if (check_io(x) || check_io(dy) || check_io(dx) || check_param(w0f)) return WT_ERR_INVALID_ARG;
    if (check_param(w0) || check_param(s0) || check_param(dw0) || check_param(ds0))
        return WT_ERR_INVALID_ARG;
    if ((b0 && !aligned(b0, 4)) || (db0 && !aligned(db0, 4))) return WT_ERR_INVALID_ARG;
    if (desc->levels > 0 && (check_param(wlf) || check_param(wl) || check_param(sl) ||
                             check_param(dwl) || check_param(dsl)))
        return WT_ERR_INVALID_ARG;
    if (ws && !aligned(ws, 256)) return WT_ERR_INVALID_ARG;
    if (ws_bytes < backward_weight_ws_bytes(*desc) || ws == nullptr) return WT_ERR_WORKSPACE;
    int launches = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = launch_forward(*desc, dy, w0f, nullptr, wlf, dx, 1, ws, ws_bytes, s, &launches);
    if (st != WT_OK) return st;
    st = launch_backward_weight(*desc, x, dy, w0, b0, s0, wl, sl, dw0, db0, ds0, dwl, dsl, ws,
                                ws_bytes, s, &launches);
    if (st == WT_OK) g_last_launches = launches;
    return st;
}

wt_status wtconv_workspace_status(const void* ws, wt_stream_t stream, int* flags) {
    if (flags) *flags = 0;
    if (ws == nullptr) return WT_ERR_INVALID_ARG;
    int words[6] = {0, 0, 0, 0, 0, 0};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(words, ws, sizeof(words), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return WT_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return WT_ERR_CUDA;
    const int f = (words[kStatusForward] ? 1 : 0) | (words[kStatusBackwardData] ? 2 : 0) |
                  (words[kStatusBackwardWeight] ? 4 : 0);
    if (flags) *flags = f;
    return f ? WT_ERR_TIMEOUT : WT_OK;
}

wt_status wtconv_debug_phase_clocks(int kernel, int reset, unsigned long long* out, int n) {
    if (out == nullptr || n < 32 || (kernel != 0 && kernel != 1)) return WT_ERR_INVALID_ARG;
    return kernel == 0 ? wt::phase_clocks_forward(reset, out)
                       : wt::phase_clocks_backward_weight(reset, out);
}

wt_status wtconv_testing_set_wait_limit_ns(unsigned long long ns) {
    g_wait_limit_ns.store(ns, std::memory_order_relaxed);
    return WT_OK;
}

const char* wtconv_status_string(wt_status status) {
    switch (status) {
        case WT_OK: return "WT_OK";
        case WT_ERR_INVALID_ARG: return "WT_ERR_INVALID_ARG: invalid shape, pointer or alignment";
        case WT_ERR_UNSUPPORTED: return "WT_ERR_UNSUPPORTED: shape or kernel size not built";
        case WT_ERR_WORKSPACE: return "WT_ERR_WORKSPACE: workspace missing or too small";
        case WT_ERR_CUDA: return "WT_ERR_CUDA: a CUDA launch or runtime call failed";
        case WT_ERR_TIMEOUT: return "WT_ERR_TIMEOUT: a kernel's bounded wait timed out";
        default: return "unknown wt_status";
    }
}

int wtconv_last_launch_count(void) { return g_last_launches; }

}  // extern "C"
