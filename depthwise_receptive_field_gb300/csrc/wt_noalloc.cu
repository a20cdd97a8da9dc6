// Backward-weight entry point that allocates nothing and takes no workspace.
//
// Some callers cannot give this library a workspace: a runtime that owns all device
// memory through its own pool and forbids raw cudaMalloc calls, or a latency-critical
// path that must not call cudaMalloc because it may synchronize the whole device. For
// them, wtconv_backward_weight_noalloc keeps its scratch in a fixed array compiled into
// the library (kNoAllocScratchBytes, 4 MiB). Every GPU that loads the library holds that
// array until the process exits.
//
// The scratch holds a 256-byte header (a status word that the plane kernel sets when one
// of its bounded waits times out, and the counter that hands planes to its CTAs; both are
// cleared with cudaMemsetAsync, which allocates nothing), the per-channel running totals
// [C][KP], the per-plane partial vectors of one chunk of images [C][nc][KP]
// (KP = k*k + 1 + 4 k*k L), and the level-2 scratch slots of the plane kernel's CTAs (when
// L >= 2). The batch is processed in chunks of nc images; each chunk runs the ordinary
// per-plane partial kernel, then a small kernel folds the chunk into the totals (the
// first chunk overwrites them, so nothing needs clearing beforehand), and finally the
// ordinary reduce + unfold kernel turns the totals into gradients; it writes NaN gradients
// if the status word was set, so that a failed call cannot pass for a result.
//
// Grid: the plane kernel runs one CTA per level-2 slot that fits in what the header,
// totals and partials leave of the 4 MiB, at most two per SM. On large planes that is far
// fewer than the workspace path's 304 CTAs (16 x 256 x 256 x 256 at k = 5, L = 5: 23 CTAs
// of 128 KB slots), so this call is correspondingly slower there.
//
// Every call shares the one array and leaves its last contents behind: two calls whose
// kernels overlap on the GPU (different streams, or different host threads on the same
// device) race on it. The first call on each device looks up the array's device address
// with cudaGetSymbolAddress (host code cannot use the symbol itself: it names a host-side
// stand-in); make that first call before any stream capture.
#include <mutex>

#include "wt_internal.h"

namespace wt {

namespace {

constexpr size_t kNoAllocScratchFloats = size_t(1) << 20;
constexpr size_t kHeaderFloats = 64;  // status word and plane counter, padded to 256 bytes
constexpr size_t kNoAllocScratchBytes = kNoAllocScratchFloats * sizeof(float);  // 4 MiB
constexpr int kMaxDevices = 64;

static_assert(kNoAllocScratchBytes == (size_t(4) << 20), "the documented size is 4 MiB");
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

std::mutex g_setup_mu;
float* g_scratch_dev_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
wt_status scratch_on_current_device(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WT_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return WT_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_dev_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return WT_ERR_CUDA;
        g_scratch_dev_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_dev_ptr[dev];
    return WT_OK;
}

// totals[c][e] = (first ? 0 : totals[c][e]) + sum_{j < nc} part[c][j][e], fixed order.
__global__ void wt_dw_accumulate_kernel(const float* part, int C, int nc, int KP, float* totals,
                                        int first) {
    const size_t n_tot = (size_t)C * KP;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n_tot;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t c = i / KP, e = i - c * KP;
        float s = first ? 0.f : totals[i];
        for (int j = 0; j < nc; ++j) s += part[(c * nc + j) * KP + e];
        totals[i] = s;
    }
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

}  // namespace wt

using namespace wt;

extern "C" wt_status wtconv_backward_weight_noalloc(const wt_desc* desc, const void* x,
                                                    const void* dy, const float* w0,
                                                    const float* b0, const float* s0,
                                                    const float* wl, const float* sl,
                                                    float* dw0, float* db0, float* ds0,
                                                    float* dwl, float* dsl,
                                                    wt_stream_t stream) {
    size_t fws = 0, bws = 0;
    wt_status st = wtconv_workspace_size(desc, &fws, nullptr, &bws);  // validates desc
    if (st != WT_OK) return st;
    if (x == nullptr || dy == nullptr || (reinterpret_cast<uintptr_t>(x) & 15u) ||
        (reinterpret_cast<uintptr_t>(dy) & 15u))
        return WT_ERR_INVALID_ARG;
    if (!w0 || !s0 || !dw0 || !ds0 || !aligned4(w0) || !aligned4(s0) || !aligned4(dw0) ||
        !aligned4(ds0) || (b0 && !aligned4(b0)) || (db0 && !aligned4(db0)))
        return WT_ERR_INVALID_ARG;
    if (desc->levels > 0 && (!wl || !sl || !dwl || !dsl || !aligned4(wl) || !aligned4(sl) ||
                             !aligned4(dwl) || !aligned4(dsl)))
        return WT_ERR_INVALID_ARG;

    // sizes: a 256-byte header (status word, plane counter), totals [C][KP], then one chunk
    // of partial vectors [C][nc][KP], then the plane kernel's level-2 scratch slots (as many
    // CTAs' as fit, up to one per plane of the chunk or two per SM, whichever is fewer; at
    // least one)
    const size_t KP = dw_partial_floats(*desc);
    const size_t per_image = (size_t)desc->c * KP;
    const size_t totals_floats = (per_image + 63) & ~size_t(63);
    const size_t slot_floats = backward_weight_slot_bytes(*desc) / sizeof(float);
    if (kHeaderFloats + totals_floats + per_image + slot_floats > kNoAllocScratchFloats)
        return WT_ERR_WORKSPACE;
    const size_t room = kNoAllocScratchFloats - kHeaderFloats - totals_floats;
    size_t want_slots = (size_t)desc->c * desc->n < 2 * (size_t)kNumSMs
                            ? (size_t)desc->c * desc->n
                            : 2 * (size_t)kNumSMs;
    if (slot_floats == 0) want_slots = 0;
    size_t nc_max = 1;
    if (room > want_slots * slot_floats + per_image)
        nc_max = (room - want_slots * slot_floats) / per_image;
    if (nc_max > (size_t)desc->n) nc_max = (size_t)desc->n;
    const size_t part_floats = (nc_max * per_image + 63) & ~size_t(63);

    float* scratch = nullptr;
    st = scratch_on_current_device(&scratch);
    if (st != WT_OK) return st;
    int* status = reinterpret_cast<int*>(scratch);  // [0] timed-out wait, [1] plane counter
    float* totals = scratch + kHeaderFloats;
    float* part = totals + totals_floats;
    float* slots = part + part_floats;
    const size_t used = kHeaderFloats + totals_floats + part_floats;
    const size_t slots_bytes =
        (kNoAllocScratchFloats > used) ? (kNoAllocScratchFloats - used) * sizeof(float) : 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // cudaMemsetAsync allocates nothing; the status word starts at zero for this call
    if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return WT_ERR_CUDA;

    const size_t esize = io_bytes(desc->io);
    const size_t image_bytes = (size_t)desc->c * desc->h * desc->w * esize;
    int launches = 0;
    for (int n0 = 0; n0 < desc->n; n0 += (int)nc_max) {
        const int nc = (desc->n - n0) < (int)nc_max ? (desc->n - n0) : (int)nc_max;
        wt_desc sub = *desc;
        sub.n = nc;
        const char* xb = static_cast<const char*>(x) + (size_t)n0 * image_bytes;
        const char* gb = static_cast<const char*>(dy) + (size_t)n0 * image_bytes;
        if (cudaMemsetAsync(status + 1, 0, sizeof(int), s) != cudaSuccess) return WT_ERR_CUDA;
        st = launch_dw_partials(sub, xb, gb, part, slots, slots_bytes, status, s, &launches);
        if (st != WT_OK) return st;
        const size_t n_tot = per_image;
        const unsigned blocks = (unsigned)((n_tot + 255) / 256 < 1024 ? (n_tot + 255) / 256 : 1024);
        wt_dw_accumulate_kernel<<<blocks, 256, 0, s>>>(part, desc->c, nc, (int)KP, totals,
                                                      n0 == 0 ? 1 : 0);
        if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
        ++launches;
    }
    st = launch_dw_reduce(*desc, totals, 1, w0, b0, s0, wl, sl, dw0, db0, ds0, dwl, dsl, status,
                          s, &launches);
    (void)fws;
    (void)bws;
    if (st == WT_OK) set_last_launch_count(launches);
    return st;
}
