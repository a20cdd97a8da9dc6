/*
 * wtconv.h -- C ABI of the GB300 (sm_103a) WTConv layer library (libwtconv.so).
 *
 * WTConv (wavelet convolution) as defined in "Fast and Memory-Efficient Wavelet
 * Convolutions via I/O-Aware Reformulation" (Aflalo, Finder, Amoyal, Treister, Freifeld),
 * §2.1 Algorithm 1: a base depthwise k x k convolution with bias and per-channel scale,
 * plus L levels of orthonormal 2-D Haar analysis (§4.1 Eq. 5), each followed by a
 * depthwise k x k convolution and a per-(channel, subband) scale on all four subbands,
 * and the inverse-Haar synthesis, summed in one closed-form pass (§4.2 Prop. 2, Eq. 7).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are caller-owned DEVICE memory unless stated otherwise, contiguous:
 *      x, y, dy, dx            [N][C][H][W] in the I/O dtype (desc->io)
 *      w0, w0f, dw0            [C][k][k]          float32
 *      b0, b0f, db0, s0, ds0   [C]                float32
 *      wl, wlf, dwl            [L][C][4][k][k]    float32, bands (LL, LH, HL, HH)
 *      sl, dsl                 [L][C][4]          float32
 *    "f" marks scale-folded parameters (§4.3 Eq. 8): w0f = s0*w0, b0f = s0*b0, wlf = sl*wl.
 *  - Depthwise convolution is cross-correlation with zero padding R = (k-1)/2.
 *  - The library allocates no device memory. Scratch comes from the caller's workspace
 *    (ws, ws_bytes); query its size with wtconv_workspace_size. A workspace may be reused
 *    by consecutive calls on one stream; calls that run concurrently on different streams
 *    need separate workspaces. State kept between calls: a per-host-thread launch counter
 *    (wtconv_last_launch_count), and the fixed 4 MiB device array of
 *    wtconv_backward_weight_noalloc, whose contents one call leaves to the next (that call
 *    clears what must start at zero, so results do not depend on it; concurrent calls of
 *    that entry point race on it).
 *  - Every call is asynchronous on `stream` (0 = legacy default stream). Argument errors
 *    are reported synchronously and nothing is launched. Launch failures are read with
 *    cudaGetLastError right after each launch and reported as WT_ERR_CUDA; faults that
 *    happen later surface on the next synchronizing CUDA call, as usual.
 *  - Gradients are written, never accumulated into.
 *  - x, y, dy and dx must be 16-byte aligned; parameter pointers 4-byte aligned.
 *  - Accepted shapes: N, C, H, W >= 1; k odd, 1 <= k <= 7; 0 <= L <= 12. Everything else
 *    returns WT_ERR_INVALID_ARG (or WT_ERR_UNSUPPORTED for a k the kernels were not built
 *    for, or a plane too large for the kernels' shared memory at that L).
 *  - Odd sides: a carrier with an odd number of rows (columns) is padded with one zero
 *    row (column) at the bottom (right) before its Haar analysis, so level l has
 *    ceil(H_{l-1} / 2) rows, and every synthesis output is cropped back to its carrier's
 *    size (the pages are silent on odd sizes; this is the plain completion of Eq. 5 and
 *    Eq. 12). It equals running the layer on X zero-padded to multiples of 2^L and keeping
 *    the top-left H x W outputs, which is how the kernels compute it.
 *  - Results are deterministic: no atomics on data (one atomic counter hands out planes to
 *    the persistent CTAs, which does not change any result); every reduction runs in a
 *    fixed order.
 */
#ifndef WTCONV_H_
#define WTCONV_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (cudaStream_t); declared here so that callers need no CUDA header. */
typedef struct CUstream_st* wt_stream_t;

typedef enum {
    WT_OK = 0,
    WT_ERR_INVALID_ARG = 1, /* bad shape, null or misaligned pointer */
    WT_ERR_UNSUPPORTED = 2, /* valid by the definition but not built (e.g. k = 9) */
    WT_ERR_WORKSPACE = 3,   /* ws too small (or NULL with ws_bytes > 0 needed) */
    WT_ERR_CUDA = 4,        /* a CUDA launch or runtime call failed */
    WT_ERR_TIMEOUT = 5      /* a kernel's bounded wait timed out (wtconv_workspace_status) */
} wt_status;

typedef enum { WT_F32 = 0, WT_BF16 = 1, WT_F16 = 2 } wt_dtype;

typedef struct {
    int n, c, h, w; /* input shape [N][C][H][W] */
    int k;          /* kernel size of every depthwise convolution (odd) */
    int levels;     /* number of Haar decomposition levels L (0 = plain depthwise conv) */
    wt_dtype io;    /* dtype of x, y, dy, dx; accumulation is always float32 */
} wt_desc;

/*
 * Workspace bytes each call needs for this shape (any pointer may be NULL to skip it).
 * fwd is also what wtconv_backward_data needs; bwd_weight is for wtconv_backward_weight;
 * the fused wtconv_backward needs max(bwd_data, bwd_weight).
 */
wt_status wtconv_workspace_size(const wt_desc* desc, size_t* fwd, size_t* bwd_data,
                                size_t* bwd_weight);

/*
 * Scale folding, §4.3 Eq. 8: w0f = s0 (.) w0, b0f = s0 (.) b0, wlf[l][c][b] = sl[l][c][b] wl[l][c][b].
 * b0 may be NULL (zero bias); then b0f is written with zeros. b0f may be NULL to skip it.
 * One small kernel. wl, sl, wlf are ignored when L = 0.
 */
wt_status wtconv_fold_scales(const wt_desc* desc, const float* w0, const float* b0,
                             const float* s0, const float* wl, const float* sl, float* w0f,
                             float* b0f, float* wlf, wt_stream_t stream);

/*
 * Forward pass, Algorithm 1 evaluated by the I/O-aware formulation of §4:
 *   y = (x *dw w0f + b0f) + sum_l synthesis_l( wlf^(l) *dw analysis_l(x) )
 * with the Haar analysis recomputed on chip (§4.1), the synthesis summed in one pass by
 * Eq. 7 (§4.2) and the scales pre-folded (§4.3; call wtconv_fold_scales first).
 * b0f may be NULL (no bias). Workspace: wtconv_workspace_size(...).fwd bytes.
 */
wt_status wtconv_forward(const wt_desc* desc, const void* x, const float* w0f,
                         const float* b0f, const float* wlf, void* y, void* ws,
                         size_t ws_bytes, wt_stream_t stream);

/*
 * Backward with respect to the input: dx = dL/dx given dy = dL/dy.
 * By §2.2 Eq. 1 (the adjoint of Haar analysis is synthesis and vice versa) and the
 * adjoint of cross-correlation, dx is the same operator applied to dy with every folded
 * kernel rotated by 180 degrees and no bias; the rotation happens inside the kernels.
 * Workspace: wtconv_workspace_size(...).bwd_data bytes.
 */
wt_status wtconv_backward_data(const wt_desc* desc, const void* dy, const float* w0f,
                               const float* wlf, void* dx, void* ws, size_t ws_bytes,
                               wt_stream_t stream);

/*
 * Backward with respect to the parameters (unfolded), §4.3 Eq. 9:
 *   dW~^(l)[c][b][u][v] = sum_{n,i,j} A_l(dy)[n][c][b][i][j] A_l(x)[n][c][b][i+u-R][j+v-R]
 *   dW~^(0)[c][u][v]    = sum_{n,y,x} dy[n][c][y][x] x[n][c][y+u-R][x+v-R],  db~[c] = sum dy
 * (A_l = level-l Haar coefficients), then
 *   dw0 = s0 dW~^(0), db0 = s0 db~, ds0 = <dW~^(0), w0> + db~ b0,
 *   dwl = sl dW~^(l),               dsl = <dW~^(l), wl>.
 * Partial sums live in the workspace (bwd_weight bytes) and are reduced in a fixed order.
 * b0 may be NULL (zero bias); db0 may be NULL to skip it. Unfolded parameters are read.
 */
wt_status wtconv_backward_weight(const wt_desc* desc, const void* x, const void* dy,
                                 const float* w0, const float* b0, const float* s0,
                                 const float* wl, const float* sl, float* dw0, float* db0,
                                 float* ds0, float* dwl, float* dsl, void* ws,
                                 size_t ws_bytes, wt_stream_t stream);

/*
 * Both backward results in one call: wtconv_backward_data followed by
 * wtconv_backward_weight on the same stream and workspace. Needs both folded (w0f, wlf)
 * and unfolded (w0, b0, s0, wl, sl) parameters.
 */
wt_status wtconv_backward(const wt_desc* desc, const void* x, const void* dy,
                          const float* w0f, const float* wlf, const float* w0,
                          const float* b0, const float* s0, const float* wl, const float* sl,
                          void* dx, float* dw0, float* db0, float* ds0, float* dwl,
                          float* dsl, void* ws, size_t ws_bytes, wt_stream_t stream);

/*
 * wtconv_backward_weight without a workspace (the paper has no counterpart: this entry
 * point exists for callers of this library that cannot provide device memory).
 * Same arguments and gradients as wtconv_backward_weight, minus ws/ws_bytes. Results are
 * deterministic and agree with wtconv_backward_weight to fp32 rounding, not bitwise: the
 * batch is summed chunk by chunk into running totals, a different fixed order.
 *
 * Who needs it: callers that cannot hand the library a workspace, e.g. a runtime that
 * owns all device memory through its own pool and forbids raw cudaMalloc, or a
 * latency-critical path that must not call cudaMalloc because it may synchronize the
 * whole device. The scratch lives in a fixed 4 MiB array compiled into the library
 * (held by every GPU that loads the library until the process exits); this call makes
 * no cudaMalloc/cudaFree and calls no allocating library routine.
 *
 * Limit, in floats (4 bytes), with KP = k*k + 1 + 4*k*k*L:
 *     64 + round64(C*KP) + C*KP + S  <=  1048576 (4 MiB)
 * where S is the level-2 scratch of one CTA (0 when L < 2, else
 * 2 * round64(4 * ceil(H/2^L) * ceil(W/2^L) * 4^(L-2)) plus, for planes whose deep levels
 * do not fit in shared memory, their carriers). Examples at k = 5, L = 5: C <= 994 for
 * 64 x 64 planes, C <= 965 for 256 x 256; at C = 1, k = 5, L = 2 square planes up to
 * 1444 x 1444.
 * Larger shapes return WT_ERR_WORKSPACE before anything is launched. The batch is
 * processed in chunks of images, and the plane kernel runs one CTA per level-2 slot that
 * fits in what is left of the 4 MiB (at most two per SM): on large planes far fewer CTAs
 * than the workspace path (16 x 256 x 256 x 256 at k = 5, L = 5: 23 instead of 304), so
 * the call is correspondingly slower there.
 *
 * Failure: if a bounded wait inside the plane kernel times out, every gradient is written
 * as NaN (the status is also WT_OK at return, since the call is asynchronous).
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Concurrency: all calls share the one array and leave its contents behind; calls whose
 * kernels overlap on the GPU (other streams or host threads on the same device) race.
 */
wt_status wtconv_backward_weight_noalloc(const wt_desc* desc, const void* x, const void* dy,
                                         const float* w0, const float* b0, const float* s0,
                                         const float* wl, const float* sl, float* dw0,
                                         float* db0, float* ds0, float* dwl, float* dsl,
                                         wt_stream_t stream);

/*
 * Device-side status of the most recent forward, backward-data and backward-weight call
 * that used this workspace (ws as passed to those calls). Every data load inside the plane
 * kernels completes on an mbarrier whose wait is bounded (1 s); a CTA whose wait runs out
 * records it in its call's status word in the workspace, waits (again bounded) for its
 * copies still in flight and leaves, so that call's outputs are incomplete.
 * This call synchronizes `stream` (the stream those calls ran on) and reads the words.
 * flags (may be NULL) receives bit 0 = forward, bit 1 = backward-data, bit 2 =
 * backward-weight timed out. Returns WT_ERR_TIMEOUT if any bit is set, WT_OK if none,
 * WT_ERR_INVALID_ARG for a NULL ws, WT_ERR_CUDA if the copy fails. Each call clears its
 * own word when it starts, so the words describe the latest call of each kind; the fused
 * wtconv_backward sets the backward-data and backward-weight words. backward-weight also
 * turns a timeout into NaN gradients, so that it cannot pass for a result.
 */
wt_status wtconv_workspace_status(const void* ws, wt_stream_t stream, int* flags);

/* Human-readable name of a status code (static string, never NULL). */
const char* wtconv_status_string(wt_status status);

/* Number of kernels the most recent successful call on this host thread launched. */
int wtconv_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* WTCONV_H_ */
