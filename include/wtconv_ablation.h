/*
 * WTConv forward as a pipeline of separate, materializing stages, and the cumulative
 * ablation variants of the three reformulations.
 *
 * Method: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware Reformulation"
 * (Aflalo et al.). §3.1 and Figure 1a describe the reference implementation: every stage of
 * Algorithm 1 is a separate primitive that reads its input from HBM and writes its output
 * back. §5.6 (Tables 8 and 9) adds the reformulations one at a time:
 *   WT_VARIANT_REFERENCE            Algorithm 1 stage by stage (§3.1). Per level: Haar
 *                                   analysis (Eq. 5), depthwise conv over the 4C coefficient
 *                                   channels, scale multiply; then, deepest level first, the
 *                                   low-pass add, the concatenation of the four bands and the
 *                                   inverse Haar transform (Eq. 12); base path conv (+ bias),
 *                                   scale multiply and the final add. Modeled HBM traffic
 *                                   Q_ref = 7N + 43/3 N (1 - 4^-L) elements (§3.1 Eq. 2).
 *   WT_VARIANT_FUSED_ANALYSIS       + one pass per level that recomputes the Haar analysis on
 *                                   chip and applies conv and scale (§4.1); it writes the
 *                                   scaled subbands Z^(l) and the raw low-pass carrier.
 *   WT_VARIANT_COLLAPSED_SYNTHESIS  + the synthesis cascade replaced by one pass indexed by
 *                                   output-coordinate bits (§4.2 Prop. 2, Eq. 7).
 *   WT_VARIANT_FOLDED               + scales folded into the weights (§4.3 Eq. 8) and the
 *                                   base-path addition fused into the final store: the
 *                                   pages' fused plan, Q_fused = 4N + 13/3 N (1 - 4^-L)
 *                                   - N 4^-L elements (§4.4 Eq. 10).
 * The fully fused single-pass forward of wtconv.h (wtconv_forward) goes one step further:
 * it keeps every Z^(l) on chip.
 *
 * Conventions are those of wtconv.h, with these differences:
 *   - fp32 I/O only (desc->io == WT_F32; WT_ERR_UNSUPPORTED otherwise); every intermediate
 *     is an fp32 tensor in the workspace, laid out as the reference materializes it:
 *     subbands [N][C][4][H_l][W_l] (band order LL, LH, HL, HH), carriers [N][C][H_l][W_l].
 *   - Parameters are the layer's unfolded ones (w0 [C][k][k], b0 [C] or NULL, s0 [C],
 *     wl [L][C][4][k][k], sl [L][C][4]); WT_VARIANT_FOLDED folds them itself into the
 *     workspace.
 *   - k in {1, 3, 5, 7}; H and W divisible by 2^L; 0 <= L <= 12.
 */
#ifndef WTCONV_ABLATION_H_
#define WTCONV_ABLATION_H_

#include <stddef.h>

#include "wtconv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    WT_VARIANT_REFERENCE = 0,
    WT_VARIANT_FUSED_ANALYSIS = 1,
    WT_VARIANT_COLLAPSED_SYNTHESIS = 2,
    WT_VARIANT_FOLDED = 3
} wt_variant;

/* Workspace bytes wtconv_forward_variant needs for (desc, variant): every intermediate the
 * variant materializes, each 256-byte aligned. WT_ERR_INVALID_ARG for a bad descriptor or
 * variant, WT_ERR_UNSUPPORTED for bf16 I/O or an unbuilt k. */
wt_status wtconv_variant_workspace_size(const wt_desc* desc, int variant, size_t* bytes);

/* y = WTConv(x) computed by `variant` (see above). x, y: [N][C][H][W] fp32 device memory,
 * 16-byte aligned; parameters fp32 device memory, 4-byte aligned (b0 may be NULL); ws:
 * device memory of at least wtconv_variant_workspace_size bytes, 256-byte aligned, whose
 * contents on entry do not matter. Launches on `stream` and returns without waiting;
 * WT_ERR_WORKSPACE for a missing or short workspace, WT_ERR_CUDA for a launch failure. */
wt_status wtconv_forward_variant(const wt_desc* desc, int variant, const void* x,
                                 const float* w0, const float* b0, const float* s0,
                                 const float* wl, const float* sl, void* y, void* ws,
                                 size_t ws_bytes, wt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* WTCONV_ABLATION_H_ */
