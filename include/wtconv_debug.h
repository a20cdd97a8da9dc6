/*
 * wtconv_debug.h -- per-phase clocks of the plane kernels, for performance analysis (not
 * part of the layer; the paper has no counterpart).
 *
 * Only a library built with -DWT_PHASE_CLOCKS records them (the package's build.py builds
 * it apart from the ordinary library: build_phase_clocks(); `python bench.py
 * --phase-clocks` prints the breakdown); the ordinary library has none of that code and
 * this call returns WT_ERR_UNSUPPORTED there.
 */
#ifndef WTCONV_DEBUG_H_
#define WTCONV_DEBUG_H_

#include "wtconv.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Copies the 32 counters of one plane kernel into out[0..31] (n >= 32): kernel 0 is the
 * forward / backward-data kernel, 1 the backward-weight kernel. Counter i < 31 is the sum,
 * over every CTA and every plane it processed, of the clock64() cycles thread 0 spent in
 * phase i (the phase numbering is documented beside the counters in the kernels' sources);
 * counter 31 is the number of planes. Accumulates over all launches since the last reset;
 * reset != 0 zeroes the counters after the copy. Synchronous (it copies from the device).
 * Returns WT_OK, WT_ERR_INVALID_ARG (out null, n < 32, kernel not 0 or 1), WT_ERR_CUDA, or
 * WT_ERR_UNSUPPORTED in a library built without the clocks.
 */
wt_status wtconv_debug_phase_clocks(int kernel, int reset, unsigned long long* out, int n);

#ifdef __cplusplus
}
#endif

#endif /* WTCONV_DEBUG_H_ */
