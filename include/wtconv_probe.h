/*
 * wtconv_probe.h -- measurement utility of libwtconv (not part of the layer).
 *
 * The WTConv kernels are bound by the FP32 pipes (their depthwise filters are packed
 * f32x2 multiply-adds), so their roofline needs the GPU's FP32 multiply-add throughput.
 * The paper has no counterpart: it reports HBM bandwidth only. This entry point runs a
 * throughput probe whose result is the measured denominator of the benchmark's roofline.
 */
#ifndef WTCONV_PROBE_H_
#define WTCONV_PROBE_H_

#include "wtconv.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Launches one FP32 multiply-add throughput probe on `stream` and returns immediately
 * (time it with events on that stream). `blocks` CTAs of 256 threads each run `iters`
 * iterations of 8 independent dependency chains per thread; `packed` = 1 uses the packed
 * two-lane form (fma.rn.f32x2, two multiply-adds per lane and instruction), 0 the scalar
 * form (fma.rn.f32). Multiply-adds issued in all: blocks * 256 * iters * 8 * (packed ? 2 : 1).
 * `out` (device, blocks * 256 floats, 4-byte aligned) receives each thread's final value so
 * that no chain can be removed. Errors: WT_ERR_INVALID_ARG for blocks < 1, iters < 1 or a
 * NULL / misaligned out; WT_ERR_CUDA if the launch fails.
 */
wt_status wtconv_fma_probe(int blocks, int iters, int packed, float* out, wt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* WTCONV_PROBE_H_ */
