// FP32 multiply-add throughput probe (the measured denominator of the kernels' roofline).
// Each thread runs 8 independent chains v <- v * m + c, with m and c kernel arguments so
// that the compiler cannot fold them; the fixed point is c / (1 - m), so values stay finite.
#include <stdint.h>

#include "wt_common.cuh"
#include "wt_internal.h"
#include "wtconv_probe.h"

namespace wt {

template <bool PACKED>
__global__ void __launch_bounds__(256) wt_fma_probe_kernel(int iters, float m, float c,
                                                           float* out) {
    const float t = 1e-3f * (float)(threadIdx.x & 63);
    if constexpr (PACKED) {
        f2x v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = pk2(t + 0.1f * j, t - 0.1f * j);
        const f2x mm = pk2(m, m), cc = pk2(c, c);
#pragma unroll 4
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = fma2(v[j], mm, cc);
        }
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float2 q = upk2(v[j]);
            s += q.x + q.y;
        }
        out[blockIdx.x * blockDim.x + threadIdx.x] = s;
    } else {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = t + 0.1f * j;
#pragma unroll 4
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                asm("fma.rn.f32 %0, %0, %1, %2;" : "+f"(v[j]) : "f"(m), "f"(c));
        }
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) s += v[j];
        out[blockIdx.x * blockDim.x + threadIdx.x] = s;
    }
}

}  // namespace wt

extern "C" wt_status wtconv_fma_probe(int blocks, int iters, int packed, float* out,
                                      wt_stream_t stream) {
    if (blocks < 1 || iters < 1 || out == nullptr ||
        (reinterpret_cast<uintptr_t>(out) & 3u) != 0)
        return WT_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float m = 0.999999f, c = 1e-6f;
    if (packed)
        wt::wt_fma_probe_kernel<true><<<blocks, 256, 0, s>>>(iters, m, c, out);
    else
        wt::wt_fma_probe_kernel<false><<<blocks, 256, 0, s>>>(iters, m, c, out);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    wt::set_last_launch_count(1);
    return WT_OK;
}
