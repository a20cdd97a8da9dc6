// Per-phase clocks of the plane kernels, for performance analysis only. Compiled in only
// when the library is built with -DWT_PHASE_CLOCKS (a separate build: build.py's
// build_phase_clocks); in the ordinary build every macro below expands to nothing.
//
// Thread 0 of each CTA reads clock64() at each phase boundary and adds the cycles since the
// previous boundary to the phase's counter in shared memory (a boundary may be crossed more
// than once a plane: its cycles accumulate); slot 31 counts the planes. When the CTA
// leaves, its counters are added to the kernel's device array. With two CTAs per SM the
// phases of one CTA are timed while the other CTA runs, so the shares describe where a
// CTA's time goes, not what each phase would cost alone.
#pragma once

#ifdef WT_PHASE_CLOCKS
namespace wt {
__device__ __forceinline__ unsigned long long* phase_counters() {
    __shared__ unsigned long long s[33];  // 31 phases, planes, last timestamp
    return s;
}
}  // namespace wt
#define WT_PHASE_BEGIN()                                                        \
    do {                                                                        \
        if (threadIdx.x == 0) {                                                 \
            unsigned long long* s_ = wt::phase_counters();                      \
            for (int i_ = 0; i_ < 32; ++i_) s_[i_] = 0;                          \
            s_[32] = clock64();                                                 \
        }                                                                       \
    } while (0)
#define WT_PHASE(i)                                                             \
    do {                                                                        \
        if (threadIdx.x == 0) {                                                 \
            unsigned long long* s_ = wt::phase_counters();                      \
            const unsigned long long n_ = clock64();                            \
            s_[(i)] += n_ - s_[32];                                             \
            s_[32] = n_;                                                        \
        }                                                                       \
    } while (0)
#define WT_PHASE_PLANE()                                                        \
    do {                                                                        \
        if (threadIdx.x == 0) wt::phase_counters()[31] += 1;                    \
    } while (0)
#define WT_PHASE_END(arr)                                                       \
    do {                                                                        \
        if (threadIdx.x == 0)                                                   \
            for (int i_ = 0; i_ < 32; ++i_) atomicAdd(&(arr)[i_], wt::phase_counters()[i_]); \
    } while (0)
#else
#define WT_PHASE_BEGIN() \
    do {                 \
    } while (0)
#define WT_PHASE(i) \
    do {            \
    } while (0)
#define WT_PHASE_PLANE() \
    do {                 \
    } while (0)
#define WT_PHASE_END(arr) \
    do {                  \
    } while (0)
#endif
