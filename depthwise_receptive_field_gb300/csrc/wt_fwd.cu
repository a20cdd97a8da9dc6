// WTConv forward and backward-data kernel for sm_103a.
//
// Method: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware Reformulation"
// (Aflalo et al.). A persistent CTA (256 threads) walks (n, c) planes and evaluates the
// whole layer on each with one read of X and one write of Y in HBM:
//
//   deep phase (L >= 2) -- a first sweep streams X through shared memory in TMA boxes
//     (several in flight) and turns every 4x4 pixel block into the four subbands of level
//     2 (§4.1 Eq. 5 twice: the level-1 carrier X^(1), then its Haar transform), stored in
//     the CTA's scratch slot; LL / 2 of them is the carrier X^(2). Levels l = 3..L then run
//     from the carriers at their own resolution, and level 2 from the stored subbands:
//     32x32 output tiles of the subbands are staged with an R-coefficient halo and
//     filtered by the four folded k x k kernels (§4.3 Eq. 8). A last pass sums Eq. 7's
//     terms of levels 2..L at level-1 resolution (§4.2 Prop. 2: coefficient address by
//     coordinate shifts, signs by coordinate bits) into the scratch slot.
//   full-resolution phase -- 64x64-pixel tiles: a TMA load brings the tile of X with a
//     2R halo (zero outside the plane) into one of two shared-memory buffers while the
//     previous tile is being computed; one pass forms the four level-1 subbands as two
//     band-pair tiles (also double-buffered, so one CTA barrier per tile suffices); each
//     warp filters the band pairs of its own coefficient rows; a last pass computes the
//     base k x k convolution straight from the raw tile (widened in registers) and
//     stores, in the same write, base + level-1 synthesis (Eq. 7's l = 1 term) + the deep
//     sum (TMA-loaded per tile).
//
// Backward-data is the same operator on dY with every kernel rotated by 180 degrees and
// no bias (§2.2 Eq. 1: the adjoint of analysis is synthesis; the adjoint of
// cross-correlation is correlation with the rotated kernel); `flip` selects it.
#include <mutex>

#include "wt_internal.h"
#include "wt_phase.cuh"
#include "wt_tile.cuh"
#include "wt_tma.cuh"

namespace wt {

constexpr int kFT = 256;  // threads per CTA
#ifdef WT_PHASE_CLOCKS
// per-phase cycle sums of the plane kernel's thread 0, all CTAs (wt_phase.cuh). Phases:
// 0 plane setup, 1 level-2 sweep and weights, 2 carriers, 3 grouped rounds, 4 level >= 3
// stage, 5 level >= 3 filter and barriers, 6 level-2 tile wait and repack (or stage),
// 7 cascade of levels >= 4 into Z^(3), 8 level-2 barrier, 9 level-2 filter, 10 level-2 deep
// sums and barrier, 11 end of the deep phase, 12 full-resolution remainder, 13 plane end,
// 14 tile wait, 15 band conversion, 16 barrier A and the next tile's issue, 17 level-1
// filter, 18 base filter, synthesis and store; 31 planes.
__device__ unsigned long long g_phase_fwd[32];
#endif

struct FwdArgs {
    CUtensorMap tmx;  // X: dims {W, H, planes}, box {XBW, XBH, 1}
    CUtensorMap tmd;  // deep sum: dims {4*W2, H2, slots}, box {64, 16, 1}
    CUtensorMap tms;  // X for the level-2 sweep: dims {W, H, planes}, box {64, SweepBox::BH, 1}
    CUtensorMap tmu;  // level-2 subbands in the slots: dims {4*W2, H2, slots}, box {4*BT, BT, 1}
    const void* x;
    void* y;
    const float* b0f;
    const float* wimg;  // per channel, the shared-memory image of its folded weights
    float* zd;         // scratch: per CTA the deep sums, then the level-2 subbands
    int* err;          // this call's status word in the workspace: set on a stuck TMA wait
    int* next;         // the word after it: the next plane to hand out (zeroed before launch)
    unsigned long long wait_ns;  // limit of every bounded wait
    long long zd_slot;  // floats of each of the two arrays of a CTA's slot
    long long slot;     // floats between consecutive CTAs' slots (2 * zd_slot + deep state)
    long long planes;
    int C, H, W, L;
    int Hp, Wp;  // the plane padded with zeros to multiples of 2^L: level l is (Hp, Wp) >> l
    int img;  // floats of one channel's weight image (a multiple of 4)
    int vec, use_tma;
    // shared-memory regions (floats): mbarriers, raw X tiles (2), weight image, band-pair
    // tiles (2), filtered level-1 band pairs, deep-sum blocks (2)
    int o_bar, o_raw, o_dblk, o_w, o_b, o_z;
    int raw_f, b_f;  // floats per raw-tile buffer and per band-pair buffer
    int b_step;      // floats between the two band-pair buffers (0: a single buffer)
    int o_dz;        // the deep levels' filtered level-2 pairs (floats)
    int car2;        // the carrier X^(2) is kept in the deep state (else re-read from u2)
    int o_u;         // level-2 tiles are TMA-staged here (over the carriers), or -1
    int small2;      // levels L..2 all fit one stacked round (small planes; L >= 3)
    // deep-level state, in shared memory or (deep_global) in the CTA's workspace slot:
    int deep_global;
    int o_car[kMaxLevels + 1];                    // carriers X^(l), l = 2..L-1
    int o_zl[kMaxLevels + 1];                     // Z^(l), l = 3..L, interleaved [Hl][Wl][4]
};

constexpr int kDBytes = 16 * 64 * 4;  // deep-sum box: 16 level-2 rows x 16 positions x 4

// Shared-memory image of each channel's folded weights, built once per call: slot 0 holds
// the base taps duplicated (w, w); slot 1 + 2(l-1) + p holds level l's band pair p as
// (w_{2p}, w_{2p+1}), each scaled by 2^-(l+1) (1/2 turns unnormalized subbands into Eq. 5's,
// 2^-l is Eq. 7's level weight). Taps are rotated by 180 degrees when `flip` (backward-data).
// The plane kernel brings a channel's image into shared memory with one bulk copy.
template <int K>
__global__ void wt_fwd_weight_image_kernel(const float* w0f, const float* wlf, int C, int L,
                                           int flip, float* img) {
    constexpr int KK = FG<K>::KK, WS = PG<K>::WS;
    const int per_c = WS * (1 + 2 * L);
    const long long n = (long long)C * per_c;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(e / per_c), o = (int)(e - (long long)c * per_c);
        const int slot = o / WS, r = o - slot * WS;
        float v = 0.f;
        if (r < 2 * KK) {
            const int uv = r >> 1, h = r & 1;
            const int src = flip ? (KK - 1 - uv) : uv;
            if (slot == 0) {
                v = w0f[(size_t)c * KK + src];
            } else {
                const int l = 1 + (slot - 1) / 2, band = 2 * ((slot - 1) & 1) + h;
                v = ldexpf(1.0f, -(l + 1)) * wlf[(((size_t)(l - 1) * C + c) * 4 + band) * KK + src];
            }
        }
        img[e] = v;
    }
}

// Box of the level-2 sweep: 64 columns x BH rows of X, 16 KB in either dtype; NBUF boxes
// are in flight (they occupy the band-pair and filtered-subband tiles, idle at that time).
// Each thread handles PPT level-2 positions of a box.
template <typename T>
struct SweepBox {
    static constexpr int BW = 64;
    static constexpr int BH = 16384 / (BW * (int)sizeof(T));
    static constexpr int BYTES = BW * BH * (int)sizeof(T);
    static constexpr int NBUF = 2;
    static constexpr int PPT = (BW / 4) * (BH / 4) / 256;
    static_assert(PPT * 256 == (BW / 4) * (BH / 4), "whole positions per thread");
};

// Level-2 sweep: the unnormalized subbands of every level-2 position go to u2
// [H/4][W/4][4] (LL, LH, HL, HH); LL / 2 of it is the carrier X^(2), also written to the
// deep state when it is kept there. TMA path: the first NBUF boxes were issued at the start
// of the plane; box t + NBUF reuses box t's buffer. Each warp releases a box on bar_e[b]
// (8 arrivals) and thread 0 refills the buffer once all have, so there is no CTA barrier
// per box. Every wait is bounded; a timeout sets *s_abort, after which no thread waits
// again, and the vote at the end returns false (uniform over the CTA).
template <typename T, bool FAST>
__device__ __forceinline__ bool level2_sweep(const FwdArgs& a, const T* xp, float* sm, float* deep,
                                             float* u2, uint64_t* bar_s, uint64_t* bar_e,
                                             uint32_t& ph_s, uint32_t& ph_e,
                                             volatile int* s_abort, long long plane,
                                             Issued& iss) {
    constexpr int BW = SweepBox<T>::BW, BH = SweepBox<T>::BH, NB = SweepBox<T>::NBUF;
    constexpr int PR = BH / 4;  // rows of level-2 positions per box
    const int H2 = a.Hp >> 2, W2 = a.Wp >> 2;
    float4* u2v = reinterpret_cast<float4*>(u2);
    float* c2 = a.car2 ? deep + a.o_car[2] : nullptr;
    const int tid = threadIdx.x;
    if (FAST || a.use_tma) {
        T* buf = reinterpret_cast<T*>(sm + a.o_b);
        const int bxn = (a.Wp + BW - 1) / BW;
        const int nbox = sweep_boxes(a.Hp, a.Wp, BW, BH);
        constexpr int PC = BW / 4;  // level-2 positions per box row
        const int pi = tid / PC, pj = tid % PC;
        bool ok = true;
        for (int t = 0; t < nbox; ++t) {
            const int b = t % NB;
            if (tid == 0 && t >= 1) {
                const int nt = t - 1 + NB, nb = (t - 1) % NB;
                if (nt < nbox && ok && *s_abort == 0) {
                    ok = mbar_wait_bounded(bar_e + nb, (ph_e >> nb) & 1u, a.wait_ns);
                    if (ok) {
                        const int ny = nt / bxn, nx = nt - ny * bxn;
                        fence_proxy_async_smem();
                        mbar_expect_tx_noted(bar_s + nb, SweepBox<T>::BYTES, iss);
                        tma_load_3d(buf + nb * (BW * BH), &a.tms, nx * BW, ny * BH, (int)plane,
                                    bar_s + nb);
                    } else {
                        *s_abort = 1;
                    }
                }
                ph_e ^= 1u << nb;
            }
            if (ok && *s_abort == 0) {
                ok = mbar_wait_bounded(bar_s + b, (ph_s >> b) & 1u, a.wait_ns);
                if (!ok) *s_abort = 1;
            }
            ph_s ^= 1u << b;
            const int by = t / bxn, bx = t - by * bxn;
#pragma unroll
            for (int k = 0; k < SweepBox<T>::PPT; ++k) {
                const int pk = pi + (256 / PC) * k;  // position row within the box
                const int i2 = by * PR + pk, j2 = bx * PC + pj;
                if (i2 < H2 && j2 < W2) {
                    const T* q = buf + b * (BW * BH) + (4 * pk) * BW + 4 * pj;
                    const float4 u = level2_block(ld4_smem<T>(q), ld4_smem<T>(q + BW),
                                                  ld4_smem<T>(q + 2 * BW),
                                                  ld4_smem<T>(q + 3 * BW));
                    if (ok) {
                        __stcg(u2v + (size_t)i2 * W2 + j2, u);
                        if (c2 != nullptr) c2[i2 * W2 + j2] = 0.5f * u.x;
                    }
                }
            }
            __syncwarp();
            if ((tid & 31) == 0) mbar_arrive(bar_e + b);
        }
        if (tid == 0) ph_e ^= 1u << ((nbox - 1) % NB);
        if (a.o_u >= 0) fence_proxy_async_global();  // u2 is read back by TMA (level-2 staging)
        if (__syncthreads_or(!ok)) return false;
    } else {
        const int n = H2 * W2;
        for (int base = tid; base < n; base += 4 * kFT) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int p = base + k * kFT;
                if (p < n) {
                    const int i2 = p / W2, j2 = p - i2 * W2;
                    float4 r[4];
                    load_block4x4<T>(xp, a.H, a.W, a.vec, 4 * i2, 4 * j2, r);
                    const float4 u = level2_block(r[0], r[1], r[2], r[3]);
                    __stcg(u2v + p, u);
                    if (c2 != nullptr) c2[p] = 0.5f * u.x;
                }
            }
        }
    }
    if (a.o_u >= 0) fence_proxy_async_global();  // u2 is read back by TMA (level-2 staging)
    return true;
}

// 2x2 block of the carrier X^(l-1), l >= 3, at (2i, 2j) of its Wp-wide grid, from cp; when
// cp is null, X^(2) as LL / 2 of the stored level-2 subbands u2.
__device__ __forceinline__ float4 carrier_block(const float* u2, const float* cp, int i, int j,
                                                int Wp) {
    const size_t o = (size_t)(2 * i) * Wp + 2 * j;
    if (cp == nullptr)
        return make_float4(0.5f * __ldcg(u2 + 4 * o), 0.5f * __ldcg(u2 + 4 * (o + 1)),
                           0.5f * __ldcg(u2 + 4 * (o + Wp)), 0.5f * __ldcg(u2 + 4 * (o + Wp + 1)));
    // o and Wp are even and the carriers 16-byte aligned: two 8-byte loads
    const float2 r0 = *reinterpret_cast<const float2*>(cp + o);
    const float2 r1 = *reinterpret_cast<const float2*>(cp + o + Wp);
    return make_float4(r0.x, r0.y, r1.x, r1.y);
}

// Carriers X^(l) = LL of X^(l-1) (normalized, Eq. 5) for l = 3..L-1, in the deep state.
// With L >= 5 and X^(2) in the deep state, X^(3) and X^(4) are formed in one pass (an X^(4)
// value recomputes its four X^(3) parents, with the same operations in the same order),
// saving a barrier; re-reading X^(2) as LL / 2 of the stored subbands instead would cost
// more than the barrier.
__device__ __forceinline__ void deep_carriers(const FwdArgs& a, const float* u2, float* deep) {
    int l0 = 3;
    if (a.L >= 5 && a.car2) {
        const float* c2 = deep + a.o_car[2];
        const int W2 = a.Wp >> 2, H3 = a.Hp >> 3, W3 = a.Wp >> 3, H4 = a.Hp >> 4, W4 = a.Wp >> 4;
        float* c3 = deep + a.o_car[3];
        float* c4 = deep + a.o_car[4];
        for (int p = threadIdx.x; p < H3 * W3 + H4 * W4; p += kFT) {
            if (p < H3 * W3) {
                const int i = p / W3, j = p - i * W3;
                const float4 q = carrier_block(u2, c2, i, j, W2);
                c3[p] = 0.5f * (q.x + q.y + q.z + q.w);
            } else {
                const int r = p - H3 * W3, i = r / W4, j = r - i * W4;
                float x3[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float4 q = carrier_block(u2, c2, 2 * i + (k >> 1), 2 * j + (k & 1), W2);
                    x3[k] = 0.5f * (q.x + q.y + q.z + q.w);
                }
                c4[r] = 0.5f * (x3[0] + x3[1] + x3[2] + x3[3]);
            }
        }
        __syncthreads();
        l0 = 5;
    }
    for (int l = l0; l < a.L; ++l) {
        const int Hl = a.Hp >> l, Wl = a.Wp >> l, Wp = a.Wp >> (l - 1);
        const float* cp = (l >= 4 || a.car2) ? deep + a.o_car[l - 1] : nullptr;
        float* cl = deep + a.o_car[l];
        for (int p = threadIdx.x; p < Hl * Wl; p += kFT) {
            const int i = p / Wl, j = p - i * Wl;
            const float4 q = carrier_block(u2, cp, i, j, Wp);
            cl[p] = 0.5f * (q.x + q.y + q.z + q.w);
        }
        __syncthreads();
    }
}

// Deep stage for level l: subbands of the 32x32 output tile at (ti0, tj0) with an R halo
// (zero outside the level grid) into the two band-pair tiles. Level 2 reads its subbands
// from the sweep's output (L2-resident), deeper levels transform the carrier X^(l-1) of the
// deep state (X^(2), when not kept there, is LL / 2 of the sweep's output). The source is
// chosen outside the loop, whose trip count is a compile-time constant so that all loads
// issue early.
template <int K, int SRC>  // SRC 0: level-2 subbands; 1: carrier cp; 2: X^(2) from u2
__device__ __forceinline__ void deep_stage_from(const FwdArgs& a, const float* u2,
                                                const float* cp, float* bs, int l, int ti0,
                                                int tj0) {
    constexpr int R = FG<K>::R, BT = FG<K>::BT;
    constexpr int PROW = PG<K>::PROW, PTILE = PG<K>::PTILE, PHALF = PG<K>::PHALF;
    constexpr int NIT = (BT * BT + kFT - 1) / kFT;
    const int Hl = a.Hp >> l, Wl = a.Wp >> l, Wp = a.Wp >> (l - 1);
    const float4* u2v = reinterpret_cast<const float4*>(u2);
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
        const int idx = threadIdx.x + it * kFT;
        if (idx >= BT * BT) break;
        const int si = idx / BT, sj = idx - si * BT;
        const int gi = ti0 - R + si, gj = tj0 - R + sj;
        float4 u = f4_zero();
        if (gi >= 0 && gi < Hl && gj >= 0 && gj < Wl) {
            if constexpr (SRC == 0) {
                u = __ldcg(u2v + (size_t)gi * Wl + gj);
            } else {
                const float4 q = carrier_block(u2, SRC == 1 ? cp : nullptr, gi, gj, Wp);
                u = haar_u(q.x, q.y, q.z, q.w);
            }
        }
        float* q = bs + si * PROW + 4 * pchunk(sj >> 1, PHALF) + 2 * (sj & 1);
        *reinterpret_cast<float2*>(q) = make_float2(u.x, u.y);
        *reinterpret_cast<float2*>(q + PTILE) = make_float2(u.z, u.w);
    }
}

template <int K>
__device__ __forceinline__ void deep_stage(const FwdArgs& a, const float* u2, float* sm,
                                           const float* deep, int l, int ti0, int tj0) {
    float* bs = sm + a.o_b;
    if (l == 2)
        deep_stage_from<K, 0>(a, u2, nullptr, bs, l, ti0, tj0);
    else if (l >= 4 || a.car2)
        deep_stage_from<K, 1>(a, u2, deep + a.o_car[l - 1], bs, l, ti0, tj0);
    else
        deep_stage_from<K, 2>(a, u2, nullptr, bs, l, ti0, tj0);
}

// Small deep levels share one stage/filter round. A group is the levels l, l-1, ..., lo >= 3
// (>= 2 with L2: small planes, below) whose grids fit one output tile, stacked in the
// band-pair tiles: level m takes 2 ceil(Hm/2) + 2R rows from row offset off_m and
// 4 ceil(Wm/4) + 2R columns, exactly the cells its 2x4-block filter reads; the stack fits
// the tile's BT rows and the blocks of all its levels fit one pass of the CTA's threads.
// Returns lo (lo = l + 1: no group, level l is filtered tile by tile).
template <int K, bool L2 = false>
__device__ __forceinline__ int deep_group(const FwdArgs& a, int l) {
    constexpr int R = FG<K>::R, BT = FG<K>::BT;
    int lo = l + 1, rows = 0, blocks = 0;
    for (int m = l; m >= (L2 ? 2 : 3); --m) {
        const int Hm = a.Hp >> m, Wm = a.Wp >> m;
        if (Hm > kCT || Wm > kCT) break;
        const int nbi = (Hm + 1) >> 1, nbj = (Wm + 3) >> 2;
        if (rows + 2 * nbi + 2 * R > BT || blocks + 2 * nbi * nbj > kFT) break;
        rows += 2 * nbi + 2 * R;
        blocks += 2 * nbi * nbj;
        lo = m;
    }
    // a lone level that fills the tile gains nothing from the compact round
    if (lo == l && rows == BT && 4 * (((a.Wp >> l) + 3) >> 2) + 2 * R == BT) lo = l + 1;
    return lo;
}

// Stage a group (levels l..lo): every level's subbands, transformed from its carrier
// X^(m-1) by Eq. 5 (with L2, level 2 read from the sweep's stored subbands), with an R halo
// and zeros outside its grid.
template <int K, bool L2 = false>
__device__ __forceinline__ void deep_group_stage(const FwdArgs& a, const float* u2,
                                                 const float* deep, float* bs, int l, int lo) {
    constexpr int R = FG<K>::R;
    constexpr int PROW = PG<K>::PROW, PTILE = PG<K>::PTILE, PHALF = PG<K>::PHALF;
    int off = 0;
    for (int m = l; m >= lo; --m) {
        const int Hm = a.Hp >> m, Wm = a.Wp >> m, Wp = a.Wp >> (m - 1);
        const int rows = 2 * ((Hm + 1) >> 1) + 2 * R, cols = 4 * ((Wm + 3) >> 2) + 2 * R;
        const float* cp = (m >= 4 || a.car2) ? deep + a.o_car[m - 1] : nullptr;
        for (int idx = threadIdx.x; idx < rows * cols; idx += kFT) {
            const int si = idx / cols, sj = idx - si * cols;
            const int gi = si - R, gj = sj - R;
            float4 u = f4_zero();
            if (gi >= 0 && gi < Hm && gj >= 0 && gj < Wm) {
                if (L2 && m == 2) {
                    u = __ldcg(reinterpret_cast<const float4*>(u2) + (size_t)gi * Wm + gj);
                } else {
                    const float4 q = carrier_block(u2, cp, gi, gj, Wp);
                    u = haar_u(q.x, q.y, q.z, q.w);
                }
            }
            float* q = bs + (off + si) * PROW + 4 * pchunk(sj >> 1, PHALF) + 2 * (sj & 1);
            *reinterpret_cast<float2*>(q) = make_float2(u.x, u.y);
            *reinterpret_cast<float2*>(q + PTILE) = make_float2(u.z, u.w);
        }
        off += rows;
    }
}

// Filter a staged group: thread t takes one 2x4 block of one band pair of one level (the
// levels' blocks numbered one after another), and writes its Z^(m) quadruples (with L2,
// level 2's into the filtered level-2 pair tiles zs, which the deep sums read).
template <int K, bool L2 = false>
__device__ __forceinline__ void deep_group_filter(const FwdArgs& a, const float* bs,
                                                  const float* wsm, float* deep, int l,
                                                  int lo, float* zs = nullptr) {
    constexpr int R = FG<K>::R;
    constexpr int PROW = PG<K>::PROW, PTILE = PG<K>::PTILE, WS = PG<K>::WS;
    int t = threadIdx.x, off = 0, lev = 0, Hm = 0, Wm = 0, nbj = 1, nb = 1;
    for (int m = l; m >= lo; --m) {
        const int h = a.Hp >> m, w = a.Wp >> m;
        const int bi_n = (h + 1) >> 1, bj_n = (w + 3) >> 2;
        if (lev == 0) {
            if (t < 2 * bi_n * bj_n) {
                lev = m;
                Hm = h;
                Wm = w;
                nbj = bj_n;
                nb = bi_n * bj_n;
            } else {
                t -= 2 * bi_n * bj_n;
                off += 2 * bi_n + 2 * R;
            }
        }
    }
    if (lev == 0) return;
    const int pp = t >= nb ? 1 : 0;
    const int r = t - pp * nb;
    const int bi = r / nbj, bj = r - bi * nbj;
    f2x acc[2][4];
    conv_pair_2x4<K>(bs + pp * PTILE + (off + 2 * bi) * PROW, bj,
                     wsm + (1 + 2 * (lev - 1) + pp) * WS, acc);
    const int gi0 = 2 * bi, gj0 = 4 * bj;
    if constexpr (L2) {
        if (lev == 2) {
            constexpr int ZROW = PG<K>::ZROW, ZTILE = PG<K>::ZTILE;
#pragma unroll
            for (int o = 0; o < 2; ++o) {
                if (gi0 + o >= Hm) continue;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j = gj0 + q;
                    if (j < Wm)
                        *reinterpret_cast<float2*>(zs + pp * ZTILE + (gi0 + o) * ZROW +
                                                   4 * zunit(j >> 1) + 2 * (j & 1)) =
                            upk2(acc[o][q]);
                }
            }
            return;
        }
    }
    float* zl = deep + a.o_zl[lev];
#pragma unroll
    for (int o = 0; o < 2; ++o) {
        if (gi0 + o >= Hm) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (gj0 + q < Wm)
                *reinterpret_cast<float2*>(zl + ((gi0 + o) * Wm + gj0 + q) * 4 + 2 * pp) =
                    upk2(acc[o][q]);
    }
}

// Levels 3..L summed once at level-3 resolution, in place over Z^(3): quadruple (i3, j3)
// becomes Eq. 7's sum over levels 3..L at its four level-2 children (a, b) = (0,0), (0,1),
// (1,0), (1,1), so that a level-2 position reads one value instead of L - 2 quadruples.
// Levels 4 and 5 are read through pointers set up once (their offsets are compile-time
// indices into the argument block); deeper levels, rare, in a loop.
__device__ __forceinline__ void deep_cascade(const FwdArgs& a, float* deep) {
    const int H3 = a.Hp >> 3, W3 = a.Wp >> 3, W4 = a.Wp >> 4, W5 = a.Wp >> 5;
    float4* z3 = reinterpret_cast<float4*>(deep + a.o_zl[3]);
    const float4* z4 = reinterpret_cast<const float4*>(deep + a.o_zl[4]);
    const float4* z5 = reinterpret_cast<const float4*>(deep + a.o_zl[5]);
#pragma unroll 2
    for (int p = threadIdx.x; p < H3 * W3; p += kFT) {
        const int i3 = p / W3, j3 = p - i3 * W3;
        float v = 0.f;
        if (a.L >= 4) v += synth_rt(z4[(i3 >> 1) * W4 + (j3 >> 1)], i3 & 1, j3 & 1);
        if (a.L >= 5) v += synth_rt(z5[(i3 >> 2) * W5 + (j3 >> 2)], (i3 >> 1) & 1, (j3 >> 1) & 1);
        for (int m = 6; m <= a.L; ++m) {
            const int sh = m - 3, Wm = a.Wp >> m;
            const float4 zm =
                reinterpret_cast<const float4*>(deep + a.o_zl[m])[(i3 >> sh) * Wm + (j3 >> sh)];
            v += synth_rt(zm, (i3 >> (m - 4)) & 1, (j3 >> (m - 4)) & 1);
        }
        const float4 z = z3[p];
        z3[p] = make_float4(synth<0, 0>(z) + v, synth<0, 1>(z) + v, synth<1, 0>(z) + v,
                            synth<1, 1>(z) + v);
    }
}

// The same sum with one loop over the levels (small planes: a few positions, compact code).
__device__ __forceinline__ void deep_cascade_loop(const FwdArgs& a, float* deep) {
    const int H3 = a.Hp >> 3, W3 = a.Wp >> 3;
    float4* z3 = reinterpret_cast<float4*>(deep + a.o_zl[3]);
    for (int p = threadIdx.x; p < H3 * W3; p += kFT) {
        const int i3 = p / W3, j3 = p - i3 * W3;
        float v = 0.f;
        for (int m = 4; m <= a.L; ++m) {
            const int sh = m - 3, Wm = a.Wp >> m;
            const float4 zm =
                reinterpret_cast<const float4*>(deep + a.o_zl[m])[(i3 >> sh) * Wm + (j3 >> sh)];
            v += synth_rt(zm, (i3 >> (m - 4)) & 1, (j3 >> (m - 4)) & 1);
        }
        const float4 z = z3[p];
        z3[p] = make_float4(synth<0, 0>(z) + v, synth<0, 1>(z) + v, synth<1, 0>(z) + v,
                            synth<1, 1>(z) + v);
    }
}

// Small planes (the host sets small2 when levels L..2, L >= 3, all fit one stacked round):
// the whole deep phase in one stage/filter round, level 2 included, then Eq. 7's sum over
// levels 2..L at level-1 resolution into the scratch slot: levels 3..L cascaded into Z^(3),
// then every level-2 position, as in the tiled level-2 pass below. Out of line, so that the
// kernel's other paths keep their own code.
template <int K>
__device__ __noinline__ void small_deep_round(const FwdArgs& a, const float* u2, float* deep,
                                              float* sm, float* zslot) {
    constexpr int ZROW = PG<K>::ZROW, ZTILE = PG<K>::ZTILE;
    float* bs = sm + a.o_b;
    float* zs = sm + a.o_dz;
    deep_group_stage<K, true>(a, u2, deep, bs, a.L, 2);
    __syncthreads();
    deep_group_filter<K, true>(a, bs, sm + a.o_w, deep, a.L, 2, zs);
    __syncthreads();
    deep_cascade_loop(a, deep);
    __syncthreads();
    float4* dsum = reinterpret_cast<float4*>(zslot);
    const int H2 = a.Hp >> 2, W2 = a.Wp >> 2;
    for (int p = threadIdx.x; p < H2 * W2; p += kFT) {
        const int i2 = p / W2, j2 = p - i2 * W2;
        const float* zc = zs + i2 * ZROW + 4 * zunit(j2 >> 1) + 2 * (j2 & 1);
        const float2 za = *reinterpret_cast<const float2*>(zc);
        const float2 zb = *reinterpret_cast<const float2*>(zc + ZTILE);
        const float4 z = make_float4(za.x, za.y, zb.x, zb.y);
        const float v = deep[a.o_zl[3] + 4 * ((i2 >> 1) * (a.Wp >> 3) + (j2 >> 1)) +
                             2 * (i2 & 1) + (j2 & 1)];
        dsum[p] = make_float4(synth<0, 0>(z) + v, synth<0, 1>(z) + v, synth<1, 0>(z) + v,
                              synth<1, 1>(z) + v);
    }
}

// A TMA-staged level-2 tile ([BT][BT] quadruples (LL, LH, HL, HH), zero outside the level
// grid) into the two band-pair tiles.
template <int K>
__device__ __forceinline__ void repack_level2(const float* ubuf, float* bs) {
    constexpr int BT = FG<K>::BT;
    constexpr int PROW = PG<K>::PROW, PTILE = PG<K>::PTILE, PHALF = PG<K>::PHALF;
    const float4* u4 = reinterpret_cast<const float4*>(ubuf);
    for (int idx = threadIdx.x; idx < BT * BT; idx += kFT) {
        const int si = idx / BT, sj = idx - si * BT;
        const float4 u = u4[idx];
        float* q = bs + si * PROW + 4 * pchunk(sj >> 1, PHALF) + 2 * (sj & 1);
        *reinterpret_cast<float2*>(q) = make_float2(u.x, u.y);
        *reinterpret_cast<float2*>(q + PTILE) = make_float2(u.z, u.w);
    }
}

// Deep levels of one plane, after the level-2 sweep: carriers X^(l >= 3), levels L..3
// filtered into the deep state, then level 2, whose filtered subbands are combined at once
// with the deeper levels into Eq. 7's sum over levels 2..L at level-1 resolution, written
// to the scratch slot: level-2 position (i2, j2) holds the sums for level-1 positions
// (2 i2 + a, 2 j2 + b) as (a, b) = (0,0), (0,1), (1,0), (1,1). The deep state (carriers,
// Z^(l >= 3)) is in shared memory (DG = false: deep is the shared-memory base) or in the
// CTA's workspace slot (DG = true).
template <int K, bool DG, bool STAGED>
__device__ __forceinline__ bool deep_levels(const FwdArgs& a, float* sm, float* deep_g,
                                            const float* u2, float* zslot, uint64_t* bar_u,
                                            uint32_t& ph_u, Issued& iss) {
    constexpr int R = FG<K>::R;
    constexpr int PROW = PG<K>::PROW, PTILE = PG<K>::PTILE, WS = PG<K>::WS;
    constexpr int ZROW = PG<K>::ZROW, ZTILE = PG<K>::ZTILE;
    float* deep = DG ? deep_g : sm;
    const float* wsm = sm + a.o_w;
    float* bs = sm + a.o_b;
    float* zs = sm + a.o_dz;  // filtered level-2 pairs
    const int tid = threadIdx.x;
    // level-2 tiles by TMA from the slot into the staging buffer (over the dead carriers),
    // the next tile's load in flight while the current one is filtered
    constexpr bool tma2 = STAGED && !DG;
    float* ubuf = sm + (tma2 ? a.o_u : 0);
    auto issue2 = [&](int ti0, int tj0) {
        mbar_expect_tx_noted(bar_u, 16u * FG<K>::BT * FG<K>::BT, iss);
        tma_load_3d(ubuf, &a.tmu, 4 * (tj0 - R), ti0 - R, (int)blockIdx.x, bar_u);
    };
    bool ok = true;
    deep_carriers(a, u2, deep);
    WT_PHASE(2);
    if (a.small2) {
        small_deep_round<K>(a, u2, deep, sm, zslot);
        return true;
    }
    for (int l = a.L; l >= 2; --l) {
        const int Hl = a.Hp >> l, Wl = a.Wp >> l;
        if (l >= 3) {
            const int lo = deep_group<K>(a, l);
            if (lo <= l) {
                deep_group_stage<K>(a, u2, deep, bs, l, lo);
                __syncthreads();
                deep_group_filter<K>(a, bs, wsm, deep, l, lo);
                __syncthreads();  // the band-pair tiles are free for the next stage
                WT_PHASE(3);
                l = lo;
                continue;
            }
        }
        if (l == 2 && tma2) {
            // every thread's generic accesses to the carriers are ordered before the load
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) issue2(0, 0);
        }
        for (int ti0 = 0; ti0 < Hl; ti0 += kCT) {
            for (int tj0 = 0; tj0 < Wl; tj0 += kCT) {
                if (l == 2 && tma2) {
                    // a timed-out wait repacks stale data; the vote below ends the kernel
                    ok = mbar_wait_bounded(bar_u, ph_u, a.wait_ns) && ok;
                    ph_u ^= 1;
                    repack_level2<K>(ubuf, bs);
                } else {
                    deep_stage<K>(a, u2, sm, deep, l, ti0, tj0);
                }
                WT_PHASE(l == 2 ? 6 : 4);
                if (l == 2 && ti0 == 0 && tj0 == 0 && a.L >= 3) deep_cascade(a, deep);
                WT_PHASE(l == 2 ? 7 : 4);
                if (l == 2 && tma2) {
                    if (__syncthreads_or(!ok)) return false;
                } else {
                    __syncthreads();
                }
                WT_PHASE(l == 2 ? 8 : 5);
                if (l == 2 && tma2 && tid == 0) {  // the next level-2 tile
                    const int nj = tj0 + kCT < Wl ? tj0 + kCT : 0;
                    const int ni = tj0 + kCT < Wl ? ti0 : ti0 + kCT;
                    if (ni < Hl) {
                        fence_proxy_async_smem();
                        issue2(ni, nj);
                    }
                }
                {
                    // band pair pp, 2x4 output block (bi, bj); at level 2 warp w takes rows
                    // 4w..4w+3 of both pairs, the rows whose deep sums it forms below
                    const int lane = tid & 31;
                    const int pp = (l == 2) ? lane >> 4 : tid >> 7;
                    const int bi = (l == 2) ? 2 * (tid >> 5) + ((lane >> 3) & 1) : (tid >> 3) & 15;
                    const int bj = tid & 7;
                    const int gi0 = ti0 + 2 * bi, gj0 = tj0 + 4 * bj;
                    if (gi0 < Hl && gj0 < Wl) {
                        f2x acc[2][4];
                        conv_pair_2x4<K>(bs + pp * PTILE + (2 * bi) * PROW, bj,
                                         wsm + (1 + 2 * (l - 1) + pp) * WS, acc);
                        if (l >= 3) {
                            float* zl = deep + a.o_zl[l];
#pragma unroll
                            for (int o = 0; o < 2; ++o) {
                                if (gi0 + o >= Hl) continue;
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    if (gj0 + q < Wl)
                                        *reinterpret_cast<float2*>(
                                            zl + ((gi0 + o) * Wl + gj0 + q) * 4 + 2 * pp) =
                                            upk2(acc[o][q]);
                            }
                        } else {
#pragma unroll
                            for (int o = 0; o < 2; ++o) {
                                float* zr = zs + pp * ZTILE + (2 * bi + o) * ZROW;
                                const float2 q0 = upk2(acc[o][0]), q1 = upk2(acc[o][1]);
                                const float2 q2 = upk2(acc[o][2]), q3 = upk2(acc[o][3]);
                                *reinterpret_cast<float4*>(zr + 4 * zunit(2 * bj)) =
                                    make_float4(q0.x, q0.y, q1.x, q1.y);
                                *reinterpret_cast<float4*>(zr + 4 * zunit(2 * bj + 1)) =
                                    make_float4(q2.x, q2.y, q3.x, q3.y);
                            }
                        }
                    }
                }
                WT_PHASE(l == 2 ? 9 : 5);
                if (l == 2) {
                    // deep sums of this level-2 tile's positions: warp w, rows 4w..4w+3
                    __syncwarp();
                    float4* dsum = reinterpret_cast<float4*>(zslot);
#pragma unroll
                    for (int k = 0; k < (kCT * kCT) / kFT; ++k) {
                        const int ti = 4 * (tid >> 5) + k, tj = tid & 31;
                        const int i2 = ti0 + ti, j2 = tj0 + tj;
                        if (i2 >= Hl || j2 >= Wl) continue;
                        const float* zc = zs + ti * ZROW + 4 * zunit(tj >> 1) + 2 * (tj & 1);
                        const float2 za = *reinterpret_cast<const float2*>(zc);
                        const float2 zb = *reinterpret_cast<const float2*>(zc + ZTILE);
                        const float4 z = make_float4(za.x, za.y, zb.x, zb.y);
                        const float v = (a.L >= 3)
                            ? deep[a.o_zl[3] + 4 * ((i2 >> 1) * (a.Wp >> 3) + (j2 >> 1)) +
                                   2 * (i2 & 1) + (j2 & 1)]
                            : 0.f;
                        dsum[(size_t)i2 * Wl + j2] =
                            make_float4(synth<0, 0>(z) + v, synth<0, 1>(z) + v,
                                        synth<1, 0>(z) + v, synth<1, 1>(z) + v);
                    }
                }
                __syncthreads();  // the band-pair tiles are free for the next stage
                WT_PHASE(l == 2 ? 10 : 5);
            }
        }
    }
    return true;
}

// MODE >= 1 (FAST): the plane is TMA-staged, has 4-aligned rows, needs no padding and
// keeps its deep state in shared memory, so those checks and the other paths are compiled
// out. MODE 2 also TMA-stages the level-2 tiles (compiled only where the layout can pick it:
// kept out of the other instantiations, whose deep levels it would slow down).
template <int K, typename T, int MODE>
__global__ void __launch_bounds__(kFT, 2) wt_fwd_plane_kernel(const __grid_constant__ FwdArgs a) {
    constexpr int R = FG<K>::R;
    constexpr int PROW = PG<K>::PROW, PTILE = PG<K>::PTILE, WS = PG<K>::WS;
    constexpr int ZROW = PG<K>::ZROW, ZTILE = PG<K>::ZTILE;
    extern __shared__ __align__(128) float4 smem_f4[];
    float* sm = reinterpret_cast<float*>(smem_f4);
    // mbarriers: X tiles (2 buffers), deep-sum blocks (2 buffers), weights, level-2 sweep
    // boxes loaded (NBUF) and released by all 8 warps (NBUF), level-2 tiles
    uint64_t* bar_x = reinterpret_cast<uint64_t*>(sm + a.o_bar);
    uint64_t* bar_d = bar_x + 2;
    uint64_t* bar_w = bar_x + 4;
    uint64_t* bar_s = bar_x + 5;
    uint64_t* bar_e = bar_s + SweepBox<T>::NBUF;
    uint64_t* bar_u = bar_e + SweepBox<T>::NBUF;  // level-2 tiles from the slot
    static_assert(SweepBox<T>::NBUF <= 2, "mbarriers below the next-plane word");
    float* dblk = sm + a.o_dblk;  // two buffers of kDBytes
    float* wsm = sm + a.o_w;
    float* zs = sm + a.o_z;
    float* zslot = a.zd + (size_t)blockIdx.x * a.slot;  // deep sums [H/4][W/4][4]
    float* u2 = zslot + a.zd_slot;                          // level-2 subbands, same shape
    constexpr bool FAST = MODE >= 1;
    const bool use_tma = FAST || a.use_tma;
    const bool deep_global = !FAST && a.deep_global;
    float* deep = deep_global ? zslot + 2 * a.zd_slot : sm;  // carriers and Z^(l >= 3)
    const size_t plane_elems = (size_t)a.H * a.W;
    const int tid = threadIdx.x;
    const bool leader = tid == 0;
    const int tiles_x = (a.W + kTile - 1) / kTile;
    const int ntiles = tiles_x * ((a.H + kTile - 1) / kTile);

    if (use_tma && leader) {
        mbar_init(bar_x, 1);
        mbar_init(bar_x + 1, 1);
        mbar_init(bar_d, 1);
        mbar_init(bar_d + 1, 1);
        mbar_init(bar_w, 1);
        for (int b = 0; b < SweepBox<T>::NBUF; ++b) {
            mbar_init(bar_s + b, 1);
            mbar_init(bar_e + b, kFT / 32);
        }
        mbar_init(bar_u, 1);
        fence_mbar_init();
    }
    Issued iss;  // phases the leader opened (for the drain after a timeout)
    WT_PHASE_BEGIN();
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + a.o_bar + 26);
    if (leader) *s_abort = 0;
    __syncthreads();
    uint32_t ph_x = 0, ph_d = 0, ph_w = 0, ph_s = 0, ph_e = 0, ph_u = 0;
    bool failed = false;
    // weights of the current plane are in shared memory (uniform over the CTA)
    auto weights_ready = [&]() -> bool {
        bool ok = true;
        if (use_tma) {
            ok = mbar_wait_bounded(bar_w, ph_w, a.wait_ns);
            ph_w ^= 1;
        }
        return !__syncthreads_or(!ok);
    };

    // planes: first blockIdx.x, then whichever is next in the shared counter (planes are
    // independent, so the order does not change any result), else a fixed stride
    int* s_next = reinterpret_cast<int*>(sm + a.o_bar + 24);
    for (long long plane = blockIdx.x; plane < a.planes;) {
        const int c = (int)(plane % a.C);
        const T* xp = reinterpret_cast<const T*>(a.x) + plane * plane_elems;
        T* yp = reinterpret_cast<T*>(a.y) + plane * plane_elems;
        // the previous plane is done with shared memory; every thread's generic accesses are
        // ordered before the TMA writes issued below and during this plane
        fence_proxy_async_smem();
        __syncthreads();
        const float bias = (a.b0f != nullptr) ? __ldg(a.b0f + c) : 0.f;
        const float* wimg = a.wimg + (size_t)c * a.img;
        if (!use_tma)
            for (int e = tid; e < a.img; e += kFT) wsm[e] = __ldg(wimg + e);
        if (leader) {
            if (use_tma) {  // this channel's weights and the first tile of this plane
                fence_proxy_async_smem();
                mbar_expect_tx_noted(bar_w, (uint32_t)a.img * 4u, iss);
                bulk_load(wsm, wimg, (uint32_t)a.img * 4u, bar_w);
                mbar_expect_tx_noted(bar_x, XBox<K, T>::BYTES, iss);
                tma_load_3d(sm + a.o_raw, &a.tmx, -XBox<K, T>::XOFF, -2 * R, (int)plane, bar_x);
            }
            if (use_tma && a.L >= 2) {  // first boxes of the level-2 sweep
                constexpr int BW = SweepBox<T>::BW, BH = SweepBox<T>::BH;
                const int bxn = (a.Wp + BW - 1) / BW, nbox = sweep_boxes(a.Hp, a.Wp, BW, BH);
                T* buf = reinterpret_cast<T*>(sm + a.o_b);
                for (int t = 0; t < SweepBox<T>::NBUF && t < nbox; ++t) {
                    const int ny = t / bxn, nx = t - ny * bxn;
                    mbar_expect_tx_noted(bar_s + t, SweepBox<T>::BYTES, iss);
                    tma_load_3d(buf + t * (BW * BH), &a.tms, nx * BW, ny * BH, (int)plane,
                                bar_s + t);
                }
            }
        }
        __syncthreads();
        WT_PHASE(0);

        // ---- deep phase (L >= 2) ----
        // carriers top-down; levels L..3 filtered into shared memory; level 2 last, its
        // filtered subbands combined at once with the deeper levels into Eq. 7's sum over
        // levels 2..L at level-1 resolution, written to the scratch slot: level-2 position
        // (i2, j2) holds the sums for level-1 positions (2i2 + a, 2j2 + b) as
        // (a, b) = (0,0), (0,1), (1,0), (1,1).
        if (a.L >= 2) {
            if (!level2_sweep<T, FAST>(a, xp, sm, deep, u2, bar_s, bar_e, ph_s, ph_e, s_abort, plane, iss) || !weights_ready()) {
                failed = true;
                break;
            }
            WT_PHASE(1);
            const bool dok =
                deep_global ? deep_levels<K, true, false>(a, sm, zslot + 2 * a.zd_slot, u2, zslot,
                                                          bar_u, ph_u, iss)
                            : deep_levels<K, false, MODE == 2>(a, sm, sm, u2, zslot, bar_u, ph_u,
                                                               iss);
            if (!dok) {
                failed = true;
                break;
            }
            fence_proxy_async_global();
            fence_proxy_async_smem();  // the deep state's space is reused by TMA (deep sums)
            __syncthreads();
            WT_PHASE(11);
        }

        // ---- full-resolution phase ----
        if (a.L < 2 && !weights_ready()) {
            failed = true;
            break;
        }
        if (a.L >= 2 && use_tma && leader) {  // deep sums of the first tile
            fence_proxy_async_smem();
            mbar_expect_tx_noted(bar_d, kDBytes, iss);
            tma_load_3d(dblk, &a.tmd, 0, 0, (int)blockIdx.x, bar_d);
        }
        // Tiles: raw X tiles and band-pair tiles are double-buffered, so one barrier per
        // tile suffices: when every thread has passed barrier A(t), all of tile t - 1 is
        // done, its buffers are free for tile t + 1 (issued right there) and a thread may
        // widen tile t + 1 while others still filter tile t.
        const int by = tid >> 4, bx = tid & 15;  // 4x4-pixel block of this thread
        bool ok_prev = true;                      // deep-sum wait of the previous tile
        for (int t = 0; t < ntiles; ++t) {
            const int ty = t / tiles_x, tx = t - ty * tiles_x;
            const int y0 = ty * kTile, x0 = tx * kTile;
            const int rb = t & 1;
            T* raw = reinterpret_cast<T*>(sm + a.o_raw + rb * a.raw_f);
            float* bs = sm + a.o_b + rb * a.b_step;
            if (a.b_step == 0 && t > 0) __syncthreads();  // one band-pair buffer: tile t - 1 is done
            float* dcur = dblk + rb * (kDBytes / 4);
            bool ok_x = true;
            if (use_tma) {
                // a timed-out wait converts stale data; the vote below ends the kernel
                ok_x = mbar_wait_bounded(bar_x + rb, (ph_x >> rb) & 1u, a.wait_ns);
                ph_x ^= 1u << rb;
            } else {
                stage_raw<K, T>(xp, a.H, a.W, raw, y0, x0);
                if (a.L >= 2) {
                    // plain copy of the 16x16 level-2 block of deep sums (zero outside)
                    const int H2 = a.Hp >> 2, W2 = a.Wp >> 2;
                    const float4* z2 = reinterpret_cast<const float4*>(zslot);
                    const int i0 = y0 >> 2, j0 = x0 >> 2;
                    const int i = tid >> 4, j = tid & 15;
                    float4 v = f4_zero();
                    if (i0 + i < H2 && j0 + j < W2) v = z2[(size_t)(i0 + i) * W2 + j0 + j];
                    reinterpret_cast<float4*>(dcur)[tid] = v;
                }
                __syncthreads();
            }
            WT_PHASE(14);
            if (a.L >= 1) convert_bands<K, T>(raw, bs);
            WT_PHASE(15);
            if (__syncthreads_or(!(ok_x && ok_prev))) {  // barrier A(t)
                failed = true;
                break;
            }
            if (use_tma && leader && t + 1 < ntiles) {  // tile t + 1: X and its deep sums
                const int ny = (t + 1) / tiles_x, nx = (t + 1) - ny * tiles_x, nb = rb ^ 1;
                mbar_expect_tx_noted(bar_x + nb, XBox<K, T>::BYTES, iss);
                tma_load_3d(sm + a.o_raw + nb * a.raw_f, &a.tmx, nx * kTile - XBox<K, T>::XOFF,
                            ny * kTile - 2 * R, (int)plane, bar_x + nb);
                if (a.L >= 2) {
                    mbar_expect_tx_noted(bar_d + nb, kDBytes, iss);
                    tma_load_3d(dblk + nb * (kDBytes / 4), &a.tmd, nx * kTile,
                                (ny * kTile) >> 2, (int)blockIdx.x, bar_d + nb);
                }
            }
            WT_PHASE(16);
            if (a.L >= 1) {
                // level-1 filters: 2 band pairs x 128 blocks of 2x4 coefficients, one per
                // thread. Warp w filters coefficient rows 4w..4w+3 of both pairs, exactly the
                // rows that its own threads' 4x4 pixel blocks synthesize below, so a warp
                // barrier hands them over.
                const int lane = tid & 31;
                const int pp = lane >> 4, bi = 2 * (tid >> 5) + ((lane >> 3) & 1), bj = lane & 7;
                if (y0 / 2 + 2 * bi < (a.H + 1) / 2 && x0 / 2 + 4 * bj < (a.W + 1) / 2) {
                    f2x acc[2][4];
                    conv_pair_2x4<K>(bs + pp * PTILE + (2 * bi) * PROW, bj, wsm + (1 + pp) * WS,
                                     acc);
#pragma unroll
                    for (int o = 0; o < 2; ++o) {
                        float* zr = zs + pp * ZTILE + (2 * bi + o) * ZROW;
                        const float2 q0 = upk2(acc[o][0]), q1 = upk2(acc[o][1]);
                        const float2 q2 = upk2(acc[o][2]), q3 = upk2(acc[o][3]);
                        *reinterpret_cast<float4*>(zr + 4 * zunit(2 * bj)) =
                            make_float4(q0.x, q0.y, q1.x, q1.y);
                        *reinterpret_cast<float4*>(zr + 4 * zunit(2 * bj + 1)) =
                            make_float4(q2.x, q2.y, q3.x, q3.y);
                    }
                }
                __syncwarp();
            }
            WT_PHASE(17);
            // the deep sums are waited for just before their use; the wait is voted on at the
            // next barrier
            bool ok_d = true;
            const int gy = y0 + 4 * by, gx = x0 + 4 * bx;
            if (gy < a.H && gx < a.W) {
                f2x acc2[4][2];
                const f2x bias2 = pk2(bias, bias);
#pragma unroll
                for (int o = 0; o < 4; ++o) acc2[o][0] = acc2[o][1] = bias2;
                conv_base_4x4_raw<K, T>(raw, by, bx, wsm, acc2);
                if (a.L >= 1) {
                    float4 d = f4_zero();
                    if (a.L >= 2) {
                        if (use_tma) ok_d = mbar_wait_bounded(bar_d + rb, (ph_d >> rb) & 1u, a.wait_ns);
                        d = reinterpret_cast<const float4*>(dcur)[tid];
                    }
                    const float dv[2][2] = {{d.x, d.y}, {d.z, d.w}};
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        // (LL, LH) and (HL, HH) of coefficients (2by+i, 2bx) and (2by+i, 2bx+1)
                        const float4 za = *reinterpret_cast<const float4*>(
                            zs + (2 * by + i) * ZROW + 4 * zunit(bx));
                        const float4 zb = *reinterpret_cast<const float4*>(
                            zs + ZTILE + (2 * by + i) * ZROW + 4 * zunit(bx));
                        const f2x s0 = add2(pk2(za.x, za.y), pk2(zb.x, zb.y));  // LL+HL, LH+HH
                        const f2x m0 = sub2(pk2(za.x, za.y), pk2(zb.x, zb.y));  // LL-HL, LH-HH
                        const f2x s1 = add2(pk2(za.z, za.w), pk2(zb.z, zb.w));
                        const f2x m1 = sub2(pk2(za.z, za.w), pk2(zb.z, zb.w));
                        const float2 S0 = upk2(s0), M0 = upk2(m0), S1 = upk2(s1), M1 = upk2(m1);
                        // Eq. 12/13 signs: (ry, rx) = (0,0): S.x+S.y, (0,1): M.x+M.y,
                        // (1,0): S.x-S.y, (1,1): M.x-M.y
                        acc2[2 * i][0] = add2(acc2[2 * i][0],
                                              pk2(S0.x + S0.y + dv[i][0], M0.x + M0.y + dv[i][0]));
                        acc2[2 * i][1] = add2(acc2[2 * i][1],
                                              pk2(S1.x + S1.y + dv[i][1], M1.x + M1.y + dv[i][1]));
                        acc2[2 * i + 1][0] = add2(acc2[2 * i + 1][0],
                                                  pk2(S0.x - S0.y + dv[i][0], M0.x - M0.y + dv[i][0]));
                        acc2[2 * i + 1][1] = add2(acc2[2 * i + 1][1],
                                                  pk2(S1.x - S1.y + dv[i][1], M1.x - M1.y + dv[i][1]));
                    }
                }
                float acc[4][4];
#pragma unroll
                for (int o = 0; o < 4; ++o) {
                    const float2 lo = upk2(acc2[o][0]), hi = upk2(acc2[o][1]);
                    acc[o][0] = lo.x; acc[o][1] = lo.y; acc[o][2] = hi.x; acc[o][3] = hi.y;
                }
                if (a.vec && gy + 4 <= a.H && gx + 4 <= a.W) {
#pragma unroll
                    for (int o = 0; o < 4; ++o)
                        IO<T>::st4(yp + (size_t)(gy + o) * a.W + gx,
                                   make_float4(acc[o][0], acc[o][1], acc[o][2], acc[o][3]));
                } else {
#pragma unroll
                    for (int o = 0; o < 4; ++o)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (gy + o < a.H && gx + q < a.W)
                                IO<T>::st(yp + (size_t)(gy + o) * a.W + gx + q, acc[o][q]);
                }
            }
            if (a.L >= 2 && use_tma) ph_d ^= 1u << rb;
            ok_prev = ok_d;
            WT_PHASE(18);
        }
        WT_PHASE(12);
        // the last tile's deep-sum wait, and every thread done with this plane's tiles
        if (!failed && __syncthreads_or(!ok_prev)) failed = true;
        if (failed) break;
        if (leader)
            *s_next = (a.next != nullptr) ? (int)gridDim.x + atomicAdd(a.next, 1) : -1;
        __syncthreads();
        plane = (a.next != nullptr) ? (long long)*s_next : plane + gridDim.x;
        WT_PHASE(13);
        WT_PHASE_PLANE();
    }
#ifdef WT_PHASE_CLOCKS
    WT_PHASE_END(g_phase_fwd);
#endif
    if (failed && leader) {
        if (a.err != nullptr) atomicExch(a.err, kErrTmaTimeout);
        // copies in flight land before the CTA leaves: X tiles, deep-sum blocks, weights,
        // sweep boxes and level-2 tiles (the release barriers take no copies)
        if (use_tma) mbar_drain_issued(iss, 0x7fu | (1u << 9), kWaitLimitNs);
    }
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------

// Tensor-map encoding through the driver entry point (no libcuda link needed).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 3-D tiled tensor map: dims {d0, d1, d2}, byte strides {s1, s2}, box {b0, b1, 1};
// reads outside the tensor return zeros.
bool encode_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base,
               unsigned long long d0, unsigned long long d1, unsigned long long d2,
               unsigned long long s1_bytes, unsigned long long s2_bytes, unsigned b0,
               unsigned b1) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    const cuuint32_t box[3] = {b0, b1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


namespace {

int round4(int v) { return (v + 3) & ~3; }
int round32(int v) { return (v + 31) & ~31; }

size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

struct FwdPlan {
    FwdArgs a;
    size_t img_bytes = 0;
    size_t smem = 0;
    int grid = 0;
    size_t ws_bytes = 0;
};

constexpr size_t kErrWordBytes = kStatusBytes;  // the workspace starts with the status words
// shared memory per CTA that still lets two CTAs share an SM
constexpr size_t kTwoCtaSmem = 228 * 1024 / 2 - 1024;

// Shared-memory layout of one CTA for nbs band-pair buffers (2: one barrier per tile; 1: an
// extra barrier before each tile's band pass) and car2 (keep the carrier X^(2) in the deep
// state, else read it as LL / 2 of the stored level-2 subbands). Returns the floats used
// with the deep state in shared memory (local_end) and without it (xend); `deep` = floats
// of the deep state.
template <int K, typename T>
void fwd_layout(FwdArgs& a, int L, int hp, int wp, int nbs, int car2, int stage_u, int& xend,
                int& local_end, int& deep) {
    int off = 0;
    a.o_bar = off;  // 0: the mbarrier region starts dynamic shared memory (wt_tma.cuh)
    off += 32;  // ten mbarriers, the next-plane and abort words and the issue bookkeeping
    a.o_raw = off;
    a.raw_f = round32((XBox<K, T>::BYTES + 3) / 4);
    off += 2 * a.raw_f;
    a.o_w = off;
    a.img = PG<K>::WS * (1 + 2 * L);
    off += a.img;
    off = round32(off);
    a.o_b = off;
    a.b_f = round32(2 * PG<K>::PTILE);
    a.b_step = (nbs == 2) ? a.b_f : 0;
    off += nbs * a.b_f;
    // the deep levels' filtered level-2 pairs: the second band-pair buffer, else the second
    // raw buffer (idle during the deep phase) when large enough, else their own space
    if (nbs == 2) {
        a.o_dz = a.o_b + a.b_f;
    } else if (a.raw_f >= 2 * PG<K>::ZTILE) {
        a.o_dz = a.o_raw + a.raw_f;
    } else {
        a.o_dz = off;
        off += 2 * PG<K>::ZTILE;
    }
    // the level-2 sweep's boxes reuse the band-pair tiles
    const int sweep_end = a.o_b + SweepBox<T>::NBUF * SweepBox<T>::BYTES / 4;
    if (off < sweep_end) off = round32(sweep_end);
    // the full-resolution phase's filtered pairs + deep-sum blocks and the deep phase's
    // carriers + Z^(l >= 3) share a region
    const int alias0 = round32(off);
    a.o_z = alias0;
    a.o_dblk = round32(alias0 + 2 * PG<K>::ZTILE);
    xend = a.o_dblk + ((L >= 2) ? 2 * kDBytes / 4 : 0);
    a.car2 = (car2 && L >= 3) ? 1 : 0;
    deep = 0;
    for (int l = 0; l <= kMaxLevels; ++l) a.o_car[l] = a.o_zl[l] = 0;
    // level-2 tiles (BT x BT subband quadruples) TMA-staged over the carriers, which are dead
    // by the time level 2 runs. Only where that measured faster than loading them directly:
    // 16-bit I/O, k <= 5 and at least two level-2 tiles (so that a load is in flight while
    // a tile is filtered; with one tile the extra barrier and the repack cost more).
    const int l2_tiles = ((hp >> 2) + kCT - 1) / kCT * (((wp >> 2) + kCT - 1) / kCT);
    const bool su = stage_u && L >= 2 && sizeof(T) == 2 && K <= 5 && l2_tiles >= 2;
    // deep-level state, each part 16-byte aligned: the carriers X^(2 or 3..L-1) and
    // Z^(3..L); with staging Z first, so that the staging buffer can overlay the carriers
    auto place_z = [&]() {
        for (int l = 3; l <= L; ++l) {
            a.o_zl[l] = deep;
            deep += 4 * (hp >> l) * (wp >> l);
        }
    };
    auto place_car = [&]() {
        for (int l = a.car2 ? 2 : 3; l < L; ++l) {
            a.o_car[l] = deep;
            deep += round4((hp >> l) * (wp >> l));
        }
    };
    a.o_u = -1;
    int dend;
    if (su) {
        place_z();
        const int zsize = deep;
        place_car();
        a.o_u = alias0 + round32(zsize);  // a TMA destination: 128-byte aligned
        const int u_end = round32(zsize) + 4 * FG<K>::BT * FG<K>::BT;
        dend = deep > u_end ? deep : u_end;
    } else {
        place_car();
        place_z();
        dend = deep;
    }
    local_end = alias0 + dend > xend ? alias0 + dend : xend;
    for (int l = 2; l <= L; ++l) {  // offsets for the shared-memory placement
        a.o_car[l] += alias0;
        a.o_zl[l] += alias0;
    }
}

// Whether levels L..2 (L >= 3) all fit one stacked round (the kernel's small_deep_round):
// every grid within one output tile, the stack within its BT rows and one 2x4 block of every
// level and band pair per thread.
template <int K>
bool small2_fits(int L, int hp, int wp) {
    if (L < 3) return false;
    constexpr int R = FG<K>::R, BT = FG<K>::BT;
    int rows = 0, blocks = 0;
    for (int m = L; m >= 2; --m) {
        const int Hm = hp >> m, Wm = wp >> m;
        if (Hm > kCT || Wm > kCT) return false;
        const int nbi = (Hm + 1) >> 1, nbj = (Wm + 3) >> 2;
        rows += 2 * nbi + 2 * R;
        blocks += 2 * nbi * nbj;
        if (rows > BT || blocks > kFT) return false;
    }
    return true;
}

template <int K, typename T>
FwdPlan fwd_plan(const wt_desc& d) {
    FwdPlan p;
    FwdArgs& a = p.a;
    const int L = d.levels;
    const int hp = padded_side(d.h, L), wp = padded_side(d.w, L);
    // Layout choice, first fit: two CTAs per SM with the deep state in shared memory (two
    // band-pair buffers before one, X^(2) kept before re-read, level-2 tiles TMA-staged
    // before loaded directly); else two CTAs per SM with the deep state in the CTA's
    // workspace slot; else one CTA per SM, deep state in shared memory if it fits, else in
    // the slot.
    static const int kOrder[8][3] = {{2, 1, 1}, {2, 1, 0}, {2, 0, 1}, {2, 0, 0},
                                     {1, 1, 1}, {1, 1, 0}, {1, 0, 1}, {1, 0, 0}};
    int xend = 0, local_end = 0, deep = 0, total = 0;
    bool chosen = false;
    for (int i = 0; i < 8 && !chosen; ++i) {
        fwd_layout<K, T>(a, L, hp, wp, kOrder[i][0], kOrder[i][1], kOrder[i][2], xend,
                         local_end, deep);
        if ((size_t)local_end * sizeof(float) <= kTwoCtaSmem) {
            a.deep_global = 0;
            total = local_end;
            chosen = true;
        }
    }
    for (int nbs = 2; nbs >= 1 && !chosen; --nbs) {
        fwd_layout<K, T>(a, L, hp, wp, nbs, 0, 0, xend, local_end, deep);
        if ((size_t)xend * sizeof(float) <= kTwoCtaSmem) {
            a.deep_global = 1;
            total = xend;
            chosen = true;
        }
    }
    for (int i = 0; i < 8 && !chosen; ++i) {
        fwd_layout<K, T>(a, L, hp, wp, kOrder[i][0], kOrder[i][1], kOrder[i][2], xend,
                         local_end, deep);
        if ((size_t)local_end * sizeof(float) <= kMaxSmemPerBlock) {
            a.deep_global = 0;
            total = local_end;
            chosen = true;
        }
    }
    if (!chosen) {
        fwd_layout<K, T>(a, L, hp, wp, 2, 0, 0, xend, local_end, deep);
        a.deep_global = 1;
        total = xend;
    }
    if (a.deep_global) {  // the deep state moves to the slot, offsets from its start
        const int alias0 = a.o_z;
        for (int l = 2; l <= L; ++l) {
            a.o_car[l] -= alias0;
            a.o_zl[l] -= alias0;
        }
    }
    if (deep == 0) a.deep_global = 0;
    a.small2 = small2_fits<K>(L, hp, wp) ? 1 : 0;
    p.smem = (size_t)total * sizeof(float);
    // per CTA: deep sums and level-2 subbands, each [H/4][W/4][4] fp32 (+ the deep state)
    a.zd_slot = (L >= 2) ? ((4LL * (hp >> 2) * (wp >> 2) + 63) & ~63LL) : 0;
    a.slot = 2 * a.zd_slot + (a.deep_global ? (((long long)deep + 63) & ~63LL) : 0);
    const long long planes = (long long)d.n * d.c;
    int occ = (int)((228 * 1024) / (p.smem + 1024));
    if (occ > 2) occ = 2;
    if (occ < 1) occ = 1;
    long long grid = (long long)kNumSMs * occ;
    if (grid > planes) grid = planes;
    p.grid = (int)grid;
    p.img_bytes = round256((size_t)d.c * a.img * sizeof(float));
    p.ws_bytes = kErrWordBytes + p.img_bytes +
                 ((L >= 2) ? (size_t)grid * (size_t)a.slot * sizeof(float) : 0);
    return p;
}

template <int K, typename T>
wt_status launch_fwd_k(const wt_desc& d, const void* x, const float* w0f, const float* b0f,
                       const float* wlf, void* y, int flip, void* ws, size_t ws_bytes,
                       cudaStream_t stream, int* launches) {
    FwdPlan p = fwd_plan<K, T>(d);
    if (p.smem > kMaxSmemPerBlock) return WT_ERR_UNSUPPORTED;
    if (ws == nullptr || ws_bytes < p.ws_bytes) return WT_ERR_WORKSPACE;
    FwdArgs& a = p.a;
    a.x = x;
    a.y = y;
    a.b0f = flip ? nullptr : b0f;
    a.err = reinterpret_cast<int*>(ws) + (flip ? kStatusBackwardData : kStatusForward);
    a.next = a.err + 1;
    a.wait_ns = wait_limit_ns();
    float* wimg = reinterpret_cast<float*>(static_cast<char*>(ws) + kErrWordBytes);
    a.wimg = wimg;
    a.zd = reinterpret_cast<float*>(static_cast<char*>(ws) + kErrWordBytes + p.img_bytes);
    a.planes = (long long)d.n * d.c;
    a.C = d.c;
    a.H = d.h;
    a.W = d.w;
    a.Hp = padded_side(d.h, d.levels);
    a.Wp = padded_side(d.w, d.levels);
    a.L = d.levels;
    a.vec = (d.w % 4 == 0) ? 1 : 0;
    // TMA needs 16-byte row strides; otherwise the tile is staged with plain loads
    const size_t esize = sizeof(T);
    const CUtensorMapDataType dt = tma_dtype<T>();
    a.use_tma = 0;
    if (((size_t)d.w * esize) % 16 == 0) {
        bool ok = encode_3d(&a.tmx, dt, x, d.w, d.h, (unsigned long long)d.n * d.c,
                            (unsigned long long)d.w * esize,
                            (unsigned long long)d.w * d.h * esize, XBox<K, T>::XBW,
                            XBox<K, T>::XBH);
        if (ok && d.levels >= 2) {
            const unsigned long long w2 = a.Wp >> 2, h2 = a.Hp >> 2;
            ok = encode_3d(&a.tmd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.zd, 4 * w2, h2,
                           (unsigned long long)p.grid, 16 * w2, (unsigned long long)a.slot * 4,
                           64, 16);
            if (ok)
                ok = encode_3d(&a.tms, dt, x, d.w, d.h, (unsigned long long)d.n * d.c,
                               (unsigned long long)d.w * esize,
                               (unsigned long long)d.w * d.h * esize, SweepBox<T>::BW,
                               SweepBox<T>::BH);
            if (ok && a.o_u >= 0)  // the slots' level-2 subbands, BT x BT positions a box
                ok = encode_3d(&a.tmu, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.zd + a.zd_slot,
                               4 * w2, h2, (unsigned long long)p.grid, 16 * w2,
                               (unsigned long long)a.slot * 4, 4 * FG<K>::BT, FG<K>::BT);
        }
        a.use_tma = ok ? 1 : 0;
    }
    if (!a.use_tma) a.o_u = -1;  // the level-2 tiles are then loaded directly
    if (cudaMemsetAsync(a.err, 0, 2 * sizeof(int), stream) != cudaSuccess) return WT_ERR_CUDA;
    {
        const long long n = (long long)d.c * a.img;
        const int blocks = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
        wt_fwd_weight_image_kernel<K><<<blocks, 256, 0, stream>>>(w0f, wlf, d.c, d.levels, flip,
                                                                  wimg);
        if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
        ++*launches;
    }
    const bool fast = a.use_tma && a.vec && a.H == a.Hp && a.W == a.Wp && !a.deep_global;
    auto kern = fast ? wt_fwd_plane_kernel<K, T, 1> : wt_fwd_plane_kernel<K, T, 0>;
    bool staged = false;
    if constexpr (K <= 5 && sizeof(T) == 2) {
        if (fast && a.o_u >= 0) {
            kern = wt_fwd_plane_kernel<K, T, 2>;
            staged = true;
        }
    }
    if (!staged) a.o_u = -1;  // level-2 tiles loaded directly
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) !=
        cudaSuccess)
        return WT_ERR_CUDA;
    kern<<<p.grid, kFT, p.smem, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    ++*launches;
    return WT_OK;
}

template <int K>
bool fwd_sizes(const wt_desc& d, size_t* smem, size_t* ws) {
    FwdPlan p = with_io_type(d.io, [&](auto t) { return fwd_plan<K, decltype(t)>(d); });
    *smem = p.smem;
    *ws = p.ws_bytes;
    return true;
}

}  // namespace

wt_status launch_forward(const wt_desc& d, const void* x, const float* w0f, const float* b0f,
                         const float* wlf, void* y, int flip, void* ws, size_t ws_bytes,
                         cudaStream_t stream, int* launches) {
    switch (d.k) {
#define WT_CASE(KV)                                                                          \
    case KV:                                                                                 \
        return with_io_type(d.io, [&](auto t) {                                              \
            return launch_fwd_k<KV, decltype(t)>(d, x, w0f, b0f, wlf, y, flip, ws, ws_bytes, \
                                                 stream, launches);                          \
        });
        WT_CASE(1)
        WT_CASE(3)
        WT_CASE(5)
        WT_CASE(7)
#undef WT_CASE
        default:
            return WT_ERR_UNSUPPORTED;
    }
}

wt_status phase_clocks_forward(int reset, unsigned long long* out) {
#ifdef WT_PHASE_CLOCKS
    if (cudaMemcpyFromSymbol(out, g_phase_fwd, sizeof(g_phase_fwd)) != cudaSuccess)
        return WT_ERR_CUDA;
    if (reset) {
        static const unsigned long long zero[32] = {0};
        if (cudaMemcpyToSymbol(g_phase_fwd, zero, sizeof(zero)) != cudaSuccess) return WT_ERR_CUDA;
    }
    return WT_OK;
#else
    (void)reset;
    (void)out;
    return WT_ERR_UNSUPPORTED;
#endif
}

bool forward_sizes(const wt_desc& d, size_t* smem, size_t* ws) {
    switch (d.k) {
        case 1: return fwd_sizes<1>(d, smem, ws);
        case 3: return fwd_sizes<3>(d, smem, ws);
        case 5: return fwd_sizes<5>(d, smem, ws);
        case 7: return fwd_sizes<7>(d, smem, ws);
        default: return false;
    }
}

}  // namespace wt
