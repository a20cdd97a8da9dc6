// WTConv backward-weight kernels for sm_103a.
//
// Method: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware Reformulation"
// (Aflalo et al.). The layer is linear in every folded kernel, so the gradient of the
// level-l folded kernel W~^(l) is the correlation of the level-l Haar coefficients of dY
// with those of X (the adjoint of the Eq. 7 synthesis is the Haar analysis, §2.2 Eq. 1):
//   dW~^(l)_b[u][v] = sum_{n,i,j} A_l(dY)_b[i][j] A_l(X)_b[i+u-R][j+v-R]
// and the base-path gradients are dW~^(0)[u][v] = sum dY[y][x] X[y+u-R][x+v-R],
// db~ = sum dY. Only X and dY are read from HBM; both Haar cascades are recomputed on chip.
//
// Kernel 1 (wt_dw_plane_kernel): a persistent grid of 256-thread CTAs walks the (n, c)
// planes. Per plane:
//   level-2 sweep (L >= 2): X and dY stream through shared memory in TMA boxes (2 to 4
//     box pairs in flight, as shared memory allows); every 4x4 pixel block becomes its
//     four level-2 subbands (Eq. 5 twice), stored for both tensors in the CTA's
//     workspace slot (L2-resident while the slots fit in L2); LL / 2 of it is the carrier
//     X^(2), dY^(2) of level 3.
//   deep levels (l >= 2): 32x32 tiles of the level's subbands of X (R halo) and dY are
//     staged as band-pair tiles, (LL, LH) and (HL, HH) (level 2 from the slot, deeper
//     levels from the carriers); threads 0-127 correlate pair 0 and 128-255 pair 1 with
//     packed f32x2 FMAs (2x4 coefficient blocks), flushed after each level by
//     recursive-halving warp reductions in a fixed order.
//   full resolution: 64x64-pixel tiles of X (2R halo) and dY arrive by TMA into two
//     buffers; the next tile's load is issued as soon as the current one's level-1
//     band pairs are formed, so it overlaps the correlations. Threads 0-127 run the base
//     correlation (4x4 pixel blocks, read from the raw tiles and widened in registers),
//     threads 128-255 the level-1 band-pair correlations (4x4 coefficient blocks). Each
//     thread keeps its partial sums in registers for the whole plane.
//   The per-plane partial vector [dW~0 | db~ | dW~^(l)_b] goes to the workspace.
// Kernel 2 (wt_dw_reduce_kernel): per channel, sums the N partial vectors in a fixed
//   order and applies the gradient unfolding of §4.3 Eq. 9.
// No atomics on data (only the counter that hands out planes): results are bitwise
// reproducible.
#include "wt_internal.h"
#include "wt_phase.cuh"
#include "wt_tile.cuh"
#include "wt_tma.cuh"

namespace wt {

constexpr int kDT = 256;  // threads per CTA
#ifdef WT_PHASE_CLOCKS
// per-phase cycle sums of the plane kernel's thread 0, all CTAs (wt_phase.cuh). Phases:
// 0 plane setup, 1 level-2 sweep, 3 tile pair wait, 4 band conversions and dY sum, 5 barrier
// B1 and the next pair's issue, 6 correlations, 7 barrier B2, 8 flush and partial vector,
// 9 plane end, 10 grouped small levels, 11 tiled level stage, 12 its first barrier, 13 its
// correlations, 14 its second barrier, 15 its flush; 31 planes.
__device__ unsigned long long g_phase_dw[32];
#endif

struct DwArgs {
    CUtensorMap tmx;  // X: dims {W, H, planes}, box {XBW, XBH, 1} (2R halo)
    CUtensorMap tmg;  // dY: dims {W, H, planes}, box {64, 64, 1}
    CUtensorMap tsx;  // X for the level-2 sweep: box {64, DwSweep::BH, 1}
    CUtensorMap tsg;  // dY for the level-2 sweep: box {64, DwSweep::BH, 1}
    const void* x;
    const void* dy;
    float* part;      // [C][N][KP]
    int* err;         // set when a TMA wait times out (may be null)
    int* next;        // the next plane to hand out (zeroed before the launch; may be null)
    unsigned long long wait_ns;  // limit of every bounded wait
    float* slots;     // per CTA: level-2 subbands of X, of dY (u2 floats each), carriers
    long long slot_floats, u2_floats;
    long long planes;
    int N, C, H, W, L;
    int Hp, Wp;  // the plane padded with zeros to multiples of 2^L: level l is (Hp, Wp) >> l
    int vec, use_tma;
    int KP;
    int nsw;  // level-2 sweep box pairs in flight (2..kMaxSweep)
    // shared memory (floats): mbarriers, raw X tiles (2 buffers of rawx_f), raw dY tiles
    // (2 of rawg_f), the partial vector, warp totals, X and dY band-pair tiles
    int o_bar, o_rawx, o_rawg, o_acc, o_red, o_xb, o_gb;
    int o_kah;  // per thread: running sum of dY and its compensation
    int rawx_f, rawg_f;
    // deep carriers X^(l), dY^(l) (l = 3..L-1; X^(2) is LL / 2 of the stored level-2
    // subbands): in shared memory, or (deep_global) in the CTA's slot after the two subband
    // arrays
    int deep_global;
    int o_carx[kMaxLevels + 1], o_cary[kMaxLevels + 1];
};

// Boxes of the level-2 sweep: 64 columns x BH rows of X or dY, 8 KB in either dtype; 2 to
// kMaxSweep (X, dY) box pairs are in flight (DwArgs::nsw, as many as shared memory allows),
// over the band-pair tiles and the carriers (idle at that time).
constexpr int kMaxSweep = 4;
template <typename T>
struct DwSweep {
    static constexpr int BW = 64;
    static constexpr int BH = sizeof(T) == 2 ? 64 : 32;
    static constexpr int BYTES = BW * BH * (int)sizeof(T);
    static constexpr int BOXF = BYTES / 4;  // floats per box
};

// dY subband-pair tiles (no halo): 32 rows x 32 cells, 16-byte chunks split even/odd.
constexpr int kGHalf = 8;             // chunks per half row
constexpr int kGRow = 8 * kGHalf;     // floats per row
constexpr int kGTile = kCT * kGRow;   // floats per pair tile

// Deep stage for level l: X subbands with an R halo into the X pair tiles, dY subbands of
// the tile's own cells into the dY pair tiles. Level 2 reads the sweep's stored subbands;
// deeper levels transform the carriers X^(l-1), dY^(l-1) (level 3: LL / 2 of the stored
// level-2 subbands) and write X^(l), dY^(l) for l < L.
template <int K>
__device__ __forceinline__ void dw_deep_stage(const DwArgs& a, const float* u2x, const float* u2g,
                                              float* sm, float* cbase, int l, int ti0,
                                              int tj0, int xoff = 0, int goff = 0) {
    constexpr int R = FG<K>::R, BT = FG<K>::BT;
    constexpr int PROW = PG<K>::PROW, PTILE = PG<K>::PTILE, PHALF = PG<K>::PHALF;
    constexpr int NIT = (BT * BT + kDT - 1) / kDT;
    const int Hl = a.Hp >> l, Wl = a.Wp >> l, Wp = a.Wp >> (l - 1);
    float* xb = sm + a.o_xb;
    float* gb = sm + a.o_gb;
    const float* cpx = (l >= 4) ? cbase + a.o_carx[l - 1] : nullptr;
    const float* cpy = (l >= 4) ? cbase + a.o_cary[l - 1] : nullptr;
    // 2x2 block of the carrier of level l - 1 >= 2 at (2gi, 2gj), transformed by Eq. 5
    auto carrier_u = [&](const float* cp, const float* u2, int gi, int gj) -> float4 {
        const size_t o = (size_t)(2 * gi) * Wp + 2 * gj;
        if (l == 3)
            return haar_u(0.5f * __ldcg(u2 + 4 * o), 0.5f * __ldcg(u2 + 4 * (o + 1)),
                          0.5f * __ldcg(u2 + 4 * (o + Wp)), 0.5f * __ldcg(u2 + 4 * (o + Wp + 1)));
        return haar_u(cp[o], cp[o + 1], cp[o + Wp], cp[o + Wp + 1]);
    };
    float* clx = (l >= 3 && l < a.L) ? cbase + a.o_carx[l] : nullptr;
    float* cly = (l >= 3 && l < a.L) ? cbase + a.o_cary[l] : nullptr;
    const float4* ux4 = reinterpret_cast<const float4*>(u2x);
    const float4* ug4 = reinterpret_cast<const float4*>(u2g);
    // a level whose grid is smaller than one tile: only the cells its correlations read,
    // 2 ceil(Hl/2) + 2R rows by 4 ceil(Wl/4) + 2R columns of X subbands (the dY subbands
    // are the inner part), zero outside the grid; from rows xoff and goff of the tiles
    // when the level is part of a group
    const int crow = 2 * ((Hl + 1) >> 1) + 2 * R, ccol = 4 * ((Wl + 3) >> 2) + 2 * R;
    if (Hl <= kCT && Wl <= kCT && (crow * ccol < BT * BT || xoff + goff > 0)) {
        for (int idx = threadIdx.x; idx < crow * ccol; idx += kDT) {
            const int si = idx / ccol, sj = idx - si * ccol;
            const int gi = si - R, gj = sj - R;
            const bool inner = si >= R && si < crow - R && sj >= R && sj < ccol - R;
            float4 ux = f4_zero(), ug = f4_zero();
            if (gi >= 0 && gi < Hl && gj >= 0 && gj < Wl) {
                if (l == 2) {
                    ux = __ldcg(ux4 + (size_t)gi * Wl + gj);
                    if (inner) ug = __ldcg(ug4 + (size_t)gi * Wl + gj);
                } else {
                    ux = carrier_u(cpx, u2x, gi, gj);
                    if (clx) clx[gi * Wl + gj] = 0.5f * ux.x;
                    ug = carrier_u(cpy, u2g, gi, gj);
                    if (cly) cly[gi * Wl + gj] = 0.5f * ug.x;
                }
            }
            float* q = xb + (xoff + si) * PROW + 4 * pchunk(sj >> 1, PHALF) + 2 * (sj & 1);
            *reinterpret_cast<float2*>(q) = make_float2(ux.x, ux.y);
            *reinterpret_cast<float2*>(q + PTILE) = make_float2(ux.z, ux.w);
            if (inner) {
                const int ci = si - R, cj = sj - R;
                float* r = gb + (goff + ci) * kGRow + 4 * pchunk(cj >> 1, kGHalf) + 2 * (cj & 1);
                *reinterpret_cast<float2*>(r) = make_float2(ug.x, ug.y);
                *reinterpret_cast<float2*>(r + kGTile) = make_float2(ug.z, ug.w);
            }
        }
        return;
    }
    if (l == 2) {  // all loads first, then all stores (loads from L2 overlap)
        float4 uxv[NIT], ugv[NIT];
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
            const int idx = threadIdx.x + it * kDT;
            const int si = idx / BT, sj = idx - si * BT;
            const int gi = ti0 - R + si, gj = tj0 - R + sj;
            const bool inner = si >= R && si < R + kCT && sj >= R && sj < R + kCT;
            const bool in = idx < BT * BT && gi >= 0 && gi < Hl && gj >= 0 && gj < Wl;
            uxv[it] = in ? __ldcg(ux4 + (size_t)gi * Wl + gj) : f4_zero();
            ugv[it] = (in && inner) ? __ldcg(ug4 + (size_t)gi * Wl + gj) : f4_zero();
        }
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
            const int idx = threadIdx.x + it * kDT;
            if (idx >= BT * BT) break;
            const int si = idx / BT, sj = idx - si * BT;
            const bool inner = si >= R && si < R + kCT && sj >= R && sj < R + kCT;
            const float4 ux = uxv[it], ug = ugv[it];
            float* q = xb + si * PROW + 4 * pchunk(sj >> 1, PHALF) + 2 * (sj & 1);
            *reinterpret_cast<float2*>(q) = make_float2(ux.x, ux.y);
            *reinterpret_cast<float2*>(q + PTILE) = make_float2(ux.z, ux.w);
            if (inner) {
                const int ci = si - R, cj = sj - R;
                float* r = gb + ci * kGRow + 4 * pchunk(cj >> 1, kGHalf) + 2 * (cj & 1);
                *reinterpret_cast<float2*>(r) = make_float2(ug.x, ug.y);
                *reinterpret_cast<float2*>(r + kGTile) = make_float2(ug.z, ug.w);
            }
        }
        return;
    }
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
        const int idx = threadIdx.x + it * kDT;
        if (idx >= BT * BT) break;
        const int si = idx / BT, sj = idx - si * BT;
        const int gi = ti0 - R + si, gj = tj0 - R + sj;
        const bool inner = si >= R && si < R + kCT && sj >= R && sj < R + kCT;
        float4 ux = f4_zero(), ug = f4_zero();
        if (gi >= 0 && gi < Hl && gj >= 0 && gj < Wl) {
            if (l == 2) {
                ux = __ldcg(ux4 + (size_t)gi * Wl + gj);
                if (inner) ug = __ldcg(ug4 + (size_t)gi * Wl + gj);
            } else {
                ux = carrier_u(cpx, u2x, gi, gj);
                if (inner) {
                    if (clx) clx[gi * Wl + gj] = 0.5f * ux.x;
                    ug = carrier_u(cpy, u2g, gi, gj);
                    if (cly) cly[gi * Wl + gj] = 0.5f * ug.x;
                }
            }
        }
        float* q = xb + si * PROW + 4 * pchunk(sj >> 1, PHALF) + 2 * (sj & 1);
        *reinterpret_cast<float2*>(q) = make_float2(ux.x, ux.y);
        *reinterpret_cast<float2*>(q + PTILE) = make_float2(ux.z, ux.w);
        if (inner) {
            const int ci = si - R, cj = sj - R;
            float* r = gb + ci * kGRow + 4 * pchunk(cj >> 1, kGHalf) + 2 * (cj & 1);
            *reinterpret_cast<float2*>(r) = make_float2(ug.x, ug.y);
            *reinterpret_cast<float2*>(r + kGTile) = make_float2(ug.z, ug.w);
        }
    }
}

// Small deep levels share one stage/correlate/flush round. A group is the levels l..hi whose
// grids fit one tile, stacked in the pair tiles (X: 2 ceil(Hm/2) + 2R rows each, dY:
// 2 ceil(Hm/2) rows each) and given whole warps per band pair (ceil(blocks / 32) each, at
// most the CTA's 8). Returns hi (hi = l: level l alone, hi < l: level l spans tiles).
template <int K>
__device__ __forceinline__ int dw_group(const DwArgs& a, int l) {
    constexpr int R = FG<K>::R, BT = FG<K>::BT;
    int hi = l - 1, rows = 0, grows = 0, warps = 0;
    for (int m = l; m <= a.L; ++m) {
        const int Hm = a.Hp >> m, Wm = a.Wp >> m;
        if (Hm > kCT || Wm > kCT) break;
        const int nbi = (Hm + 1) >> 1, nbj = (Wm + 3) >> 2;
        const int nw = 2 * ((nbi * nbj + 31) >> 5);
        if (rows + 2 * nbi + 2 * R > BT || grows + 2 * nbi > kCT || warps + nw > kDT / 32) break;
        rows += 2 * nbi + 2 * R;
        grows += 2 * nbi;
        warps += nw;
        hi = m;
    }
    return hi;
}

// Level-2 sweep of X and dY: the unnormalized level-2 subbands of every position go to
// u2x / u2g [H/4][W/4][4] (LL, LH, HL, HH). TMA path: the first NB box pairs were issued at
// the start of the plane; pair t + NB reuses pair t's buffers. With NB >= 3 a CTA barrier
// after each pair's wait frees the previous pair's buffers. With NB = 2 there is no CTA
// barrier per pair: every warp arrives on bar_e[b] (8 arrivals) when it is done with
// buffer b, and thread 0 waits for that before refilling it, so warps may run apart. Every
// wait is bounded; a timeout sets *s_abort, after which no thread waits again, and the vote
// at the end returns false (uniform over the CTA).
template <typename T, bool FAST>
__device__ __forceinline__ bool dw_sweep(const DwArgs& a, const T* xp, const T* gp, float* sm,
                                         float* u2x, float* u2g, uint64_t* bar_s,
                                         uint64_t* bar_e, uint32_t& ph_s, uint32_t& ph_e,
                                         volatile int* s_abort, long long plane, Issued& iss) {
    using S = DwSweep<T>;
    constexpr int BW = S::BW, BH = S::BH, PR = BH / 4, PC = BW / 4;
    const int NB = a.nsw;
    const int H2 = a.Hp >> 2, W2 = a.Wp >> 2;
    float4* ux4 = reinterpret_cast<float4*>(u2x);
    float4* ug4 = reinterpret_cast<float4*>(u2g);
    const int tid = threadIdx.x;
    if (FAST || a.use_tma) {
        T* buf = reinterpret_cast<T*>(sm + a.o_xb);  // X boxes 0..NB-1, then dY boxes
        const int bxn = (a.Wp + BW - 1) / BW;
        const int nbox = sweep_boxes(a.Hp, a.Wp, BW, BH);
        const int pi = tid / PC, pj = tid % PC;
        // this thread's level-2 position of pair t (in buffers b)
        auto pair = [&](int t, int b) {
            const int by = t / bxn, bx = t - by * bxn;
            const int i2 = by * PR + pi, j2 = bx * PC + pj;
            if (pi < PR && i2 < H2 && j2 < W2) {
                const T* q = buf + b * (BW * BH) + (4 * pi) * BW + 4 * pj;
                const float4 ux = level2_block(ld4_smem<T>(q), ld4_smem<T>(q + BW),
                                               ld4_smem<T>(q + 2 * BW), ld4_smem<T>(q + 3 * BW));
                const T* r = q + NB * (BW * BH);
                const float4 ug = level2_block(ld4_smem<T>(r), ld4_smem<T>(r + BW),
                                               ld4_smem<T>(r + 2 * BW), ld4_smem<T>(r + 3 * BW));
                const size_t o = (size_t)i2 * W2 + j2;
                __stcg(ux4 + o, ux);
                __stcg(ug4 + o, ug);
            }
        };
        auto refill = [&](int nt, int nb) {  // pair nt into buffers nb
            const int ny = nt / bxn, nx = nt - ny * bxn;
            mbar_expect_tx_noted(bar_s + nb, 2 * S::BYTES, iss);
            tma_load_3d(buf + nb * (BW * BH), &a.tsx, nx * BW, ny * BH, (int)plane, bar_s + nb);
            tma_load_3d(buf + (NB + nb) * (BW * BH), &a.tsg, nx * BW, ny * BH, (int)plane,
                        bar_s + nb);
        };
        if (NB >= 3) {
            // three or more pairs in flight: one CTA barrier per pair (measured faster here
            // than the per-warp releases below, which win with two pairs)
            for (int t = 0, b = 0, nb = NB - 1; t < nbox; ++t) {
                const bool okb = mbar_wait_bounded(bar_s + b, (ph_s >> b) & 1u, a.wait_ns);
                ph_s ^= 1u << b;
                if (__syncthreads_or(!okb)) return false;
                // every thread is past pair t - 1: refill its buffers with pair t - 1 + NB
                if (tid == 0 && t >= 1 && t - 1 + NB < nbox) refill(t - 1 + NB, nb);
                pair(t, b);
                nb = b;
                b = (b + 1 == NB) ? 0 : b + 1;
            }
            return true;
        }
        bool ok = true;
        for (int t = 0, b = 0, nb = NB - 1; t < nbox; ++t) {  // b = t % NB, nb = (t - 1) % NB
            if (tid == 0 && t >= 1) {
                // pair t - 1 + NB into the buffers of pair t - 1 once every warp released them
                const int nt = t - 1 + NB;
                if (nt < nbox && ok && *s_abort == 0) {
                    ok = mbar_wait_bounded(bar_e + nb, (ph_e >> nb) & 1u, a.wait_ns);
                    if (ok)
                        refill(nt, nb);
                    else
                        *s_abort = 1;
                }
                ph_e ^= 1u << nb;  // the release of pair t - 1 (waited for or not)
            }
            if (ok && *s_abort == 0) {
                ok = mbar_wait_bounded(bar_s + b, (ph_s >> b) & 1u, a.wait_ns);
                if (!ok) *s_abort = 1;
            }
            ph_s ^= 1u << b;
            if (ok) pair(t, b);
            __syncwarp();
            if ((tid & 31) == 0) mbar_arrive(bar_e + b);
            nb = b;
            b = (b + 1 == NB) ? 0 : b + 1;
        }
        if (tid == 0) ph_e ^= 1u << ((nbox - 1) % NB);  // the release of the last pair
        if (__syncthreads_or(!ok)) return false;
    } else {
        const int n = H2 * W2;
        for (int p = tid; p < n; p += kDT) {
            const int i2 = p / W2, j2 = p - i2 * W2;
            float4 r[4];
            load_block4x4<T>(xp, a.H, a.W, a.vec, 4 * i2, 4 * j2, r);
            const float4 ux = level2_block(r[0], r[1], r[2], r[3]);
            load_block4x4<T>(gp, a.H, a.W, a.vec, 4 * i2, 4 * j2, r);
            const float4 ug = level2_block(r[0], r[1], r[2], r[3]);
            __stcg(ux4 + p, ux);
            __stcg(ug4 + p, ug);
        }
    }
    return true;
}

// Level-1 unnormalized subbands of the raw dY tile (64x64, no halo) into the dY pair tiles
// (when `bands`); returns this thread's sum of the dY values it read. One item = 2x4 pixels.
template <typename T>
__device__ __forceinline__ float convert_raw_dy(const T* raw, float* gb, bool bands) {
    float sum = 0.f;
    // items in storage order (unit u of a pair-tile row holds chunk m), so that a
    // quarter-warp's 16-byte stores are contiguous (no bank conflicts)
    for (int idx = threadIdx.x; idx < kCT * (kCT / 2); idx += blockDim.x) {
        const int ci = idx >> 4, u = idx & 15;
        const int m = (u < kGHalf) ? 2 * u : 2 * (u - kGHalf) + 1;
        const T* r0 = raw + (2 * ci) * kTile + 4 * m;
        const float4 ra = ld4_smem<T>(r0), rb = ld4_smem<T>(r0 + kTile);
        sum += ((ra.x + ra.y) + (ra.z + ra.w)) + ((rb.x + rb.y) + (rb.z + rb.w));
        if (bands) {
            const float4 h0 = haar_u(ra.x, ra.y, rb.x, rb.y);
            const float4 h1 = haar_u(ra.z, ra.w, rb.z, rb.w);
            float* q = gb + ci * kGRow + 4 * u;
            *reinterpret_cast<float4*>(q) = make_float4(h0.x, h0.y, h1.x, h1.y);
            *reinterpret_cast<float4*>(q + kGTile) = make_float4(h0.z, h0.w, h1.z, h1.w);
        }
    }
    return sum;
}

// One compensated (Kahan) step of this thread's running sum kah[tid] (with its
// compensation in kah[blockDim.x + tid]): sum += v. In shared memory, not registers: the
// correlation loops need every register.
__device__ __forceinline__ void kahan_add(float* kah, float v) {
    const int t = threadIdx.x, n = blockDim.x;
    const float s = kah[t], c = kah[n + t];
    const float y = v - c;
    const float u = s + y;
    kah[n + t] = (u - s) - y;
    kah[t] = u;
}

// Recursive-halving warp reduction of 32 values: lane l ends with the warp total of
// entry l in v[0]. 31 shuffles per lane instead of 160 for an all-to-all butterfly.
__device__ __forceinline__ void warp_reduce32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 0; s < 5; ++s) {
        const int mask = 16 >> s;
        const int half = 16 >> s;
        const bool upper = (lane & mask) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float keep = upper ? v[i + half] : v[i];
            const float send = upper ? v[i] : v[i + half];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
    }
}

// Warp totals of NV values (pairs of packed accumulators, then an optional extra
// scalar) into red[e], e < NV, 32 entries at a time.
template <int NQ, int NV>
__device__ __forceinline__ void warp_totals_to(const f2x (&acc)[NQ], float extra, float* red) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int c0 = 0; c0 < NV; c0 += 32) {
        float t[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int e = c0 + j;
            if (e < 2 * NQ) {
                const float2 p = upk2(acc[e >> 1]);
                t[j] = (e & 1) ? p.y : p.x;
            } else {
                t[j] = (e == 2 * NQ && e < NV) ? extra : 0.f;
            }
        }
        warp_reduce32(t);
        if (c0 + lane < NV) red[c0 + lane] = t[0];
    }
}

// FAST: the plane is TMA-staged, has 4-aligned rows, needs no padding and keeps its deep
// carriers in shared memory, so those checks and the other paths are compiled out.
template <int K, typename T, bool FAST>
__global__ void __launch_bounds__(kDT, (K >= 7) ? 1 : 2) wt_dw_plane_kernel(const __grid_constant__ DwArgs a) {
    constexpr int R = FG<K>::R, KK = FG<K>::KK;
    constexpr int PROW = PG<K>::PROW, PTILE = PG<K>::PTILE;
    using S = DwSweep<T>;
    extern __shared__ __align__(128) float4 smem_f4[];
    float* sm = reinterpret_cast<float*>(smem_f4);
    // mbarriers: the full-resolution tile pairs (2 buffers), then the level-2 sweep's box
    // pairs
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + a.o_bar);
    uint64_t* bar_s = bar + 2;           // sweep pairs loaded
    uint64_t* bar_e = bar_s + kMaxSweep;  // sweep pairs released by all 8 warps
    static_assert(2 + 2 * kMaxSweep <= 12, "mbarriers below the next-plane word");
    float* acc_sm = sm + a.o_acc;
    float* red = sm + a.o_red;  // [8 warps][128]
    float* xb = sm + a.o_xb;
    float* gb = sm + a.o_gb;
    const int tid = threadIdx.x, warp = tid >> 5;
    const bool leader = tid == 0;
    const bool use_tma = FAST || a.use_tma;
    float* slot = a.slots + (size_t)blockIdx.x * a.slot_floats;
    float* u2x = slot;
    float* u2g = slot + a.u2_floats;
    float* cbase = (!FAST && a.deep_global) ? slot + 2 * a.u2_floats : sm;  // carriers
    const size_t plane_elems = (size_t)a.H * a.W;
    const int tiles_x = (a.W + kTile - 1) / kTile;
    const int ntiles = tiles_x * ((a.H + kTile - 1) / kTile);
    constexpr int BYTES = XBox<K, T>::BYTES + kTile * kTile * (int)sizeof(T);

    if (use_tma && leader) {
        mbar_init(bar, 1);
        mbar_init(bar + 1, 1);
        for (int b = 0; b < a.nsw; ++b) {
            mbar_init(bar_s + b, 1);
            mbar_init(bar_e + b, kDT / 32);
        }
        fence_mbar_init();
    }
    Issued iss;  // phases the leader opened (for the drain after a timeout)
    WT_PHASE_BEGIN();
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + a.o_bar + 26);  // a wait timed out
    if (leader) *s_abort = 0;
    __syncthreads();
    uint32_t ph = 0, ph_s = 0, ph_e = 0;
    bool failed = false;

    // planes: first blockIdx.x, then whichever is next in the shared counter (planes are
    // independent, so the order does not change any result), else a fixed stride
    int* s_next = reinterpret_cast<int*>(sm + a.o_bar + 24);
    int ticket = 0;  // the leader's reservation of the plane after the current one
    for (long long plane = blockIdx.x; plane < a.planes;) {
        const int n = (int)(plane / a.C), c = (int)(plane - (long long)n * a.C);
        const T* xp = reinterpret_cast<const T*>(a.x) + plane * plane_elems;
        const T* gp = reinterpret_cast<const T*>(a.dy) + plane * plane_elems;
        // the previous plane is done with shared memory; every thread's generic accesses are
        // ordered before the TMA writes issued below and during this plane
        fence_proxy_async_smem();
        __syncthreads();
        // the plane after this one is reserved now; the atomic's latency hides behind the
        // plane's work (its result is read only at the end of the plane)
        if (leader && a.next != nullptr) ticket = atomicAdd(a.next, 1);
        for (int e = tid; e < a.KP; e += kDT) acc_sm[e] = 0.f;
        if (use_tma && leader) {
            // the first full-resolution tile pair, in flight during the deep levels, and the
            // first box pairs of the level-2 sweep
            fence_proxy_async_smem();
            mbar_expect_tx_noted(bar, BYTES, iss);
            tma_load_3d(sm + a.o_rawx, &a.tmx, -XBox<K, T>::XOFF, -2 * R, (int)plane, bar);
            tma_load_3d(sm + a.o_rawg, &a.tmg, 0, 0, (int)plane, bar);
            if (a.L >= 2) {
                constexpr int BW = S::BW, BH = S::BH;
                const int bxn = (a.Wp + BW - 1) / BW, nbox = sweep_boxes(a.Hp, a.Wp, BW, BH);
                T* buf = reinterpret_cast<T*>(sm + a.o_xb);
                for (int t = 0; t < a.nsw && t < nbox; ++t) {
                    const int ny = t / bxn, nx = t - ny * bxn;
                    mbar_expect_tx_noted(bar_s + t, 2 * S::BYTES, iss);
                    tma_load_3d(buf + t * (BW * BH), &a.tsx, nx * BW, ny * BH, (int)plane,
                                bar_s + t);
                    tma_load_3d(buf + (a.nsw + t) * (BW * BH), &a.tsg, nx * BW, ny * BH,
                                (int)plane, bar_s + t);
                }
            }
        }
        __syncthreads();
        WT_PHASE(0);

        // ---- deep levels l = 2..L: band pair pp = tid / 128, 2x4 block per thread ----
        if (a.L >= 2) {
            if (!dw_sweep<T, FAST>(a, xp, gp, sm, u2x, u2g, bar_s, bar_e, ph_s, ph_e, s_abort,
                                   plane, iss)) {
                failed = true;
                break;
            }
            __syncthreads();
        }
        WT_PHASE(1);
        for (int l = 2; l <= a.L; ++l) {
            const int Hl = a.Hp >> l, Wl = a.Wp >> l;
            const int hi = dw_group<K>(a, l);
            if (hi > l) {
                // stage levels l..hi (level m + 1 >= 4 reads the carrier level m writes)
                int xoff = 0, goff = 0;
                for (int m = l; m <= hi; ++m) {
                    dw_deep_stage<K>(a, u2x, u2g, sm, cbase, m, 0, 0, xoff, goff);
                    const int nbi = ((a.Hp >> m) + 1) >> 1;
                    xoff += 2 * nbi + 2 * R;
                    goff += 2 * nbi;
                    if (m >= 3 && m < hi) __syncthreads();
                }
                __syncthreads();
                // this warp's unit: level lev, band pair pp, blocks from 32 * (warp - w0)
                int lev = 0, pp = 0, w0 = 0, nbj = 1, nbk = 0, Hm = 0, Wm = 0;
                xoff = goff = 0;
                {
                    int wn = 0, xo = 0, go = 0;
                    for (int m = l; m <= hi; ++m) {
                        const int h = a.Hp >> m, w = a.Wp >> m;
                        const int bi_n = (h + 1) >> 1, bj_n = (w + 3) >> 2;
                        const int nw = (bi_n * bj_n + 31) >> 5;
                        for (int q = 0; q < 2; ++q) {
                            if (lev == 0 && warp < wn + nw) {
                                lev = m;
                                pp = q;
                                w0 = wn;
                                nbj = bj_n;
                                nbk = bi_n * bj_n;
                                Hm = h;
                                Wm = w;
                                xoff = xo;
                                goff = go;
                            }
                            wn += nw;
                        }
                        xo += 2 * bi_n + 2 * R;
                        go += 2 * bi_n;
                    }
                }
                if (lev != 0) {
                    f2x accd[KK];
#pragma unroll
                    for (int q = 0; q < KK; ++q) accd[q] = 0ull;
                    const int r = 32 * (warp - w0) + (tid & 31);
                    const int bi = r / nbj, bj = r - bi * nbj;
                    if (r < nbk && 2 * bi < Hm && 4 * bj < Wm) {
                        f2x g[2][4];
#pragma unroll
                        for (int o = 0; o < 2; ++o) {
                            const float* gr = gb + pp * kGTile + (goff + 2 * bi + o) * kGRow;
                            const float4 t0 = *reinterpret_cast<const float4*>(gr + 4 * bj);
                            const float4 t1 = *reinterpret_cast<const float4*>(gr + 4 * (kGHalf + bj));
                            g[o][0] = pk2(t0.x, t0.y);
                            g[o][1] = pk2(t0.z, t0.w);
                            g[o][2] = pk2(t1.x, t1.y);
                            g[o][3] = pk2(t1.z, t1.w);
                        }
                        corr_pair<K, 2>(xb + pp * PTILE + (xoff + 2 * bi) * PROW, bj, g, accd);
                    }
                    warp_totals_to<KK, 2 * KK>(accd, 0.f, red + warp * 128);
                }
                __syncthreads();
                // fixed-order sum of each unit's warps into acc_sm
                {
                    int wn = 0;
                    for (int m = l; m <= hi; ++m) {
                        const int bi_n = ((a.Hp >> m) + 1) >> 1, bj_n = ((a.Wp >> m) + 3) >> 2;
                        const int nw = (bi_n * bj_n + 31) >> 5;
                        for (int e = tid; e < 4 * KK; e += kDT) {
                            const int p2 = e / (2 * KK), k = e - p2 * 2 * KK;
                            float sacc = 0.f;
                            for (int w = 0; w < nw; ++w) sacc += red[(wn + p2 * nw + w) * 128 + k];
                            acc_sm[KK + 1 + (m - 1) * 4 * KK + (2 * p2 + (k & 1)) * KK + (k >> 1)] += sacc;
                        }
                        wn += 2 * nw;
                    }
                }
                __syncthreads();
                WT_PHASE(10);
                l = hi;
                continue;
            }
            const int pp = tid >> 7, bi = (tid >> 3) & 15, bj = tid & 7;
            f2x accd[KK];
#pragma unroll
            for (int q = 0; q < KK; ++q) accd[q] = 0ull;
            for (int ti0 = 0; ti0 < Hl; ti0 += kCT) {
                for (int tj0 = 0; tj0 < Wl; tj0 += kCT) {
                    dw_deep_stage<K>(a, u2x, u2g, sm, cbase, l, ti0, tj0);
                    WT_PHASE(11);
                    __syncthreads();
                    WT_PHASE(12);
                    if (ti0 + 2 * bi < Hl && tj0 + 4 * bj < Wl) {
                        f2x g[2][4];
#pragma unroll
                        for (int o = 0; o < 2; ++o) {
                            const float* gr = gb + pp * kGTile + (2 * bi + o) * kGRow;
                            const float4 t0 = *reinterpret_cast<const float4*>(gr + 4 * bj);
                            const float4 t1 = *reinterpret_cast<const float4*>(gr + 4 * (kGHalf + bj));
                            g[o][0] = pk2(t0.x, t0.y);
                            g[o][1] = pk2(t0.z, t0.w);
                            g[o][2] = pk2(t1.x, t1.y);
                            g[o][3] = pk2(t1.z, t1.w);
                        }
                        corr_pair<K, 2>(xb + pp * PTILE + (2 * bi) * PROW, bj, g, accd);
                    }
                    WT_PHASE(13);
                    __syncthreads();
                    WT_PHASE(14);
                }
            }
            // flush: warps 4pp..4pp+3 hold band pair pp; fixed-order sum into acc_sm
            warp_totals_to<KK, 2 * KK>(accd, 0.f, red + warp * 128);
            __syncthreads();
            for (int e = tid; e < 4 * KK; e += kDT) {
                const int p2 = e / (2 * KK), k = e - p2 * 2 * KK;  // k = 2*tap + band-in-pair
                float s = 0.f;
                for (int w = 0; w < 4; ++w) s += red[(4 * p2 + w) * 128 + k];
                acc_sm[KK + 1 + (l - 1) * 4 * KK + (2 * p2 + (k & 1)) * KK + (k >> 1)] += s;
            }
            __syncthreads();
            WT_PHASE(15);
        }
        fence_proxy_async_smem();  // warp totals may sit in raw X buffer 1, refilled by TMA

        // ---- full resolution: warps 0-3 base path, warps 4-7 level-1 band pairs ----
        const bool base_role = (a.L == 0) || (tid < 128);
        f2x acc[KK];
#pragma unroll
        for (int q = 0; q < KK; ++q) acc[q] = 0ull;
        // sum of dY, taken while converting the dY tiles: a register partial over at most 16
        // tiles, folded into a compensated (Kahan) running sum so that planes of millions of
        // pixels keep the fp32 sum accurate to a few ulps
        float* kah = sm + a.o_kah;
        kah[tid] = 0.f;
        kah[kDT + tid] = 0.f;
        float dpart = 0.f;
        // Raw tiles are double-buffered: tile t + 1's pair is issued as soon as tile t's is
        // converted (barrier B1), into the buffers tile t - 1 freed at its barrier B2.
        for (int t = 0; t < ntiles; ++t) {
            const int ty = t / tiles_x, tx = t - ty * tiles_x;
            const int y0 = ty * kTile, x0 = tx * kTile;
            const int rb = t & 1;
            const T* rawx = reinterpret_cast<const T*>(sm + a.o_rawx + rb * a.rawx_f);
            const T* rawg = reinterpret_cast<const T*>(sm + a.o_rawg + rb * a.rawg_f);
            bool ok = true;
            if (use_tma) {
                // a timed-out wait converts stale data; the vote below ends the kernel
                ok = mbar_wait_bounded(bar + rb, (ph >> rb) & 1u, a.wait_ns);
                ph ^= 1u << rb;
            } else {
                stage_raw<K, T>(xp, a.H, a.W, const_cast<T*>(rawx), y0, x0);
                stage_raw_tile<T>(gp, a.H, a.W, const_cast<T*>(rawg), y0, x0);
                __syncthreads();
            }
            WT_PHASE(3);
            if (a.L >= 1) convert_bands<K, T>(rawx, xb);
            dpart += convert_raw_dy<T>(rawg, gb, a.L >= 1);
            WT_PHASE(4);
            if (__syncthreads_or(!ok)) {  // B1(t)
                failed = true;
                break;
            }
            if (use_tma && leader && t + 1 < ntiles) {
                const int ny = (t + 1) / tiles_x, nx = (t + 1) - ny * tiles_x, nb = rb ^ 1;
                mbar_expect_tx_noted(bar + nb, BYTES, iss);
                tma_load_3d(sm + a.o_rawx + nb * a.rawx_f, &a.tmx, nx * kTile - XBox<K, T>::XOFF,
                            ny * kTile - 2 * R, (int)plane, bar + nb);
                tma_load_3d(sm + a.o_rawg + nb * a.rawg_f, &a.tmg, nx * kTile, ny * kTile,
                            (int)plane, bar + nb);
            }
            WT_PHASE(5);
            if ((t & 15) == 15 || t + 1 == ntiles) {
                kahan_add(kah, dpart);
                dpart = 0.f;
            }
            if (base_role) {
                const int nb = (a.L == 0) ? 1 : 2;
                for (int k = 0; k < nb; ++k) {
                    const int blk = tid + kDT / 2 * k;  // L == 0: tid covers all 256 blocks
                    const int by = blk >> 4, bx = blk & 15;
                    if (y0 + 4 * by >= a.H || x0 + 4 * bx >= a.W) continue;
                    corr_base_4x4_raw<K, T>(rawx, rawg, by, bx, acc);
                }
            } else {
                const int t2 = tid - 128, pp = t2 >> 6, bi = (t2 >> 3) & 7, bj = t2 & 7;
                if (y0 / 2 + 4 * bi < (a.H + 1) / 2 && x0 / 2 + 4 * bj < (a.W + 1) / 2) {
                    f2x g[4][4];
#pragma unroll
                    for (int o = 0; o < 4; ++o) {
                        const float* gr = gb + pp * kGTile + (4 * bi + o) * kGRow;
                        const float4 t0 = *reinterpret_cast<const float4*>(gr + 4 * bj);
                        const float4 t1 = *reinterpret_cast<const float4*>(gr + 4 * (kGHalf + bj));
                        g[o][0] = pk2(t0.x, t0.y);
                        g[o][1] = pk2(t0.z, t0.w);
                        g[o][2] = pk2(t1.x, t1.y);
                        g[o][3] = pk2(t1.z, t1.w);
                    }
                    corr_pair<K, 4>(xb + pp * PTILE + (4 * bi) * PROW, bj, g, acc);
                }
            }
            WT_PHASE(6);
            __syncthreads();  // B2(t): the band-pair tiles and raw buffer rb are free
            WT_PHASE(7);
        }
        if (failed) break;

        // ---- flush: fixed-order reductions into acc_sm, then the partial vector ----
        const float dbs = kah[tid] - kah[kDT + tid];
        __syncthreads();  // every thread has read its sum before `red` takes the warp totals
        warp_totals_to<KK, 2 * KK + 1>(acc, dbs, red + warp * 128);
        __syncthreads();
        const int nbase = (a.L == 0) ? 8 : 4;
        for (int e = tid; e <= KK; e += kDT) {
            // base taps: both lanes of each base warp's accumulators; e == KK: the sum of dY,
            // which every warp holds a share of (it is taken while converting the dY tiles)
            float s = 0.f;
            if (e < KK) {
                for (int w = 0; w < nbase; ++w) s += red[w * 128 + 2 * e] + red[w * 128 + 2 * e + 1];
            } else {
                for (int w = 0; w < kDT / 32; ++w) s += red[w * 128 + 2 * KK];
            }
            acc_sm[e] += s;
        }
        if (a.L >= 1) {
            for (int e = tid; e < 4 * KK; e += kDT) {
                // band pair pp lives in warps 4 + 2pp and 5 + 2pp
                const int p2 = e / (2 * KK), k = e - p2 * 2 * KK;
                const float s = red[(4 + 2 * p2) * 128 + k] + red[(5 + 2 * p2) * 128 + k];
                acc_sm[KK + 1 + (2 * p2 + (k & 1)) * KK + (k >> 1)] += s;
            }
        }
        __syncthreads();
        float* out = a.part + ((size_t)c * a.N + n) * a.KP;
        for (int e = tid; e < a.KP; e += kDT) out[e] = acc_sm[e];
        WT_PHASE(8);
        if (leader)
            *s_next = (a.next != nullptr) ? (int)gridDim.x + ticket : -1;
        __syncthreads();
        plane = (a.next != nullptr) ? (long long)*s_next : plane + gridDim.x;
        WT_PHASE(9);
        WT_PHASE_PLANE();
    }
#ifdef WT_PHASE_CLOCKS
    WT_PHASE_END(g_phase_dw);
#endif
    if (failed && leader) {
        if (a.err != nullptr) atomicExch(a.err, kErrTmaTimeout);
        // copies in flight land before the CTA leaves: the tile pairs and the sweep pairs
        // (the release barriers take no copies)
        if (use_tma) mbar_drain_issued(iss, 0x3u | (((1u << a.nsw) - 1u) << 2), kWaitLimitNs);
    }
}

// Per channel: fixed-order sum of the N partial vectors, then §4.3 Eq. 9. When the plane
// kernel recorded a timed-out wait (*err != 0), every gradient is written as NaN instead,
// so that the failure cannot pass for a result.
__global__ void wt_dw_reduce_kernel(const float* part, int C, int G, int KP, int K, int L,
                                    const float* w0, const float* b0, const float* s0,
                                    const float* wl, const float* sl, float* dw0, float* db0,
                                    float* ds0, float* dwl, float* dsl, const int* err) {
    extern __shared__ float tot[];
    const int c = blockIdx.x;
    const int KK = K * K;
    const bool bad = err != nullptr && *reinterpret_cast<const volatile int*>(err) != 0;
    for (int e = threadIdx.x; e < KP; e += blockDim.x) {
        float s = 0.f;
        for (int gi = 0; gi < G; ++gi) s += part[((size_t)c * G + gi) * KP + e];
        // level entries were accumulated from unnormalized subbands on both sides (4x)
        tot[e] = bad ? __int_as_float(0x7fc00000) : (e > KK) ? 0.25f * s : s;
    }
    __syncthreads();
    const float s0c = s0[c];
    for (int e = threadIdx.x; e < KK; e += blockDim.x) dw0[(size_t)c * KK + e] = s0c * tot[e];
    if (threadIdx.x == 0) {
        float d = 0.f;
        for (int e = 0; e < KK; ++e) d = fmaf(tot[e], w0[(size_t)c * KK + e], d);
        d = fmaf(tot[KK], b0 ? b0[c] : 0.f, d);
        ds0[c] = d;
        if (db0) db0[c] = s0c * tot[KK];
    }
    for (int e = threadIdx.x; e < L * 4 * KK; e += blockDim.x) {
        const int l = e / (4 * KK), rem = e - l * 4 * KK;
        const int b = rem / KK, uv = rem - b * KK;
        const size_t pi = ((size_t)l * C + c) * 4 + b;
        dwl[pi * KK + uv] = sl[pi] * tot[KK + 1 + e];
    }
    for (int e = threadIdx.x; e < L * 4; e += blockDim.x) {
        const int l = e / 4, b = e - l * 4;
        const size_t pi = ((size_t)l * C + c) * 4 + b;
        float d = 0.f;
        for (int uv = 0; uv < KK; ++uv)
            d = fmaf(tot[KK + 1 + (l * 4 + b) * KK + uv], wl[pi * KK + uv], d);
        dsl[pi] = d;
    }
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
namespace {

int round4(int v) { return (v + 3) & ~3; }
int round32(int v) { return (v + 31) & ~31; }

constexpr size_t kDwErrBytes = kStatusBytes;  // the workspace starts with the status words
constexpr size_t kTwoCtaSmem = 228 * 1024 / 2 - 1024;  // two CTAs per SM still fit

size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

// Shared-memory layout, slot layout and grid of the plane kernel for d.
struct DwPlan {
    DwArgs a;
    size_t smem = 0;
    int grid = 0;            // persistent CTAs
    size_t slot_bytes = 0;   // workspace per CTA (0 when L < 2)
};

template <int K, typename T>
DwPlan dw_layout(const wt_desc& d) {
    constexpr int KK = FG<K>::KK;
    DwPlan p;
    DwArgs& a = p.a;
    const int L = d.levels;
    const int hp = padded_side(d.h, L), wp = padded_side(d.w, L);
    a.KP = KK + 1 + 4 * KK * L;
    int off = 0;
    a.o_bar = off;  // 0: the mbarrier region starts dynamic shared memory (wt_tma.cuh)
    off += 32;  // mbarriers, the next-plane and abort words and the issue bookkeeping
    a.o_rawx = off;
    a.rawx_f = round32((XBox<K, T>::BYTES + 3) / 4);
    off += 2 * a.rawx_f;
    a.o_rawg = off;
    a.rawg_f = round32(kTile * kTile * (int)sizeof(T) / 4);
    off += 2 * a.rawg_f;
    a.o_acc = off;
    off += round32(a.KP);
    // warp totals of the flushes, 8 x 128 floats, with the dY sum's Kahan words in their
    // first 2 x 256 (read before the full-resolution flush overwrites them); where that
    // would cost the second CTA per SM, the totals use the second raw X buffer instead (idle
    // at flush time: the deep levels run before tile 1 is issued, the full-resolution flush
    // after the last tile) and the Kahan words get their own 2 x 256
    static_assert(8 * 128 <= (XBox<K, T>::BYTES) / 4, "warp totals fit a raw X buffer");
    const int tiles_rest = 2 * PG<K>::PTILE + 4 + 2 * kGTile;  // band-pair tiles (+ padding)
    const int sweep_min = 2 * 2 * DwSweep<T>::BOXF;  // two box pairs
    const int tail = tiles_rest > sweep_min ? tiles_rest : sweep_min;
    if ((size_t)(off + 8 * 128 + tail + 32) * sizeof(float) <= kTwoCtaSmem) {
        a.o_red = off;
        a.o_kah = off;
        off += 8 * 128;
    } else {
        a.o_red = a.o_rawx + a.rawx_f;
        a.o_kah = off;
        off += 2 * kDT;
    }
    a.o_xb = off;
    off += 2 * PG<K>::PTILE;
    off = round4(off);
    a.o_gb = off;
    off += 2 * kGTile;
    // the deep-level carriers X^(l), dY^(l), l = 3..L-1, after the band-pair tiles
    off = round32(off);
    const int alias0 = off;
    int cp = 0;
    for (int l = 0; l <= kMaxLevels; ++l) a.o_carx[l] = a.o_cary[l] = 0;
    for (int l = 3; l < L; ++l) {
        const int sz = round4((hp >> l) * (wp >> l));
        a.o_carx[l] = cp;
        cp += sz;
        a.o_cary[l] = cp;
        cp += sz;
    }
    // The level-2 sweep's nsw box pairs overlay the band-pair tiles, the carriers and
    // whatever space follows (all idle during the sweep). First fit, preferring carriers in
    // shared memory (the FAST instantiation) and then more box pairs: two CTAs per SM (k <=
    // 5) with carriers in shared memory and 4 or 3 pairs; with carriers in the CTA's
    // workspace slot and 4 or 3 pairs; either placement with 2 pairs; else one CTA per SM.
    const size_t two = (K >= 7) ? kMaxSmemPerBlock : kTwoCtaSmem;
    auto end_of = [&](int nsw, bool dg) {
        const int e = dg ? alias0 : alias0 + cp;
        const int sw = a.o_xb + 2 * nsw * DwSweep<T>::BOXF;
        return e > sw ? e : sw;
    };
    static const int kTry[6][2] = {{4, 0}, {3, 0}, {4, 1}, {3, 1}, {2, 0}, {2, 1}};
    int total = -1;
    for (size_t lim : {two, kMaxSmemPerBlock}) {
        for (int i = 0; i < 6 && total < 0; ++i) {
            const bool dg = kTry[i][1] != 0;
            if (dg && cp == 0) continue;
            if ((size_t)end_of(kTry[i][0], dg) * sizeof(float) <= lim) {
                a.nsw = kTry[i][0];
                a.deep_global = dg ? 1 : 0;
                total = end_of(a.nsw, dg);
            }
        }
        if (total >= 0) break;
    }
    if (total < 0) {  // too large for shared memory: reported as unsupported by the caller
        a.nsw = 2;
        a.deep_global = cp > 0 ? 1 : 0;
        total = end_of(2, a.deep_global != 0);
    }
    if (!a.deep_global)
        for (int l = 3; l < L; ++l) {
            a.o_carx[l] += alias0;
            a.o_cary[l] += alias0;
        }
    p.smem = (size_t)total * sizeof(float);
    // per CTA: the level-2 subbands of X and of dY, [H/4][W/4][4] fp32 each (+ carriers)
    a.u2_floats = (L >= 2) ? ((4LL * (hp >> 2) * (wp >> 2) + 63) & ~63LL) : 0;
    a.slot_floats = 2 * a.u2_floats + (a.deep_global ? (((long long)cp + 63) & ~63LL) : 0);
    p.slot_bytes = (size_t)a.slot_floats * sizeof(float);
    const long long planes = (long long)d.n * d.c;
    int occ = (int)((228 * 1024) / (p.smem + 1024));
    const int occ_max = (K >= 7) ? 1 : 2;
    if (occ > occ_max) occ = occ_max;
    if (occ < 1) occ = 1;
    long long grid = (long long)kNumSMs * occ;
    if (grid > planes) grid = planes;
    p.grid = (int)grid;
    return p;
}

// Fill the kernel arguments (pointers, tensor maps) for one launch with `grid` CTAs.
template <int K, typename T>
bool dw_prepare(const wt_desc& d, const void* x, const void* dy, float* part, float* slots,
                int* err, DwPlan& p) {
    DwArgs& a = p.a;
    if (p.smem > kMaxSmemPerBlock) return false;
    if (p.slot_bytes > 0 && slots == nullptr) return false;
    a.slots = slots;
    a.x = x;
    a.dy = dy;
    a.part = part;
    a.err = err;
    a.next = (err != nullptr) ? err + 1 : nullptr;
    a.wait_ns = wait_limit_ns();
    a.planes = (long long)d.n * d.c;
    a.N = d.n;
    a.C = d.c;
    a.H = d.h;
    a.W = d.w;
    a.Hp = padded_side(d.h, d.levels);
    a.Wp = padded_side(d.w, d.levels);
    a.L = d.levels;
    a.vec = (d.w % 4 == 0) ? 1 : 0;
    a.use_tma = 0;
    const size_t esize = sizeof(T);
    if (((size_t)d.w * esize) % 16 == 0) {
        const CUtensorMapDataType dt = tma_dtype<T>();
        const unsigned long long planes = (unsigned long long)d.n * d.c;
        const unsigned long long s1 = (unsigned long long)d.w * esize;
        const unsigned long long s2 = (unsigned long long)d.w * d.h * esize;
        bool ok =
            encode_3d(&a.tmx, dt, x, d.w, d.h, planes, s1, s2, XBox<K, T>::XBW, XBox<K, T>::XBH) &&
            encode_3d(&a.tmg, dt, dy, d.w, d.h, planes, s1, s2, kTile, kTile);
        if (ok && d.levels >= 2)
            ok = encode_3d(&a.tsx, dt, x, d.w, d.h, planes, s1, s2, DwSweep<T>::BW,
                           DwSweep<T>::BH) &&
                 encode_3d(&a.tsg, dt, dy, d.w, d.h, planes, s1, s2, DwSweep<T>::BW,
                           DwSweep<T>::BH);
        a.use_tma = ok ? 1 : 0;
    }
    return true;
}

template <int K, typename T>
wt_status launch_dw_plane(const DwPlan& p, cudaStream_t stream, int* launches) {
    const DwArgs& a = p.a;
    const bool fast = a.use_tma && a.vec && a.H == a.Hp && a.W == a.Wp && !a.deep_global;
    auto kern = fast ? wt_dw_plane_kernel<K, T, true> : wt_dw_plane_kernel<K, T, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) !=
        cudaSuccess)
        return WT_ERR_CUDA;
    kern<<<(unsigned)p.grid, kDT, p.smem, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    ++*launches;
    return WT_OK;
}

template <int K, typename T>
wt_status launch_dw_k(const wt_desc& d, const void* x, const void* dy, const float* w0,
                      const float* b0, const float* s0, const float* wl, const float* sl,
                      float* dw0, float* db0, float* ds0, float* dwl, float* dsl, void* ws,
                      size_t ws_bytes, cudaStream_t stream, int* launches) {
    const int KP = FG<K>::KK + 1 + 4 * FG<K>::KK * d.levels;
    const size_t part_bytes = round256((size_t)d.c * d.n * KP * sizeof(float));
    DwPlan p = dw_layout<K, T>(d);
    const size_t need = kDwErrBytes + part_bytes + (size_t)p.grid * p.slot_bytes;
    if (ws == nullptr || ws_bytes < need) return WT_ERR_WORKSPACE;
    int* err = reinterpret_cast<int*>(ws) + kStatusBackwardWeight;
    float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + kDwErrBytes);
    float* slots = reinterpret_cast<float*>(static_cast<char*>(ws) + kDwErrBytes + part_bytes);
    if (!dw_prepare<K, T>(d, x, dy, part, slots, err, p)) return WT_ERR_UNSUPPORTED;
    if (cudaMemsetAsync(err, 0, 2 * sizeof(int), stream) != cudaSuccess) return WT_ERR_CUDA;
    wt_status st = launch_dw_plane<K, T>(p, stream, launches);
    if (st != WT_OK) return st;
    wt_dw_reduce_kernel<<<(unsigned)d.c, 128, (size_t)p.a.KP * sizeof(float), stream>>>(
        part, d.c, d.n, p.a.KP, K, d.levels, w0, b0, s0, wl, sl, dw0, db0, ds0, dwl, dsl, err);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    ++*launches;
    return WT_OK;
}

// Partial vectors only (no reduce), with the CTAs' slots in [slots, slots + slot_bytes_max):
// the grid shrinks to the slots that fit.
template <int K, typename T>
wt_status launch_dw_partials_k(const wt_desc& d, const void* x, const void* dy, float* part,
                               float* slots, size_t slots_bytes, int* err, cudaStream_t stream,
                               int* launches) {
    DwPlan p = dw_layout<K, T>(d);
    if (p.slot_bytes > 0) {
        const size_t fit = slots_bytes / p.slot_bytes;
        if (fit == 0) return WT_ERR_WORKSPACE;
        if ((size_t)p.grid > fit) p.grid = (int)fit;
    }
    if (!dw_prepare<K, T>(d, x, dy, part, slots, err, p)) return WT_ERR_UNSUPPORTED;
    return launch_dw_plane<K, T>(p, stream, launches);
}

}  // namespace

wt_status launch_dw_partials(const wt_desc& d, const void* x, const void* dy, float* part,
                             float* slots, size_t slots_bytes, int* err, cudaStream_t stream,
                             int* launches) {
    switch (d.k) {
#define WT_CASE(KV)                                                                           \
    case KV:                                                                                  \
        return with_io_type(d.io, [&](auto t) {                                               \
            return launch_dw_partials_k<KV, decltype(t)>(d, x, dy, part, slots, slots_bytes,  \
                                                         err, stream, launches);              \
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

wt_status launch_dw_reduce(const wt_desc& d, const float* part, int groups, const float* w0,
                           const float* b0, const float* s0, const float* wl, const float* sl,
                           float* dw0, float* db0, float* ds0, float* dwl, float* dsl,
                           const int* err, cudaStream_t stream, int* launches) {
    const int KP = (int)dw_partial_floats(d);
    wt_dw_reduce_kernel<<<(unsigned)d.c, 128, (size_t)KP * sizeof(float), stream>>>(
        part, d.c, groups, KP, d.k, d.levels, w0, b0, s0, wl, sl, dw0, db0, ds0, dwl, dsl, err);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    ++*launches;
    return WT_OK;
}

wt_status phase_clocks_backward_weight(int reset, unsigned long long* out) {
#ifdef WT_PHASE_CLOCKS
    if (cudaMemcpyFromSymbol(out, g_phase_dw, sizeof(g_phase_dw)) != cudaSuccess)
        return WT_ERR_CUDA;
    if (reset) {
        static const unsigned long long zero[32] = {0};
        if (cudaMemcpyToSymbol(g_phase_dw, zero, sizeof(zero)) != cudaSuccess) return WT_ERR_CUDA;
    }
    return WT_OK;
#else
    (void)reset;
    (void)out;
    return WT_ERR_UNSUPPORTED;
#endif
}

size_t dw_partial_floats(const wt_desc& d) {
    const int KK = d.k * d.k;
    return (size_t)KK + 1 + 4 * (size_t)KK * d.levels;
}

namespace {
// Plan of the plane kernel for d (shared memory, slots, grid).
bool dw_plan(const wt_desc& d, DwPlan& p) {
    switch (d.k) {
#define WT_CASE(KV)                                                                          \
    case KV:                                                                                 \
        p = with_io_type(d.io, [&](auto t) { return dw_layout<KV, decltype(t)>(d); });       \
        return true;
        WT_CASE(1)
        WT_CASE(3)
        WT_CASE(5)
        WT_CASE(7)
#undef WT_CASE
        default: return false;
    }
}
}  // namespace

size_t backward_weight_ws_bytes(const wt_desc& d) {
    DwPlan p;
    if (!dw_plan(d, p)) return 0;
    return kDwErrBytes + round256((size_t)d.c * d.n * dw_partial_floats(d) * sizeof(float)) +
           (size_t)p.grid * p.slot_bytes;
}

size_t backward_weight_slot_bytes(const wt_desc& d) {
    DwPlan p;
    if (!dw_plan(d, p)) return 0;
    return p.slot_bytes;
}

size_t backward_weight_smem_bytes(const wt_desc& d) {
    DwPlan p;
    if (!dw_plan(d, p)) return 0;
    return p.smem;
}

wt_status launch_backward_weight(const wt_desc& d, const void* x, const void* dy,
                                 const float* w0, const float* b0, const float* s0,
                                 const float* wl, const float* sl, float* dw0, float* db0,
                                 float* ds0, float* dwl, float* dsl, void* ws, size_t ws_bytes,
                                 cudaStream_t stream, int* launches) {
    switch (d.k) {
#define WT_CASE(KV)                                                                          \
    case KV:                                                                                 \
        return with_io_type(d.io, [&](auto t) {                                              \
            return launch_dw_k<KV, decltype(t)>(d, x, dy, w0, b0, s0, wl, sl, dw0, db0, ds0, \
                                                dwl, dsl, ws, ws_bytes, stream, launches);   \
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

}  // namespace wt
