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
// Kernel 1 (wt_dw_plane_kernel): one CTA (256 threads) per (c, n) plane.
//   deep levels (l >= 2): 32x32 tiles of the level's subbands of X (R halo) and dY are
//     staged as band-pair tiles, (LL, LH) and (HL, HH), from on-chip carriers (level 2
//     from the 4x4 pixel blocks of X and dY); threads 0-127 correlate pair 0 and threads
//     128-255 pair 1 with packed f32x2 FMAs (2x4 coefficient blocks), and the sums are
//     flushed after each level by recursive-halving warp reductions in a fixed order.
//   full resolution: 64x64-pixel tiles of X (2R halo) and dY arrive by TMA; the next
//     tile's load is issued as soon as the current one has been widened to fp32, so it
//     overlaps the correlations. Threads 0-127 run the base correlation (4x4 pixel
//     blocks), threads 128-255 the level-1 band-pair correlations (4x4 coefficient
//     blocks). Each thread keeps its partial sums in registers for the whole plane.
//   The per-plane partial vector [dW~0 | db~ | dW~^(l)_b] goes to the workspace.
// Kernel 2 (wt_dw_reduce_kernel): per channel, sums the N partial vectors in a fixed
//   order and applies the gradient unfolding of §4.3 Eq. 9.
// No atomics anywhere: results are bitwise reproducible.
#include "wt_internal.h"
#include "wt_tile.cuh"
#include "wt_tma.cuh"

namespace wt {

constexpr int kDT = 256;  // threads per CTA

struct DwArgs {
    CUtensorMap tmx;  // X: dims {W, H, planes}, box {XBW, XBH, 1} (2R halo)
    CUtensorMap tmg;  // dY: dims {W, H, planes}, box {64, 64, 1}
    const void* x;
    const void* dy;
    float* part;  // [C][N][KP]
    int* err;     // set when a TMA wait times out (may be null)
    int N, C, H, W, L;
    int Hp, Wp;  // the plane padded with zeros to multiples of 2^L: level l is (Hp, Wp) >> l
    int vec, use_tma;
    int KP;
    int o_bar, o_rawx, o_rawg, o_acc, o_red, o_xb, o_gb, o_x, o_g;  // shared memory (floats)
    // deep carriers X^(l), dY^(l) (l = 2..L-1): in shared memory, or (deep_global) in a
    // per-plane region of car_floats floats at car + plane * car_floats
    int deep_global;
    float* car;
    long long car_floats;
    int o_carx[kMaxLevels + 1], o_cary[kMaxLevels + 1];
};

// dY subband-pair tiles (no halo): 32 rows x 32 cells, 16-byte chunks split even/odd.
constexpr int kGHalf = 8;             // chunks per half row
constexpr int kGRow = 8 * kGHalf;     // floats per row
constexpr int kGTile = kCT * kGRow;   // floats per pair tile

// Deep stage for level l: X subbands with an R halo into the X pair tiles, dY subbands of
// the tile's own cells into the dY pair tiles; carriers X^(l), dY^(l) for l < L.
template <int K, typename T, bool FAST>
__device__ __forceinline__ void dw_deep_stage(const DwArgs& a, const T* xp, const T* gp,
                                              float* sm, float* cbase, int l, int ti0,
                                              int tj0) {
    constexpr int R = FG<K>::R, BT = FG<K>::BT;
    constexpr int PROW = PG<K>::PROW, PTILE = PG<K>::PTILE, PHALF = PG<K>::PHALF;
    constexpr int NIT = (BT * BT + kDT - 1) / kDT;
    const int Hl = a.Hp >> l, Wl = a.Wp >> l, Wp = a.Wp >> (l - 1);
    float* xb = sm + a.o_xb;
    float* gb = sm + a.o_gb;
    const float* cpx = (l >= 3) ? cbase + a.o_carx[l - 1] : nullptr;
    const float* cpy = (l >= 3) ? cbase + a.o_cary[l - 1] : nullptr;
    float* clx = (l < a.L) ? cbase + a.o_carx[l] : nullptr;
    float* cly = (l < a.L) ? cbase + a.o_cary[l] : nullptr;
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
        const int idx = threadIdx.x + it * kDT;
        if (idx >= BT * BT) break;
        const int si = idx / BT, sj = idx - si * BT;
        const int gi = ti0 - R + si, gj = tj0 - R + sj;
        const bool inner = si >= R && si < R + kCT && sj >= R && sj < R + kCT;
        float4 ux = f4_zero(), ug = f4_zero();
        if (gi >= 0 && gi < Hl && gj >= 0 && gj < Wl) {
            float ca, cb, cc, cd;
            carrier_block<T, FAST>(l, xp, a.H, a.W, a.vec, cpx, Wp, gi, gj, ca, cb, cc, cd);
            ux = haar_u(ca, cb, cc, cd);
            if (inner) {
                if (clx) clx[gi * Wl + gj] = 0.5f * ux.x;
                carrier_block<T, FAST>(l, gp, a.H, a.W, a.vec, cpy, Wp, gi, gj, ca, cb, cc, cd);
                ug = haar_u(ca, cb, cc, cd);
                if (cly) cly[gi * Wl + gj] = 0.5f * ug.x;
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

// Widen the TMA-staged raw dY tile (64x64) to the fp32 dY tile and, when `bands`, form
// its level-1 unnormalized subbands in the dY pair tiles. One item = 2x4 pixels. Returns
// this thread's sum of the dY values it converted.
template <typename T>
__device__ __forceinline__ float convert_raw_dy(const T* raw, float* gs, float* gb, bool bands) {
    float sum = 0.f;
    for (int idx = threadIdx.x; idx < kCT * (kCT / 2); idx += blockDim.x) {
        const int ci = idx >> 4, m = idx & 15;
        const T* r0 = raw + (2 * ci) * kTile + 4 * m;
        const float2 a0 = ld2_smem<T>(r0), a1 = ld2_smem<T>(r0 + 2);
        const float2 b0 = ld2_smem<T>(r0 + kTile), b1 = ld2_smem<T>(r0 + kTile + 2);
        float* d0 = gs + (2 * ci) * kTile + 4 * m;
        *reinterpret_cast<float4*>(d0) = make_float4(a0.x, a0.y, a1.x, a1.y);
        *reinterpret_cast<float4*>(d0 + kTile) = make_float4(b0.x, b0.y, b1.x, b1.y);
        sum += ((a0.x + a0.y) + (a1.x + a1.y)) + ((b0.x + b0.y) + (b1.x + b1.y));
        if (bands) {
            const float4 u = haar_u(a0.x, a0.y, b0.x, b0.y);
            const float4 v = haar_u(a1.x, a1.y, b1.x, b1.y);
            float* q = gb + ci * kGRow + 4 * pchunk(m, kGHalf);
            *reinterpret_cast<float4*>(q) = make_float4(u.x, u.y, v.x, v.y);
            *reinterpret_cast<float4*>(q + kGTile) = make_float4(u.z, u.w, v.z, v.w);
        }
    }
    return sum;
}

// Non-TMA staging of the dY tile (fp32 tile + pair tiles), zero outside the plane.
// Returns this thread's sum of the dY values it staged.
template <typename T>
__device__ __forceinline__ float stage_dy_plain(const T* gp, int H, int W, float* gs, float* gb,
                                                bool bands, int y0, int x0) {
    float sum = 0.f;
    for (int idx = threadIdx.x; idx < kCT * kCT; idx += blockDim.x) {
        const int ci = idx / kCT, cj = idx - ci * kCT;
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int gy = y0 + 2 * ci + (e >> 1), gx = x0 + 2 * cj + (e & 1);
            v[e] = (gy < H && gx < W) ? IO<T>::ld(gp + (size_t)gy * W + gx) : 0.f;
        }
        float* d0 = gs + (2 * ci) * kTile + 2 * cj;
        d0[0] = v[0]; d0[1] = v[1]; d0[kTile] = v[2]; d0[kTile + 1] = v[3];
        sum += (v[0] + v[1]) + (v[2] + v[3]);
        if (bands) {
            const float4 u = haar_u(v[0], v[1], v[2], v[3]);
            float* q = gb + ci * kGRow + 4 * pchunk(cj >> 1, kGHalf) + 2 * (cj & 1);
            *reinterpret_cast<float2*>(q) = make_float2(u.x, u.y);
            *reinterpret_cast<float2*>(q + kGTile) = make_float2(u.z, u.w);
        }
    }
    return sum;
}

// One compensated (Kahan) step of this thread's running sum red[tid] (with its
// compensation in red[blockDim.x + tid]): sum += v.
__device__ __forceinline__ void kahan_add(float* red, float v) {
    const int t = threadIdx.x, n = blockDim.x;
    const float s = red[t], c = red[n + t];
    const float y = v - c;
    const float u = s + y;
    red[n + t] = (u - s) - y;
    red[t] = u;
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
    constexpr int R = FG<K>::R, KK = FG<K>::KK, PAD = FG<K>::PAD, XP = FG<K>::XPITCH;
    constexpr int PROW = PG<K>::PROW, PTILE = PG<K>::PTILE;
    extern __shared__ __align__(128) float4 smem_f4[];
    float* sm = reinterpret_cast<float*>(smem_f4);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + a.o_bar);
    T* rawx = reinterpret_cast<T*>(sm + a.o_rawx);
    T* rawg = reinterpret_cast<T*>(sm + a.o_rawg);
    float* acc_sm = sm + a.o_acc;
    float* red = sm + a.o_red;  // [8 warps][64]
    float* xb = sm + a.o_xb;
    float* gb = sm + a.o_gb;
    float* xs = sm + a.o_x;
    float* gs = sm + a.o_g;
    const int tid = threadIdx.x, warp = tid >> 5;
    const bool leader = tid == 0;
    const bool use_tma = FAST || a.use_tma;

    const int c = blockIdx.x, n = blockIdx.y;
    const long long plane = (long long)n * a.C + c;
    const size_t plane_elems = (size_t)a.H * a.W;
    const T* xp = reinterpret_cast<const T*>(a.x) + plane * plane_elems;
    const T* gp = reinterpret_cast<const T*>(a.dy) + plane * plane_elems;
    const int tiles_x = (a.W + kTile - 1) / kTile;
    const int ntiles = tiles_x * ((a.H + kTile - 1) / kTile);
    constexpr int BYTES = XBox<K, T>::BYTES + kTile * kTile * (int)sizeof(T);

    for (int e = tid; e < a.KP; e += kDT) acc_sm[e] = 0.f;
    if (use_tma && leader) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (use_tma && leader) {  // first tile, in flight during the deep levels
        mbar_arrive_expect_tx(bar, BYTES);
        tma_load_3d(rawx, &a.tmx, -XBox<K, T>::XOFF, -2 * R, (int)plane, bar);
        tma_load_3d(rawg, &a.tmg, 0, 0, (int)plane, bar);
    }
    uint32_t ph = 0;

    // ---- deep levels l = 2..L: band pair pp = tid / 128, 2x4 block per thread ----
    float* cbase = (!FAST && a.deep_global) ? a.car + plane * a.car_floats : sm;  // carriers
    for (int l = 2; l <= a.L; ++l) {
        const int Hl = a.Hp >> l, Wl = a.Wp >> l;
        const int pp = tid >> 7, bi = (tid >> 3) & 15, bj = tid & 7;
        f2x accd[KK];
#pragma unroll
        for (int q = 0; q < KK; ++q) accd[q] = 0ull;
        for (int ti0 = 0; ti0 < Hl; ti0 += kCT) {
            for (int tj0 = 0; tj0 < Wl; tj0 += kCT) {
                dw_deep_stage<K, T, FAST>(a, xp, gp, sm, cbase, l, ti0, tj0);
                __syncthreads();
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
                __syncthreads();
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
    }

    // ---- full resolution: warps 0-3 base path, warps 4-7 level-1 band pairs ----
    const bool base_role = (a.L == 0) || (tid < 128);
    f2x acc[KK];
#pragma unroll
    for (int q = 0; q < KK; ++q) acc[q] = 0ull;
    // sum of dY, taken while converting the dY tiles: a register partial over at most 16
    // tiles, folded into a compensated (Kahan) running sum so that planes of millions of
    // pixels keep the fp32 sum accurate to a few ulps. The running sum and its compensation
    // live in this thread's two words of `red` (idle until the final flush).
    red[tid] = 0.f;
    red[kDT + tid] = 0.f;
    float dpart = 0.f;
    bool failed = false;
    for (int t = 0; t < ntiles; ++t) {
        const int ty = t / tiles_x, tx = t - ty * tiles_x;
        const int y0 = ty * kTile, x0 = tx * kTile;
        if (use_tma) {
            const bool ok = mbar_wait_bounded(bar, ph);
            ph ^= 1;
            if (__syncthreads_or(!ok)) {
                failed = true;
                break;
            }
            convert_raw<K, T>(rawx, xs, xb, a.L >= 1);
            dpart += convert_raw_dy<T>(rawg, gs, gb, a.L >= 1);
            __syncthreads();
            if (leader && t + 1 < ntiles) {
                const int ny = (t + 1) / tiles_x, nx = (t + 1) - ny * tiles_x;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, BYTES);
                tma_load_3d(rawx, &a.tmx, nx * kTile - XBox<K, T>::XOFF, ny * kTile - 2 * R,
                            (int)plane, bar);
                tma_load_3d(rawg, &a.tmg, nx * kTile, ny * kTile, (int)plane, bar);
            }
        } else {
            stage_tile<K, T>(xp, a.H, a.W, a.vec, xs, y0, x0);
            dpart += stage_dy_plain<T>(gp, a.H, a.W, gs, gb, a.L >= 1, y0, x0);
            __syncthreads();
            if (a.L >= 1) {
                pair_bands_from_tile<K>(xs, xb);
                __syncthreads();
            }
        }
        if ((t & 15) == 15 || t + 1 == ntiles) {
            kahan_add(red, dpart);
            dpart = 0.f;
        }
        if (base_role) {
            const int nb = (a.L == 0) ? 1 : 2;
            for (int k = 0; k < nb; ++k) {
                const int blk = tid + kDT / 2 * k;  // L == 0: tid covers all 256 blocks
                const int by = blk >> 4, bx = blk & 15;
                if (y0 + 4 * by >= a.H || x0 + 4 * bx >= a.W) continue;
                f2x g[4][2];
#pragma unroll
                for (int o = 0; o < 4; ++o) {
                    const float4 tv = *reinterpret_cast<const float4*>(gs + (4 * by + o) * kTile + 4 * bx);
                    g[o][0] = pk2(tv.x, tv.y);
                    g[o][1] = pk2(tv.z, tv.w);
                }
                corr_base_4x4<K>(xs + (4 * by + R) * XP + 4 * bx + R + PAD, XP, g, acc);
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
        __syncthreads();
    }
    if (failed) {
        if (leader && a.err != nullptr) atomicExch(a.err, kErrTmaTimeout);
        return;
    }

    // ---- flush: fixed-order reductions into acc_sm, then the partial vector ----
    const float dbs = red[tid] - red[kDT + tid];
    __syncthreads();  // every thread has read its sum before `red` takes the warp totals
    warp_totals_to<KK, 2 * KK + 1>(acc, dbs, red + warp * 128);
    __syncthreads();
    const int nbase = (a.L == 0) ? 8 : 4;
    for (int e = tid; e <= KK; e += kDT) {
        // base taps: even + odd column halves of each base warp; e == KK: the sum of dY,
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
}

// Per channel: fixed-order sum of the N partial vectors, then §4.3 Eq. 9.
__global__ void wt_dw_reduce_kernel(const float* part, int C, int G, int KP, int K, int L,
                                    const float* w0, const float* b0, const float* s0,
                                    const float* wl, const float* sl, float* dw0, float* db0,
                                    float* ds0, float* dwl, float* dsl) {
    extern __shared__ float tot[];
    const int c = blockIdx.x;
    const int KK = K * K;
    for (int e = threadIdx.x; e < KP; e += blockDim.x) {
        float s = 0.f;
        for (int gi = 0; gi < G; ++gi) s += part[((size_t)c * G + gi) * KP + e];
        // level entries were accumulated from unnormalized subbands on both sides (4x)
        tot[e] = (e > KK) ? 0.25f * s : s;
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

constexpr size_t kDwErrBytes = 256;  // the workspace starts with a status word
constexpr size_t kTwoCtaSmem = 228 * 1024 / 2 - 1024;  // two CTAs per SM still fit

size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

template <int K, typename T>
void dw_layout(const wt_desc& d, DwArgs& a, size_t& smem_bytes) {
    constexpr int KK = FG<K>::KK;
    const int L = d.levels;
    a.KP = KK + 1 + 4 * KK * L;
    int off = 0;
    a.o_bar = off;
    off += 32;
    a.o_rawx = off;
    off += round32((XBox<K, T>::BYTES + 3) / 4);
    a.o_rawg = off;
    off += round32(kTile * kTile * (int)sizeof(T) / 4);
    a.o_acc = off;
    off += round32(a.KP);
    a.o_red = off;
    off += 8 * 128;
    a.o_xb = off;
    off += 2 * PG<K>::PTILE;
    off = round4(off);
    a.o_gb = off;
    off += 2 * kGTile;
    // the fp32 X and dY tiles share their region with the deep-level carriers
    const int alias0 = off;
    a.o_x = off;
    off += FG<K>::XROWS * FG<K>::XPITCH;
    off = round4(off);
    a.o_g = off;
    off += kTile * kTile;
    int cp = 0;
    for (int l = 0; l <= kMaxLevels; ++l) a.o_carx[l] = a.o_cary[l] = 0;
    for (int l = 2; l < L; ++l) {
        const int sz = round4((padded_side(d.h, d.levels) >> l) *
                              (padded_side(d.w, d.levels) >> l));
        a.o_carx[l] = cp;
        cp += sz;
        a.o_cary[l] = cp;
        cp += sz;
    }
    // the carriers stay in shared memory unless they would lower the occupancy the tiles
    // alone allow (two CTAs per SM for k <= 5 when the tiles fit it, else one) or not fit
    // at all; then they move to the workspace
    const size_t two = (K >= 7) ? kMaxSmemPerBlock : kTwoCtaSmem;
    const size_t limit = ((size_t)off * sizeof(float) <= two) ? two : kMaxSmemPerBlock;
    const int local_end = alias0 + cp > off ? alias0 + cp : off;
    a.deep_global = (cp > 0 && (size_t)local_end * sizeof(float) > limit) ? 1 : 0;
    a.car_floats = a.deep_global ? (((long long)cp + 63) & ~63LL) : 0;
    if (!a.deep_global)
        for (int l = 2; l < L; ++l) {
            a.o_carx[l] += alias0;
            a.o_cary[l] += alias0;
        }
    const int total = a.deep_global ? off : local_end;
    smem_bytes = (size_t)total * sizeof(float);
}

// Fill the kernel arguments (layout, pointers, tensor maps) for one launch.
template <int K, typename T>
bool dw_prepare(const wt_desc& d, const void* x, const void* dy, float* part, float* car,
                int* err, DwArgs& a, size_t& smem) {
    dw_layout<K, T>(d, a, smem);
    if (smem > kMaxSmemPerBlock) return false;
    if (a.deep_global && car == nullptr) return false;
    a.car = car;
    a.x = x;
    a.dy = dy;
    a.part = part;
    a.err = err;
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
        const bool ok =
            encode_3d(&a.tmx, dt, x, d.w, d.h, planes, s1, s2, XBox<K, T>::XBW, XBox<K, T>::XBH) &&
            encode_3d(&a.tmg, dt, dy, d.w, d.h, planes, s1, s2, kTile, kTile);
        a.use_tma = ok ? 1 : 0;
    }
    return true;
}

template <int K, typename T>
wt_status launch_dw_plane(const DwArgs& a, size_t smem, const wt_desc& d, cudaStream_t stream,
                          int* launches) {
    const bool fast = a.use_tma && a.vec && a.H == a.Hp && a.W == a.Wp && !a.deep_global;
    auto kern = fast ? wt_dw_plane_kernel<K, T, true> : wt_dw_plane_kernel<K, T, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return WT_ERR_CUDA;
    kern<<<dim3((unsigned)d.c, (unsigned)d.n), kDT, smem, stream>>>(a);
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
    DwArgs a;
    size_t smem = 0;
    dw_layout<K, T>(d, a, smem);
    const size_t need = kDwErrBytes + part_bytes +
                        (size_t)d.c * d.n * (size_t)a.car_floats * sizeof(float);
    if (ws == nullptr || ws_bytes < need) return WT_ERR_WORKSPACE;
    int* err = reinterpret_cast<int*>(ws);
    float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + kDwErrBytes);
    float* car = reinterpret_cast<float*>(static_cast<char*>(ws) + kDwErrBytes + part_bytes);
    if (!dw_prepare<K, T>(d, x, dy, part, car, err, a, smem)) return WT_ERR_UNSUPPORTED;
    if (cudaMemsetAsync(err, 0, sizeof(int), stream) != cudaSuccess) return WT_ERR_CUDA;
    wt_status st = launch_dw_plane<K, T>(a, smem, d, stream, launches);
    if (st != WT_OK) return st;
    wt_dw_reduce_kernel<<<(unsigned)d.c, 128, (size_t)a.KP * sizeof(float), stream>>>(
        part, d.c, d.n, a.KP, K, d.levels, w0, b0, s0, wl, sl, dw0, db0, ds0, dwl, dsl);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    ++*launches;
    return WT_OK;
}

template <int K, typename T>
wt_status launch_dw_partials_k(const wt_desc& d, const void* x, const void* dy, float* part,
                               cudaStream_t stream, int* launches) {
    DwArgs a;
    size_t smem = 0;
    // (no carrier region here: shapes whose carriers need the workspace are unsupported)
    if (!dw_prepare<K, T>(d, x, dy, part, nullptr, nullptr, a, smem)) return WT_ERR_UNSUPPORTED;
    return launch_dw_plane<K, T>(a, smem, d, stream, launches);
}

}  // namespace

wt_status launch_dw_partials(const wt_desc& d, const void* x, const void* dy, float* part,
                             cudaStream_t stream, int* launches) {
    switch (d.k) {
#define WT_CASE(KV)                                                                           \
    case KV:                                                                                  \
        return with_io_type(d.io, [&](auto t) {                                               \
            return launch_dw_partials_k<KV, decltype(t)>(d, x, dy, part, stream, launches);   \
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
                           cudaStream_t stream, int* launches) {
    const int KP = (int)dw_partial_floats(d);
    wt_dw_reduce_kernel<<<(unsigned)d.c, 128, (size_t)KP * sizeof(float), stream>>>(
        part, d.c, groups, KP, d.k, d.levels, w0, b0, s0, wl, sl, dw0, db0, ds0, dwl, dsl);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    ++*launches;
    return WT_OK;
}

size_t dw_partial_floats(const wt_desc& d) {
    const int KK = d.k * d.k;
    return (size_t)KK + 1 + 4 * (size_t)KK * d.levels;
}

namespace {
// Layout of the plane kernel for d (shared memory bytes and the carriers' placement).
bool dw_plan(const wt_desc& d, DwArgs& a, size_t& smem) {
    switch (d.k) {
#define WT_CASE(KV)                                                                          \
    case KV:                                                                                 \
        with_io_type(d.io, [&](auto t) { dw_layout<KV, decltype(t)>(d, a, smem); return 0; }); \
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
    DwArgs a;
    size_t smem = 0;
    if (!dw_plan(d, a, smem)) return 0;
    return kDwErrBytes + round256((size_t)d.c * d.n * dw_partial_floats(d) * sizeof(float)) +
           (size_t)d.c * d.n * (size_t)a.car_floats * sizeof(float);
}

size_t backward_weight_smem_bytes(const wt_desc& d) {
    DwArgs a;
    size_t smem = 0;
    if (!dw_plan(d, a, smem)) return 0;
    return smem;
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
