// WTConv forward and backward-data kernel for sm_103a.
//
// Method: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware Reformulation"
// (Aflalo et al.). A persistent CTA (256 threads) walks (n, c) planes and evaluates the
// whole layer on each with one read of X and one write of Y in HBM:
//
//   deep phase (L >= 2) -- levels l = 2..L run at their own resolution: 32x32 output
//     tiles of the level's Haar subbands (§4.1 Eq. 5, recomputed on chip from the low-pass
//     carrier X^(l-1); level 2 reads X itself in 4x4 pixel blocks) are staged in shared
//     memory with an R-coefficient halo and filtered by the four folded k x k kernels
//     (§4.3 Eq. 8). The filtered subbands Z^(l) go to this CTA's scratch slot (tens of KB,
//     L2-resident). A last pass sums Eq. 7's terms of levels 2..L at level-1 resolution
//     (§4.2 Prop. 2: coefficient address by coordinate shifts, signs by coordinate bits)
//     and writes that sum in place of Z^(2).
//   full-resolution phase -- 64x64-pixel tiles: a TMA load brings the tile of X with a
//     2R halo (zero outside the plane) into shared memory while the previous tile is being
//     computed; one pass widens it to fp32 and forms the four level-1 subbands; four
//     streaming 4x4-block passes filter the subbands; a last pass computes the base k x k
//     convolution and stores, in the same write, base + level-1 synthesis (Eq. 7's l = 1
//     term) + the deep sum (TMA-loaded per tile).
//
// Backward-data is the same operator on dY with every kernel rotated by 180 degrees and
// no bias (§2.2 Eq. 1: the adjoint of analysis is synthesis; the adjoint of
// cross-correlation is correlation with the rotated kernel); `flip` selects it.
#include <mutex>

#include "wt_internal.h"
#include "wt_tile.cuh"
#include "wt_tma.cuh"

namespace wt {

constexpr int kFT = 256;  // threads per CTA

struct FwdArgs {
    CUtensorMap tmx;  // X: dims {W, H, planes}, box {XBW, XBH, 1}
    CUtensorMap tmd;  // deep sum: dims {4*W2, H2, slots}, box {64, 16, 1}
    const void* x;
    void* y;
    const float* w0f;
    const float* b0f;
    const float* wlf;
    float* zd;         // scratch: one slot of zd_slot floats per CTA (the deep sums)
    int* err;          // first word of the workspace: set on a stuck TMA wait
    long long zd_slot;
    long long planes;
    int C, H, W, L;
    int flip, vec, use_tma;
    int o_bar, o_raw, o_dblk, o_w, o_b, o_x, o_z;  // shared-memory regions (floats)
    int o_car[kMaxLevels + 1];                    // carriers X^(l), l = 2..L-1
    int o_zl[kMaxLevels + 1];                     // Z^(l), l = 3..L, interleaved [Hl][Wl][4]
};

constexpr int kDBytes = 16 * 64 * 4;  // deep-sum box: 16 level-2 rows x 16 positions x 4

// Folded weights of channel c into shared memory as packed pairs: slot 0 holds the base
// taps duplicated (w, w); slot 1 + 2(l-1) + p holds level l's band pair p as
// (w_{2p}, w_{2p+1}), each scaled by 2^-(l+1) (1/2 turns unnormalized subbands into
// Eq. 5's, 2^-l is Eq. 7's level weight). Taps are rotated by 180 degrees when `flip`.
template <int K>
__device__ __forceinline__ void load_weights(const FwdArgs& a, int c, float* wsm) {
    constexpr int KK = FG<K>::KK, WS = PG<K>::WS;
    const int nk = 1 + 4 * a.L;  // base + 4 bands per level
    for (int e = threadIdx.x; e < nk * KK; e += blockDim.x) {
        const int s = e / KK, uv = e - s * KK;
        const int src = a.flip ? (KK - 1 - uv) : uv;
        if (s == 0) {
            const float v = __ldg(a.w0f + (size_t)c * KK + src);
            wsm[2 * uv] = v;
            wsm[2 * uv + 1] = v;
        } else {
            const int l = 1 + (s - 1) / 4, b = (s - 1) & 3;
            const float v = ldexpf(1.0f, -(l + 1)) *
                            __ldg(a.wlf + (((size_t)(l - 1) * a.C + c) * 4 + b) * KK + src);
            wsm[(1 + 2 * (l - 1) + (b >> 1)) * WS + 2 * uv + (b & 1)] = v;
        }
    }
}

// Deep stage for level l: subbands of the 32x32 output tile at (ti0, tj0) with an R halo
// (zero outside the level grid) into the two band-pair tiles. Level 2 reads the 4x4
// pixel blocks of X (L2-resident), deeper levels the carrier X^(l-1) in shared memory.
// The trip count is a compile-time constant so that the loads of all cells issue early.
template <int K, typename T>
__device__ __forceinline__ void deep_stage(const FwdArgs& a, const T* xp, float* sm, int l,
                                           int ti0, int tj0) {
    constexpr int R = FG<K>::R, BT = FG<K>::BT;
    constexpr int PROW = PG<K>::PROW, PTILE = PG<K>::PTILE, PHALF = PG<K>::PHALF;
    constexpr int NIT = (BT * BT + kFT - 1) / kFT;
    const int Hl = a.H >> l, Wl = a.W >> l, Wp = a.W >> (l - 1);
    float* bs = sm + a.o_b;
    const float* carp = (l >= 3) ? sm + a.o_car[l - 1] : nullptr;
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
        const int idx = threadIdx.x + it * kFT;
        if (idx >= BT * BT) break;
        const int si = idx / BT, sj = idx - si * BT;
        const int gi = ti0 - R + si, gj = tj0 - R + sj;
        float4 u = f4_zero();
        if (gi >= 0 && gi < Hl && gj >= 0 && gj < Wl) {
            float ca, cb, cc, cd;
            carrier_block<T>(l, xp, a.W, carp, Wp, gi, gj, ca, cb, cc, cd);
            u = haar_u(ca, cb, cc, cd);
        }
        float* q = bs + si * PROW + 4 * pchunk(sj >> 1, PHALF) + 2 * (sj & 1);
        *reinterpret_cast<float2*>(q) = make_float2(u.x, u.y);
        *reinterpret_cast<float2*>(q + PTILE) = make_float2(u.z, u.w);
    }
}

// Low-pass carriers for the deep levels: X^(2) from the 4x4 pixel blocks of X (through
// the level-1 carrier, Eq. 5's LL twice), then X^(l) from X^(l-1) for l = 3..L-1.
template <typename T>
__device__ __forceinline__ void deep_carriers(const FwdArgs& a, const T* xp, float* sm) {
    {
        const int H2 = a.H >> 2, W2 = a.W >> 2, n = H2 * W2;
        float* c2 = sm + a.o_car[2];
        for (int base = threadIdx.x; base < n; base += 4 * kFT) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int p = base + u * kFT;
                if (p < n) {
                    const int i2 = p / W2, j2 = p - i2 * W2;
                    float ca, cb, cc, cd;
                    carrier_block<T>(2, xp, a.W, nullptr, 0, i2, j2, ca, cb, cc, cd);
                    c2[p] = 0.5f * (ca + cb + cc + cd);
                }
            }
        }
    }
    __syncthreads();
    for (int l = 3; l < a.L; ++l) {
        const int Hl = a.H >> l, Wl = a.W >> l, Wp = a.W >> (l - 1);
        const float* cp = sm + a.o_car[l - 1];
        float* cl = sm + a.o_car[l];
        for (int p = threadIdx.x; p < Hl * Wl; p += kFT) {
            const int i = p / Wl, j = p - i * Wl;
            const float* q = cp + (size_t)(2 * i) * Wp + 2 * j;
            cl[p] = 0.5f * (q[0] + q[1] + q[Wp] + q[Wp + 1]);
        }
        __syncthreads();
    }
}

template <int K, typename T>
__global__ void __launch_bounds__(kFT, 2) wt_fwd_plane_kernel(const __grid_constant__ FwdArgs a) {
    constexpr int R = FG<K>::R, PAD = FG<K>::PAD, XP = FG<K>::XPITCH;
    constexpr int PROW = PG<K>::PROW, PTILE = PG<K>::PTILE, WS = PG<K>::WS;
    constexpr int ZROW = PG<K>::ZROW, ZTILE = PG<K>::ZTILE;
    extern __shared__ __align__(128) float4 smem_f4[];
    float* sm = reinterpret_cast<float*>(smem_f4);
    uint64_t* bar_x = reinterpret_cast<uint64_t*>(sm + a.o_bar);
    uint64_t* bar_d = bar_x + 1;
    T* raw = reinterpret_cast<T*>(sm + a.o_raw);
    float* dblk = sm + a.o_dblk;
    float* wsm = sm + a.o_w;
    float* xs = sm + a.o_x;
    float* bs = sm + a.o_b;
    float* zs = sm + a.o_z;
    float* zslot = a.zd + (size_t)blockIdx.x * a.zd_slot;
    const size_t plane_elems = (size_t)a.H * a.W;
    const int tid = threadIdx.x;
    const bool leader = tid == 0;
    const int tiles_x = (a.W + kTile - 1) / kTile;
    const int ntiles = tiles_x * ((a.H + kTile - 1) / kTile);

    if (a.use_tma && leader) {
        mbar_init(bar_x, 1);
        mbar_init(bar_d, 1);
        fence_mbar_init();
    }
    __syncthreads();
    uint32_t ph_x = 0, ph_d = 0;
    bool failed = false;

    for (long long plane = blockIdx.x; plane < a.planes; plane += gridDim.x) {
        const int c = (int)(plane % a.C);
        const T* xp = reinterpret_cast<const T*>(a.x) + plane * plane_elems;
        T* yp = reinterpret_cast<T*>(a.y) + plane * plane_elems;
        __syncthreads();  // the previous plane is done with shared memory
        load_weights<K>(a, c, wsm);
        const float bias = (a.b0f != nullptr) ? __ldg(a.b0f + c) : 0.f;
        if (leader) {
            const long long nxt = plane + gridDim.x;
            if (a.use_tma && nxt < a.planes) {
                // next plane of this CTA: bring it into L2 while this one is computed
                const char* np =
                    reinterpret_cast<const char*>(a.x) + (size_t)nxt * plane_elems * sizeof(T);
                const size_t bytes = plane_elems * sizeof(T);
                for (size_t o = 0; o < bytes; o += (1u << 20)) {
                    const size_t nb = (bytes - o) < (1u << 20) ? (bytes - o) : (1u << 20);
                    prefetch_l2_bulk(np + o, (uint32_t)nb);
                }
            }
            if (a.use_tma) {  // first tile of this plane
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar_x, XBox<K, T>::BYTES);
                tma_load_3d(raw, &a.tmx, -XBox<K, T>::XOFF, -2 * R, (int)plane, bar_x);
            }
        }
        __syncthreads();

        // ---- deep phase (L >= 2) ----
        // carriers top-down; levels L..3 filtered into shared memory; level 2 last, its
        // filtered subbands combined at once with the deeper levels into Eq. 7's sum over
        // levels 2..L at level-1 resolution, written to the scratch slot: level-2 position
        // (i2, j2) holds the sums for level-1 positions (2i2 + a, 2j2 + b) as
        // (a, b) = (0,0), (0,1), (1,0), (1,1).
        if (a.L >= 2) {
            if (a.L >= 3) deep_carriers<T>(a, xp, sm);
            for (int l = a.L; l >= 2; --l) {
                const int Hl = a.H >> l, Wl = a.W >> l;
                for (int ti0 = 0; ti0 < Hl; ti0 += kCT) {
                    for (int tj0 = 0; tj0 < Wl; tj0 += kCT) {
                        deep_stage<K, T>(a, xp, sm, l, ti0, tj0);
                        __syncthreads();
                        {
                            // band pair pp = tid / 128, 2x4 output block (bi, bj)
                            const int pp = tid >> 7, bi = (tid >> 3) & 15, bj = tid & 7;
                            const int gi0 = ti0 + 2 * bi, gj0 = tj0 + 4 * bj;
                            if (gi0 < Hl && gj0 < Wl) {
                                f2x acc[2][4];
                                conv_pair_2x4<K>(bs + pp * PTILE + (2 * bi) * PROW, bj,
                                                 wsm + (1 + 2 * (l - 1) + pp) * WS, acc);
                                if (l >= 3) {
                                    float* zl = sm + a.o_zl[l];
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
                                        float* zr = zs + pp * ZTILE + (2 * bi + o) * ZROW + 8 * bj;
                                        const float2 q0 = upk2(acc[o][0]), q1 = upk2(acc[o][1]);
                                        const float2 q2 = upk2(acc[o][2]), q3 = upk2(acc[o][3]);
                                        reinterpret_cast<float4*>(zr)[0] = make_float4(q0.x, q0.y, q1.x, q1.y);
                                        reinterpret_cast<float4*>(zr)[1] = make_float4(q2.x, q2.y, q3.x, q3.y);
                                    }
                                }
                            }
                        }
                        __syncthreads();
                        if (l == 2) {
                            // deep sums of this level-2 tile's positions
                            float4* dsum = reinterpret_cast<float4*>(zslot);
#pragma unroll
                            for (int k = 0; k < (kCT * kCT) / kFT; ++k) {
                                const int p = tid + k * kFT, ti = p >> 5, tj = p & 31;
                                const int i2 = ti0 + ti, j2 = tj0 + tj;
                                if (i2 >= Hl || j2 >= Wl) continue;
                                const float2 za = *reinterpret_cast<const float2*>(zs + ti * ZROW + 2 * tj);
                                const float2 zb = *reinterpret_cast<const float2*>(zs + ZTILE + ti * ZROW + 2 * tj);
                                const float4 z = make_float4(za.x, za.y, zb.x, zb.y);
                                float v = 0.f;
                                for (int m = 3; m <= a.L; ++m) {
                                    const int sh = m - 2, Wm = a.W >> m;
                                    const float4 zm = reinterpret_cast<const float4*>(sm + a.o_zl[m])
                                        [(i2 >> sh) * Wm + (j2 >> sh)];
                                    v += synth_rt(zm, (i2 >> (m - 3)) & 1, (j2 >> (m - 3)) & 1);
                                }
                                dsum[(size_t)i2 * Wl + j2] =
                                    make_float4(synth<0, 0>(z) + v, synth<0, 1>(z) + v,
                                                synth<1, 0>(z) + v, synth<1, 1>(z) + v);
                            }
                        }
                    }
                }
            }
            fence_proxy_async_global();
            __syncthreads();
        }

        // ---- full-resolution phase ----
        const int by = tid >> 4, bx = tid & 15;  // 4x4-pixel block of this thread
        for (int t = 0; t < ntiles; ++t) {
            const int ty = t / tiles_x, tx = t - ty * tiles_x;
            const int y0 = ty * kTile, x0 = tx * kTile;
            if (a.L >= 2) {
                if (a.use_tma) {
                    if (leader) {
                        fence_proxy_async_smem();
                        mbar_arrive_expect_tx(bar_d, kDBytes);
                        tma_load_3d(dblk, &a.tmd, x0, y0 >> 2, (int)blockIdx.x, bar_d);
                    }
                } else {
                    // plain copy of the 16x16 level-2 block of deep sums (zero outside)
                    const int H2 = a.H >> 2, W2 = a.W >> 2;
                    const float4* z2 = reinterpret_cast<const float4*>(zslot);
                    const int i0 = y0 >> 2, j0 = x0 >> 2;
                    const int i = tid >> 4, j = tid & 15;
                    float4 v = f4_zero();
                    if (i0 + i < H2 && j0 + j < W2) v = z2[(size_t)(i0 + i) * W2 + j0 + j];
                    reinterpret_cast<float4*>(dblk)[tid] = v;
                }
            }
            if (a.use_tma) {
                const bool ok = mbar_wait_bounded(bar_x, ph_x);
                ph_x ^= 1;
                if (__syncthreads_or(!ok)) {
                    failed = true;
                    break;
                }
                convert_raw<K, T>(raw, xs, bs, a.L >= 1);
                __syncthreads();
                if (leader && t + 1 < ntiles) {  // prefetch the next tile of this plane
                    const int ny = (t + 1) / tiles_x, nx = (t + 1) - ny * tiles_x;
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(bar_x, XBox<K, T>::BYTES);
                    tma_load_3d(raw, &a.tmx, nx * kTile - XBox<K, T>::XOFF, ny * kTile - 2 * R,
                                (int)plane, bar_x);
                }
            } else {
                stage_tile<K, T>(xp, a.H, a.W, a.vec, xs, y0, x0);
                __syncthreads();
                if (a.L >= 1) {
                    pair_bands_from_tile<K>(xs, bs);
                    __syncthreads();
                }
            }
            if (a.L >= 1) {
                // level-1 filters: 2 band pairs x 128 blocks of 2x4 coefficients, one per thread
                const int pp = tid >> 7, bi = (tid >> 3) & 15, bj = tid & 7;
                if (y0 / 2 + 2 * bi < a.H / 2 && x0 / 2 + 4 * bj < a.W / 2) {
                    f2x acc[2][4];
                    conv_pair_2x4<K>(bs + pp * PTILE + (2 * bi) * PROW, bj, wsm + (1 + pp) * WS,
                                     acc);
#pragma unroll
                    for (int o = 0; o < 2; ++o) {
                        float* zr = zs + pp * ZTILE + (2 * bi + o) * ZROW + 8 * bj;
                        const float2 q0 = upk2(acc[o][0]), q1 = upk2(acc[o][1]);
                        const float2 q2 = upk2(acc[o][2]), q3 = upk2(acc[o][3]);
                        reinterpret_cast<float4*>(zr)[0] = make_float4(q0.x, q0.y, q1.x, q1.y);
                        reinterpret_cast<float4*>(zr)[1] = make_float4(q2.x, q2.y, q3.x, q3.y);
                    }
                }
                __syncthreads();
            }
            if (a.L >= 2 && a.use_tma) {
                const bool ok = mbar_wait_bounded(bar_d, ph_d);
                ph_d ^= 1;
                if (__syncthreads_or(!ok)) {
                    failed = true;
                    break;
                }
            }
            const int gy = y0 + 4 * by, gx = x0 + 4 * bx;
            if (gy < a.H && gx < a.W) {
                f2x acc2[4][2];
                const f2x bias2 = pk2(bias, bias);
#pragma unroll
                for (int o = 0; o < 4; ++o) acc2[o][0] = acc2[o][1] = bias2;
                conv_base_4x4<K>(xs + (4 * by + R) * XP + 4 * bx + R + PAD, XP, wsm, acc2);
                if (a.L >= 1) {
                    float4 d = f4_zero();
                    if (a.L >= 2) d = reinterpret_cast<const float4*>(dblk)[tid];
                    const float dv[2][2] = {{d.x, d.y}, {d.z, d.w}};
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        // (LL, LH) and (HL, HH) of coefficients (2by+i, 2bx) and (2by+i, 2bx+1)
                        const float4 za = *reinterpret_cast<const float4*>(
                            zs + (2 * by + i) * ZROW + 4 * bx);
                        const float4 zb = *reinterpret_cast<const float4*>(
                            zs + ZTILE + (2 * by + i) * ZROW + 4 * bx);
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
            __syncthreads();
        }
        if (failed) break;
    }
    if (failed && leader && a.err != nullptr) atomicExch(a.err, kErrTmaTimeout);
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

struct FwdPlan {
    FwdArgs a;
    size_t smem = 0;
    int grid = 0;
    size_t ws_bytes = 0;
};

constexpr size_t kErrWordBytes = 256;  // the workspace starts with the error word

template <int K, typename T>
FwdPlan fwd_plan(const wt_desc& d) {
    FwdPlan p;
    FwdArgs& a = p.a;
    const int L = d.levels;
    int off = 0;
    a.o_bar = off;
    off += 32;  // two mbarriers, padded to 128 bytes
    a.o_raw = off;
    off += round32((XBox<K, T>::BYTES + 3) / 4);
    a.o_dblk = off;
    off += (L >= 2) ? kDBytes / 4 : 0;
    a.o_w = off;
    off += PG<K>::WS * (1 + 2 * L);
    off = round32(off);
    a.o_b = off;
    off += 2 * PG<K>::PTILE;
    off = round4(off);
    a.o_z = off;
    off += 2 * PG<K>::ZTILE;
    // the full-resolution X tile and the deep-phase carriers + Z^(l >= 3) share a region
    const int alias0 = off;
    a.o_x = off;
    const int xend = off + FG<K>::XROWS * FG<K>::XPITCH;
    int cp = alias0;
    for (int l = 0; l <= kMaxLevels; ++l) a.o_car[l] = a.o_zl[l] = 0;
    for (int l = 2; l < L; ++l) {
        a.o_car[l] = cp;
        cp += round4((d.h >> l) * (d.w >> l));
    }
    for (int l = 3; l <= L; ++l) {
        a.o_zl[l] = cp;
        cp += 4 * (d.h >> l) * (d.w >> l);
    }
    const int total = xend > cp ? xend : cp;
    p.smem = (size_t)total * sizeof(float);
    // deep-sum slot: [H/4][W/4][4] fp32
    a.zd_slot = (L >= 2) ? ((4LL * (d.h >> 2) * (d.w >> 2) + 63) & ~63LL) : 0;
    const long long planes = (long long)d.n * d.c;
    int occ = (int)((228 * 1024) / (p.smem + 1024));
    if (occ > 2) occ = 2;
    if (occ < 1) occ = 1;
    long long grid = (long long)kNumSMs * occ;
    if (grid > planes) grid = planes;
    p.grid = (int)grid;
    p.ws_bytes =
        kErrWordBytes + ((L >= 2) ? (size_t)grid * (size_t)a.zd_slot * sizeof(float) : 0);
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
    a.w0f = w0f;
    a.b0f = flip ? nullptr : b0f;
    a.wlf = wlf;
    a.err = reinterpret_cast<int*>(ws);
    a.zd = reinterpret_cast<float*>(static_cast<char*>(ws) + kErrWordBytes);
    a.planes = (long long)d.n * d.c;
    a.C = d.c;
    a.H = d.h;
    a.W = d.w;
    a.L = d.levels;
    a.flip = flip;
    a.vec = (d.w % 4 == 0) ? 1 : 0;
    // TMA needs 16-byte row strides; otherwise the tile is staged with plain loads
    const size_t esize = sizeof(T);
    const CUtensorMapDataType dt =
        sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    a.use_tma = 0;
    if (((size_t)d.w * esize) % 16 == 0) {
        bool ok = encode_3d(&a.tmx, dt, x, d.w, d.h, (unsigned long long)d.n * d.c,
                            (unsigned long long)d.w * esize,
                            (unsigned long long)d.w * d.h * esize, XBox<K, T>::XBW,
                            XBox<K, T>::XBH);
        if (ok && d.levels >= 2) {
            const unsigned long long w2 = d.w >> 2, h2 = d.h >> 2;
            ok = encode_3d(&a.tmd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.zd, 4 * w2, h2,
                           (unsigned long long)p.grid, 16 * w2, (unsigned long long)a.zd_slot * 4,
                           64, 16);
        }
        a.use_tma = ok ? 1 : 0;
    }
    if (cudaMemsetAsync(a.err, 0, sizeof(int), stream) != cudaSuccess) return WT_ERR_CUDA;
    auto kern = wt_fwd_plane_kernel<K, T>;
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
    FwdPlan p = (d.io == WT_BF16) ? fwd_plan<K, __nv_bfloat16>(d) : fwd_plan<K, float>(d);
    *smem = p.smem;
    *ws = p.ws_bytes;
    return true;
}

}  // namespace

wt_status launch_forward(const wt_desc& d, const void* x, const float* w0f, const float* b0f,
                         const float* wlf, void* y, int flip, void* ws, size_t ws_bytes,
                         cudaStream_t stream, int* launches) {
    const bool bf = d.io == WT_BF16;
    switch (d.k) {
#define WT_CASE(KV)                                                                          \
    case KV:                                                                                 \
        return bf ? launch_fwd_k<KV, __nv_bfloat16>(d, x, w0f, b0f, wlf, y, flip, ws,        \
                                                    ws_bytes, stream, launches)              \
                  : launch_fwd_k<KV, float>(d, x, w0f, b0f, wlf, y, flip, ws, ws_bytes,      \
                                            stream, launches);
        WT_CASE(1)
        WT_CASE(3)
        WT_CASE(5)
        WT_CASE(7)
#undef WT_CASE
        default:
            return WT_ERR_UNSUPPORTED;
    }
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
