// WTConv backward-weight kernels for sm_103a.
//
// Method: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware Reformulation"
// (Aflalo et al.). The layer is linear in every folded kernel, so the gradient of the
// level-l folded kernel W~^(l) is the correlation of the level-l Haar coefficients of dY
// with those of X (the adjoint of the Eq. 7 synthesis is the Haar analysis, §2.2 Eq. 1):
//   dW~^(l)_b[u][v] = sum_{n,i,j} A_l(dY)_b[i][j] A_l(X)_b[i+u-R][j+v-R]
// and the base gradients are dW~^(0)[u][v] = sum dY[y][x] X[y+u-R][x+v-R], db~ = sum dY.
// Nothing but X and dY is read from HBM: both Haar cascades are recomputed on chip.
//
// Kernel 1 (wt_dw_plane_kernel): CTA (c, g) walks the planes n = g, g+G, ... of channel
//   c. Levels >= 2 are staged from on-chip carriers exactly like the forward's deep phase;
//   level 1 and the base path come from full-resolution tiles. Each thread keeps its
//   partial sums in registers; they are reduced by warp shuffles and then across warps
//   in a fixed order into a per-CTA vector, written to the workspace.
// Kernel 2 (wt_dw_reduce_kernel): per channel, sums the G partial vectors in a fixed
//   order and applies the gradient unfolding of §4.3 Eq. 9.
// No atomics anywhere: the result is bitwise reproducible.
#include "wt_common.cuh"
#include "wt_internal.h"

namespace wt {

struct DwArgs {
    const void* x;
    const void* dy;
    float* part;  // [C][G][KP]
    int N, C, H, W, L, G;
    int vec;
    int tileH, tileW;
    int KP;
    // shared-memory layout, floats
    int o_acc, o_red;
    int o_carx[kMaxLevels + 1], o_cary[kMaxLevels + 1];
    int o_stx, o_sty, stx_half, sty_half;
    int o_px, px_pitch, o_py;
    int o_bx, bx_half, o_by, by_half;
};

constexpr int kDwDeepTile = 32;

template <int K>
struct DGeo {
    static constexpr int R = (K - 1) / 2;
    static constexpr int KK = K * K;
    static constexpr int PAD = (4 - (R % 4)) % 4;
    static constexpr int WIN = K + 3;
    static constexpr int NV4 = (WIN + 3) / 4;
    static constexpr int CW = 2 + 2 * R;
};

// Warp-level sum over lanes that share (lane & (step0 - 1)); then the per-warp results
// are combined across warps in a fixed order and added into acc_sm[off + e].
template <int NV>
__device__ __forceinline__ void block_flush(float (&v)[NV], int lane_groups, float* red,
                                            float* acc_sm, int off) {
    // lane_groups = 1: all lanes share one sum; 2: lanes split by parity (pair index)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
#pragma unroll
    for (int e = 0; e < NV; ++e) {
        float s = v[e];
        for (int m = lane_groups; m < 32; m <<= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
        v[e] = s;
    }
    if (lane < lane_groups) {
#pragma unroll
        for (int e = 0; e < NV; ++e) red[(warp * lane_groups + lane) * NV + e] = v[e];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < lane_groups * NV; e += blockDim.x) {
        const int grp = e / NV, k = e - grp * NV;
        float s = 0.f;
        for (int w = 0; w < nwarps; ++w) s += red[(w * lane_groups + grp) * NV + k];
        acc_sm[off + e] += s;
    }
    __syncthreads();
}

// Correlation of one 2x2 block of dY coefficients (bands 2p, 2p+1) with the X window.
template <int K>
__device__ __forceinline__ void corr_item(const float4* xs, int xpitch, int xhalf,
                                          const float4* gs, int gpitch, int ghalf, int bi,
                                          int bj, int p, float (&acc)[2][K * K]) {
    constexpr int CW = DGeo<K>::CW;
    float2 g[2][2];
#pragma unroll
    for (int oi = 0; oi < 2; ++oi)
#pragma unroll
        for (int oj = 0; oj < 2; ++oj) {
            const float4 t = gs[(2 * bi + oi) * gpitch + bj + oj * ghalf];
            g[oi][oj] = p ? make_float2(t.z, t.w) : make_float2(t.x, t.y);
        }
    const float4* xb = xs + (2 * bi) * xpitch + bj;
#pragma unroll
    for (int i = 0; i < CW; ++i) {
#pragma unroll
        for (int j = 0; j < CW; ++j) {
            const float4 t = xb[i * xpitch + (j >> 1) + (j & 1) * xhalf];
            const float2 xv = p ? make_float2(t.z, t.w) : make_float2(t.x, t.y);
#pragma unroll
            for (int oi = 0; oi < 2; ++oi)
#pragma unroll
                for (int oj = 0; oj < 2; ++oj) {
                    const int u = i - oi, v = j - oj;
                    if (u >= 0 && u < K && v >= 0 && v < K) {
                        acc[0][u * K + v] = fmaf(g[oi][oj].x, xv.x, acc[0][u * K + v]);
                        acc[1][u * K + v] = fmaf(g[oi][oj].y, xv.y, acc[1][u * K + v]);
                    }
                }
        }
    }
}

// Deep-level stage: X subbands with an R halo, dY subbands without, both unnormalized;
// carriers X^(l), dY^(l) written for l < L.
template <int K, typename T>
__device__ __forceinline__ void dw_deep_stage(const DwArgs& a, const T* xp, const T* gp,
                                              float* sm, int l, int ti0, int tj0) {
    constexpr int R = DGeo<K>::R;
    constexpr int SR = kDwDeepTile + 2 * R;
    const int Hl = a.H >> l, Wl = a.W >> l;
    const int Wp = a.W >> (l - 1);
    float4* stx = reinterpret_cast<float4*>(sm + a.o_stx);
    float4* sty = reinterpret_cast<float4*>(sm + a.o_sty);
    const int xpitch = 2 * a.stx_half, gpitch = 2 * a.sty_half;
    for (int idx = threadIdx.x; idx < SR * SR; idx += blockDim.x) {
        const int si = idx / SR, sj = idx - si * SR;
        const int gi = ti0 - R + si, gj = tj0 - R + sj;
        const bool inner = si >= R && si < R + kDwDeepTile && sj >= R && sj < R + kDwDeepTile;
        float4 ux = f4_zero(), ug = f4_zero();
        if (gi >= 0 && gi < Hl && gj >= 0 && gj < Wl) {
#pragma unroll
            for (int src = 0; src < 2; ++src) {
                if (src == 1 && !inner) break;  // dY is needed without halo only
                float ca, cb, cc, cd;
                if (l == 2) {
                    const T* p = (src ? gp : xp) + (size_t)(4 * gi) * a.W + 4 * gj;
                    const float4 r0 = IO<T>::ld4(p);
                    const float4 r1 = IO<T>::ld4(p + a.W);
                    const float4 r2 = IO<T>::ld4(p + 2 * (size_t)a.W);
                    const float4 r3 = IO<T>::ld4(p + 3 * (size_t)a.W);
                    ca = 0.5f * (r0.x + r0.y + r1.x + r1.y);
                    cb = 0.5f * (r0.z + r0.w + r1.z + r1.w);
                    cc = 0.5f * (r2.x + r2.y + r3.x + r3.y);
                    cd = 0.5f * (r2.z + r2.w + r3.z + r3.w);
                } else {
                    const float* q = sm + (src ? a.o_cary[l - 1] : a.o_carx[l - 1]) +
                                     (size_t)(2 * gi) * Wp + 2 * gj;
                    ca = q[0];
                    cb = q[1];
                    cc = q[Wp];
                    cd = q[Wp + 1];
                }
                const float4 u = haar_u(ca, cb, cc, cd);
                if (src == 0) ux = u; else ug = u;
                if (l < a.L && inner)
                    sm[(src ? a.o_cary[l] : a.o_carx[l]) + (size_t)gi * Wl + gj] = 0.5f * u.x;
            }
        }
        stx[si * xpitch + split_col(sj, a.stx_half)] = ux;
        if (inner) sty[(si - R) * gpitch + split_col(sj - R, a.sty_half)] = ug;
    }
}

template <int K, typename T>
__global__ void __launch_bounds__(256) wt_dw_plane_kernel(const DwArgs a) {
    constexpr int R = DGeo<K>::R, KK = DGeo<K>::KK, PAD = DGeo<K>::PAD;
    constexpr int WIN = DGeo<K>::WIN, NV4 = DGeo<K>::NV4;
    extern __shared__ float4 smem_f4[];
    float* sm = reinterpret_cast<float*>(smem_f4);
    float* acc_sm = sm + a.o_acc;
    float* red = sm + a.o_red;

    const int c = blockIdx.x, g = blockIdx.y;
    const size_t plane_elems = (size_t)a.H * a.W;
    for (int e = threadIdx.x; e < a.KP; e += blockDim.x) acc_sm[e] = 0.f;

    float acc0[KK + 1];  // base kernel taps + bias
#pragma unroll
    for (int q = 0; q <= KK; ++q) acc0[q] = 0.f;
    const int pair = threadIdx.x & 1;  // blockDim is even: pair index is fixed per thread
    __syncthreads();

    for (int n = g; n < a.N; n += a.G) {
        const size_t plane = (size_t)n * a.C + c;
        const T* xp = reinterpret_cast<const T*>(a.x) + plane * plane_elems;
        const T* gp = reinterpret_cast<const T*>(a.dy) + plane * plane_elems;

        // ---- levels 2..L ----
        for (int l = 2; l <= a.L; ++l) {
            float accp[2][KK];
#pragma unroll
            for (int q = 0; q < KK; ++q) accp[0][q] = accp[1][q] = 0.f;
            const int Hl = a.H >> l, Wl = a.W >> l;
            for (int ti0 = 0; ti0 < Hl; ti0 += kDwDeepTile) {
                for (int tj0 = 0; tj0 < Wl; tj0 += kDwDeepTile) {
                    dw_deep_stage<K, T>(a, xp, gp, sm, l, ti0, tj0);
                    __syncthreads();
                    constexpr int BPR = kDwDeepTile / 2;
                    for (int it = threadIdx.x; it < BPR * BPR * 2; it += blockDim.x) {
                        const int blk = it >> 1;
                        const int bi = blk / BPR, bj = blk - bi * BPR;
                        if (ti0 + 2 * bi >= Hl || tj0 + 2 * bj >= Wl) continue;
                        corr_item<K>(reinterpret_cast<const float4*>(sm + a.o_stx),
                                     2 * a.stx_half, a.stx_half,
                                     reinterpret_cast<const float4*>(sm + a.o_sty),
                                     2 * a.sty_half, a.sty_half, bi, bj, pair, accp);
                    }
                    __syncthreads();
                }
            }
            float flat[2 * KK];
#pragma unroll
            for (int q = 0; q < KK; ++q) {
                flat[q] = accp[0][q];
                flat[KK + q] = accp[1][q];
            }
            // lanes of equal parity hold the same band pair; layout [pair][band][tap]
            block_flush<2 * KK>(flat, 2, red, acc_sm, KK + 1 + (l - 1) * 4 * KK);
        }

        // ---- level 1 and the base path, full-resolution tiles ----
        float accp[2][KK];
#pragma unroll
        for (int q = 0; q < KK; ++q) accp[0][q] = accp[1][q] = 0.f;
        float* spx = sm + a.o_px;
        float* spy = sm + a.o_py;
        float4* sbx = reinterpret_cast<float4*>(sm + a.o_bx);
        float4* sby = reinterpret_cast<float4*>(sm + a.o_by);
        const int bpr = a.tileW >> 2;
        const int nblk = (a.tileH >> 2) * bpr;
        for (int y0 = 0; y0 < a.H; y0 += a.tileH) {
            for (int x0 = 0; x0 < a.W; x0 += a.tileW) {
                // stage X with a 2R halo and dY without, zero outside the plane
                {
                    const int rows = a.tileH + 4 * R, cols = a.tileW + 4 * R;
                    const int c_lo = x0 - 2 * R;
                    for (int idx = threadIdx.x; idx < rows * cols; idx += blockDim.x) {
                        const int r = idx / cols, cc = idx - r * cols;
                        const int gy = y0 - 2 * R + r, gx = c_lo + cc;
                        float v = 0.f;
                        if (gy >= 0 && gy < a.H && gx >= 0 && gx < a.W)
                            v = IO<T>::ld(xp + (size_t)gy * a.W + gx);
                        spx[r * a.px_pitch + PAD + cc] = v;
                    }
                    const int tw = a.tileW;
                    if (a.vec) {
                        const int tw4 = tw >> 2;
                        for (int idx = threadIdx.x; idx < a.tileH * tw4; idx += blockDim.x) {
                            const int r = idx / tw4, q = idx - r * tw4;
                            const int gy = y0 + r, gx = x0 + 4 * q;
                            float4 v = f4_zero();
                            if (gy < a.H && gx < a.W) v = IO<T>::ld4(gp + (size_t)gy * a.W + gx);
                            *reinterpret_cast<float4*>(spy + r * tw + 4 * q) = v;
                        }
                    } else {
                        for (int idx = threadIdx.x; idx < a.tileH * tw; idx += blockDim.x) {
                            const int r = idx / tw, cc = idx - r * tw;
                            const int gy = y0 + r, gx = x0 + cc;
                            float v = 0.f;
                            if (gy < a.H && gx < a.W) v = IO<T>::ld(gp + (size_t)gy * a.W + gx);
                            spy[r * tw + cc] = v;
                        }
                    }
                }
                __syncthreads();
                if (a.L >= 1) {
                    const int crow = a.tileH / 2 + 2 * R, ccol = a.tileW / 2 + 2 * R;
                    for (int idx = threadIdx.x; idx < crow * ccol; idx += blockDim.x) {
                        const int ci = idx / ccol, cj = idx - ci * ccol;
                        const float* p = spx + (2 * ci) * a.px_pitch + PAD + 2 * cj;
                        sbx[ci * 2 * a.bx_half + split_col(cj, a.bx_half)] =
                            haar_u(p[0], p[1], p[a.px_pitch], p[a.px_pitch + 1]);
                    }
                    const int grow = a.tileH / 2, gcol = a.tileW / 2;
                    for (int idx = threadIdx.x; idx < grow * gcol; idx += blockDim.x) {
                        const int ci = idx / gcol, cj = idx - ci * gcol;
                        const float* p = spy + (2 * ci) * a.tileW + 2 * cj;
                        sby[ci * 2 * a.by_half + split_col(cj, a.by_half)] =
                            haar_u(p[0], p[1], p[a.tileW], p[a.tileW + 1]);
                    }
                    __syncthreads();
                }
                // base path: dW~0 and db~
                for (int blk = threadIdx.x; blk < nblk; blk += blockDim.x) {
                    const int by = blk / bpr, bx = blk - by * bpr;
                    const int py = 4 * by, px = 4 * bx;
                    if (y0 + py >= a.H || x0 + px >= a.W) continue;
                    float gv[4][4];
#pragma unroll
                    for (int o = 0; o < 4; ++o) {
                        const float4 t = *reinterpret_cast<const float4*>(spy + (py + o) * a.tileW + px);
                        gv[o][0] = t.x; gv[o][1] = t.y; gv[o][2] = t.z; gv[o][3] = t.w;
                        acc0[KK] += (t.x + t.y) + (t.z + t.w);
                    }
#pragma unroll
                    for (int rr = 0; rr < WIN; ++rr) {
                        const float4* rowp = reinterpret_cast<const float4*>(
                            spx + (py + R + rr) * a.px_pitch + px + R + PAD);
                        float v[4 * NV4];
#pragma unroll
                        for (int q = 0; q < NV4; ++q) {
                            const float4 t = rowp[q];
                            v[4 * q] = t.x; v[4 * q + 1] = t.y; v[4 * q + 2] = t.z; v[4 * q + 3] = t.w;
                        }
#pragma unroll
                        for (int o = 0; o < 4; ++o) {
                            const int u = rr - o;
                            if (u < 0 || u >= K) continue;
#pragma unroll
                            for (int oc = 0; oc < 4; ++oc)
#pragma unroll
                                for (int vv = 0; vv < K; ++vv)
                                    acc0[u * K + vv] = fmaf(gv[o][oc], v[oc + vv], acc0[u * K + vv]);
                        }
                    }
                }
                // level 1
                if (a.L >= 1) {
                    for (int it = threadIdx.x; it < nblk * 2; it += blockDim.x) {
                        const int blk = it >> 1;
                        const int by = blk / bpr, bx = blk - by * bpr;
                        if (y0 + 4 * by >= a.H || x0 + 4 * bx >= a.W) continue;
                        corr_item<K>(sbx, 2 * a.bx_half, a.bx_half, sby, 2 * a.by_half,
                                     a.by_half, by, bx, pair, accp);
                    }
                }
                __syncthreads();
            }
        }
        if (a.L >= 1) {
            float flat[2 * KK];
#pragma unroll
            for (int q = 0; q < KK; ++q) {
                flat[q] = accp[0][q];
                flat[KK + q] = accp[1][q];
            }
            block_flush<2 * KK>(flat, 2, red, acc_sm, KK + 1);
        }
    }
    block_flush<KK + 1>(acc0, 1, red, acc_sm, 0);
    float* out = a.part + ((size_t)c * a.G + g) * a.KP;
    for (int e = threadIdx.x; e < a.KP; e += blockDim.x) out[e] = acc_sm[e];
}

// Per channel: fixed-order sum of the G partial vectors, then §4.3 Eq. 9.
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
    // level layout inside one level: [pair][band-in-pair][tap] == [band][tap]
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
        for (int uv = 0; uv < KK; ++uv) d = fmaf(tot[KK + 1 + (l * 4 + b) * KK + uv], wl[pi * KK + uv], d);
        dsl[pi] = d;
    }
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
namespace {

int round4(int v) { return (v + 3) & ~3; }

int choose_groups(const wt_desc& d) {
    const int target = 4 * kNumSMs;
    int need = (target + d.c - 1) / d.c;
    if (need < 1) need = 1;
    if (need >= d.n) return d.n;
    for (int gsz = need; gsz <= d.n; ++gsz)
        if (d.n % gsz == 0) return gsz;
    return d.n;
}

template <int K>
void dw_layout(const wt_desc& d, DwArgs& a, int& nthreads, size_t& smem_bytes) {
    constexpr int R = DGeo<K>::R, KK = DGeo<K>::KK, PAD = DGeo<K>::PAD;
    const int L = d.levels;
    const int H4 = round4(d.h), W4 = round4(d.w);
    if ((H4 / 4) * (W4 / 4) <= 256) {
        a.tileH = H4;
        a.tileW = W4;
    } else {
        a.tileW = W4 >= 64 ? 64 : W4;
        a.tileH = 64 * 64 / a.tileW;
        if (a.tileH > H4) a.tileH = H4;
    }
    const int nblk = (a.tileH / 4) * (a.tileW / 4);
    nthreads = ((nblk + 31) / 32) * 32;
    if (nthreads > 256) nthreads = 256;
    if (nthreads < 64) nthreads = 64;
    a.KP = KK + 1 + 4 * KK * L;
    int off = 0;
    a.o_acc = off;
    off += round4(a.KP);
    a.o_red = off;
    off += round4((nthreads / 32) * 2 * 2 * KK);
    const int u0 = off;
    int dp = u0;
    for (int l = 0; l <= kMaxLevels; ++l) a.o_carx[l] = a.o_cary[l] = 0;
    for (int l = 2; l < L; ++l) {
        const int sz = round4((d.h >> l) * (d.w >> l));
        a.o_carx[l] = dp;
        dp += sz;
        a.o_cary[l] = dp;
        dp += sz;
    }
    a.stx_half = (kDwDeepTile + 2 * R + 1) / 2;
    a.sty_half = kDwDeepTile / 2;
    a.o_stx = dp;
    a.o_sty = dp;
    if (L >= 2) {
        dp += 4 * (kDwDeepTile + 2 * R) * 2 * a.stx_half;
        a.o_sty = dp;
        dp += 4 * kDwDeepTile * 2 * a.sty_half;
    }
    int fp = u0;
    a.px_pitch = round4(PAD + a.tileW + 4 * R + 4);
    a.o_px = fp;
    fp += (a.tileH + 4 * R) * a.px_pitch;
    a.o_py = fp;
    fp += a.tileH * a.tileW;
    a.bx_half = (a.tileW / 2 + 2 * R + 1) / 2;
    a.by_half = (a.tileW / 2 + 1) / 2;
    a.o_bx = fp;
    a.o_by = fp;
    if (L >= 1) {
        fp += 4 * (a.tileH / 2 + 2 * R) * 2 * a.bx_half;
        a.o_by = fp;
        fp += 4 * (a.tileH / 2) * 2 * a.by_half;
    }
    const int total = dp > fp ? dp : fp;
    smem_bytes = (size_t)total * sizeof(float);
}

template <int K, typename T>
wt_status launch_dw_k(const wt_desc& d, const void* x, const void* dy, const float* w0,
                      const float* b0, const float* s0, const float* wl, const float* sl,
                      float* dw0, float* db0, float* ds0, float* dwl, float* dsl, void* ws,
                      size_t ws_bytes, cudaStream_t stream, int* launches) {
    DwArgs a;
    int nthreads = 0;
    size_t smem = 0;
    dw_layout<K>(d, a, nthreads, smem);
    if (smem > kMaxSmemPerBlock) return WT_ERR_UNSUPPORTED;
    a.G = choose_groups(d);
    const size_t need = (size_t)d.c * a.G * a.KP * sizeof(float);
    if (ws == nullptr || ws_bytes < need) return WT_ERR_WORKSPACE;
    a.x = x;
    a.dy = dy;
    a.part = reinterpret_cast<float*>(ws);
    a.N = d.n;
    a.C = d.c;
    a.H = d.h;
    a.W = d.w;
    a.L = d.levels;
    a.vec = (d.w % 4 == 0) ? 1 : 0;
    auto kern = wt_dw_plane_kernel<K, T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return WT_ERR_CUDA;
    kern<<<dim3((unsigned)d.c, (unsigned)a.G), nthreads, smem, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    ++*launches;
    wt_dw_reduce_kernel<<<(unsigned)d.c, 128, (size_t)a.KP * sizeof(float), stream>>>(
        a.part, d.c, a.G, a.KP, K, d.levels, w0, b0, s0, wl, sl, dw0, db0, ds0, dwl, dsl);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    ++*launches;
    return WT_OK;
}

}  // namespace

size_t backward_weight_ws_bytes(const wt_desc& d) {
    const int KK = d.k * d.k;
    const size_t KP = (size_t)KK + 1 + 4 * (size_t)KK * d.levels;
    return (size_t)d.c * choose_groups(d) * KP * sizeof(float);
}

size_t backward_weight_smem_bytes(const wt_desc& d) {
    DwArgs a;
    int nt = 0;
    size_t smem = 0;
    switch (d.k) {
        case 1: dw_layout<1>(d, a, nt, smem); break;
        case 3: dw_layout<3>(d, a, nt, smem); break;
        case 5: dw_layout<5>(d, a, nt, smem); break;
        case 7: dw_layout<7>(d, a, nt, smem); break;
        default: return 0;
    }
    return smem;
}

wt_status launch_backward_weight(const wt_desc& d, const void* x, const void* dy,
                                 const float* w0, const float* b0, const float* s0,
                                 const float* wl, const float* sl, float* dw0, float* db0,
                                 float* ds0, float* dwl, float* dsl, void* ws, size_t ws_bytes,
                                 cudaStream_t stream, int* launches) {
    const bool bf = d.io == WT_BF16;
    switch (d.k) {
#define WT_CASE(KV)                                                                          \
    case KV:                                                                                 \
        return bf ? launch_dw_k<KV, __nv_bfloat16>(d, x, dy, w0, b0, s0, wl, sl, dw0, db0,   \
                                                   ds0, dwl, dsl, ws, ws_bytes, stream,      \
                                                   launches)                                 \
                  : launch_dw_k<KV, float>(d, x, dy, w0, b0, s0, wl, sl, dw0, db0, ds0, dwl, \
                                           dsl, ws, ws_bytes, stream, launches);
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
