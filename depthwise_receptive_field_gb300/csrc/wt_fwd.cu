// WTConv forward and backward-data kernel for sm_103a.
//
// Method: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware Reformulation"
// (Aflalo et al.). One CTA owns one (n, c) plane and evaluates the whole layer on it
// with one read of X and one write of Y in HBM:
//
//   deep phase (L >= 2) -- the levels l = 2..L run at their own resolution entirely in
//     shared memory: the Haar butterfly of §4.1 Eq. 5 is recomputed from the low-pass
//     carrier X^(l-1) into a halo-padded coefficient tile, the four k x k filters
//     (scales folded, §4.3 Eq. 8) are applied, and the filtered coefficients Z^(l) stay
//     on chip. The level-2 tiles read X itself (4x4 pixel blocks, L2-resident after the
//     first pass), so the level-1 carrier is never materialized anywhere.
//   full-resolution phase -- 64x64-pixel tiles of X (halo 2R) are staged once; each
//     thread owns a 4x4 pixel block and computes the base k x k convolution, the level-1
//     Haar coefficients' k x k filters for its 2x2 coefficient block, and the closed-form
//     bit-indexed synthesis of §4.2 Prop. 2 / Eq. 7 over all L levels (level 1 from
//     registers, levels >= 2 from shared memory), adding the base path in the same store.
//
// Backward-data is the same operator on dY with every kernel rotated by 180 degrees and
// no bias (adjoint of Eq. 5 is Eq. 12 by §2.2 Eq. 1; adjoint of cross-correlation is
// correlation with the rotated kernel); `flip` selects it.
#include "wt_common.cuh"
#include "wt_internal.h"

namespace wt {

struct FwdArgs {
    const void* x;
    void* y;
    const float* w0f;
    const float* b0f;
    const float* wlf;
    int C, H, W, L;
    int flip;
    int vec;           // 1: rows may be read/written 4 elements at a time
    int tileH, tileW;  // full-resolution tile, pixels (multiples of 4)
    // shared-memory layout, in floats
    int o_w0, o_wl;
    int o_zd[kMaxLevels + 1];
    int o_car[kMaxLevels + 1];
    int o_stage, st_half;
    int o_px, px_pitch;
    int o_bd, bd_half;
};

constexpr int kDeepTile = 32;  // deep-phase output tile (coefficients per side)

template <int K>
struct Geo {
    static constexpr int R = (K - 1) / 2;
    static constexpr int KK = K * K;
    static constexpr int PAD = (4 - (R % 4)) % 4;     // aligns each thread's pixel window
    static constexpr int WIN = K + 3;                 // window rows/cols for a 4-wide block
    static constexpr int NV4 = (WIN + 3) / 4;         // float4 loads per window row
    static constexpr int CW = 2 + 2 * R;              // coefficient window for a 2x2 block
};

// Stage the level-l coefficient tile (unnormalized subbands, zero outside the grid) for
// outputs [ti0, ti0+kDeepTile) x [tj0, tj0+kDeepTile) with an R-coefficient halo; also
// write the normalized carrier X^(l) for the tile's own positions when l < L.
template <int K, typename T>
__device__ __forceinline__ void deep_stage(const FwdArgs& a, const T* xp, float* sm, int l,
                                           int ti0, int tj0) {
    constexpr int R = Geo<K>::R;
    constexpr int SR = kDeepTile + 2 * R;
    const int Hl = a.H >> l, Wl = a.W >> l;
    float4* stage = reinterpret_cast<float4*>(sm + a.o_stage);
    const int pitch = 2 * a.st_half;
    const float* carp = (l >= 3) ? sm + a.o_car[l - 1] : nullptr;
    float* carl = (l < a.L) ? sm + a.o_car[l] : nullptr;
    const int Wp = a.W >> (l - 1);  // width of X^(l-1)
    for (int idx = threadIdx.x; idx < SR * SR; idx += blockDim.x) {
        const int si = idx / SR, sj = idx - si * SR;
        const int gi = ti0 - R + si, gj = tj0 - R + sj;
        float4 u = f4_zero();
        if (gi >= 0 && gi < Hl && gj >= 0 && gj < Wl) {
            float ca, cb, cc, cd;
            if (l == 2) {
                // X^(1) 2x2 block from the 4x4 pixel block of X at (4gi, 4gj)
                const T* p = xp + (size_t)(4 * gi) * a.W + 4 * gj;
                const float4 r0 = IO<T>::ld4(p);
                const float4 r1 = IO<T>::ld4(p + a.W);
                const float4 r2 = IO<T>::ld4(p + 2 * (size_t)a.W);
                const float4 r3 = IO<T>::ld4(p + 3 * (size_t)a.W);
                ca = 0.5f * (r0.x + r0.y + r1.x + r1.y);
                cb = 0.5f * (r0.z + r0.w + r1.z + r1.w);
                cc = 0.5f * (r2.x + r2.y + r3.x + r3.y);
                cd = 0.5f * (r2.z + r2.w + r3.z + r3.w);
            } else {
                const float* q = carp + (size_t)(2 * gi) * Wp + 2 * gj;
                ca = q[0];
                cb = q[1];
                cc = q[Wp];
                cd = q[Wp + 1];
            }
            u = haar_u(ca, cb, cc, cd);
            if (carl && si >= R && si < R + kDeepTile && sj >= R && sj < R + kDeepTile)
                carl[(size_t)gi * Wl + gj] = 0.5f * u.x;
        }
        stage[si * pitch + split_col(sj, a.st_half)] = u;
    }
}

// Filter one staged tile: each thread computes 2x2 output cells (4 bands each).
template <int K>
__device__ __forceinline__ void deep_conv(const FwdArgs& a, float* sm, int l, int ti0, int tj0,
                                          const float4 (&wr)[K * K]) {
    constexpr int CW = Geo<K>::CW;
    const int Hl = a.H >> l, Wl = a.W >> l;
    const float4* stage = reinterpret_cast<const float4*>(sm + a.o_stage);
    float4* zd = reinterpret_cast<float4*>(sm + a.o_zd[l]);
    const int pitch = 2 * a.st_half;
    constexpr int BPR = kDeepTile / 2;  // 2x2 blocks per tile row
    for (int blk = threadIdx.x; blk < BPR * BPR; blk += blockDim.x) {
        const int bi = blk / BPR, bj = blk - bi * BPR;
        const int oi0 = 2 * bi, oj0 = 2 * bj;
        if (ti0 + oi0 >= Hl || tj0 + oj0 >= Wl) continue;
        float4 z[2][2];
#pragma unroll
        for (int q = 0; q < 4; ++q) z[q >> 1][q & 1] = f4_zero();
#pragma unroll
        for (int i = 0; i < CW; ++i) {
#pragma unroll
            for (int j = 0; j < CW; ++j) {
                const float4 s = stage[(oi0 + i) * pitch + bj + (j >> 1) + (j & 1) * a.st_half];
#pragma unroll
                for (int oi = 0; oi < 2; ++oi) {
#pragma unroll
                    for (int oj = 0; oj < 2; ++oj) {
                        const int u = i - oi, v = j - oj;
                        if (u >= 0 && u < K && v >= 0 && v < K) f4_fma(z[oi][oj], wr[u * K + v], s);
                    }
                }
            }
        }
#pragma unroll
        for (int oi = 0; oi < 2; ++oi) {
#pragma unroll
            for (int oj = 0; oj < 2; ++oj) {
                const int gi = ti0 + oi0 + oi, gj = tj0 + oj0 + oj;
                if (gi < Hl && gj < Wl) zd[(size_t)gi * Wl + gj] = z[oi][oj];
            }
        }
    }
}

// Stage the full-resolution pixel tile [y0-2R, y0+tileH+2R) x [x0-2R, x0+tileW+2R),
// zero outside the plane.
template <int K, typename T>
__device__ __forceinline__ void stage_pixels(const FwdArgs& a, const T* xp, float* spx, int y0,
                                             int x0) {
    constexpr int R = Geo<K>::R, PAD = Geo<K>::PAD;
    const int rows = a.tileH + 4 * R, cols = a.tileW + 4 * R;
    const int c_lo = x0 - 2 * R;
    if (a.vec) {
        const int g_lo = (c_lo >= 0) ? (c_lo & ~3) : -((-c_lo + 3) & ~3);
        const int ngroups = (x0 + a.tileW + 2 * R - g_lo + 3) >> 2;
        for (int idx = threadIdx.x; idx < rows * ngroups; idx += blockDim.x) {
            const int r = idx / ngroups, g = idx - r * ngroups;
            const int gy = y0 - 2 * R + r, gx = g_lo + 4 * g;
            float4 v = f4_zero();
            if (gy >= 0 && gy < a.H && gx >= 0 && gx < a.W) v = IO<T>::ld4(xp + (size_t)gy * a.W + gx);
            float* dst = spx + r * a.px_pitch + PAD - c_lo;
            const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int cc = gx + q - c_lo;
                if (cc >= 0 && cc < cols) dst[gx + q] = e[q];
            }
        }
    } else {
        for (int idx = threadIdx.x; idx < rows * cols; idx += blockDim.x) {
            const int r = idx / cols, cc = idx - r * cols;
            const int gy = y0 - 2 * R + r, gx = c_lo + cc;
            float v = 0.f;
            if (gy >= 0 && gy < a.H && gx >= 0 && gx < a.W) v = IO<T>::ld(xp + (size_t)gy * a.W + gx);
            spx[r * a.px_pitch + PAD + cc] = v;
        }
    }
}

// Level-1 unnormalized subbands of the staged tile: cell (ci, cj) is the 2x2 pixel block
// at tile rows 2ci.., cols 2cj.. (coefficient y0/2 - R + ci, x0/2 - R + cj).
template <int K>
__device__ __forceinline__ void stage_bands(const FwdArgs& a, const float* spx, float4* sbd) {
    constexpr int R = Geo<K>::R, PAD = Geo<K>::PAD;
    const int crow = a.tileH / 2 + 2 * R, ccol = a.tileW / 2 + 2 * R;
    const int pitch = 2 * a.bd_half;
    for (int idx = threadIdx.x; idx < crow * ccol; idx += blockDim.x) {
        const int ci = idx / ccol, cj = idx - ci * ccol;
        const float* p = spx + (2 * ci) * a.px_pitch + PAD + 2 * cj;
        sbd[ci * pitch + split_col(cj, a.bd_half)] =
            haar_u(p[0], p[1], p[a.px_pitch], p[a.px_pitch + 1]);
    }
}

template <int K, typename T>
__global__ void __launch_bounds__(256) wt_fwd_plane_kernel(const FwdArgs a) {
    constexpr int R = Geo<K>::R, KK = Geo<K>::KK, PAD = Geo<K>::PAD;
    constexpr int WIN = Geo<K>::WIN, NV4 = Geo<K>::NV4, CW = Geo<K>::CW;
    extern __shared__ float4 smem_f4[];
    float* sm = reinterpret_cast<float*>(smem_f4);

    const int plane = blockIdx.x;
    const int c = plane % a.C;
    const size_t plane_elems = (size_t)a.H * a.W;
    const T* xp = reinterpret_cast<const T*>(a.x) + (size_t)plane * plane_elems;
    T* yp = reinterpret_cast<T*>(a.y) + (size_t)plane * plane_elems;

    // ---- folded weights -> shared memory; power-of-two factors and rotation applied ----
    float* w0s = sm + a.o_w0;
    float4* wls = reinterpret_cast<float4*>(sm + a.o_wl);
    for (int e = threadIdx.x; e < KK * (1 + a.L); e += blockDim.x) {
        const int lvl = e / KK, uv = e - lvl * KK;
        const int src = a.flip ? (KK - 1 - uv) : uv;
        if (lvl == 0) {
            w0s[uv] = __ldg(a.w0f + (size_t)c * KK + src);
        } else {
            // Z'^(l) = 2^-(l+1) W~^(l) U: 1/2 turns U back into Y, 2^-l is Eq. 7's weight
            const float sc = ldexpf(1.0f, -(lvl + 1));
            const float* wb = a.wlf + (((size_t)(lvl - 1) * a.C + c) * 4) * KK + src;
            wls[(lvl - 1) * KK + uv] =
                make_float4(sc * __ldg(wb), sc * __ldg(wb + KK), sc * __ldg(wb + 2 * KK),
                            sc * __ldg(wb + 3 * KK));
        }
    }
    const float bias = (a.b0f != nullptr) ? __ldg(a.b0f + c) : 0.f;
    __syncthreads();

    // ---- deep phase: levels 2..L on chip ----
    for (int l = 2; l <= a.L; ++l) {
        float4 wr[KK];
#pragma unroll
        for (int q = 0; q < KK; ++q) wr[q] = wls[(l - 1) * KK + q];
        const int Hl = a.H >> l, Wl = a.W >> l;
        for (int ti0 = 0; ti0 < Hl; ti0 += kDeepTile) {
            for (int tj0 = 0; tj0 < Wl; tj0 += kDeepTile) {
                deep_stage<K, T>(a, xp, sm, l, ti0, tj0);
                __syncthreads();
                deep_conv<K>(a, sm, l, ti0, tj0, wr);
                __syncthreads();
            }
        }
    }

    // ---- full-resolution phase ----
    float w0r[KK];
#pragma unroll
    for (int q = 0; q < KK; ++q) w0r[q] = w0s[q];
    float4 w1r[KK];
    if (a.L >= 1) {
#pragma unroll
        for (int q = 0; q < KK; ++q) w1r[q] = wls[q];
    }
    float* spx = sm + a.o_px;
    float4* sbd = reinterpret_cast<float4*>(sm + a.o_bd);
    const int bd_pitch = 2 * a.bd_half;
    const int bpr = a.tileW >> 2;                   // 4x4 pixel blocks per tile row
    const int nblk = (a.tileH >> 2) * bpr;

    for (int y0 = 0; y0 < a.H; y0 += a.tileH) {
        for (int x0 = 0; x0 < a.W; x0 += a.tileW) {
            stage_pixels<K, T>(a, xp, spx, y0, x0);
            __syncthreads();
            if (a.L >= 1) {
                stage_bands<K>(a, spx, sbd);
                __syncthreads();
            }
            for (int blk = threadIdx.x; blk < nblk; blk += blockDim.x) {
                const int by = blk / bpr, bx = blk - by * bpr;
                const int py = 4 * by, px = 4 * bx;
                const int gy = y0 + py, gx = x0 + px;
                if (gy >= a.H || gx >= a.W) continue;

                // base path: k x k on X plus folded bias
                float acc[4][4];
#pragma unroll
                for (int o = 0; o < 4; ++o)
#pragma unroll
                    for (int oc = 0; oc < 4; ++oc) acc[o][oc] = bias;
#pragma unroll
                for (int rr = 0; rr < WIN; ++rr) {
                    const float4* rowp =
                        reinterpret_cast<const float4*>(spx + (py + R + rr) * a.px_pitch + px + R + PAD);
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
                                acc[o][oc] = fmaf(w0r[u * K + vv], v[oc + vv], acc[o][oc]);
                    }
                }

                if (a.L >= 1) {
                    // level 1: k x k on the four subbands of the 2x2 coefficient block
                    float4 z[2][2];
#pragma unroll
                    for (int q = 0; q < 4; ++q) z[q >> 1][q & 1] = f4_zero();
                    const float4* cb = sbd + (2 * by) * bd_pitch + bx;
#pragma unroll
                    for (int i = 0; i < CW; ++i) {
#pragma unroll
                        for (int j = 0; j < CW; ++j) {
                            const float4 s = cb[i * bd_pitch + (j >> 1) + (j & 1) * a.bd_half];
#pragma unroll
                            for (int oi = 0; oi < 2; ++oi)
#pragma unroll
                                for (int oj = 0; oj < 2; ++oj) {
                                    const int u = i - oi, v = j - oj;
                                    if (u >= 0 && u < K && v >= 0 && v < K)
                                        f4_fma(z[oi][oj], w1r[u * K + v], s);
                                }
                        }
                    }
                    // levels >= 2: Eq. 7 terms, addressed by coordinate bits
                    float dsum[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
                    const int gci = gy >> 1, gcj = gx >> 1;  // even
                    for (int l = 2; l <= a.L; ++l) {
                        const int Wl = a.W >> l;
                        const float4 zl = reinterpret_cast<const float4*>(sm + a.o_zd[l])
                            [(size_t)(gci >> (l - 1)) * Wl + (gcj >> (l - 1))];
#pragma unroll
                        for (int oi = 0; oi < 2; ++oi)
#pragma unroll
                            for (int oj = 0; oj < 2; ++oj)
                                dsum[oi][oj] += synth_rt(zl, ((gci + oi) >> (l - 2)) & 1,
                                                         ((gcj + oj) >> (l - 2)) & 1);
                    }
#pragma unroll
                    for (int oi = 0; oi < 2; ++oi)
#pragma unroll
                        for (int oj = 0; oj < 2; ++oj) {
                            const float d = dsum[oi][oj];
                            acc[2 * oi][2 * oj] += synth<0, 0>(z[oi][oj]) + d;
                            acc[2 * oi][2 * oj + 1] += synth<0, 1>(z[oi][oj]) + d;
                            acc[2 * oi + 1][2 * oj] += synth<1, 0>(z[oi][oj]) + d;
                            acc[2 * oi + 1][2 * oj + 1] += synth<1, 1>(z[oi][oj]) + d;
                        }
                }

                // store the 4x4 block
                if (a.vec && gy + 4 <= a.H && gx + 4 <= a.W) {
#pragma unroll
                    for (int o = 0; o < 4; ++o)
                        IO<T>::st4(yp + (size_t)(gy + o) * a.W + gx,
                                   make_float4(acc[o][0], acc[o][1], acc[o][2], acc[o][3]));
                } else {
#pragma unroll
                    for (int o = 0; o < 4; ++o)
#pragma unroll
                        for (int oc = 0; oc < 4; ++oc)
                            if (gy + o < a.H && gx + oc < a.W)
                                IO<T>::st(yp + (size_t)(gy + o) * a.W + gx + oc, acc[o][oc]);
                }
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------

namespace {

int round4(int v) { return (v + 3) & ~3; }

template <int K>
bool fwd_layout(const wt_desc& d, FwdArgs& a, int& nthreads, size_t& smem_bytes) {
    constexpr int R = Geo<K>::R, KK = Geo<K>::KK, PAD = Geo<K>::PAD;
    const int L = d.levels;
    // tile: whole plane when it has at most 256 4x4 blocks, else 64x64 pixels
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

    int off = 0;
    a.o_w0 = off;
    off += round4(KK);
    a.o_wl = off;
    off += 4 * KK * L;
    for (int l = 0; l <= kMaxLevels; ++l) a.o_zd[l] = a.o_car[l] = 0;
    for (int l = 2; l <= L; ++l) {
        a.o_zd[l] = off;
        off += 4 * (d.h >> l) * (d.w >> l);
    }
    const int u0 = off;
    // deep-phase scratch (aliases the full-resolution tile buffers)
    int dp = u0;
    for (int l = 2; l < L; ++l) {
        a.o_car[l] = dp;
        dp += round4((d.h >> l) * (d.w >> l));
    }
    a.st_half = (kDeepTile + 2 * R + 1) / 2;
    a.o_stage = dp;
    if (L >= 2) dp += 4 * (kDeepTile + 2 * R) * 2 * a.st_half;
    // full-resolution tile buffers
    int fp = u0;
    a.px_pitch = round4(PAD + a.tileW + 4 * R + 4);
    a.o_px = fp;
    fp += (a.tileH + 4 * R) * a.px_pitch;
    a.bd_half = (a.tileW / 2 + 2 * R + 1) / 2;
    a.o_bd = fp;
    if (L >= 1) fp += 4 * (a.tileH / 2 + 2 * R) * 2 * a.bd_half;
    const int total = dp > fp ? dp : fp;
    smem_bytes = (size_t)total * sizeof(float);
    return true;
}

template <int K, typename T>
wt_status launch_fwd_k(const wt_desc& d, const void* x, const float* w0f, const float* b0f,
                       const float* wlf, void* y, int flip, cudaStream_t stream, int* launches) {
    FwdArgs a;
    int nthreads = 0;
    size_t smem = 0;
    fwd_layout<K>(d, a, nthreads, smem);
    if (smem > kMaxSmemPerBlock) return WT_ERR_UNSUPPORTED;
    a.x = x;
    a.y = y;
    a.w0f = w0f;
    a.b0f = flip ? nullptr : b0f;
    a.wlf = wlf;
    a.C = d.c;
    a.H = d.h;
    a.W = d.w;
    a.L = d.levels;
    a.flip = flip;
    a.vec = (d.w % 4 == 0) ? 1 : 0;
    auto kern = wt_fwd_plane_kernel<K, T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return WT_ERR_CUDA;
    const long planes = (long)d.n * d.c;
    kern<<<(unsigned)planes, nthreads, smem, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    ++*launches;
    return WT_OK;
}

}  // namespace

wt_status launch_forward(const wt_desc& d, const void* x, const float* w0f, const float* b0f,
                         const float* wlf, void* y, int flip, cudaStream_t stream,
                         int* launches) {
    const bool bf = d.io == WT_BF16;
    switch (d.k) {
#define WT_CASE(KV)                                                                         \
    case KV:                                                                                \
        return bf ? launch_fwd_k<KV, __nv_bfloat16>(d, x, w0f, b0f, wlf, y, flip, stream,   \
                                                    launches)                               \
                  : launch_fwd_k<KV, float>(d, x, w0f, b0f, wlf, y, flip, stream, launches);
        WT_CASE(1)
        WT_CASE(3)
        WT_CASE(5)
        WT_CASE(7)
#undef WT_CASE
        default:
            return WT_ERR_UNSUPPORTED;
    }
}

size_t forward_smem_bytes(const wt_desc& d) {
    FwdArgs a;
    int nt = 0;
    size_t smem = 0;
    switch (d.k) {
        case 1: fwd_layout<1>(d, a, nt, smem); break;
        case 3: fwd_layout<3>(d, a, nt, smem); break;
        case 5: fwd_layout<5>(d, a, nt, smem); break;
        case 7: fwd_layout<7>(d, a, nt, smem); break;
        default: return 0;
    }
    return smem;
}

}  // namespace wt
