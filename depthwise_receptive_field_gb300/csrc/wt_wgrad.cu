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
// Kernel 1 (wt_dw_plane_kernel): one CTA per (c, n) plane.
//   deep levels (l >= 2): 32x32 tiles of the level's subbands of X (R halo) and dY are
//     staged from on-chip carriers (level 2 from the 4x4 pixel blocks of X and dY); warp w
//     correlates band w and reduces its 25 sums with warp shuffles after each level.
//   full resolution: 64x64-pixel tiles; warps 0-1 run the base correlation (8x4 pixel
//     blocks, dY read straight into registers), warps 2-3 the level-1 subband correlations
//     (16 lanes per band, 4x4 coefficient blocks). Each thread keeps its 25 partial sums
//     in registers for the whole plane.
//   The per-plane partial vector [dW~0 | db~ | dW~^(l)_b] goes to the workspace.
// Kernel 2 (wt_dw_reduce_kernel): per channel, sums the N partial vectors in a fixed
//   order and applies the gradient unfolding of §4.3 Eq. 9.
// No atomics anywhere: results are bitwise reproducible.
#include "wt_internal.h"
#include "wt_tile.cuh"

namespace wt {

constexpr int kDT = 128;  // threads per CTA

struct DwArgs {
    const void* x;
    const void* dy;
    float* part;  // [C][N][KP]
    int N, C, H, W, L;
    int vec;
    int KP;
    int o_acc, o_red, o_xb, o_gb, o_x;  // shared-memory regions (floats)
    int o_carx[kMaxLevels + 1], o_cary[kMaxLevels + 1];
};

// Deep stage for level l: X subbands with an R halo into xb (band-major, BPITCH) and the
// dY subbands of the tile's own 32x32 cells into gb ([4][32][32]); carriers for l < L.
template <int K, typename T>
__device__ __forceinline__ void dw_deep_stage(const DwArgs& a, const T* xp, const T* gp,
                                              float* sm, int l, int ti0, int tj0) {
    constexpr int R = FG<K>::R, BT = FG<K>::BT, BP = FG<K>::BPITCH, BAND = FG<K>::BAND;
    constexpr int ZAND = FG<K>::ZAND;
    const int Hl = a.H >> l, Wl = a.W >> l, Wp = a.W >> (l - 1);
    float* xb = sm + a.o_xb;
    float* gb = sm + a.o_gb;
    const float* cpx = (l >= 3) ? sm + a.o_carx[l - 1] : nullptr;
    const float* cpy = (l >= 3) ? sm + a.o_cary[l - 1] : nullptr;
    float* clx = (l < a.L) ? sm + a.o_carx[l] : nullptr;
    float* cly = (l < a.L) ? sm + a.o_cary[l] : nullptr;
    for (int idx = threadIdx.x; idx < BT * BT; idx += blockDim.x) {
        const int si = idx / BT, sj = idx - si * BT;
        const int gi = ti0 - R + si, gj = tj0 - R + sj;
        const bool inner = si >= R && si < R + kCT && sj >= R && sj < R + kCT;
        float4 ux = f4_zero(), ug = f4_zero();
        if (gi >= 0 && gi < Hl && gj >= 0 && gj < Wl) {
            float ca, cb, cc, cd;
            carrier_block<T>(l, xp, a.W, cpx, Wp, gi, gj, ca, cb, cc, cd);
            ux = haar_u(ca, cb, cc, cd);
            if (inner) {
                if (clx) clx[(size_t)gi * Wl + gj] = 0.5f * ux.x;
                carrier_block<T>(l, gp, a.W, cpy, Wp, gi, gj, ca, cb, cc, cd);
                ug = haar_u(ca, cb, cc, cd);
                if (cly) cly[(size_t)gi * Wl + gj] = 0.5f * ug.x;
            }
        }
        float* q = xb + si * BP + sj;
        q[0] = ux.x;
        q[BAND] = ux.y;
        q[2 * BAND] = ux.z;
        q[3 * BAND] = ux.w;
        if (inner) {
            float* r = gb + (si - R) * kCT + (sj - R);
            r[0] = ug.x;
            r[ZAND] = ug.y;
            r[2 * ZAND] = ug.z;
            r[3 * ZAND] = ug.w;
        }
    }
}

// Sum v[] over all 32 lanes (xor butterfly); every lane ends with the totals.
template <int NV>
__device__ __forceinline__ void warp_sum(float (&v)[NV], int lanes) {
#pragma unroll
    for (int e = 0; e < NV; ++e) {
        float s = v[e];
        for (int m = 1; m < lanes; m <<= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
        v[e] = s;
    }
}

template <int K, typename T>
__global__ void __launch_bounds__(kDT, 3) wt_dw_plane_kernel(const DwArgs a) {
    constexpr int R = FG<K>::R, KK = FG<K>::KK, PAD = FG<K>::PAD;
    constexpr int XP = FG<K>::XPITCH, BP = FG<K>::BPITCH, BAND = FG<K>::BAND;
    constexpr int ZAND = FG<K>::ZAND;
    extern __shared__ float4 smem_f4[];
    float* sm = reinterpret_cast<float*>(smem_f4);
    float* acc_sm = sm + a.o_acc;
    float* red = sm + a.o_red;
    float* xb = sm + a.o_xb;
    float* gb = sm + a.o_gb;
    float* xs = sm + a.o_x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    const int c = blockIdx.x, n = blockIdx.y;
    const size_t plane = (size_t)n * a.C + c;
    const size_t plane_elems = (size_t)a.H * a.W;
    const T* xp = reinterpret_cast<const T*>(a.x) + plane * plane_elems;
    const T* gp = reinterpret_cast<const T*>(a.dy) + plane * plane_elems;
    for (int e = threadIdx.x; e < a.KP; e += blockDim.x) acc_sm[e] = 0.f;
    __syncthreads();

    // ---- deep levels: warp w correlates band w ----
    for (int l = 2; l <= a.L; ++l) {
        const int Hl = a.H >> l, Wl = a.W >> l;
        float accd[KK];
#pragma unroll
        for (int q = 0; q < KK; ++q) accd[q] = 0.f;
        for (int ti0 = 0; ti0 < Hl; ti0 += kCT) {
            for (int tj0 = 0; tj0 < Wl; tj0 += kCT) {
                dw_deep_stage<K, T>(a, xp, gp, sm, l, ti0, tj0);
                __syncthreads();
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int blk = lane + 32 * k, bi = blk >> 3, bj = blk & 7;
                    if (ti0 + 4 * bi >= Hl || tj0 + 4 * bj >= Wl) continue;
                    float g[4][4];
                    const float* gr = gb + warp * ZAND + (4 * bi) * kCT + 4 * bj;
#pragma unroll
                    for (int o = 0; o < 4; ++o) {
                        const float4 t = *reinterpret_cast<const float4*>(gr + o * kCT);
                        g[o][0] = t.x; g[o][1] = t.y; g[o][2] = t.z; g[o][3] = t.w;
                    }
                    corr_rows<K, 4>(xb + warp * BAND + (4 * bi) * BP + 4 * bj, BP, g, accd);
                }
                __syncthreads();
            }
        }
        warp_sum<KK>(accd, 32);
        float* dst = acc_sm + KK + 1 + (l - 1) * 4 * KK + warp * KK;
#pragma unroll
        for (int e = 0; e < KK; ++e)
            if (lane == (e & 31)) dst[e] += accd[e];
    }

    // ---- level 1 and the base path ----
    const bool base_role = (a.L == 0) || (warp < 2);
    float acc[KK + 1];  // taps (+ bias sum for the base role)
#pragma unroll
    for (int q = 0; q <= KK; ++q) acc[q] = 0.f;
    for (int y0 = 0; y0 < a.H; y0 += kTile) {
        for (int x0 = 0; x0 < a.W; x0 += kTile) {
            stage_tile<K, T>(xp, a.H, a.W, a.vec, xs, y0, x0);
            if (a.L >= 1) {
                // dY subbands of the tile's 32x32 coefficients (no halo needed)
                for (int idx = threadIdx.x; idx < kCT * kCT; idx += blockDim.x) {
                    const int ci = idx / kCT, cj = idx - ci * kCT;
                    const int gy = y0 + 2 * ci, gx = x0 + 2 * cj;
                    float4 u = f4_zero();
                    if (gy < a.H && gx < a.W) {
                        const float2 r0 = IO<T>::ld2(gp + (size_t)gy * a.W + gx);
                        const float2 r1 = IO<T>::ld2(gp + (size_t)(gy + 1) * a.W + gx);
                        u = haar_u(r0.x, r0.y, r1.x, r1.y);
                    }
                    float* r = gb + ci * kCT + cj;
                    r[0] = u.x;
                    r[ZAND] = u.y;
                    r[2 * ZAND] = u.z;
                    r[3 * ZAND] = u.w;
                }
            }
            __syncthreads();
            if (a.L >= 1) {
                bands_from_tile<K>(xs, xb);
                __syncthreads();
            }
            if (base_role) {
                const int nb = (a.L == 0) ? 1 : 2;
                for (int k = 0; k < nb; ++k) {
                    const int blk = (a.L == 0) ? threadIdx.x : threadIdx.x + 64 * k;
                    const int by = blk >> 4, bx = blk & 15;
                    const int gy = y0 + 8 * by, gx = x0 + 4 * bx;
                    if (gy >= a.H || gx >= a.W) continue;
                    float g[8][4];
#pragma unroll
                    for (int o = 0; o < 8; ++o) {
                        if (a.vec && gy + o < a.H) {
                            const float4 t = IO<T>::ld4(gp + (size_t)(gy + o) * a.W + gx);
                            g[o][0] = t.x; g[o][1] = t.y; g[o][2] = t.z; g[o][3] = t.w;
                        } else {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                g[o][q] = (gy + o < a.H && gx + q < a.W)
                                              ? IO<T>::ld(gp + (size_t)(gy + o) * a.W + gx + q)
                                              : 0.f;
                        }
                        acc[KK] += (g[o][0] + g[o][1]) + (g[o][2] + g[o][3]);
                    }
                    corr_rows<K, 8>(xs + (8 * by + R) * XP + 4 * bx + R + PAD, XP, g, acc);
                }
            } else {
                const int b = (threadIdx.x - 64) >> 4, j = (threadIdx.x - 64) & 15;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int blk = j + 16 * k, bi = blk >> 3, bj = blk & 7;
                    if (y0 / 2 + 4 * bi >= a.H / 2 || x0 / 2 + 4 * bj >= a.W / 2) continue;
                    float g[4][4];
                    const float* gr = gb + b * ZAND + (4 * bi) * kCT + 4 * bj;
#pragma unroll
                    for (int o = 0; o < 4; ++o) {
                        const float4 t = *reinterpret_cast<const float4*>(gr + o * kCT);
                        g[o][0] = t.x; g[o][1] = t.y; g[o][2] = t.z; g[o][3] = t.w;
                    }
                    corr_rows<K, 4>(xb + b * BAND + (4 * bi) * BP + 4 * bj, BP, g, acc);
                }
            }
            __syncthreads();
        }
    }

    // ---- flush: fixed-order reductions into acc_sm, then the partial vector ----
    if (base_role) {
        warp_sum<KK + 1>(acc, 32);
        if (lane == 0) {
#pragma unroll
            for (int e = 0; e <= KK; ++e) red[warp * (KK + 1) + e] = acc[e];
        }
    } else {
        warp_sum<KK + 1>(acc, 16);  // lanes 0-15 and 16-31 hold one band each
        const int b = (threadIdx.x - 64) >> 4;
        float* dst = acc_sm + KK + 1 + b * KK;
        if ((lane & 15) == 0) {
#pragma unroll
            for (int e = 0; e < KK; ++e) dst[e] += acc[e];
        }
    }
    __syncthreads();
    const int nbase = (a.L == 0) ? 4 : 2;
    for (int e = threadIdx.x; e <= KK; e += blockDim.x) {
        float s = 0.f;
        for (int w = 0; w < nbase; ++w) s += red[w * (KK + 1) + e];
        acc_sm[e] += s;
    }
    __syncthreads();
    float* out = a.part + ((size_t)c * a.N + n) * a.KP;
    for (int e = threadIdx.x; e < a.KP; e += blockDim.x) out[e] = acc_sm[e];
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

template <int K>
void dw_layout(const wt_desc& d, DwArgs& a, size_t& smem_bytes) {
    constexpr int KK = FG<K>::KK;
    const int L = d.levels;
    a.KP = KK + 1 + 4 * KK * L;
    int off = 0;
    a.o_acc = off;
    off += round4(a.KP);
    a.o_red = off;
    off += round4(4 * (KK + 1));
    a.o_xb = off;
    off += 4 * FG<K>::BAND;
    a.o_gb = off;
    off += 4 * FG<K>::ZAND;
    a.o_x = off;
    const int alias0 = off;
    off += FG<K>::XROWS * FG<K>::XPITCH;
    int cp = alias0;
    for (int l = 0; l <= kMaxLevels; ++l) a.o_carx[l] = a.o_cary[l] = 0;
    for (int l = 2; l < L; ++l) {
        const int sz = round4((d.h >> l) * (d.w >> l));
        a.o_carx[l] = cp;
        cp += sz;
        a.o_cary[l] = cp;
        cp += sz;
    }
    const int total = off > cp ? off : cp;
    smem_bytes = (size_t)total * sizeof(float);
}

template <int K, typename T>
wt_status launch_dw_k(const wt_desc& d, const void* x, const void* dy, const float* w0,
                      const float* b0, const float* s0, const float* wl, const float* sl,
                      float* dw0, float* db0, float* ds0, float* dwl, float* dsl, void* ws,
                      size_t ws_bytes, cudaStream_t stream, int* launches) {
    DwArgs a;
    size_t smem = 0;
    dw_layout<K>(d, a, smem);
    if (smem > kMaxSmemPerBlock) return WT_ERR_UNSUPPORTED;
    const size_t need = (size_t)d.c * d.n * a.KP * sizeof(float);
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
    kern<<<dim3((unsigned)d.c, (unsigned)d.n), kDT, smem, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    ++*launches;
    wt_dw_reduce_kernel<<<(unsigned)d.c, 128, (size_t)a.KP * sizeof(float), stream>>>(
        a.part, d.c, d.n, a.KP, K, d.levels, w0, b0, s0, wl, sl, dw0, db0, ds0, dwl, dsl);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    ++*launches;
    return WT_OK;
}

template <int K, typename T>
wt_status launch_dw_partials_k(const wt_desc& d, const void* x, const void* dy, float* part,
                               cudaStream_t stream, int* launches) {
    DwArgs a;
    size_t smem = 0;
    dw_layout<K>(d, a, smem);
    if (smem > kMaxSmemPerBlock) return WT_ERR_UNSUPPORTED;
    a.x = x;
    a.dy = dy;
    a.part = part;
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
    kern<<<dim3((unsigned)d.c, (unsigned)d.n), kDT, smem, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return WT_ERR_CUDA;
    ++*launches;
    return WT_OK;
}

}  // namespace

wt_status launch_dw_partials(const wt_desc& d, const void* x, const void* dy, float* part,
                             cudaStream_t stream, int* launches) {
    const bool bf = d.io == WT_BF16;
    switch (d.k) {
#define WT_CASE(KV)                                                                          \
    case KV:                                                                                 \
        return bf ? launch_dw_partials_k<KV, __nv_bfloat16>(d, x, dy, part, stream, launches) \
                  : launch_dw_partials_k<KV, float>(d, x, dy, part, stream, launches);
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

size_t backward_weight_ws_bytes(const wt_desc& d) {
    const int KK = d.k * d.k;
    const size_t KP = (size_t)KK + 1 + 4 * (size_t)KK * d.levels;
    return (size_t)d.c * d.n * KP * sizeof(float);
}

size_t backward_weight_smem_bytes(const wt_desc& d) {
    DwArgs a;
    size_t smem = 0;
    switch (d.k) {
        case 1: dw_layout<1>(d, a, smem); break;
        case 3: dw_layout<3>(d, a, smem); break;
        case 5: dw_layout<5>(d, a, smem); break;
        case 7: dw_layout<7>(d, a, smem); break;
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
