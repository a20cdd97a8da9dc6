// WTConv forward and backward-data kernel for sm_103a.
//
// Method: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware Reformulation"
// (Aflalo et al.). A persistent CTA walks (n, c) planes and evaluates the whole layer on
// each with one read of X and one write of Y in HBM:
//
//   deep phase (L >= 2) -- levels l = 2..L run at their own resolution: 32x32 output
//     tiles of the level's Haar subbands (§4.1 Eq. 5, recomputed on chip from the
//     low-pass carrier X^(l-1); level 2 reads X itself in 4x4 pixel blocks) are staged in
//     shared memory with an R-coefficient halo, the four folded k x k filters (§4.3 Eq. 8)
//     are applied, and the filtered subbands Z^(l) go to this CTA's private scratch slot
//     (a few tens of KB per CTA: L2-resident, never a full-tensor HBM round trip).
//   full-resolution phase -- 64x64-pixel tiles of X (halo 2R) are staged once; the four
//     level-1 subbands of the tile are formed in shared memory; each subband is filtered
//     by a streaming register-blocked k x k pass (4x4 outputs per thread), and a final pass
//     computes the base k x k convolution (8x4 pixels per thread) and adds, in the same
//     store, the closed-form bit-indexed synthesis of §4.2 Prop. 2 / Eq. 7 over all levels
//     (level 1 from the tile, levels >= 2 from the scratch slot).
//
// Every k x k filter is a streaming stencil: one window row at a time in registers,
// k*k weights in registers, independent accumulators innermost. Shared-memory accesses
// are 16-byte vectors at consecutive addresses across lanes (no bank conflicts).
//
// Backward-data is the same operator on dY with every kernel rotated by 180 degrees and
// no bias (§2.2 Eq. 1: the adjoint of analysis is synthesis; the adjoint of
// cross-correlation is correlation with the rotated kernel); `flip` selects it.
#include "wt_internal.h"
#include "wt_tile.cuh"

namespace wt {

constexpr int kFT = 128;        // threads per CTA
struct FwdArgs {
    const void* x;
    void* y;
    const float* w0f;
    const float* b0f;
    const float* wlf;
    float* zd;             // deep scratch, one slot of zd_slot floats per CTA
    long long zd_slot;
    long long zd_off[kMaxLevels + 1];  // offset of Z^(l) inside a slot, band-major [4][Hl][Wl]
    long long planes;
    int C, H, W, L;
    int flip, vec;
    int o_w, o_x, o_b, o_z;            // shared-memory regions (floats)
    int o_car[kMaxLevels + 1];         // carriers X^(l), l = 2..L-1
};

// ---------------------------------------------------------------------------------
// phases
// ---------------------------------------------------------------------------------

// Folded weights of channel c into shared memory: base kernel, then level l band b at
// slot 1 + 4(l-1) + b, each scaled by 2^-(l+1) (1/2 turns the unnormalized subbands back
// into Eq. 5's, 2^-l is Eq. 7's level weight) and rotated when `flip`.
template <int K>
__device__ __forceinline__ void load_weights(const FwdArgs& a, int c, float* wsm) {
    constexpr int KK = FG<K>::KK, KKP = FG<K>::KKP;
    const int nk = 1 + 4 * a.L;
    for (int e = threadIdx.x; e < nk * KK; e += blockDim.x) {
        const int s = e / KK, uv = e - s * KK;
        const int src = a.flip ? (KK - 1 - uv) : uv;
        float v;
        if (s == 0) {
            v = __ldg(a.w0f + (size_t)c * KK + src);
        } else {
            const int l = 1 + (s - 1) / 4, b = (s - 1) & 3;
            v = ldexpf(1.0f, -(l + 1)) *
                __ldg(a.wlf + (((size_t)(l - 1) * a.C + c) * 4 + b) * KK + src);
        }
        wsm[s * KKP + uv] = v;
    }
}

// Deep phase stage for level l: subbands of the 32x32 output tile at (ti0, tj0) with an
// R halo (zero outside the level grid), band-major; carrier X^(l) for the tile's own
// positions when l < L.
template <int K, typename T>
__device__ __forceinline__ void deep_stage(const FwdArgs& a, const T* xp, float* sm, int l,
                                           int ti0, int tj0) {
    constexpr int R = FG<K>::R, BT = FG<K>::BT, BP = FG<K>::BPITCH, BAND = FG<K>::BAND;
    const int Hl = a.H >> l, Wl = a.W >> l, Wp = a.W >> (l - 1);
    float* bs = sm + a.o_b;
    const float* carp = (l >= 3) ? sm + a.o_car[l - 1] : nullptr;
    float* carl = (l < a.L) ? sm + a.o_car[l] : nullptr;
    for (int idx = threadIdx.x; idx < BT * BT; idx += blockDim.x) {
        const int si = idx / BT, sj = idx - si * BT;
        const int gi = ti0 - R + si, gj = tj0 - R + sj;
        float4 u = f4_zero();
        if (gi >= 0 && gi < Hl && gj >= 0 && gj < Wl) {
            float ca, cb, cc, cd;
            carrier_block<T>(l, xp, a.W, carp, Wp, gi, gj, ca, cb, cc, cd);
            u = haar_u(ca, cb, cc, cd);
            if (carl && si >= R && si < R + kCT && sj >= R && sj < R + kCT)
                carl[(size_t)gi * Wl + gj] = 0.5f * u.x;
        }
        float* q = bs + si * BP + sj;
        q[0] = u.x;
        q[BAND] = u.y;
        q[2 * BAND] = u.z;
        q[3 * BAND] = u.w;
    }
}

template <int K, typename T>
__global__ void __launch_bounds__(kFT, 4) wt_fwd_plane_kernel(const FwdArgs a) {
    constexpr int R = FG<K>::R, KKP = FG<K>::KKP, PAD = FG<K>::PAD;
    constexpr int XP = FG<K>::XPITCH, BP = FG<K>::BPITCH, BAND = FG<K>::BAND;
    extern __shared__ float4 smem_f4[];
    float* sm = reinterpret_cast<float*>(smem_f4);
    float* wsm = sm + a.o_w;
    float* xs = sm + a.o_x;
    float* bs = sm + a.o_b;
    float* zs = sm + a.o_z;
    float* zslot = a.zd + (size_t)blockIdx.x * a.zd_slot;
    const size_t plane_elems = (size_t)a.H * a.W;

    for (long long plane = blockIdx.x; plane < a.planes; plane += gridDim.x) {
        const int c = (int)(plane % a.C);
        const T* xp = reinterpret_cast<const T*>(a.x) + plane * plane_elems;
        T* yp = reinterpret_cast<T*>(a.y) + plane * plane_elems;
        __syncthreads();  // previous plane is done with shared memory and weights
        load_weights<K>(a, c, wsm);
        const float bias = (a.b0f != nullptr) ? __ldg(a.b0f + c) : 0.f;
        __syncthreads();

        // ---- deep phase: Z^(l), l = 2..L, into the scratch slot ----
        for (int l = 2; l <= a.L; ++l) {
            const int Hl = a.H >> l, Wl = a.W >> l;
            float* zl = zslot + a.zd_off[l];
            for (int ti0 = 0; ti0 < Hl; ti0 += kCT) {
                for (int tj0 = 0; tj0 < Wl; tj0 += kCT) {
                    deep_stage<K, T>(a, xp, sm, l, ti0, tj0);
                    __syncthreads();
                    for (int it = threadIdx.x; it < 4 * 64; it += blockDim.x) {
                        const int b = it >> 6, bi = (it >> 3) & 7, bj = it & 7;
                        const int gi0 = ti0 + 4 * bi, gj0 = tj0 + 4 * bj;
                        if (gi0 >= Hl || gj0 >= Wl) continue;
                        float acc[4][4];
                        conv4x4<K>(bs + b * BAND + (4 * bi) * BP + 4 * bj, BP,
                                   wsm + (1 + 4 * (l - 1) + b) * KKP, acc);
                        float* zb = zl + (size_t)b * Hl * Wl;
#pragma unroll
                        for (int o = 0; o < 4; ++o) {
                            if (gi0 + o >= Hl) continue;
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                if (gj0 + q < Wl) zb[(size_t)(gi0 + o) * Wl + gj0 + q] = acc[o][q];
                        }
                    }
                    __syncthreads();
                }
            }
        }

        // ---- full-resolution phase ----
        const int by = threadIdx.x >> 4, bx = threadIdx.x & 15;  // 8x4-pixel base block
        for (int y0 = 0; y0 < a.H; y0 += kTile) {
            for (int x0 = 0; x0 < a.W; x0 += kTile) {
                stage_tile<K, T>(xp, a.H, a.W, a.vec, xs, y0, x0);
                __syncthreads();
                if (a.L >= 1) {
                    bands_from_tile<K>(xs, bs);
                    __syncthreads();
                    // level-1 filters: 4 bands x 64 blocks of 4x4 coefficients
                    for (int it = threadIdx.x; it < 4 * 64; it += blockDim.x) {
                        const int b = it >> 6, bi = (it >> 3) & 7, bj = it & 7;
                        if (y0 / 2 + 4 * bi >= (a.H + 1) / 2 || x0 / 2 + 4 * bj >= (a.W + 1) / 2)
                            continue;
                        float acc[4][4];
                        conv4x4<K>(bs + b * BAND + (4 * bi) * BP + 4 * bj, BP,
                                   wsm + (1 + b) * KKP, acc);
#pragma unroll
                        for (int o = 0; o < 4; ++o)
                            *reinterpret_cast<float4*>(zs + b * (kCT * kCT) + (4 * bi + o) * kCT + 4 * bj) =
                                make_float4(acc[o][0], acc[o][1], acc[o][2], acc[o][3]);
                    }
                    __syncthreads();
                }
                const int gy = y0 + 8 * by, gx = x0 + 4 * bx;
                if (gy < a.H && gx < a.W) {
                    float acc[8][4];
#pragma unroll
                    for (int o = 0; o < 8; ++o)
#pragma unroll
                        for (int q = 0; q < 4; ++q) acc[o][q] = bias;
                    conv8x4<K>(xs + (8 * by + R) * XP + 4 * bx + R + PAD, XP, wsm, acc);
                    if (a.L >= 1) {
                        // Eq. 7: level 1 from the z tile, levels >= 2 from the scratch slot
                        float d[4][2];
#pragma unroll
                        for (int i = 0; i < 4; ++i) d[i][0] = d[i][1] = 0.f;
                        const int gci0 = gy >> 1, gcj0 = gx >> 1;  // gci0 % 4 == 0, gcj0 even
                        for (int l = 2; l <= a.L; ++l) {
                            const int Hl = a.H >> l, Wl = a.W >> l;
                            const float* zl = zslot + a.zd_off[l];
                            const size_t bst = (size_t)Hl * Wl;
                            const int sh = l - 1;
                            const int jl = gcj0 >> sh;
                            const int sx = (gcj0 >> (l - 2)) & 1;  // l >= 3: same for both columns
#pragma unroll
                            for (int half = 0; half < 2; ++half) {
                                // l == 2: rows gci0/2 and gci0/2 + 1; l >= 3: one row
                                if (l >= 3 && half == 1) break;
                                const int il = (gci0 >> sh) + half;
                                if (il >= Hl) break;  // rows past H (H = 4 mod 8) are not stored
                                const float* zp = zl + (size_t)il * Wl + jl;
                                const float4 z = make_float4(zp[0], zp[bst], zp[2 * bst], zp[3 * bst]);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    if (l == 2 && (i >> 1) != half) continue;
                                    const int syb = (l == 2) ? (i & 1)
                                                  : (l == 3) ? ((i >> 1) & 1)
                                                             : ((gci0 >> (l - 2)) & 1);
#pragma unroll
                                    for (int j = 0; j < 2; ++j) {
                                        const int sxb = (l == 2) ? j : sx;
                                        d[i][j] += synth_rt(z, syb, sxb);
                                    }
                                }
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float z1[2][4];
                            const float* zr = zs + (4 * by + i) * kCT + 2 * bx;
#pragma unroll
                            for (int b = 0; b < 4; ++b) {
                                const float2 t = *reinterpret_cast<const float2*>(zr + b * (kCT * kCT));
                                z1[0][b] = t.x;
                                z1[1][b] = t.y;
                            }
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const float4 z = make_float4(z1[j][0], z1[j][1], z1[j][2], z1[j][3]);
                                acc[2 * i][2 * j] += synth<0, 0>(z) + d[i][j];
                                acc[2 * i][2 * j + 1] += synth<0, 1>(z) + d[i][j];
                                acc[2 * i + 1][2 * j] += synth<1, 0>(z) + d[i][j];
                                acc[2 * i + 1][2 * j + 1] += synth<1, 1>(z) + d[i][j];
                            }
                        }
                    }
                    if (a.vec && gy + 8 <= a.H && gx + 4 <= a.W) {
#pragma unroll
                        for (int o = 0; o < 8; ++o)
                            IO<T>::st4(yp + (size_t)(gy + o) * a.W + gx,
                                       make_float4(acc[o][0], acc[o][1], acc[o][2], acc[o][3]));
                    } else {
#pragma unroll
                        for (int o = 0; o < 8; ++o)
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                if (gy + o < a.H && gx + q < a.W)
                                    IO<T>::st(yp + (size_t)(gy + o) * a.W + gx + q, acc[o][q]);
                    }
                }
                __syncthreads();
            }
        }
    }
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------

namespace {

int round4(int v) { return (v + 3) & ~3; }

struct FwdPlan {
    FwdArgs a;
    size_t smem = 0;
    int grid = 0;
    size_t ws_bytes = 0;
};

template <int K>
FwdPlan fwd_plan(const wt_desc& d) {
    FwdPlan p;
    FwdArgs& a = p.a;
    const int L = d.levels;
    int off = 0;
    a.o_w = off;
    off += FG<K>::KKP * (1 + 4 * L);
    off = round4(off);
    // the F-phase buffers; the deep carriers alias the X and z tiles
    a.o_b = off;
    off += 4 * FG<K>::BAND;
    const int alias0 = off;
    a.o_x = off;
    off += FG<K>::XROWS * FG<K>::XPITCH;
    a.o_z = off;
    off += 4 * FG<K>::ZAND;
    int cp = alias0;
    for (int l = 0; l <= kMaxLevels; ++l) a.o_car[l] = 0;
    for (int l = 2; l < L; ++l) {
        a.o_car[l] = cp;
        cp += round4((d.h >> l) * (d.w >> l));
    }
    const int total = off > cp ? off : cp;
    p.smem = (size_t)total * sizeof(float);
    // deep scratch slot: Z^(l) band-major for l = 2..L
    long long zo = 0;
    for (int l = 0; l <= kMaxLevels; ++l) a.zd_off[l] = 0;
    for (int l = 2; l <= L; ++l) {
        a.zd_off[l] = zo;
        zo += 4LL * (d.h >> l) * (d.w >> l);
    }
    a.zd_slot = (zo + 63) & ~63LL;  // 256-byte aligned slots
    const long long planes = (long long)d.n * d.c;
    int occ = (int)((228 * 1024) / (p.smem + 1024));
    if (occ > 4) occ = 4;
    if (occ < 1) occ = 1;
    long long grid = (long long)kNumSMs * occ;
    if (grid > planes) grid = planes;
    p.grid = (int)grid;
    p.ws_bytes = (L >= 2) ? (size_t)grid * (size_t)a.zd_slot * sizeof(float) : 0;
    return p;
}

template <int K, typename T>
wt_status launch_fwd_k(const wt_desc& d, const void* x, const float* w0f, const float* b0f,
                       const float* wlf, void* y, int flip, void* ws, size_t ws_bytes,
                       cudaStream_t stream, int* launches) {
    FwdPlan p = fwd_plan<K>(d);
    if (p.smem > kMaxSmemPerBlock) return WT_ERR_UNSUPPORTED;
    if (p.ws_bytes > 0 && (ws == nullptr || ws_bytes < p.ws_bytes)) return WT_ERR_WORKSPACE;
    FwdArgs& a = p.a;
    a.x = x;
    a.y = y;
    a.w0f = w0f;
    a.b0f = flip ? nullptr : b0f;
    a.wlf = wlf;
    a.zd = reinterpret_cast<float*>(ws);
    a.planes = (long long)d.n * d.c;
    a.C = d.c;
    a.H = d.h;
    a.W = d.w;
    a.L = d.levels;
    a.flip = flip;
    a.vec = (d.w % 4 == 0) ? 1 : 0;
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
    FwdPlan p = fwd_plan<K>(d);
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
