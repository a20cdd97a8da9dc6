// WTConv forward as separate materializing stages, and the cumulative ablation variants.
//
// Method: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware Reformulation"
// (Aflalo et al.). The reference pipeline follows §3.1 / Figure 1a: every stage of
// Algorithm 1 reads its input tensor from HBM and writes its output tensor back. The
// variants add, cumulatively, the reformulations of §4 in the order of §5.6: the per-level
// fused analysis + conv + scale pass (§4.1), the single bit-indexed synthesis pass (§4.2
// Prop. 2, Eq. 7), and scale folding with the base add fused into the final store (§4.3).
// These kernels exist to measure what each reformulation saves (time and HBM traffic, the
// analogue of the pages' Tables 8 and 11); the production forward is wt_fwd.cu.
//
// All stages are fp32. Kernels are plain grid-stride or shared-memory-tiled CUDA: each
// stage is coalesced and reads / writes its tensors once, like the framework primitives the
// reference chains together.
#include <stdint.h>

#include "wt_common.cuh"
#include "wt_internal.h"
#include "wtconv_ablation.h"

namespace wt {

namespace {

constexpr int kEwThreads = 256;

int ew_blocks(long long n) {
    long long b = (n + kEwThreads - 1) / kEwThreads;
    if (b > 8 * kNumSMs * 8) b = 8 * kNumSMs * 8;
    return (int)(b < 1 ? 1 : b);
}

// ---------------------------------------------------------------------------------
// Reference stages
// ---------------------------------------------------------------------------------

// Eq. 5 Haar analysis: in plane p at in + p * in_ps ([2Ho][2Wo]) -> out [P][4][Ho][Wo].
__global__ void k_haar_analysis(const float* in, long long in_ps, int Ho, int Wo, long long P,
                                float* out) {
    const long long n = P * Ho * Wo;
    const int Wi = 2 * Wo;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        const long long p = e / ((long long)Ho * Wo);
        const int r = (int)(e - p * Ho * Wo), i = r / Wo, j = r - i * Wo;
        const float* q = in + p * in_ps + (size_t)(2 * i) * Wi + 2 * j;
        const float a = q[0], b = q[1], c = q[Wi], d = q[Wi + 1];
        float* o = out + (p * 4) * Ho * Wo + r;
        const long long bs = (long long)Ho * Wo;
        o[0] = 0.5f * (a + b + c + d);
        o[bs] = 0.5f * (a + b - c - d);
        o[2 * bs] = 0.5f * (a - b + c - d);
        o[3 * bs] = 0.5f * (a - b - c + d);
    }
}

// Eq. 12 inverse Haar (the reference's transposed stride-2 conv): in [P][4][Ho][Wo] ->
// out [P][2Ho][2Wo].
__global__ void k_haar_synthesis(const float* in, int Ho, int Wo, long long P, float* out) {
    const long long n = P * Ho * Wo;
    const long long bs = (long long)Ho * Wo;
    const int Wi = 2 * Wo;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        const long long p = e / bs;
        const int r = (int)(e - p * bs), i = r / Wo, j = r - i * Wo;
        const float* z = in + p * 4 * bs + r;
        const float ll = z[0], lh = z[bs], hl = z[2 * bs], hh = z[3 * bs];
        float* o = out + p * 4 * bs + (size_t)(2 * i) * Wi + 2 * j;
        o[0] = 0.5f * (ll + lh + hl + hh);
        o[1] = 0.5f * (ll + lh - hl - hh);
        o[Wi] = 0.5f * (ll - lh + hl - hh);
        o[Wi + 1] = 0.5f * (ll - lh - hl + hh);
    }
}

// out[p][i] = a[p * a_ps + i] + (b ? b[p * b_ps + i] : 0) over planes of n elements.
__global__ void k_add_planes(const float* a, long long a_ps, const float* b, long long b_ps,
                             long long n, long long P, float* out) {
    const long long tot = P * n;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < tot;
         e += (long long)gridDim.x * blockDim.x) {
        const long long p = e / n, i = e - p * n;
        float v = a[p * a_ps + i];
        if (b != nullptr) v += b[p * b_ps + i];
        out[e] = v;
    }
}

// out[p][i] = in[p][i] * s[p % nch] over planes of n elements; float4 access when
// n % 4 == 0 (vec4), else one element per thread.
__global__ void k_scale_planes(const float* in, const float* s, int nch, long long n,
                               long long P, int vec4, float* out) {
    if (vec4) {
        const long long n4 = n / 4, tot = P * n4;
        for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < tot;
             e += (long long)gridDim.x * blockDim.x) {
            const float sc = s[(e / n4) % nch];
            float4 v = reinterpret_cast<const float4*>(in)[e];
            v.x *= sc; v.y *= sc; v.z *= sc; v.w *= sc;
            reinterpret_cast<float4*>(out)[e] = v;
        }
    } else {
        const long long tot = P * n;
        for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < tot;
             e += (long long)gridDim.x * blockDim.x)
            out[e] = in[e] * s[(e / n) % nch];
    }
}

// Launch of k_scale_planes sized to its access width.
void scale_planes(const float* in, const float* s, int nch, long long n, long long P, float* out,
                  cudaStream_t st) {
    const int vec4 = (n % 4 == 0) ? 1 : 0;
    k_scale_planes<<<ew_blocks(vec4 ? P * n / 4 : P * n), kEwThreads, 0, st>>>(in, s, nch, n, P,
                                                                               vec4, out);
}

// Concatenation of the summed low-pass band with the three high bands:
// out[p][0] = xll[p], out[p][b] = z[p][b] for b = 1..3 (planes of n elements).
__global__ void k_concat(const float* xll, const float* z, long long n, long long P, float* out) {
    const long long tot = P * 4 * n;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < tot;
         e += (long long)gridDim.x * blockDim.x) {
        const long long q = e / n, i = e - q * n;  // q = 4 p + band
        const long long p = q >> 2;
        out[e] = ((q & 3) == 0) ? xll[p * n + i] : z[e];
    }
}

// Zero-padded "same" depthwise k x k cross-correlation, one plane per (p): out plane p at
// out + p * out_ps = sum_{u,v} w[p % nch][u][v] in[y+u-R][x+v-R] (+ bias[p % nch]).
// Tiles of 32 x 64 outputs staged with an R halo in shared memory; 8 outputs per thread.
constexpr int kCTY = 32, kCTX = 64;

template <int K>
__global__ void __launch_bounds__(256) k_dwconv(const float* in, long long in_ps,
                                                const float* w, const float* bias, int nch,
                                                int H, int W, long long P, float* out,
                                                long long out_ps) {
    constexpr int R = (K - 1) / 2, KK = K * K;
    constexpr int SR = kCTY + 2 * R, SC = kCTX + 2 * R, SP = SC + 1;
    __shared__ float tile[SR * SP];
    __shared__ float wsh[KK];
    const int tx = (W + kCTX - 1) / kCTX, ty = (H + kCTY - 1) / kCTY;
    const long long nblk = P * tx * ty;
    const int r = threadIdx.x >> 3, c0 = (threadIdx.x & 7) * 8;
    for (long long blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        const long long p = blk / (tx * ty);
        const int t = (int)(blk - p * tx * ty), by = t / tx, bx = t - by * tx;
        const int y0 = by * kCTY, x0 = bx * kCTX;
        const int ch = (int)(p % nch);
        __syncthreads();  // the previous tile is done with shared memory
        if (threadIdx.x < KK) wsh[threadIdx.x] = w[(size_t)ch * KK + threadIdx.x];
        const float* ip = in + p * in_ps;
        for (int e = threadIdx.x; e < SR * SC; e += blockDim.x) {
            const int rr = e / SC, cc = e - rr * SC;
            const int gy = y0 - R + rr, gx = x0 - R + cc;
            tile[rr * SP + cc] =
                (gy >= 0 && gy < H && gx >= 0 && gx < W) ? ip[(size_t)gy * W + gx] : 0.f;
        }
        __syncthreads();
        const float b0 = bias ? bias[ch] : 0.f;
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = b0;
#pragma unroll
        for (int u = 0; u < K; ++u) {
            float v[8 + 2 * R];
#pragma unroll
            for (int m = 0; m < 8 + 2 * R; ++m) v[m] = tile[(r + u) * SP + c0 + m];
#pragma unroll
            for (int vv = 0; vv < K; ++vv) {
                const float wt = wsh[u * K + vv];
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = fmaf(wt, v[q + vv], acc[q]);
            }
        }
        const int gy = y0 + r;
        if (gy < H) {
            float* op = out + p * out_ps + (size_t)gy * W + x0 + c0;
            if ((W & 3) == 0 && x0 + c0 + 8 <= W) {
                reinterpret_cast<float4*>(op)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                reinterpret_cast<float4*>(op)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (x0 + c0 + q < W) op[q] = acc[q];
            }
        }
    }
}

// ---------------------------------------------------------------------------------
// Fused stages
// ---------------------------------------------------------------------------------

// §4.1: one level in one pass. The Haar subbands of the carrier xin ([P][2Ho][2Wo]) are
// recomputed on chip for a 32 x 32 coefficient tile with an R halo, filtered per band by
// wl_l[c][b] (k x k), multiplied by sl_l[c][b] when sl_l is given (else the weights are
// folded), and written to z [P][4][Ho][Wo]; the raw LL band goes to carrier [P][Ho][Wo]
// when carrier != nullptr.
constexpr int kFLT = 32;

template <int K>
__global__ void __launch_bounds__(256) k_fused_level(const float* xin, const float* wl_l,
                                                     const float* sl_l, int C, int Ho, int Wo,
                                                     long long P, float* z, float* carrier) {
    constexpr int R = (K - 1) / 2, KK = K * K;
    constexpr int BT = kFLT + 2 * R, BP = BT + 1;
    __shared__ float bands[4][BT * BP];
    __shared__ float wsh[4 * KK];
    __shared__ float ssh[4];
    const int tx = (Wo + kFLT - 1) / kFLT, ty = (Ho + kFLT - 1) / kFLT;
    const long long nblk = P * tx * ty;
    const int Wi = 2 * Wo;
    const long long bs = (long long)Ho * Wo;
    const int band = threadIdx.x >> 6, row = (threadIdx.x & 63) >> 1,
              c0 = (threadIdx.x & 1) * 16;
    for (long long blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        const long long p = blk / (tx * ty);
        const int t = (int)(blk - p * tx * ty), by = t / tx, bx = t - by * tx;
        const int i0 = by * kFLT, j0 = bx * kFLT;
        const int c = (int)(p % C);
        __syncthreads();
        for (int e = threadIdx.x; e < 4 * KK; e += blockDim.x)
            wsh[e] = wl_l[(size_t)c * 4 * KK + e];
        if (threadIdx.x < 4) ssh[threadIdx.x] = sl_l ? sl_l[(size_t)c * 4 + threadIdx.x] : 1.f;
        const float* xp = xin + p * (long long)(2 * Ho) * Wi;
        for (int e = threadIdx.x; e < BT * BT; e += blockDim.x) {
            const int si = e / BT, sj = e - si * BT;
            const int gi = i0 - R + si, gj = j0 - R + sj;
            float ll = 0.f, lh = 0.f, hl = 0.f, hh = 0.f;
            if (gi >= 0 && gi < Ho && gj >= 0 && gj < Wo) {
                const float* q = xp + (size_t)(2 * gi) * Wi + 2 * gj;
                const float a = q[0], b = q[1], cc = q[Wi], d = q[Wi + 1];
                ll = 0.5f * (a + b + cc + d);
                lh = 0.5f * (a + b - cc - d);
                hl = 0.5f * (a - b + cc - d);
                hh = 0.5f * (a - b - cc + d);
                if (carrier != nullptr && si >= R && si < R + kFLT && sj >= R && sj < R + kFLT)
                    carrier[p * bs + (size_t)gi * Wo + gj] = ll;
            }
            bands[0][si * BP + sj] = ll;
            bands[1][si * BP + sj] = lh;
            bands[2][si * BP + sj] = hl;
            bands[3][si * BP + sj] = hh;
        }
        __syncthreads();
        float acc[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) acc[q] = 0.f;
        const float* bp = bands[band];
#pragma unroll
        for (int u = 0; u < K; ++u) {
            float v[16 + 2 * R];
#pragma unroll
            for (int m = 0; m < 16 + 2 * R; ++m) v[m] = bp[(row + u) * BP + c0 + m];
#pragma unroll
            for (int vv = 0; vv < K; ++vv) {
                const float wt = wsh[band * KK + u * K + vv];
#pragma unroll
                for (int q = 0; q < 16; ++q) acc[q] = fmaf(wt, v[q + vv], acc[q]);
            }
        }
        const int gi = i0 + row;
        if (gi < Ho) {
            const float sc = ssh[band];
            float* op = z + (p * 4 + band) * bs + (size_t)gi * Wo + j0 + c0;
#pragma unroll
            for (int q = 0; q < 16; ++q)
                if (j0 + c0 + q < Wo) op[q] = sl_l ? acc[q] * sc : acc[q];
        }
    }
}

// §4.2 Prop. 2 / Eq. 7: out[p][y][x] = (base ? base[p][y][x] : 0)
//   + sum_l 2^-l (Z_LL + s_y Z_LH + s_x Z_HL + s_y s_x Z_HH)^(l) at (y >> l, x >> l),
// s_y = (-1)^(bit l-1 of y), s_x likewise. One thread per level-1 position (a 2 x 2 output
// block); z[l-1] is level l's [P][4][H_l][W_l] subband tensor.
struct SynthArgs {
    const float* z[kMaxLevels];
};

__global__ void k_collapsed_synthesis(const __grid_constant__ SynthArgs za, int L, int H, int W, long long P,
                                      const float* base, float* out) {
    const int H1 = H >> 1, W1 = W >> 1;
    const long long n = P * H1 * W1;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        const long long p = e / ((long long)H1 * W1);
        const int r = (int)(e - p * H1 * W1), i = r / W1, j = r - i * W1;
        float o[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        for (int l = 1; l <= L; ++l) {
            const int Hl = H >> l, Wl = W >> l, sh = l - 1;
            const long long bs = (long long)Hl * Wl;
            const float* zl = za.z[l - 1] + p * 4 * bs + (size_t)(i >> sh) * Wl + (j >> sh);
            const float ll = zl[0], lh = zl[bs], hl = zl[2 * bs], hh = zl[3 * bs];
            const float f = ldexpf(1.0f, -l);
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    // coordinate bit l-1 of y = 2i + a, x = 2j + b
                    const int by = (l == 1) ? a : ((i >> (l - 2)) & 1);
                    const int bx = (l == 1) ? b : ((j >> (l - 2)) & 1);
                    const float t0 = by ? (ll - lh) : (ll + lh);
                    const float t1 = by ? (hl - hh) : (hl + hh);
                    o[a][b] += f * (bx ? (t0 - t1) : (t0 + t1));
                }
        }
        const size_t o0 = (size_t)p * H * W + (size_t)(2 * i) * W + 2 * j;
#pragma unroll
        for (int a = 0; a < 2; ++a) {
            float2 v = make_float2(o[a][0], o[a][1]);
            if (base != nullptr) {
                const float2 bv = *reinterpret_cast<const float2*>(base + o0 + (size_t)a * W);
                v.x += bv.x;
                v.y += bv.y;
            }
            *reinterpret_cast<float2*>(out + o0 + (size_t)a * W) = v;
        }
    }
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------

// Bump allocator over the workspace; with base == nullptr it only measures.
struct Arena {
    char* base;
    size_t off = 0;
    float* take(size_t floats) {
        float* p = base ? reinterpret_cast<float*>(base + off) : nullptr;
        off += (floats * sizeof(float) + 255) & ~size_t(255);
        return p;
    }
};

struct Plan {
    // per level l (index l - 1)
    float* y[kMaxLevels] = {};       // Haar subbands Y^(l) (reference)
    float* conv[kMaxLevels] = {};    // conv output (reference)
    float* z[kMaxLevels] = {};       // scaled subbands Z^(l)
    float* car[kMaxLevels] = {};     // raw LL carriers (fused variants)
    float* xll[kMaxLevels] = {};     // summed low-pass band (synthesis cascade)
    float* cat[kMaxLevels] = {};     // concatenated bands (synthesis cascade)
    float* nxt[kMaxLevels] = {};     // inverse-Haar output (synthesis cascade)
    float* sum = nullptr;                    // collapsed level sum (variant 2)
    float* bconv = nullptr;                  // base conv output
    float* bscaled = nullptr;                // base conv * s0
    float* w0f = nullptr;                    // folded parameters (variant 3)
    float* b0f = nullptr;
    float* wlf = nullptr;
};

Plan plan_variant(const wt_desc& d, int v, Arena& ar) {
    Plan pl;
    const long long P = (long long)d.n * d.c;
    const long long N = P * d.h * d.w;
    const int L = d.levels, KK = d.k * d.k;
    for (int l = 1; l <= L; ++l) {
        const long long Nl = P * 4 * (long long)(d.h >> l) * (d.w >> l);  // N_l elements
        if (v == WT_VARIANT_REFERENCE) {
            pl.y[l - 1] = ar.take(Nl);
            pl.conv[l - 1] = ar.take(Nl);
        } else if (l < L) {
            pl.car[l - 1] = ar.take(Nl / 4);
        }
        pl.z[l - 1] = ar.take(Nl);
        if (v <= WT_VARIANT_FUSED_ANALYSIS) {
            pl.xll[l - 1] = ar.take(Nl / 4);
            pl.cat[l - 1] = ar.take(Nl);
            pl.nxt[l - 1] = ar.take(Nl);
        }
    }
    if (v == WT_VARIANT_COLLAPSED_SYNTHESIS && L >= 1) pl.sum = ar.take(N);
    pl.bconv = ar.take(N);
    if (v != WT_VARIANT_FOLDED) pl.bscaled = ar.take(N);
    if (v == WT_VARIANT_FOLDED) {
        pl.w0f = ar.take((size_t)d.c * KK);
        pl.b0f = ar.take((size_t)d.c);
        pl.wlf = ar.take((size_t)L * d.c * 4 * KK + 1);
    }
    return pl;
}

template <int K>
wt_status run_variant(const wt_desc& d, int v, const float* x, const float* w0, const float* b0,
                      const float* s0, const float* wl, const float* sl, float* y,
                      const Plan& pl, cudaStream_t s, int* launches) {
    const long long P = (long long)d.n * d.c;
    const int L = d.levels, C = d.c;
    constexpr int KK = K * K;
    const long long HW = (long long)d.h * d.w;
    auto ok = [&]() -> bool {
        ++*launches;
        return cudaGetLastError() == cudaSuccess;
    };
    const int conv_grid = 4 * kNumSMs * 8;

    const float* wlv = wl;
    const float* slv = sl;
    const float* w0v = w0;
    const float* b0v = b0;
    if (v == WT_VARIANT_FOLDED) {
        wt_status st = launch_fold(d, w0, b0, s0, wl, sl, pl.w0f, pl.b0f, pl.wlf, s, launches);
        if (st != WT_OK) return st;
        wlv = pl.wlf;
        slv = nullptr;
        w0v = pl.w0f;
        b0v = pl.b0f;
    }

    // ---- analysis, level by level ----
    const float* cur = x;
    long long cur_ps = HW;
    for (int l = 1; l <= L; ++l) {
        const int Hl = d.h >> l, Wl = d.w >> l;
        const long long bs = (long long)Hl * Wl;
        const float* wl_l = wlv + (size_t)(l - 1) * C * 4 * KK;
        const float* sl_l = slv ? slv + (size_t)(l - 1) * C * 4 : nullptr;
        if (v == WT_VARIANT_REFERENCE) {
            k_haar_analysis<<<ew_blocks(P * bs), kEwThreads, 0, s>>>(cur, cur_ps, Hl, Wl, P,
                                                                     pl.y[l - 1]);
            if (!ok()) return WT_ERR_CUDA;
            const int tiles = ((Hl + kCTY - 1) / kCTY) * ((Wl + kCTX - 1) / kCTX);
            long long blocks = 4 * P * tiles;
            if (blocks > conv_grid) blocks = conv_grid;
            k_dwconv<K><<<(int)blocks, 256, 0, s>>>(pl.y[l - 1], bs, wl_l, nullptr, 4 * C, Hl, Wl,
                                                    4 * P, pl.conv[l - 1], bs);
            if (!ok()) return WT_ERR_CUDA;
            scale_planes(pl.conv[l - 1], sl_l, 4 * C, bs, 4 * P, pl.z[l - 1], s);
            if (!ok()) return WT_ERR_CUDA;
            cur = pl.y[l - 1];  // the LL band of Y^(l), read in place by the next level
            cur_ps = 4 * bs;
        } else {
            const int tiles = ((Hl + kFLT - 1) / kFLT) * ((Wl + kFLT - 1) / kFLT);
            long long blocks = P * tiles;
            if (blocks > conv_grid) blocks = conv_grid;
            k_fused_level<K><<<(int)blocks, 256, 0, s>>>(cur, wl_l, sl_l, C, Hl, Wl, P,
                                                         pl.z[l - 1],
                                                         l < L ? pl.car[l - 1] : nullptr);
            if (!ok()) return WT_ERR_CUDA;
            cur = pl.car[l - 1];
            cur_ps = bs;
        }
    }

    // ---- synthesis ----
    const float* levels_sum = nullptr;  // full-resolution sum of the level terms
    if (L >= 1 && v <= WT_VARIANT_FUSED_ANALYSIS) {
        const float* nxt = nullptr;  // R^(l+1) at level-l resolution
        for (int l = L; l >= 1; --l) {
            const int Hl = d.h >> l, Wl = d.w >> l;
            const long long bs = (long long)Hl * Wl;
            k_add_planes<<<ew_blocks(P * bs), kEwThreads, 0, s>>>(pl.z[l - 1], 4 * bs, nxt, bs,
                                                                  bs, P, pl.xll[l - 1]);
            if (!ok()) return WT_ERR_CUDA;
            k_concat<<<ew_blocks(4 * P * bs), kEwThreads, 0, s>>>(pl.xll[l - 1], pl.z[l - 1],
                                                                  bs, P, pl.cat[l - 1]);
            if (!ok()) return WT_ERR_CUDA;
            k_haar_synthesis<<<ew_blocks(P * bs), kEwThreads, 0, s>>>(pl.cat[l - 1], Hl, Wl, P,
                                                                      pl.nxt[l - 1]);
            if (!ok()) return WT_ERR_CUDA;
            nxt = pl.nxt[l - 1];
        }
        levels_sum = nxt;
    } else if (L >= 1 && v == WT_VARIANT_COLLAPSED_SYNTHESIS) {
        SynthArgs za{};
        for (int l = 1; l <= L; ++l) za.z[l - 1] = pl.z[l - 1];
        k_collapsed_synthesis<<<ew_blocks(P * HW / 4), kEwThreads, 0, s>>>(za, L, d.h, d.w, P,
                                                                          nullptr, pl.sum);
        if (!ok()) return WT_ERR_CUDA;
        levels_sum = pl.sum;
    }

    // ---- base path ----
    const bool base_is_output = (v == WT_VARIANT_FOLDED && L == 0);
    {
        const int tiles = ((d.h + kCTY - 1) / kCTY) * ((d.w + kCTX - 1) / kCTX);
        long long blocks = P * tiles;
        if (blocks > conv_grid) blocks = conv_grid;
        k_dwconv<K><<<(int)blocks, 256, 0, s>>>(x, HW, w0v, b0v, C, d.h, d.w, P,
                                                base_is_output ? y : pl.bconv, HW);
        if (!ok()) return WT_ERR_CUDA;
    }
    if (v == WT_VARIANT_FOLDED) {
        if (L >= 1) {  // base + Eq. 7 level sum, written once
            SynthArgs za{};
            for (int l = 1; l <= L; ++l) za.z[l - 1] = pl.z[l - 1];
            k_collapsed_synthesis<<<ew_blocks(P * HW / 4), kEwThreads, 0, s>>>(
                za, L, d.h, d.w, P, pl.bconv, y);
            if (!ok()) return WT_ERR_CUDA;
        }
        return WT_OK;
    }
    scale_planes(pl.bconv, s0, C, HW, P, pl.bscaled, s);
    if (!ok()) return WT_ERR_CUDA;
    k_add_planes<<<ew_blocks(P * HW), kEwThreads, 0, s>>>(pl.bscaled, HW, levels_sum, HW, HW, P,
                                                          y);
    if (!ok()) return WT_ERR_CUDA;
    return WT_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

wt_status check_variant(const wt_desc* desc, int variant) {
    size_t a = 0, b = 0, c = 0;
    wt_status st = wtconv_workspace_size(desc, &a, &b, &c);  // validates the descriptor
    if (st != WT_OK) return st;
    if (variant < WT_VARIANT_REFERENCE || variant > WT_VARIANT_FOLDED) return WT_ERR_INVALID_ARG;
    if (desc->io != WT_F32) return WT_ERR_UNSUPPORTED;
    if (desc->levels > kMaxLevels) return WT_ERR_UNSUPPORTED;
    // the staged pipelines materialize every level at exactly half the size of the last
    const int m = 1 << desc->levels;
    if ((desc->h % m) != 0 || (desc->w % m) != 0) return WT_ERR_UNSUPPORTED;
    return WT_OK;
}

}  // namespace

}  // namespace wt

using namespace wt;

extern "C" wt_status wtconv_variant_workspace_size(const wt_desc* desc, int variant,
                                                   size_t* bytes) {
    wt_status st = check_variant(desc, variant);
    if (st != WT_OK) return st;
    if (bytes == nullptr) return WT_ERR_INVALID_ARG;
    Arena ar{nullptr};
    plan_variant(*desc, variant, ar);
    *bytes = ar.off;
    return WT_OK;
}

extern "C" wt_status wtconv_forward_variant(const wt_desc* desc, int variant, const void* x,
                                            const float* w0, const float* b0, const float* s0,
                                            const float* wl, const float* sl, void* y, void* ws,
                                            size_t ws_bytes, wt_stream_t stream) {
    wt_status st = check_variant(desc, variant);
    if (st != WT_OK) return st;
    if (x == nullptr || y == nullptr || !aligned(x, 16) || !aligned(y, 16))
        return WT_ERR_INVALID_ARG;
    if (!w0 || !s0 || !aligned(w0, 4) || !aligned(s0, 4) || (b0 && !aligned(b0, 4)))
        return WT_ERR_INVALID_ARG;
    if (desc->levels > 0 && (!wl || !sl || !aligned(wl, 4) || !aligned(sl, 4)))
        return WT_ERR_INVALID_ARG;
    Arena measure{nullptr};
    plan_variant(*desc, variant, measure);
    if (ws == nullptr || ws_bytes < measure.off || !aligned(ws, 256)) return WT_ERR_WORKSPACE;
    Arena ar{static_cast<char*>(ws)};
    const Plan pl = plan_variant(*desc, variant, ar);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int launches = 0;
    const float* xf = static_cast<const float*>(x);
    float* yf = static_cast<float*>(y);
    switch (desc->k) {
        case 1: st = run_variant<1>(*desc, variant, xf, w0, b0, s0, wl, sl, yf, pl, s, &launches); break;
        case 3: st = run_variant<3>(*desc, variant, xf, w0, b0, s0, wl, sl, yf, pl, s, &launches); break;
        case 5: st = run_variant<5>(*desc, variant, xf, w0, b0, s0, wl, sl, yf, pl, s, &launches); break;
        case 7: st = run_variant<7>(*desc, variant, xf, w0, b0, s0, wl, sl, yf, pl, s, &launches); break;
        default: st = WT_ERR_UNSUPPORTED;
    }
    if (st == WT_OK) set_last_launch_count(launches);
    return st;
}
