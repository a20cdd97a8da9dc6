// Tile geometry and streaming register-blocked k x k stencils shared by the forward /
// backward-data kernel and the backward-weight kernel (sm_103a).
//
// A full-resolution tile is 64x64 pixels staged with a 2R-pixel halo (R = (k-1)/2), so
// that its 32x32 level-1 Haar coefficients (§4.1 Eq. 5 of "Fast and Memory-Efficient
// Wavelet Convolutions via I/O-Aware Reformulation") can be formed with an R-coefficient
// halo. Every k x k filter (or its weight-gradient correlation) streams one window row at
// a time through registers with the k*k taps in registers and independent accumulators
// innermost. Shared-memory rows are read as 16-byte vectors at consecutive addresses
// across the lanes of a warp (no bank conflicts).
#pragma once

#include "wt_common.cuh"

namespace wt {

constexpr int kTile = 64;       // full-resolution tile side, pixels
constexpr int kCT = kTile / 2;  // coefficient tile side; also the deep-level output tile

template <int K>
struct FG {
    static constexpr int R = (K - 1) / 2;
    static constexpr int KK = K * K;
    static constexpr int BT = kCT + 2 * R;  // coefficient tile side with halo
};

// ---------------------------------------------------------------------------------
// Band-pair tiles for packed (f32x2) filtering: the four subbands are stored as two
// tiles of interleaved pairs, (LL, LH) and (HL, HH), so that one packed FMA applies the
// two bands' own taps to their own coefficients. A row holds BT cells (2 floats each);
// 16-byte chunks of 2 cells are laid out even chunks first, then odd chunks, so that the
// lanes of a warp, which own 4-cell-wide blocks, read consecutive 16-byte words.
// ---------------------------------------------------------------------------------
template <int K>
struct PG {
    static constexpr int R = FG<K>::R, BT = FG<K>::BT, KK = FG<K>::KK;
    static constexpr int NCR = BT / 2;                 // chunks per row
    static constexpr int PHALF = (NCR + 1) / 2;        // start of the odd chunks
    static constexpr int PROW = 8 * PHALF;             // floats per row
    static constexpr int PTILE = BT * PROW;            // floats per pair tile
    static constexpr int NCH = 2 + R;                  // chunks per window row (2x4 block)
    static constexpr int WS = (2 * KK + 3) & ~3;       // floats per weight-pair slot
    static constexpr int ZROW = 2 * kCT;               // floats per row of a filtered pair tile
    static constexpr int ZTILE = kCT * ZROW;
};

__device__ __forceinline__ int pchunk(int c, int half) { return (c >> 1) + (c & 1) * half; }

// Filtered pair tiles (ZROW floats = 16 16-byte units a row): chunk c (two coefficients of a
// band pair) is stored at unit c ^ (c / 8), a permutation. Writers store chunks 2j and
// 2j + 1 (j = 0..7 in a quarter-warp), readers chunk j or j + 8: each of these sets of 8
// lands on 8 distinct bank groups, so neither side has bank conflicts.
__device__ __forceinline__ int zunit(int c) { return c ^ ((c >> 3) & 1); }

// Packed k x k filter of a 2x4 block of one band pair: acc[o][q] = sum_{u,v} w[u][v] (.)
// cell[o+u][q+v], two bands at once. `rows` = pair tile + (first window row) * PROW;
// the block's window starts at cell 4*bj. wsl = KK taps as (w_b0, w_b1) pairs.
template <int K>
__device__ __forceinline__ void conv_pair_2x4(const float* rows, int bj, const float* wsl,
                                              f2x (&acc)[2][4]) {
    constexpr int R = PG<K>::R, KK = PG<K>::KK, NCH = PG<K>::NCH, PROW = PG<K>::PROW;
    constexpr int PHALF = PG<K>::PHALF;
    f2x w[KK];
#pragma unroll
    for (int q = 0; q + 1 < KK; q += 2) {
        const float4 t = *reinterpret_cast<const float4*>(wsl + 2 * q);
        w[q] = pk2(t.x, t.y);
        w[q + 1] = pk2(t.z, t.w);
    }
    if constexpr (KK & 1) {
        const float2 t = *reinterpret_cast<const float2*>(wsl + 2 * (KK - 1));
        w[KK - 1] = pk2(t.x, t.y);
    }
#pragma unroll
    for (int o = 0; o < 2; ++o)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[o][q] = 0ull;
#pragma unroll
    for (int r = 0; r < 2 + 2 * R; ++r) {
        const float* rp = rows + r * PROW;
        f2x v[2 * NCH];
#pragma unroll
        for (int m = 0; m < NCH; ++m) {
            const float4 t = *reinterpret_cast<const float4*>(
                rp + 4 * (bj + (m >> 1) + (m & 1) * PHALF));
            v[2 * m] = pk2(t.x, t.y);
            v[2 * m + 1] = pk2(t.z, t.w);
        }
        // taps outermost: consecutive packed FMAs update different accumulators
#pragma unroll
        for (int vv = 0; vv < K; ++vv)
#pragma unroll
            for (int o = 0; o < 2; ++o) {
                const int u = r - o;
                if (u < 0 || u >= K) continue;
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[o][q] = fma2(w[u * K + vv], v[q + vv], acc[o][q]);
            }
    }
}

// Packed weight-gradient correlation of a ROWS x 4 block of one band pair:
// acc[u*K+v] += sum_{o,q} g[o][q] (.) cell[o+u][q+v], two bands at once. `rows` = pair
// tile + (first window row) * PROW; the window starts at cell 4*bj.
template <int K, int ROWS>
__device__ __forceinline__ void corr_pair(const float* rows, int bj, const f2x (&g)[ROWS][4],
                                          f2x (&acc)[K * K]) {
    constexpr int R = PG<K>::R, NCH = PG<K>::NCH, PROW = PG<K>::PROW, PHALF = PG<K>::PHALF;
#pragma unroll
    for (int r = 0; r < ROWS + 2 * R; ++r) {
        const float* rp = rows + r * PROW;
        f2x v[2 * NCH];
#pragma unroll
        for (int m = 0; m < NCH; ++m) {
            const float4 t = *reinterpret_cast<const float4*>(
                rp + 4 * (bj + (m >> 1) + (m & 1) * PHALF));
            v[2 * m] = pk2(t.x, t.y);
            v[2 * m + 1] = pk2(t.z, t.w);
        }
#pragma unroll
        for (int o = 0; o < ROWS; ++o) {
            const int u = r - o;
            if (u < 0 || u >= K) continue;
#pragma unroll
            for (int vv = 0; vv < K; ++vv)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    acc[u * K + vv] = fma2(g[o][q], v[q + vv], acc[u * K + vv]);
        }
    }
}

// TMA box of a staged tile with a 2R halo: columns from x0 - XOFF (16-byte aligned
// start), XBW wide; rows from y0 - 2R, XBH high.
template <int K, typename T>
struct XBox {
    static constexpr int R = FG<K>::R;
    static constexpr int A = 16 / (int)sizeof(T);             // elements per 16 bytes
    static constexpr int XOFF = ((2 * R + A - 1) / A) * A;
    static constexpr int XBW = ((kTile + 2 * R + XOFF + A - 1) / A) * A;
    static constexpr int XBH = kTile + 4 * R;
    static constexpr int C0 = XOFF - 2 * R;                   // raw column of tile column 0
    static constexpr int BYTES = XBW * XBH * (int)sizeof(T);
};

template <typename T>
__device__ __forceinline__ float2 ld2_smem(const T* p);
template <>
__device__ __forceinline__ float2 ld2_smem<float>(const float* p) {
    return *reinterpret_cast<const float2*>(p);
}
template <>
__device__ __forceinline__ float2 ld2_smem<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// Four consecutive elements from shared memory, widened (8-byte aligned for bfloat16,
// 16-byte aligned for fp32).
template <typename T>
__device__ __forceinline__ float4 ld4_smem(const T* p);
template <>
__device__ __forceinline__ float4 ld4_smem<float>(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 ld4_smem<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

template <>
__device__ __forceinline__ float2 ld2_smem<__half>(const __half* p) {
    return __half22float2(*reinterpret_cast<const __half2*>(p));
}
template <>
__device__ __forceinline__ float4 ld4_smem<__half>(const __half* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// The 4x4 pixel block of a plane at (r0, c0), zero outside H x W (the padding of a plane
// whose sides are not multiples of 2^L); vector loads when the block lies inside the plane
// and rows start on 4-element boundaries (vec: W % 4 == 0).
template <typename T>
__device__ __forceinline__ void load_block4x4(const T* xp, int H, int W, int vec, int r0, int c0,
                                              float4 (&r)[4]) {
    if (vec && r0 + 3 < H && c0 + 3 < W) {
#pragma unroll
        for (int q = 0; q < 4; ++q) r[q] = IO<T>::ld4(xp + (size_t)(r0 + q) * W + c0);
    } else {  // edge of the plane or unaligned rows: element loads
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float e[4];
#pragma unroll
            for (int m = 0; m < 4; ++m)
                e[m] = (r0 + q < H && c0 + m < W) ? IO<T>::ld(xp + (size_t)(r0 + q) * W + c0 + m)
                                                  : 0.f;
            r[q] = make_float4(e[0], e[1], e[2], e[3]);
        }
    }
}

// The level-1 band-pair tiles alone from the raw tile (the base filter reads the raw tile
// itself): one item = two horizontally adjacent cells (a 2x4 pixel block).
template <int K, typename T>
__device__ __forceinline__ void convert_bands(const T* raw, float* bs) {
    constexpr int BT = FG<K>::BT;
    constexpr int NCR = PG<K>::NCR, PROW = PG<K>::PROW, PTILE = PG<K>::PTILE;
    constexpr int PHALF = PG<K>::PHALF;
    constexpr int RW = XBox<K, T>::XBW, C0 = XBox<K, T>::C0;
    // items in storage order (unit u of a pair-tile row holds chunk m, pchunk(m) = u), so
    // that a quarter-warp's 16-byte stores are contiguous (no bank conflicts)
    for (int idx = threadIdx.x; idx < BT * NCR; idx += blockDim.x) {
        const int ci = idx / NCR, u = idx - ci * NCR;
        const int m = (u < PHALF) ? 2 * u : 2 * (u - PHALF) + 1;
        const T* r0 = raw + (2 * ci) * RW + C0 + 4 * m;
        float2 a0, a1, b0, b1;
        if constexpr (C0 % 4 == 0) {  // 4-element aligned: one vector load per row
            const float4 ra = ld4_smem<T>(r0), rb = ld4_smem<T>(r0 + RW);
            a0 = make_float2(ra.x, ra.y); a1 = make_float2(ra.z, ra.w);
            b0 = make_float2(rb.x, rb.y); b1 = make_float2(rb.z, rb.w);
        } else {
            a0 = ld2_smem<T>(r0); a1 = ld2_smem<T>(r0 + 2);
            b0 = ld2_smem<T>(r0 + RW); b1 = ld2_smem<T>(r0 + RW + 2);
        }
        const float4 h0 = haar_u(a0.x, a0.y, b0.x, b0.y);
        const float4 h1 = haar_u(a1.x, a1.y, b1.x, b1.y);
        float* q = bs + ci * PROW + 4 * u;
        *reinterpret_cast<float4*>(q) = make_float4(h0.x, h0.y, h1.x, h1.y);
        *reinterpret_cast<float4*>(q + PTILE) = make_float4(h0.z, h0.w, h1.z, h1.w);
    }
}

// Non-TMA staging of a raw tile: element (rr, cc) of the XBox layout is pixel
// (y0 - 2R + rr, x0 - XOFF + cc) of the plane, zero outside it (element loads: any row
// alignment).
template <int K, typename T>
__device__ __forceinline__ void stage_raw(const T* xp, int H, int W, T* raw, int y0, int x0) {
    constexpr int R = FG<K>::R, RW = XBox<K, T>::XBW, RH = XBox<K, T>::XBH;
    constexpr int XOFF = XBox<K, T>::XOFF;
    for (int idx = threadIdx.x; idx < RH * RW; idx += blockDim.x) {
        const int rr = idx / RW, cc = idx - rr * RW;
        const int gy = y0 - 2 * R + rr, gx = x0 - XOFF + cc;
        raw[idx] = (gy >= 0 && gy < H && gx >= 0 && gx < W) ? xp[(size_t)gy * W + gx]
                                                             : static_cast<T>(0.f);
    }
}

// N consecutive raw elements v[i] = p[S + i], widened to float, read as 4-element vectors
// from the 4-element-aligned offset S & ~3: 8-byte loads for 16-bit types, 16-byte loads for
// fp32 (p must be that aligned). A half-warp's 16 pixel blocks then read one contiguous
// 128 / 256 bytes per load, with no bank conflicts between the two half-warps' rows.
template <typename T, int N, int S>
__device__ __forceinline__ void load_raw_vec(const T* p, float (&v)[N]) {
    constexpr int A0 = S & ~3;
    constexpr int NL = (S - A0 + N + 3) / 4;
    float e[4 * NL];
#pragma unroll
    for (int j = 0; j < NL; ++j) {
        const float4 t = ld4_smem<T>(p + A0 + 4 * j);
        e[4 * j] = t.x;
        e[4 * j + 1] = t.y;
        e[4 * j + 2] = t.z;
        e[4 * j + 3] = t.w;
    }
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = e[S - A0 + i];
}

// Base k x k filter of the 4x4 pixel block (by, bx) of a tile, read from the raw tile
// (widened in registers), accumulating onto acc[o][p] = (pixel (o, 2p), pixel (o, 2p+1)).
// Window row r is raw row 4by + R + r; window column j is raw column 4bx + XOFF - R + j.
// wdup = KK taps as (w, w) pairs. Scalar FMAs for k >= 5 (the packed form would pair the
// window at odd offsets with moves: measured 14% slower at k = 5, 11% at k = 7), packed
// for k <= 3 (4% faster there).
template <int K, typename T>
__device__ __forceinline__ void conv_base_4x4_raw(const T* raw, int by, int bx,
                                                  const float* wdup, f2x (&acc)[4][2]) {
    constexpr int R = FG<K>::R, KK = FG<K>::KK;
    constexpr int RW = XBox<K, T>::XBW, S = XBox<K, T>::XOFF - R;
    constexpr int NV = 4 + 2 * R;
    const T* base = raw + (4 * by + R) * RW + 4 * bx;
    if constexpr (K >= 5) {
        float w[KK];
#pragma unroll
        for (int q = 0; q + 1 < KK; q += 2) {
            const float4 t = *reinterpret_cast<const float4*>(wdup + 2 * q);
            w[q] = t.x;
            w[q + 1] = t.z;
        }
        if constexpr (KK & 1) w[KK - 1] = wdup[2 * (KK - 1)];
        float a[4][4];
#pragma unroll
        for (int o = 0; o < 4; ++o) {
            const float2 lo = upk2(acc[o][0]), hi = upk2(acc[o][1]);
            a[o][0] = lo.x; a[o][1] = lo.y; a[o][2] = hi.x; a[o][3] = hi.y;
        }
#pragma unroll
        for (int r = 0; r < 4 + 2 * R; ++r) {
            float v[NV];
            load_raw_vec<T, NV, S>(base + r * RW, v);
            // taps outermost: consecutive FMAs update different accumulators
#pragma unroll
            for (int vv = 0; vv < K; ++vv)
#pragma unroll
                for (int o = 0; o < 4; ++o) {
                    const int u = r - o;
                    if (u < 0 || u >= K) continue;
#pragma unroll
                    for (int q = 0; q < 4; ++q) a[o][q] = fmaf(w[u * K + vv], v[q + vv], a[o][q]);
                }
        }
#pragma unroll
        for (int o = 0; o < 4; ++o) {
            acc[o][0] = pk2(a[o][0], a[o][1]);
            acc[o][1] = pk2(a[o][2], a[o][3]);
        }
    } else {
        f2x w[KK];
#pragma unroll
        for (int q = 0; q + 1 < KK; q += 2) {
            const float4 t = *reinterpret_cast<const float4*>(wdup + 2 * q);
            w[q] = pk2(t.x, t.y);
            w[q + 1] = pk2(t.z, t.w);
        }
        if constexpr (KK & 1) {
            const float2 t = *reinterpret_cast<const float2*>(wdup + 2 * (KK - 1));
            w[KK - 1] = pk2(t.x, t.y);
        }
#pragma unroll
        for (int r = 0; r < 4 + 2 * R; ++r) {
            float v[NV];
            load_raw_vec<T, NV, S>(base + r * RW, v);
            f2x A[NV / 2], B[NV / 2 - 1];
#pragma unroll
            for (int m = 0; m < NV / 2; ++m) A[m] = pk2(v[2 * m], v[2 * m + 1]);
#pragma unroll
            for (int m = 0; m < NV / 2 - 1; ++m) B[m] = pk2(v[2 * m + 1], v[2 * m + 2]);
#pragma unroll
            for (int vv = 0; vv < K; ++vv)
#pragma unroll
                for (int o = 0; o < 4; ++o) {
                    const int u = r - o;
                    if (u < 0 || u >= K) continue;
#pragma unroll
                    for (int pp = 0; pp < 2; ++pp) {
                        const int idx = 2 * pp + vv;
                        const f2x in = (idx & 1) ? B[(idx - 1) >> 1] : A[idx >> 1];
                        acc[o][pp] = fma2(w[u * K + vv], in, acc[o][pp]);
                    }
                }
        }
    }
}

// Base weight-gradient correlation of the 4x4 pixel block (by, bx), read from the raw tiles
// and widened in registers: X in the layout above (window row r is raw row 4by + R + r,
// window column j raw column 4bx + XOFF - R + j) and the 64x64 dY tile. acc[u*K+v]
// accumulates sum_{o,q} dY[o][q] X[o+u][q+v] over its two lanes (add them at the end):
// with 16-bit I/O and k = 5 all of it in the low lane by scalar FMAs (the packed form pairs
// the window at odd offsets with moves: measured 9% slower in isolation, 2.7% on the whole
// 16x256x256x256 backward-weight), else the even and odd columns packed,
// g[o][p] = (dY[o][2p], dY[o][2p+1]) (at k = 7, whose kernel runs one CTA per SM with
// twice the accumulators, the scalar form measured 6% slower; fp32 and k = 3 gain nothing).
template <int K, typename T>
__device__ __forceinline__ void corr_base_4x4_raw(const T* rawx, const T* rawg, int by, int bx,
                                                  f2x (&acc)[K * K]) {
    constexpr int R = FG<K>::R;
    constexpr int RW = XBox<K, T>::XBW, S = XBox<K, T>::XOFF - R;
    constexpr int NV = 4 + 2 * R;
    const T* base = rawx + (4 * by + R) * RW + 4 * bx;
    if constexpr (K == 5 && sizeof(T) == 2) {
        float g[4][4];
#pragma unroll
        for (int o = 0; o < 4; ++o) {
            const float4 t = ld4_smem<T>(rawg + (4 * by + o) * kTile + 4 * bx);
            g[o][0] = t.x; g[o][1] = t.y; g[o][2] = t.z; g[o][3] = t.w;
        }
#pragma unroll
        for (int r = 0; r < 4 + 2 * R; ++r) {
            float v[NV];
            load_raw_vec<T, NV, S>(base + r * RW, v);
#pragma unroll
            for (int o = 0; o < 4; ++o) {
                const int u = r - o;
                if (u < 0 || u >= K) continue;
#pragma unroll
                for (int vv = 0; vv < K; ++vv)
#pragma unroll
                    for (int q = 0; q < 4; ++q) fma_lo(acc[u * K + vv], g[o][q], v[q + vv]);
            }
        }
    } else {
        f2x g[4][2];
#pragma unroll
        for (int o = 0; o < 4; ++o) {
            const float4 t = ld4_smem<T>(rawg + (4 * by + o) * kTile + 4 * bx);
            g[o][0] = pk2(t.x, t.y);
            g[o][1] = pk2(t.z, t.w);
        }
#pragma unroll
        for (int r = 0; r < 4 + 2 * R; ++r) {
            float v[NV];
            load_raw_vec<T, NV, S>(base + r * RW, v);
            f2x A[NV / 2], B[NV / 2 - 1];
#pragma unroll
            for (int m = 0; m < NV / 2; ++m) A[m] = pk2(v[2 * m], v[2 * m + 1]);
#pragma unroll
            for (int m = 0; m < NV / 2 - 1; ++m) B[m] = pk2(v[2 * m + 1], v[2 * m + 2]);
#pragma unroll
            for (int o = 0; o < 4; ++o) {
                const int u = r - o;
                if (u < 0 || u >= K) continue;
#pragma unroll
                for (int vv = 0; vv < K; ++vv)
#pragma unroll
                    for (int pp = 0; pp < 2; ++pp) {
                        const int idx = 2 * pp + vv;
                        const f2x in = (idx & 1) ? B[(idx - 1) >> 1] : A[idx >> 1];
                        acc[u * K + vv] = fma2(g[o][pp], in, acc[u * K + vv]);
                    }
            }
        }
    }
}

// Non-TMA staging of a 64x64 raw tile without halo: element (rr, cc) is pixel
// (y0 + rr, x0 + cc) of the plane, zero outside it.
template <typename T>
__device__ __forceinline__ void stage_raw_tile(const T* p, int H, int W, T* raw, int y0, int x0) {
    for (int idx = threadIdx.x; idx < kTile * kTile; idx += blockDim.x) {
        const int rr = idx / kTile, cc = idx - rr * kTile;
        const int gy = y0 + rr, gx = x0 + cc;
        raw[idx] = (gy < H && gx < W) ? p[(size_t)gy * W + gx] : static_cast<T>(0.f);
    }
}

// Number of bw x bh boxes that tile an H x W plane.
__device__ __forceinline__ int sweep_boxes(int H, int W, int bw, int bh) {
    return ((W + bw - 1) / bw) * ((H + bh - 1) / bh);
}

// Level-2 subbands (unnormalized) and carrier of the 4x4 pixel block r0..r3 (Eq. 5 applied
// to the pixels gives X^(1) = LL; applied again to the 2x2 block of X^(1) it gives level 2).
__device__ __forceinline__ float4 level2_block(const float4& r0, const float4& r1,
                                               const float4& r2, const float4& r3) {
    const float ca = 0.5f * (r0.x + r0.y + r1.x + r1.y);
    const float cb = 0.5f * (r0.z + r0.w + r1.z + r1.w);
    const float cc = 0.5f * (r2.x + r2.y + r3.x + r3.y);
    const float cd = 0.5f * (r2.z + r2.w + r3.z + r3.w);
    return haar_u(ca, cb, cc, cd);
}

}  // namespace wt
