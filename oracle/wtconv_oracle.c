/*
 * CPU oracle for the WTConv layer (wavelet convolution): TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may call this
 * file. The product path (the CUDA library) shares no code with it.
 *
 * Source: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware Reformulation"
 * (Aflalo, Finder, Amoyal, Treister, Freifeld), abbreviated "WTConv-IO" below.
 *
 * Everything is plain loops in double precision, one plane at a time, with every
 * intermediate tensor of the method materialized exactly as the paper's Algorithm 1
 * states it. No blocking, fusion or reordering beyond what the definitions state.
 *
 * Layouts (all row-major, contiguous):
 *   x, y, dy, dx   [n][c][h][w]
 *   w0             [c][k][k]      base depthwise kernel W^(0)
 *   b0             [c]            base bias b (NULL means zero)
 *   s0             [c]            base scale s^(0)
 *   wl             [L][c][4][k][k] level kernels W^(l), band order (LL, LH, HL, HH)
 *   sl             [L][c][4]      level scales s^(l)
 *
 * Readings of points the paper leaves open (each is listed in the design notes):
 *   - one k x k kernel and one scale per (channel, band) at every level: the level
 *     convolution runs over the 4C-channel coefficient tensor (WTConv-IO §3.1);
 *   - depthwise convolution is cross-correlation with zero padding R = (k-1)/2 so that
 *     the resolution is preserved (WTConv-IO §2.1), odd k only;
 *   - the bias sits inside the base scale: s0 * (X *dw W0 + b) (Algorithm 1, return line);
 *   - the level scale multiplies after the convolution (Algorithm 1, "filter, then scale");
 *   - a carrier with an odd number of rows (columns) is padded with one zero row (column)
 *     at the bottom (right) before its analysis, so level l has ceil(h_{l-1} / 2) rows,
 *     and each synthesis output is cropped back to the carrier's size (the pages are
 *     silent on odd sizes; this is the plainest completion of Eq. 5 / Eq. 12).
 *
 * Parity pins: none of these functions is trusted on its own; the pytest suite under
 * tests/ pins them against Prop. 1, Eq. 5, Eq. 13, library convolutions with autograd,
 * exact reconstruction, finite differences and a brute-force operator matrix.
 */
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int n, c, h, w, k, levels;
} wo_desc;

/* 0 = ok, 1 = invalid arguments, 2 = out of memory */
static int wo_check(const wo_desc* d) {
    if (!d) return 1;
    if (d->n < 0 || d->c <= 0 || d->h <= 0 || d->w <= 0) return 1;
    if (d->k < 1 || d->k > 31 || (d->k % 2) == 0) return 1;
    if (d->levels < 0 || d->levels > 30) return 1;
    return 0;
}

/* ---------------------------------------------------------------------------------
 * Building blocks
 * ------------------------------------------------------------------------------- */

/* Pixel (r, c) of an h x w plane, zero outside it (the padding of odd carriers). */
static double px(const double* in, int h, int w, int r, int c) {
    return (r < h && c < w) ? in[(size_t)r * w + c] : 0.0;
}

/*
 * One level of orthonormal 2-D Haar analysis (WTConv-IO §4.1, Eq. 5), applied to every
 * non-overlapping 2x2 block [a b; c d] of a plane of size h x w:
 *   LL = (a+b+c+d)/2, LH = (a+b-c-d)/2, HL = (a-b+c-d)/2, HH = (a-b-c+d)/2.
 * a is (2i, 2j), b is (2i, 2j+1), c is (2i+1, 2j), d is (2i+1, 2j+1); pixels past an odd
 * edge are zero. out is [4][ceil(h/2)][ceil(w/2)] in band order (LL, LH, HL, HH).
 */
void wo_haar_analysis(int h, int w, const double* in, double* out) {
    const int h2 = (h + 1) / 2, w2 = (w + 1) / 2;
    const size_t band = (size_t)h2 * w2;
    for (int i = 0; i < h2; ++i) {
        for (int j = 0; j < w2; ++j) {
            const double a = px(in, h, w, 2 * i, 2 * j);
            const double b = px(in, h, w, 2 * i, 2 * j + 1);
            const double c = px(in, h, w, 2 * i + 1, 2 * j);
            const double dd = px(in, h, w, 2 * i + 1, 2 * j + 1);
            const size_t o = (size_t)i * w2 + j;
            out[0 * band + o] = 0.5 * (a + b + c + dd);
            out[1 * band + o] = 0.5 * (a + b - c - dd);
            out[2 * band + o] = 0.5 * (a - b + c - dd);
            out[3 * band + o] = 0.5 * (a - b - c + dd);
        }
    }
}

/*
 * One level of Haar synthesis (WTConv-IO App. A, Eq. 12): the value at within-block
 * position (ry, rx) of block (i, j) is
 *   (LL + (-1)^ry LH + (-1)^rx HL + (-1)^(ry+rx) HH) / 2,
 * cropped to an ho x wo plane (ho in {2 h2 - 1, 2 h2}): in is [4][h2][w2], out [ho][wo].
 */
static void haar_synthesis_crop(int h2, int w2, int ho, int wo, const double* in,
                                double* out) {
    const size_t band = (size_t)h2 * w2;
    for (int i = 0; i < h2; ++i) {
        for (int j = 0; j < w2; ++j) {
            const size_t o = (size_t)i * w2 + j;
            const double ll = in[0 * band + o], lh = in[1 * band + o];
            const double hl = in[2 * band + o], hh = in[3 * band + o];
            for (int ry = 0; ry < 2; ++ry) {
                for (int rx = 0; rx < 2; ++rx) {
                    if (2 * i + ry >= ho || 2 * j + rx >= wo) continue;
                    const double sy = ry ? -1.0 : 1.0;
                    const double sx = rx ? -1.0 : 1.0;
                    out[(size_t)(2 * i + ry) * wo + 2 * j + rx] =
                        0.5 * (ll + sy * lh + sx * hl + sy * sx * hh);
                }
            }
        }
    }
}

/* Eq. 12 without cropping: in is [4][h2][w2]; out is [2*h2][2*w2]. */
void wo_haar_synthesis(int h2, int w2, const double* in, double* out) {
    haar_synthesis_crop(h2, w2, 2 * h2, 2 * w2, in, out);
}

/*
 * Depthwise k x k convolution of one plane, as deep-learning frameworks define it:
 * cross-correlation with zero padding R = (k-1)/2 (WTConv-IO §2.1 "zero-padded to
 * preserve resolution"):
 *   out[i][j] = sum_{u,v} wt[u][v] * in[i+u-R][j+v-R], in = 0 outside the plane.
 */
void wo_dwconv(int h, int w, int k, const double* in, const double* wt, double* out) {
    const int r = (k - 1) / 2;
    for (int i = 0; i < h; ++i) {
        for (int j = 0; j < w; ++j) {
            double acc = 0.0;
            for (int u = 0; u < k; ++u) {
                const int ii = i + u - r;
                if (ii < 0 || ii >= h) continue;
                for (int v = 0; v < k; ++v) {
                    const int jj = j + v - r;
                    if (jj < 0 || jj >= w) continue;
                    acc += wt[u * k + v] * in[(size_t)ii * w + jj];
                }
            }
            out[(size_t)i * w + j] = acc;
        }
    }
}

/* Adjoint of wo_dwconv with respect to its input: gin[p][q] += sum wt[u][v] g[p-u+R][q-v+R]. */
static void dwconv_adjoint_input(int h, int w, int k, const double* g, const double* wt,
                                 double* gin) {
    const int r = (k - 1) / 2;
    for (int i = 0; i < h; ++i) {
        for (int j = 0; j < w; ++j) {
            const double gij = g[(size_t)i * w + j];
            for (int u = 0; u < k; ++u) {
                const int ii = i + u - r;
                if (ii < 0 || ii >= h) continue;
                for (int v = 0; v < k; ++v) {
                    const int jj = j + v - r;
                    if (jj < 0 || jj >= w) continue;
                    gin[(size_t)ii * w + jj] += wt[u * k + v] * gij;
                }
            }
        }
    }
}

/* Adjoint of wo_dwconv with respect to its kernel: gwt[u][v] += sum_{i,j} g[i][j] in[i+u-R][j+v-R]. */
static void dwconv_adjoint_weight(int h, int w, int k, const double* g, const double* in,
                                  double* gwt) {
    const int r = (k - 1) / 2;
    for (int i = 0; i < h; ++i) {
        for (int j = 0; j < w; ++j) {
            const double gij = g[(size_t)i * w + j];
            for (int u = 0; u < k; ++u) {
                const int ii = i + u - r;
                if (ii < 0 || ii >= h) continue;
                for (int v = 0; v < k; ++v) {
                    const int jj = j + v - r;
                    if (jj < 0 || jj >= w) continue;
                    gwt[u * k + v] += gij * in[(size_t)ii * w + jj];
                }
            }
        }
    }
}

/* Adjoint of one cropped synthesis level (transpose of Eq. 12 and of the crop, entry by
 * entry): g is [ho][wo], gin [4][h2][w2]. */
static void synthesis_adjoint(int h2, int w2, int ho, int wo, const double* g, double* gin) {
    const size_t band = (size_t)h2 * w2;
    for (int i = 0; i < h2; ++i) {
        for (int j = 0; j < w2; ++j) {
            const size_t o = (size_t)i * w2 + j;
            double acc[4] = {0.0, 0.0, 0.0, 0.0};
            for (int ry = 0; ry < 2; ++ry) {
                for (int rx = 0; rx < 2; ++rx) {
                    if (2 * i + ry >= ho || 2 * j + rx >= wo) continue;
                    const double sy = ry ? -1.0 : 1.0;
                    const double sx = rx ? -1.0 : 1.0;
                    const double gv = g[(size_t)(2 * i + ry) * wo + 2 * j + rx];
                    acc[0] += 0.5 * gv;
                    acc[1] += 0.5 * sy * gv;
                    acc[2] += 0.5 * sx * gv;
                    acc[3] += 0.5 * sy * sx * gv;
                }
            }
            for (int b = 0; b < 4; ++b) gin[b * band + o] = acc[b];
        }
    }
}

/* Adjoint of one padded analysis level (transpose of Eq. 5 and of the zero padding,
 * entry by entry): g is [4][ceil(h/2)][ceil(w/2)], gin [h][w]; accumulates. */
static void analysis_adjoint(int h, int w, const double* g, double* gin) {
    const int h2 = (h + 1) / 2, w2 = (w + 1) / 2;
    const size_t band = (size_t)h2 * w2;
    for (int i = 0; i < h2; ++i) {
        for (int j = 0; j < w2; ++j) {
            const size_t o = (size_t)i * w2 + j;
            const double ll = g[0 * band + o], lh = g[1 * band + o];
            const double hl = g[2 * band + o], hh = g[3 * band + o];
            /* column of Eq. 5 for a, b, c, d respectively; padded pixels have no gradient */
            const double col[4] = {0.5 * (ll + lh + hl + hh), 0.5 * (ll + lh - hl - hh),
                                   0.5 * (ll - lh + hl - hh), 0.5 * (ll - lh - hl + hh)};
            for (int q = 0; q < 4; ++q) {
                const int r = 2 * i + (q >> 1), c = 2 * j + (q & 1);
                if (r < h && c < w) gin[(size_t)r * w + c] += col[q];
            }
        }
    }
}

/* ---------------------------------------------------------------------------------
 * Forward pass of one plane: Algorithm 1, every intermediate materialized.
 * ------------------------------------------------------------------------------- */

typedef struct {
    int L, k;
    int* hl;     /* hl[0] = h, hl[l] = ceil(hl[l-1] / 2), l = 1..L */
    int* wl;
    double** X;  /* X[l]: carrier at level l, [hl][wl], X[0] = input */
    double** Y;  /* Y[l]: analysis coefficients of X[l-1], [4][hl][wl], l = 1..L */
    double** Cv; /* Cv[l]: Y[l] *dw W^(l) before scaling, [4][hl][wl] */
    double** Z;  /* Z[l] = s^(l) * Cv[l] */
    double* base_conv; /* X *dw W^(0) + b, [h][w] */
} plane_tape;

static void tape_free(plane_tape* t) {
    if (!t->hl) return;
    for (int l = 0; l <= t->L; ++l) {
        if (l > 0) free(t->X[l]);
        free(t->Y[l]);
        free(t->Cv[l]);
        free(t->Z[l]);
    }
    free(t->X); free(t->Y); free(t->Cv); free(t->Z);
    free(t->base_conv);
    free(t->hl); free(t->wl);
    memset(t, 0, sizeof(*t));
}

static int tape_alloc(plane_tape* t, int h, int w, int k, int L) {
    memset(t, 0, sizeof(*t));
    t->L = L; t->k = k;
    t->hl = (int*)calloc((size_t)L + 1, sizeof(int));
    t->wl = (int*)calloc((size_t)L + 1, sizeof(int));
    t->X = (double**)calloc((size_t)L + 1, sizeof(double*));
    t->Y = (double**)calloc((size_t)L + 1, sizeof(double*));
    t->Cv = (double**)calloc((size_t)L + 1, sizeof(double*));
    t->Z = (double**)calloc((size_t)L + 1, sizeof(double*));
    t->base_conv = (double*)calloc((size_t)h * w, sizeof(double));
    if (!t->hl || !t->wl || !t->X || !t->Y || !t->Cv || !t->Z || !t->base_conv) return 2;
    for (int l = 0; l <= L; ++l) {
        t->hl[l] = (l == 0) ? h : (t->hl[l - 1] + 1) / 2;
        t->wl[l] = (l == 0) ? w : (t->wl[l - 1] + 1) / 2;
        if (l == 0) continue;
        const size_t sz = (size_t)t->hl[l] * t->wl[l];
        t->X[l] = (double*)calloc(sz, sizeof(double));
        t->Y[l] = (double*)calloc(4 * sz, sizeof(double));
        t->Cv[l] = (double*)calloc(4 * sz, sizeof(double));
        t->Z[l] = (double*)calloc(4 * sz, sizeof(double));
        if (!t->X[l] || !t->Y[l] || !t->Cv[l] || !t->Z[l]) return 2;
    }
    return 0;
}

/*
 * Downward loop of Algorithm 1 for one plane of channel ch:
 *   Y^(l) = A X^(l-1);  Z^(l) = s^(l) * (Y^(l) *dw W^(l));  X^(l) = [Y^(l)]_LL
 * and the base convolution X *dw W^(0) + b.
 */
static void plane_down(const wo_desc* d, int ch, const double* xin, const double* w0,
                       const double* b0, const double* wl, const double* sl, plane_tape* t) {
    const int k = d->k, L = d->levels, C = d->c, kk = k * k;
    t->X[0] = (double*)xin;
    for (int l = 1; l <= L; ++l) {
        const int hh = t->hl[l], ww = t->wl[l];
        const size_t band = (size_t)hh * ww;
        wo_haar_analysis(t->hl[l - 1], t->wl[l - 1], t->X[l - 1], t->Y[l]);
        for (int b = 0; b < 4; ++b) {
            const double* kern = wl + (((size_t)(l - 1) * C + ch) * 4 + b) * kk;
            const double s = sl[((size_t)(l - 1) * C + ch) * 4 + b];
            wo_dwconv(hh, ww, k, t->Y[l] + b * band, kern, t->Cv[l] + b * band);
            for (size_t e = 0; e < band; ++e) t->Z[l][b * band + e] = s * t->Cv[l][b * band + e];
        }
        memcpy(t->X[l], t->Y[l], band * sizeof(double)); /* raw, unfiltered LL */
    }
    wo_dwconv(d->h, d->w, k, xin, w0 + (size_t)ch * kk, t->base_conv);
    const double bias = b0 ? b0[ch] : 0.0;
    for (size_t e = 0; e < (size_t)d->h * d->w; ++e) t->base_conv[e] += bias;
}

/*
 * Upward loop of Algorithm 1 (cascade):
 *   R^(L+1) = 0;  R^(l) = A^T( ([Z^(l)]_LL + R^(l+1)) || [Z^(l)]_H ), cropped to X^(l-1)'s size;
 * then out = s0 * base_conv + R^(1).
 */
static int plane_up_cascade(const wo_desc* d, int ch, const double* s0, const plane_tape* t,
                            double* out) {
    const int L = d->levels;
    const size_t npix = (size_t)d->h * d->w;
    double* R = NULL; /* R^(l+1), at resolution hl[l] x wl[l] */
    for (int l = L; l >= 1; --l) {
        const int hh = t->hl[l], ww = t->wl[l];
        const size_t band = (size_t)hh * ww;
        double* U = (double*)malloc(4 * band * sizeof(double));
        double* Rn = (double*)malloc((size_t)t->hl[l - 1] * t->wl[l - 1] * sizeof(double));
        if (!U || !Rn) { free(U); free(Rn); free(R); return 2; }
        memcpy(U, t->Z[l], 4 * band * sizeof(double));
        if (R) for (size_t e = 0; e < band; ++e) U[e] += R[e];
        haar_synthesis_crop(hh, ww, t->hl[l - 1], t->wl[l - 1], U, Rn);
        free(U);
        free(R);
        R = Rn;
    }
    for (size_t e = 0; e < npix; ++e) out[e] = s0[ch] * t->base_conv[e] + (R ? R[e] : 0.0);
    free(R);
    return 0;
}

/*
 * Closed-form single-pass synthesis (WTConv-IO Prop. 2, Eq. 6-7):
 *   R[y][x] = sum_l 2^-l ( Z_LL + s_y Z_LH + s_x Z_HL + s_y s_x Z_HH )^(l)[y>>l][x>>l],
 *   s_y = (-1)^(floor(y / 2^(l-1)) mod 2), s_x likewise,
 * then out = s0 * base_conv + R.
 */
static void plane_up_closed(const wo_desc* d, int ch, const double* s0, const plane_tape* t,
                            double* out) {
    const int L = d->levels;
    for (int y = 0; y < d->h; ++y) {
        for (int x = 0; x < d->w; ++x) {
            double r = 0.0;
            for (int l = 1; l <= L; ++l) {
                const int ww = t->wl[l];
                const size_t band = (size_t)t->hl[l] * ww;
                const size_t o = (size_t)(y >> l) * ww + (x >> l);
                const double sy = ((y >> (l - 1)) & 1) ? -1.0 : 1.0;
                const double sx = ((x >> (l - 1)) & 1) ? -1.0 : 1.0;
                double scale = 1.0;
                for (int q = 0; q < l; ++q) scale *= 0.5;
                r += scale * (t->Z[l][o] + sy * t->Z[l][band + o] + sx * t->Z[l][2 * band + o] +
                              sy * sx * t->Z[l][3 * band + o]);
            }
            const size_t e = (size_t)y * d->w + x;
            out[e] = s0[ch] * t->base_conv[e] + r;
        }
    }
}

/*
 * WTConv forward. mode 0: Algorithm 1 with the level-by-level cascade (reference form).
 * mode 1: the same Z^(l) summed with the closed form of Eq. 7.
 * Returns 0 on success, 1 on invalid arguments, 2 when out of memory.
 */
int wo_forward(const wo_desc* d, const double* x, const double* w0, const double* b0,
               const double* s0, const double* wl, const double* sl, double* y, int mode) {
    if (wo_check(d) || !x || !w0 || !s0 || !y || (d->levels > 0 && (!wl || !sl))) return 1;
    const size_t npix = (size_t)d->h * d->w;
    const long planes = (long)d->n * d->c;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (long p = 0; p < planes; ++p) {
        const int ch = (int)(p % d->c);
        plane_tape t;
        if (tape_alloc(&t, d->h, d->w, d->k, d->levels)) { tape_free(&t); err |= 2; continue; }
        plane_down(d, ch, x + (size_t)p * npix, w0, b0, wl, sl, &t);
        if (mode == 1) {
            plane_up_closed(d, ch, s0, &t, y + (size_t)p * npix);
        } else {
            err |= plane_up_cascade(d, ch, s0, &t, y + (size_t)p * npix);
        }
        tape_free(&t);
    }
    return err;
}

/*
 * WTConv backward: the literal reverse-mode derivative of Algorithm 1, stage by stage.
 * Haar steps use the transpose of their own matrices (WTConv-IO §2.2 Eq. 1 states that
 * this is analysis for synthesis and synthesis for analysis), convolutions use their
 * input and weight adjoints, and the scales and bias use the product rule. Gradients
 * are taken directly with respect to the unfolded parameters (W, b, s); nothing here
 * uses the scale folding of §4.3.
 *
 * Outputs (all written, not accumulated): dx [n][c][h][w], dw0 [c][k][k], db0 [c],
 * ds0 [c], dwl [L][c][4][k][k], dsl [L][c][4]. db0 may be NULL.
 */
int wo_backward(const wo_desc* d, const double* x, const double* dy, const double* w0,
                const double* b0, const double* s0, const double* wl, const double* sl,
                double* dx, double* dw0, double* db0, double* ds0, double* dwl, double* dsl) {
    if (wo_check(d) || !x || !dy || !w0 || !s0 || !dx || !dw0 || !ds0 ||
        (d->levels > 0 && (!wl || !sl || !dwl || !dsl)))
        return 1;
    const int k = d->k, kk = k * k, L = d->levels, C = d->c;
    const size_t npix = (size_t)d->h * d->w;
    int err = 0;
    /* one channel per iteration: its parameter gradients sum over the batch in a fixed order */
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int ch = 0; ch < C; ++ch) {
        double gw0[1024], gb = 0.0, gs0 = 0.0; /* k <= 31 */
        double* gwl = (double*)calloc((size_t)(L > 0 ? L : 1) * 4 * kk, sizeof(double));
        double* gsl = (double*)calloc((size_t)(L > 0 ? L : 1) * 4, sizeof(double));
        memset(gw0, 0, sizeof(gw0));
        if (!gwl || !gsl) { free(gwl); free(gsl); err |= 2; continue; }
        for (int nn = 0; nn < d->n; ++nn) {
            const size_t p = (size_t)nn * C + ch;
            const double* xin = x + p * npix;
            const double* g = dy + p * npix;
            double* gx = dx + p * npix;
            plane_tape t;
            if (tape_alloc(&t, d->h, d->w, k, L)) { tape_free(&t); err |= 2; break; }
            plane_down(d, ch, xin, w0, b0, wl, sl, &t);

            /* out = s0 * base_conv + R^(1) */
            double* gbase = (double*)malloc(npix * sizeof(double));
            if (!gbase) { tape_free(&t); err |= 2; break; }
            for (size_t e = 0; e < npix; ++e) {
                gs0 += g[e] * t.base_conv[e];
                gbase[e] = s0[ch] * g[e];
                gb += gbase[e];
            }
            dwconv_adjoint_weight(d->h, d->w, k, gbase, xin, gw0);
            memset(gx, 0, npix * sizeof(double));
            dwconv_adjoint_input(d->h, d->w, k, gbase, w0 + (size_t)ch * kk, gx);
            free(gbase);

            /* reverse of the upward loop: gradients of Z^(l) for l = 1..L */
            double** gZ = (double**)calloc((size_t)L + 1, sizeof(double*));
            const double* gR = g; /* gradient of R^(1) */
            double* gR_owned = NULL;
            for (int l = 1; l <= L; ++l) {
                const size_t band = (size_t)t.hl[l] * t.wl[l];
                gZ[l] = (double*)malloc(4 * band * sizeof(double));
                /* grad of the concatenation */
                synthesis_adjoint(t.hl[l], t.wl[l], t.hl[l - 1], t.wl[l - 1], gR, gZ[l]);
                double* next = (double*)malloc(band * sizeof(double));
                memcpy(next, gZ[l], band * sizeof(double)); /* R^(l+1) was added to LL */
                free(gR_owned);
                gR_owned = next;
                gR = next;
            }
            free(gR_owned);

            /* reverse of the downward loop, l = L..1 */
            double* gXl = NULL; /* gradient of carrier X^(l) */
            for (int l = L; l >= 1; --l) {
                const int hh = t.hl[l], ww = t.wl[l];
                const size_t band = (size_t)hh * ww;
                double* gY = (double*)calloc(4 * band, sizeof(double));
                for (int b = 0; b < 4; ++b) {
                    const size_t pi = ((size_t)(l - 1) * C + ch) * 4 + b;
                    const double s = sl[pi];
                    double* gC = (double*)malloc(band * sizeof(double));
                    for (size_t e = 0; e < band; ++e) {
                        gsl[(size_t)(l - 1) * 4 + b] += gZ[l][b * band + e] * t.Cv[l][b * band + e];
                        gC[e] = s * gZ[l][b * band + e];
                    }
                    dwconv_adjoint_weight(hh, ww, k, gC, t.Y[l] + b * band,
                                          gwl + ((size_t)(l - 1) * 4 + b) * kk);
                    dwconv_adjoint_input(hh, ww, k, gC, wl + pi * kk, gY + b * band);
                    free(gC);
                }
                if (gXl) { /* X^(l) = [Y^(l)]_LL */
                    for (size_t e = 0; e < band; ++e) gY[e] += gXl[e];
                    free(gXl);
                }
                double* gprev;
                if (l > 1) {
                    gprev = (double*)calloc((size_t)t.hl[l - 1] * t.wl[l - 1], sizeof(double));
                } else {
                    gprev = gx; /* accumulate into dx on top of the base-path gradient */
                }
                analysis_adjoint(t.hl[l - 1], t.wl[l - 1], gY, gprev);
                free(gY);
                gXl = (l > 1) ? gprev : NULL;
            }
            for (int l = 1; l <= L; ++l) free(gZ[l]);
            free(gZ);
            tape_free(&t);
        }
        for (int e = 0; e < kk; ++e) dw0[(size_t)ch * kk + e] = gw0[e];
        if (db0) db0[ch] = gb;
        ds0[ch] = gs0;
        for (int l = 1; l <= L; ++l) {
            for (int b = 0; b < 4; ++b) {
                const size_t pi = ((size_t)(l - 1) * C + ch) * 4 + b;
                memcpy(dwl + pi * kk, gwl + ((size_t)(l - 1) * 4 + b) * kk, kk * sizeof(double));
                dsl[pi] = gsl[(size_t)(l - 1) * 4 + b];
            }
        }
        free(gwl);
        free(gsl);
    }
    return err;
}

int wo_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the following calls (n >= 1); only the timed CPU baseline changes it. */
void wo_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
