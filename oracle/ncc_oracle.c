/*
 * ncc_oracle.c -- plain, slow, obviously correct CPU oracle for normalized
 * cross-correlation (NCC) template matching of 8-bit images.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline and reference legs may load this code.  It shares nothing with
 * the CUDA library (no headers, helpers, tables or constants) and never
 * calls into it.
 *
 * What it follows (The CUDA Handbook, chapter 15, "Image Processing:
 * Normalized Correlation"):
 *   - "Image in shared memory", Listing 15-5: for every shift the kernel
 *     forms three integer sums over the wT x hT window whose top-left pixel
 *     is the shift -- the pixel sum, the sum of squared pixels and the sum of
 *     pixel*template products -- and turns them, with the template's own
 *     sum and the pixel count, into one correlation coefficient.
 *   - Section 15.8, "The Denominator: Summed Area Tables": S(x,y) accumulates
 *     every pixel above and to the left of (x,y); a second table Q does the
 *     same for I^2; both are 64-bit; a rectangle's sum is the four-corner
 *     difference of the box-sum equation, with corners in row -1 or column -1
 *     read as zero (Figure 15-7).
 *
 * Readings where the pages are silent:
 *   - The tables are inclusive: S[y][x] = sum over j<=y, i<=x of I[j][i].
 *   - The coefficient routine's body is not printed.  The coefficient is the
 *     Pearson correlation of window and template, in exact-integer form:
 *       num = N*SumIT - SumI*SumT,  vI = N*SumI2 - SumI^2,
 *       vT  = N*SumT2 - SumT^2,     r  = num / sqrt(vI*vT),
 *     r = 0 when vI == 0 or vT == 0, and r is clamped to [-1, 1]; N = wT*hT.
 *     num, vI, vT are exact in int64; r is evaluated in double.
 *   - Outputs cover the valid shifts only: Ox = W-wT+1 columns by
 *     Oy = H-hT+1 rows; out[t][y][x] is the window with top-left pixel (x,y).
 *
 * Each function is the definition written out: no blocking, no fusion and
 * no reordering.  Parity is pinned by the not-gpu tests (brute-force sums,
 * closed forms, library routines); see the test module for the list.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)

static size_t at(int W, int x, int y) { return (size_t)y * (size_t)W + (size_t)x; }

/* ---------------------------------------------------------------------- */
/* Summed-area tables.                                                    */
/* ---------------------------------------------------------------------- */

/* S[y][x] = S[y-1][x] + (I[y][0] + ... + I[y][x]); the same for Q with I^2.
 * One pass in row order, every quantity in int64. */
int ncc_oracle_sat(const uint8_t *img, int W, int H, int64_t *S, int64_t *Q)
{
    if (!img || !S || !Q || W <= 0 || H <= 0) return ORACLE_BAD_ARG;
    for (int y = 0; y < H; y++) {
        int64_t run_i = 0;  /* I[y][0..x]   */
        int64_t run_q = 0;  /* I[y][0..x]^2 */
        for (int x = 0; x < W; x++) {
            int64_t p = (int64_t)img[at(W, x, y)];
            run_i += p;
            run_q += p * p;
            int64_t above_i = (y > 0) ? S[at(W, x, y - 1)] : 0;
            int64_t above_q = (y > 0) ? Q[at(W, x, y - 1)] : 0;
            S[at(W, x, y)] = above_i + run_i;
            Q[at(W, x, y)] = above_q + run_q;
        }
    }
    return ORACLE_OK;
}

/* Table value at (x,y), with row -1 and column -1 reading as zero. */
static int64_t table_at(const int64_t *S, int W, int x, int y)
{
    if (x < 0 || y < 0) return 0;
    return S[at(W, x, y)];
}

/* Sum over the half-open box [x0,x1) x [y0,y1) by the four-corner equation:
 * S(x1-1,y1-1) - S(x0-1,y1-1) - S(x1-1,y0-1) + S(x0-1,y0-1). */
int64_t ncc_oracle_sat_box(const int64_t *S, int W, int x0, int y0, int x1, int y1)
{
    return table_at(S, W, x1 - 1, y1 - 1) - table_at(S, W, x0 - 1, y1 - 1)
         - table_at(S, W, x1 - 1, y0 - 1) + table_at(S, W, x0 - 1, y0 - 1);
}

/* ---------------------------------------------------------------------- */
/* Per-template constants and per-shift sums.                              */
/* ---------------------------------------------------------------------- */

/* SumT and SumT2 of one wT x hT template (row-major). */
void ncc_oracle_template_stats(const uint8_t *T, int wT, int hT,
                               int64_t *sumT, int64_t *sumT2)
{
    int64_t a = 0, b = 0;
    for (int k = 0; k < wT * hT; k++) {
        int64_t t = (int64_t)T[k];
        a += t;
        b += t * t;
    }
    *sumT = a;
    *sumT2 = b;
}

/* SumI, SumI2 and SumIT of the window with top-left pixel (x,y): the direct
 * double loop over the window, in int64. */
void ncc_oracle_window_sums(const uint8_t *img, int W, const uint8_t *T,
                            int wT, int hT, int x, int y,
                            int64_t *sI, int64_t *sI2, int64_t *sIT)
{
    int64_t s1 = 0, s2 = 0, s3 = 0;
    for (int dy = 0; dy < hT; dy++) {
        for (int dx = 0; dx < wT; dx++) {
            int64_t p = (int64_t)img[at(W, x + dx, y + dy)];
            int64_t t = (int64_t)T[at(wT, dx, dy)];
            s1 += p;
            s2 += p * p;
            s3 += p * t;
        }
    }
    *sI = s1;
    *sI2 = s2;
    *sIT = s3;
}

/* Pearson coefficient from exact integer sums (see the header). */
double ncc_oracle_coefficient(int64_t N, int64_t sI, int64_t sI2, int64_t sIT,
                              int64_t sT, int64_t sT2)
{
    int64_t num = N * sIT - sI * sT;
    int64_t vI = N * sI2 - sI * sI;
    int64_t vT = N * sT2 - sT * sT;
    if (vI == 0 || vT == 0) return 0.0;
    double r = (double)num / sqrt((double)vI * (double)vT);
    if (r > 1.0) return 1.0;
    if (r < -1.0) return -1.0;
    return r;
}

static int shapes_ok(const uint8_t *img, int W, int H, const uint8_t *T,
                     int wT, int hT, int nT)
{
    return img && T && W > 0 && H > 0 && nT > 0 && wT > 0 && hT > 0 &&
           wT <= W && hT <= H;
}

/* Every valid shift of every template.  out is [nT][Oy][Ox] doubles; the
 * three sum arrays are optional (NULL skips them) and share out's layout.
 * Output rows are independent, so with n_threads > 1 they are spread over
 * OpenMP threads; each value is still the per-shift double loop above. */
int ncc_oracle_correlate(const uint8_t *img, int W, int H, const uint8_t *T,
                         int wT, int hT, int nT, double *out,
                         int64_t *sumI, int64_t *sumI2, int64_t *sumIT,
                         int n_threads)
{
    if (!shapes_ok(img, W, H, T, wT, hT, nT) || !out) return ORACLE_BAD_ARG;
    const int Ox = W - wT + 1, Oy = H - hT + 1;
    const int64_t N = (int64_t)wT * hT;
    (void)n_threads;
    for (int t = 0; t < nT; t++) {
        const uint8_t *Tt = T + (size_t)t * wT * hT;
        int64_t sT, sT2;
        ncc_oracle_template_stats(Tt, wT, hT, &sT, &sT2);
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads > 0 ? n_threads : 1)
#endif
        for (int y = 0; y < Oy; y++) {
            for (int x = 0; x < Ox; x++) {
                int64_t a, b, c;
                ncc_oracle_window_sums(img, W, Tt, wT, hT, x, y, &a, &b, &c);
                size_t o = ((size_t)t * Oy + y) * Ox + x;
                out[o] = ncc_oracle_coefficient(N, a, b, c, sT, sT2);
                if (sumI) sumI[o] = a;
                if (sumI2) sumI2[o] = b;
                if (sumIT) sumIT[o] = c;
            }
        }
    }
    return ORACLE_OK;
}

/* The same quantities at n listed shifts (xs[k], ys[k]) for every template.
 * out and the optional sum arrays are [nT][n]. */
int ncc_oracle_correlate_at(const uint8_t *img, int W, int H, const uint8_t *T,
                            int wT, int hT, int nT, const int32_t *xs,
                            const int32_t *ys, int n, double *out,
                            int64_t *sumI, int64_t *sumI2, int64_t *sumIT,
                            int n_threads)
{
    if (!shapes_ok(img, W, H, T, wT, hT, nT) || !out || !xs || !ys || n < 0)
        return ORACLE_BAD_ARG;
    const int Ox = W - wT + 1, Oy = H - hT + 1;
    for (int k = 0; k < n; k++)
        if (xs[k] < 0 || xs[k] >= Ox || ys[k] < 0 || ys[k] >= Oy) return ORACLE_BAD_ARG;
    const int64_t N = (int64_t)wT * hT;
    (void)n_threads;
    for (int t = 0; t < nT; t++) {
        const uint8_t *Tt = T + (size_t)t * wT * hT;
        int64_t sT, sT2;
        ncc_oracle_template_stats(Tt, wT, hT, &sT, &sT2);
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 64) num_threads(n_threads > 0 ? n_threads : 1)
#endif
        for (int k = 0; k < n; k++) {
            int64_t a, b, c;
            ncc_oracle_window_sums(img, W, Tt, wT, hT, xs[k], ys[k], &a, &b, &c);
            size_t o = (size_t)t * n + k;
            out[o] = ncc_oracle_coefficient(N, a, b, c, sT, sT2);
            if (sumI) sumI[o] = a;
            if (sumI2) sumI2[o] = b;
            if (sumIT) sumIT[o] = c;
        }
    }
    return ORACLE_OK;
}

/* 1 when this build was compiled with OpenMP, else 0. */
int ncc_oracle_has_openmp(void)
{
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}
