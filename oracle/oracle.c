/*
 * oracle.c -- plain CPU oracle for tile-based rasterization of projected 2D
 * Gaussian splats.  TEST INFRASTRUCTURE ONLY: used by tests/, the smoke check
 * and the benchmark's CPU-baseline leg; never by the product path.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared oracle.c -lm
 * (-ffp-contract=off matters: the float32 binning below must round after
 * every operation, exactly as written.)
 *
 * The pages (see oracle.h) fix the model's names and shapes but print no
 * equation.  The readings taken here, each the plainest one consistent with
 * front-to-back alpha compositing of 2D Gaussians in 16x16 tiles:
 *   R1 pixel (x, y) is sampled at its centre (x + 0.5, y + 0.5);
 *   R2 conic (a, b, c) is the inverse covariance [[a, b], [b, c]];
 *      sigma = (a dx^2 + c dy^2) / 2 + b dx dy,  G = exp(-sigma),  d = p - mean;
 *   R3 alpha = min(0.99, opacity * G); a splat is skipped at a pixel when
 *      alpha < 1/255;
 *   R4 T starts at 1; for each unskipped splat in list order T' = T (1 - alpha);
 *      if T' < 1e-4 the pixel stops before blending it, else C += rgb alpha T
 *      and T = T';
 *   R5 image = C + T_final * bg;
 *   R6 last_contrib = 1 + list position of the last blended splat (0: none);
 *   R7 binning: a splat touches the tiles of the AABB of the ellipse where
 *      alpha >= 1/255 is possible, {d : d^T conic d <= 2 ln(255 o)}, whose
 *      half widths are sqrt(k c / det), sqrt(k a / det);
 *   R8 a splat is culled (no pairs) unless every input is finite, depth > 0,
 *      a > 0, c > 0, det = ac - b^2 > 0, and 1/255 <= opacity (255 o finite);
 *   R9 pair key = tile << 32 | float bits of depth; list order is (tile,
 *      depth, splat index) ascending;
 *   R10 backward: the exact partial derivatives of L = sum dL/dimage * image
 *      with respect to the stored mean, conic (a, b, c as stored, so db is
 *      the full partial of the off-diagonal entry), opacity and rgb; through
 *      the 0.99 clamp the alpha derivative is 0;
 *   R11 accumulated weight of a splat = sum over pixels of alpha T (the sum;
 *      an average is the caller's division);
 *   R12 median depth = depth of the last blended splat whose T before
 *      blending was > 0.5 (0 when none was blended);
 *   R13 per-splat weight statistics: the maximum over pixels of the blend
 *      weight alpha T, and the number of pixels that blended the splat (the
 *      "Avg" accumulated weight is R11's sum divided by that count).
 *   R17 depth distortion of a pixel (the "distortion" option, whose per-pixel
 *      totals the backward keeps): D = sum over pairs i < j of the pixel's
 *      blended splats of w_i w_j (z_i - z_j)^2, w = alpha T, z the splat's
 *      depth; its upstream gradient dL/dD per pixel adds to the backward,
 *      which then also gives dL/ddepth.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ALPHA_MIN (1.0 / 255.0)
#define ALPHA_MAX 0.99
#define T_EPS 1e-4
#define MAX_AMB ORC_MAX_AMB

/* Margins of the binning ellipse (R7): k is widened by a relative and an
 * absolute 2^-10 so that float32 rounding of ln, products and square roots
 * can never shrink the covered set. */
#define K_REL (1.0f + 1.0f / 1024.0f)
#define K_ABS (1.0f / 1024.0f)

/* Unit roundoff of float32: the error model of the GPU's float evaluation
 * that decides which pixels are knife edges. */
#define U32 (1.0 / 16777216.0)
/* Relative error of the hardware base-2 exponential (ex2.approx.f32, whose
 * documented bound is 2^-22), taken with a factor 2. */
#define EX2_REL (1.0 / 2097152.0)
/* First-order bounds are used below; this factor covers the neglected
 * higher-order terms (of relative size n u, n the operations chained). */
#define FIRST_ORDER 1.05

void orc_constants(double out[4])
{
    out[0] = ALPHA_MIN;
    out[1] = ALPHA_MAX;
    out[2] = T_EPS;
    out[3] = ORC_TILE;
}

/* ln(x) for a positive, finite, normal float32, in float32 arithmetic:
 * x = m 2^e with m in [1, 2), ln x = e ln2 + 2 atanh(t), t = (m - 1)/(m + 1)
 * in [0, 1/3), and atanh(t) = t (1 + t^2/3 + t^4/5 + ... + t^14/15) by
 * Horner.  The truncated tail is below 2e-9; every operation is one IEEE
 * rounding, so the result is reproducible anywhere IEEE float32 is. */
float orc_ln(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    const int e = (int)((u >> 23) & 0xffu) - 127;
    const uint32_t mu = (u & 0x007fffffu) | 0x3f800000u;
    float m;
    memcpy(&m, &mu, 4);
    const float t = (m - 1.0f) / (m + 1.0f);
    const float t2 = t * t;
    float p = 1.0f / 15.0f;
    p = p * t2 + 1.0f / 13.0f;
    p = p * t2 + 1.0f / 11.0f;
    p = p * t2 + 1.0f / 9.0f;
    p = p * t2 + 1.0f / 7.0f;
    p = p * t2 + 1.0f / 5.0f;
    p = p * t2 + 1.0f / 3.0f;
    p = p * t2 + 1.0f;
    const float lnm = 2.0f * (t * p);
    return (float)e * 0.69314718055994531f + lnm;
}

int orc_splat_rect(const orc_splats_f *s, int64_t i, int32_t W, int32_t H, int32_t r[4])
{
    const float mx = s->mean2d[2 * i], my = s->mean2d[2 * i + 1];
    const float a = s->conic[3 * i], b = s->conic[3 * i + 1], c = s->conic[3 * i + 2];
    const float o = s->opacity[i], d = s->depth[i];
    const float *col = s->rgb + 3 * i;
    if (!isfinite(mx) || !isfinite(my) || !isfinite(a) || !isfinite(b) || !isfinite(c) ||
        !isfinite(o) || !isfinite(d) || !isfinite(col[0]) || !isfinite(col[1]) ||
        !isfinite(col[2]))
        return -1;
    if (!(d > 0.0f) || !(a > 0.0f) || !(c > 0.0f))
        return -1;
    const float det = a * c - b * b;
    if (!(det > 0.0f))
        return -1;
    if (!(o >= (float)ALPHA_MIN))
        return -1;
    const float x = 255.0f * o;
    if (isinf(x))
        return -1;
    float k = 2.0f * orc_ln(x);
    k = k * K_REL + K_ABS;
    const float rx = sqrtf(k * c / det);
    const float ry = sqrtf(k * a / det);
    if (rx != rx || ry != ry)
        return -1;
    const int32_t tiles_x = (W + ORC_TILE - 1) / ORC_TILE;
    const int32_t tiles_y = (H + ORC_TILE - 1) / ORC_TILE;
    float x0 = floorf((mx - rx) * 0.0625f), x1 = floorf((mx + rx) * 0.0625f);
    float y0 = floorf((my - ry) * 0.0625f), y1 = floorf((my + ry) * 0.0625f);
    x0 = fmaxf(x0, 0.0f);
    y0 = fmaxf(y0, 0.0f);
    x1 = fminf(x1, (float)(tiles_x - 1));
    y1 = fminf(y1, (float)(tiles_y - 1));
    if (x0 > x1 || y0 > y1)
        return 0;
    r[0] = (int32_t)x0;
    r[1] = (int32_t)y0;
    r[2] = (int32_t)x1;
    r[3] = (int32_t)y1;
    return 1;
}

int64_t orc_bin(const orc_splats_f *s, int32_t W, int32_t H, uint64_t *keys, uint32_t *vals,
                int64_t capacity, int64_t *culled)
{
    const int32_t tiles_x = (W + ORC_TILE - 1) / ORC_TILE;
    int64_t count = 0, nculled = 0;
    for (int64_t i = 0; i < s->n; ++i) {
        int32_t r[4];
        const int v = orc_splat_rect(s, i, W, H, r);
        if (v < 0) {
            ++nculled;
            continue;
        }
        if (v == 0)
            continue;
        uint32_t dbits;
        memcpy(&dbits, &s->depth[i], 4);
        for (int32_t ty = r[1]; ty <= r[3]; ++ty)
            for (int32_t tx = r[0]; tx <= r[2]; ++tx) {
                if (count < capacity) {
                    const uint64_t tile = (uint64_t)ty * (uint64_t)tiles_x + (uint64_t)tx;
                    keys[count] = (tile << 32) | dbits;
                    vals[count] = (uint32_t)i;
                }
                ++count;
            }
    }
    if (culled)
        *culled = nculled;
    return count;
}

typedef struct {
    uint64_t key;
    uint32_t val;
} pair_t;

static int cmp_pair(const void *pa, const void *pb)
{
    const pair_t *a = pa, *b = pb;
    if (a->key != b->key)
        return a->key < b->key ? -1 : 1;
    if (a->val != b->val)
        return a->val < b->val ? -1 : 1;
    return 0;
}

/* Order of R9: ascending (key, splat index) with the C library's qsort. */
void orc_sort(uint64_t *keys, uint32_t *vals, int64_t n)
{
    if (n <= 0)
        return;
    pair_t *p = malloc((size_t)n * sizeof(pair_t));
    for (int64_t i = 0; i < n; ++i) {
        p[i].key = keys[i];
        p[i].val = vals[i];
    }
    qsort(p, (size_t)n, sizeof(pair_t), cmp_pair);
    for (int64_t i = 0; i < n; ++i) {
        keys[i] = p[i].key;
        vals[i] = p[i].val;
    }
    free(p);
}

/* CSR ranges: offs[t] = number of pairs whose tile is < t. */
int orc_offsets(const uint64_t *keys, int64_t n, int32_t n_tiles, uint32_t *offs)
{
    memset(offs, 0, sizeof(uint32_t) * ((size_t)n_tiles + 1));
    for (int64_t i = 0; i < n; ++i) {
        const uint64_t t = keys[i] >> 32;
        if (t >= (uint64_t)n_tiles)
            return -1;
        offs[t + 1] += 1;
    }
    for (int32_t t = 0; t < n_tiles; ++t)
        offs[t + 1] += offs[t];
    return 0;
}

/* ---------------------------------------------------------------- forward */

typedef struct {
    int64_t pos;       /* position in the tile's list */
    double alpha, G;
    double T;          /* transmittance before blending */
    double mrel;       /* relative error bound of a float32 alpha here */
    double relT;       /* relative error bound of a float32 T before blending */
    int clamped;
} blend_rec;

typedef struct {
    blend_rec *rec;
    int64_t n;
    double C[3];
    double T;          /* T_final */
    double relT;       /* relative error bound of a float32 product for T */
    double median;
    uint32_t last;
    int n_amb;
    int64_t amb_pos[MAX_AMB];
    int amb_kind[MAX_AMB];
} pix_run;

/* Error bounds of a float32 evaluation of a (pixel, splat).  The GPU takes
 * the exponent in base 2, e2 = A dx^2 + B dx dy + C dy^2 with A, B, C the
 * float32 products of -log2(e)/2, -log2(e) (each itself rounded) with a, b,
 * c, dx and dy rounded differences, two products and two fused multiply-adds:
 * every term carries at most 7 roundings, so |e2_f - e2| <= 7 u log2(e) tau
 * with tau = |a| dx^2 / 2 + |b dx dy| + |c| dy^2 / 2 (u = 2^-24, first order).
 *
 * skip_margin: the floor decision compares e2 with thr = -log2f(fl(255 o)),
 * whose error is one rounding of 255 o (log2(1 + u) < 1.45 u) plus log2f's
 * documented 1 ulp (<= 2 u |thr|).  A float32 decision can differ from the
 * exact one only if |ln(255 alpha)| <= ln 2 (|e2 error| + |thr error|)
 * <= 7 u tau + 2 u ln(255 o) + u; the returned relative margin on alpha
 * covers that with the first-order factor.
 *
 * value_margin: relative error of the float32 alpha = fl(o ex2(e2_f)):
 * ln 2 |e2 error| + the exponential's EX2_REL + one rounding, plus the
 * float32 cap 0.99f (0.16 u above 0.99).
 *
 * A decision whose distance to its threshold is inside these bounds may be
 * taken either way by a float32 evaluation: a knife edge. */
static double sigma_terms(double a, double b, double c, double dx, double dy)
{
    return 0.5 * fabs(a) * dx * dx + 0.5 * fabs(c) * dy * dy + fabs(b * dx * dy);
}

static double skip_margin(double tau, double o)
{
    const double l = log(255.0 * o);
    return FIRST_ORDER * U32 * (7.0 * tau + 2.0 * fabs(l) + 1.0);
}

static double value_margin(double tau)
{
    return FIRST_ORDER * (7.0 * U32 * tau + EX2_REL + 1.5 * U32);
}

void orc_margins(double a, double b, double c, double dx, double dy, double o, double out[2])
{
    const double tau = sigma_terms(a, b, c, dx, dy);
    out[0] = skip_margin(tau, o);
    out[1] = value_margin(tau);
}

void orc_margins_n(int64_t n, const double *a, const double *b, const double *c,
                   const double *dx, const double *dy, const double *o, double *skip,
                   double *value)
{
    for (int64_t i = 0; i < n; ++i) {
        double m[2];
        orc_margins(a[i], b[i], c[i], dx[i], dy[i], o[i], m);
        skip[i] = m[0];
        value[i] = m[1];
    }
}

static void note_amb(pix_run *r, int64_t pos, int kind)
{
    if (r->n_amb < MAX_AMB) {
        r->amb_pos[r->n_amb] = pos;
        r->amb_kind[r->n_amb] = kind;
    }
    r->n_amb++;
}

/* Composite one pixel front to back over a tile's list (R1-R6, R12).  When
 * flip_pos >= 0 the decision of kind flip_kind at that list position is taken
 * the other way, giving an alternative outcome of a knife-edge pixel. */
static void run_pixel(const orc_splats_d *s, const uint32_t *list, int64_t len, double px,
                      double py, int64_t flip_pos, int flip_kind, pix_run *r)
{
    r->n = 0;
    r->C[0] = r->C[1] = r->C[2] = 0.0;
    r->T = 1.0;
    r->relT = 0.0;
    r->median = 0.0;
    r->last = 0;
    r->n_amb = 0;
    for (int64_t k = 0; k < len; ++k) {
        const int64_t i = list[k];
        const double a = s->conic[3 * i], b = s->conic[3 * i + 1], c = s->conic[3 * i + 2];
        const double dx = px - s->mean2d[2 * i], dy = py - s->mean2d[2 * i + 1];
        const double sigma = 0.5 * (a * dx * dx + c * dy * dy) + b * dx * dy;
        const double G = exp(-sigma);
        const double oG = s->opacity[i] * G;
        const double tau = sigma_terms(a, b, c, dx, dy);
        const double mrel = value_margin(tau);

        int clamped = oG > ALPHA_MAX;
        if (fabs(oG - ALPHA_MAX) <= mrel * ALPHA_MAX)
            note_amb(r, k, ORC_AMB_CLAMP);
        if (k == flip_pos && flip_kind == ORC_AMB_CLAMP)
            clamped = !clamped;
        const double alpha = clamped ? ALPHA_MAX : oG;

        /* the floor is decided on the unclamped exponent (alpha >= 1/255
         * holds or fails for o G and min(0.99, o G) alike) */
        int skip = alpha < ALPHA_MIN;
        if (fabs(oG - ALPHA_MIN) <= skip_margin(tau, s->opacity[i]) * oG)
            note_amb(r, k, ORC_AMB_ALPHA);
        if (k == flip_pos && flip_kind == ORC_AMB_ALPHA)
            skip = !skip;
        if (skip)
            continue;

        /* T' = fl(T fl(1 - alpha)): the subtraction carries alpha's error
         * (alpha mrel / (1 - alpha)) and one rounding, the product one more;
         * the threshold 1e-4f lies 0.42 u below 1e-4 */
        const double Tn = r->T * (1.0 - alpha);
        const double rel_om = alpha * mrel / (1.0 - alpha) + U32;
        int stop = Tn < T_EPS;
        if (fabs(Tn - T_EPS) <= FIRST_ORDER * (r->relT + rel_om + 2.0 * U32) * Tn)
            note_amb(r, k, ORC_AMB_TERM);
        if (k == flip_pos && flip_kind == ORC_AMB_TERM)
            stop = !stop;
        if (stop)
            break;

        int med = r->T > 0.5;
        if (fabs(r->T - 0.5) <= FIRST_ORDER * r->relT * r->T)
            note_amb(r, k, ORC_AMB_MEDIAN);
        if (k == flip_pos && flip_kind == ORC_AMB_MEDIAN)
            med = !med;
        if (med)
            r->median = s->depth[i];

        const double w = alpha * r->T;
        for (int ch = 0; ch < 3; ++ch)
            r->C[ch] += s->rgb[3 * i + ch] * w;
        blend_rec *e = &r->rec[r->n++];
        e->pos = k;
        e->alpha = alpha;
        e->G = G;
        e->T = r->T;
        e->mrel = mrel;
        e->relT = r->relT;
        e->clamped = clamped;
        r->T = Tn;
        r->relT += rel_om + U32;
        r->last = (uint32_t)(k + 1);
    }
}

/* Test accessor: one pixel's compositing as run_pixel does it, with the
 * error bounds the knife-edge decisions use.  out[k] (k < min(n, cap))
 * receives the k-th blended splat: list position, alpha, G, T before it,
 * its alpha error bound and the bound on T before it.  tail = (T_final, the
 * bound on T_final, last_contrib, number of knife-edge decisions); amb
 * receives up to ORC_MAX_AMB (position, kind) pairs.  Returns n. */
int64_t orc_trace_pixel(const orc_splats_d *s, const uint32_t *list, int64_t len, double px,
                        double py, orc_trace_rec *out, int64_t cap, double tail[4],
                        int32_t *amb)
{
    pix_run r;
    r.rec = malloc(sizeof(blend_rec) * (size_t)(len > 0 ? len : 1));
    run_pixel(s, list, len, px, py, -1, 0, &r);
    for (int64_t k = 0; k < r.n && k < cap; ++k) {
        out[k].pos = r.rec[k].pos;
        out[k].alpha = r.rec[k].alpha;
        out[k].G = r.rec[k].G;
        out[k].T = r.rec[k].T;
        out[k].mrel = r.rec[k].mrel;
        out[k].relT = r.rec[k].relT;
        out[k].clamped = r.rec[k].clamped;
        out[k].pad = 0;
    }
    tail[0] = r.T;
    tail[1] = r.relT;
    tail[2] = (double)r.last;
    tail[3] = (double)r.n_amb;
    const int na = r.n_amb < MAX_AMB ? r.n_amb : MAX_AMB;
    for (int j = 0; j < na && amb; ++j) {
        amb[2 * j] = (int32_t)r.amb_pos[j];
        amb[2 * j + 1] = r.amb_kind[j];
    }
    const int64_t n = r.n;
    free(r.rec);
    return n;
}

/* R17 by its definition: the double sum over pairs of blended splats.
 * err receives a bound on the error of a float32 evaluation by running
 * totals of depths taken relative to the first blended splat's.  For the
 * k-th blended splat i (k = 0, 1, ...) with the totals A, D1', D2' of the
 * splats before it:
 *   (16 + k) u w_i (z'_i^2 A + 2 |z'_i| |D1'| + D2') -- its term's roundings
 *     and those the totals gathered: each is a float32 running sum of k
 *     non-negative terms (depths are ascending, so z' >= 0), off by at
 *     most k u of itself;
 *   w_i E_i (2 relT + mrel_i + 4 u (n + 2)), E_i = sum over the other blended
 *     splats j of w_j (z_i - z_j)^2 -- the weights' own errors (a pair's
 *     product carries both weights' errors, so each weight's error is
 *     weighed against its pairs with earlier and later splats alike) and
 *     the rounding of the sum of the n terms into D. */
static double pixel_dist(const orc_splats_d *s, const uint32_t *list, const pix_run *r,
                         double *err)
{
    double D = 0.0;
    for (int64_t i = 0; i < r->n; ++i)
        for (int64_t j = 0; j < i; ++j) {
            const double wi = r->rec[i].alpha * r->rec[i].T, wj = r->rec[j].alpha * r->rec[j].T;
            const double dz = s->depth[list[r->rec[i].pos]] - s->depth[list[r->rec[j].pos]];
            D += wi * wj * dz * dz;
        }
    if (err) {
        double e = 0.0, A = 0.0, D1 = 0.0, D2 = 0.0;
        const double z0 = r->n ? s->depth[list[r->rec[0].pos]] : 0.0;
        for (int64_t i = 0; i < r->n; ++i) {
            const double w = r->rec[i].alpha * r->rec[i].T;
            const double zi = s->depth[list[r->rec[i].pos]];
            const double z = zi - z0;
            double E = 0.0;
            for (int64_t j = 0; j < r->n; ++j) {
                const double dz = zi - s->depth[list[r->rec[j].pos]];
                E += r->rec[j].alpha * r->rec[j].T * dz * dz;
            }
            const double relw = 2.0 * r->relT + r->rec[i].mrel + 4.0 * U32 * (double)(r->n + 2);
            e += (16.0 + (double)i) * U32 * w * (z * z * A + 2.0 * fabs(z) * fabs(D1) + D2) +
                 w * E * relw;
            A += w;
            D1 += w * z;
            D2 += w * z * z;
        }
        *err = e;
    }
    return D;
}

static int64_t max_list(const orc_frame *f, int32_t n_tiles)
{
    int64_t m = 1;
    for (int32_t t = 0; t < n_tiles; ++t) {
        const int64_t len = (int64_t)f->offs[t + 1] - (int64_t)f->offs[t];
        if (len > m)
            m = len;
    }
    return m;
}

int64_t orc_forward(const orc_splats_d *s, const orc_frame *f, orc_fwd_out *out,
                    orc_alt *alts, int64_t alt_capacity)
{
    const int32_t W = f->W, H = f->H;
    const int32_t tiles_x = (W + ORC_TILE - 1) / ORC_TILE;
    const int32_t tiles_y = (H + ORC_TILE - 1) / ORC_TILE;
    const int64_t HW = (int64_t)W * H;
    const int64_t mlen = max_list(f, tiles_x * tiles_y);
    pix_run r, r2;
    r.rec = malloc(sizeof(blend_rec) * (size_t)mlen);
    r2.rec = malloc(sizeof(blend_rec) * (size_t)mlen);
    int64_t n_alt = 0;
    for (int32_t ty = 0; ty < tiles_y; ++ty)
        for (int32_t tx = 0; tx < tiles_x; ++tx) {
            const int32_t t = ty * tiles_x + tx;
            if (f->tile_mask && !f->tile_mask[t])
                continue;
            const uint32_t *list = f->vals + f->offs[t];
            const int64_t len = (int64_t)f->offs[t + 1] - (int64_t)f->offs[t];
            for (int32_t y = ty * ORC_TILE; y < (ty + 1) * ORC_TILE && y < H; ++y)
                for (int32_t x = tx * ORC_TILE; x < (tx + 1) * ORC_TILE && x < W; ++x) {
                    const int64_t p = (int64_t)y * W + x;
                    run_pixel(s, list, len, x + 0.5, y + 0.5, -1, 0, &r);
                    if (out->image)
                        for (int ch = 0; ch < 3; ++ch)
                            out->image[ch * HW + p] = r.C[ch] + r.T * f->bg[ch];
                    if (out->T_final)
                        out->T_final[p] = r.T;
                    if (out->last)
                        out->last[p] = r.last;
                    if (out->median)
                        out->median[p] = r.median;
                    if (out->n_amb)
                        out->n_amb[p] = (uint8_t)(r.n_amb > 255 ? 255 : r.n_amb);
                    if (out->dist)
                        out->dist[p] = pixel_dist(s, list, &r, out->dist_err ? &out->dist_err[p] : NULL);
                    for (int64_t k = 0; k < r.n; ++k) {   /* R13 */
                        const int64_t i = list[r.rec[k].pos];
                        const double w = r.rec[k].alpha * r.rec[k].T;
                        if (out->max_w && w > out->max_w[i])
                            out->max_w[i] = w;
                        if (out->count)
                            out->count[i] += 1;
                        if (out->splat_amb && r.n_amb)
                            out->splat_amb[i] = 1;
                    }
                    const int na = r.n_amb < MAX_AMB ? r.n_amb : MAX_AMB;
                    for (int j = 0; j < na; ++j) {
                        if (alts && n_alt < alt_capacity) {
                            run_pixel(s, list, len, x + 0.5, y + 0.5, r.amb_pos[j],
                                      r.amb_kind[j], &r2);
                            orc_alt *e = &alts[n_alt];
                            e->pixel = (int32_t)p;
                            e->kind = r.amb_kind[j];
                            e->list_pos = (int32_t)r.amb_pos[j];
                            e->last = r2.last;
                            for (int ch = 0; ch < 3; ++ch)
                                e->image[ch] = r2.C[ch] + r2.T * f->bg[ch];
                            e->T_final = r2.T;
                            e->median = r2.median;
                            e->dist = pixel_dist(s, list, &r2, NULL);
                            if (out->splat_amb)
                                for (int64_t k = 0; k < r2.n; ++k)
                                    out->splat_amb[list[r2.rec[k].pos]] = 1;
                        }
                        ++n_alt;
                    }
                }
        }
    free(r.rec);
    free(r2.rec);
    return n_alt;
}

/* --------------------------------------------------------------- backward */

enum { F_MX, F_MY, F_A, F_B, F_C, F_O, F_R, F_G, F_BL, F_W, F_Z, NF };


/* Gradient contributions of one pixel by the plain definition (R10, R11):
 * with T_k the transmittance before blended splat k, w_k = alpha_k T_k and
 * S_k = sum over later blended splats j of rgb_j w_j,
 *   dL/drgb_k   = g w_k
 *   dL/dalpha_k = sum_ch g_ch (rgb_k,ch T_k - (S_k,ch + T_final bg_ch) / (1 - alpha_k))
 *   dL/dsigma_k = -alpha_k dL/dalpha_k         (d alpha / d sigma = -o G)
 *   dL/do_k     = G_k dL/dalpha_k
 *   dL/dmean    = dL/dsigma * (-(a dx + b dy), -(b dx + c dy))
 *   dL/d(a,b,c) = dL/dsigma * (dx^2 / 2, dx dy, dy^2 / 2)
 * written to out[k][F_*]; out[k][F_W] = w_k.
 * With an upstream gradient gD of the distortion D (R17), D's own terms add:
 * with E_k = dD/dw_k = sum_j w_j (z_k - z_j)^2 and dw_i/dalpha_k = T_k (i = k),
 * -w_i / (1 - alpha_k) (i after k),
 *   dL/dalpha_k += gD (E_k T_k - sum_{i after k} w_i E_i / (1 - alpha_k))
 *   dL/dz_k      = gD sum_j 2 w_k w_j (z_k - z_j)                  (out[k][F_Z]). */
static void pixel_backward(const orc_splats_d *s, const uint32_t *list, const pix_run *r,
                           double px, double py, const double g[3], const double bg[3],
                           double gD, double *out)
{
    double S[3] = {0.0, 0.0, 0.0};
    double SE = 0.0;   /* sum over later blended splats of w E */
    for (int64_t k = r->n - 1; k >= 0; --k) {
        const blend_rec *e = &r->rec[k];
        const int64_t i = list[e->pos];
        const double *col = s->rgb + 3 * i;
        const double w = e->alpha * e->T;
        double dL_dalpha = 0.0;
        for (int ch = 0; ch < 3; ++ch)
            dL_dalpha += g[ch] * (col[ch] * e->T - (S[ch] + r->T * bg[ch]) / (1.0 - e->alpha));
        double E = 0.0, dz_sum = 0.0;
        if (gD != 0.0) {
            const double zk = s->depth[i];
            for (int64_t j = 0; j < r->n; ++j) {
                const double wj = r->rec[j].alpha * r->rec[j].T;
                const double dz = zk - s->depth[list[r->rec[j].pos]];
                E += wj * dz * dz;
                dz_sum += 2.0 * w * wj * dz;
            }
            dL_dalpha += gD * (E * e->T - SE / (1.0 - e->alpha));
        }
        double *o = out + NF * k;
        o[F_Z] = gD * dz_sum;
        for (int ch = 0; ch < 3; ++ch)
            o[F_R + ch] = g[ch] * w;
        o[F_W] = w;
        if (!e->clamped) {
            const double a = s->conic[3 * i], b = s->conic[3 * i + 1], c = s->conic[3 * i + 2];
            const double dx = px - s->mean2d[2 * i], dy = py - s->mean2d[2 * i + 1];
            const double dL_dsigma = -e->alpha * dL_dalpha;
            o[F_MX] = dL_dsigma * -(a * dx + b * dy);
            o[F_MY] = dL_dsigma * -(b * dx + c * dy);
            o[F_A] = dL_dsigma * 0.5 * dx * dx;
            o[F_B] = dL_dsigma * dx * dy;
            o[F_C] = dL_dsigma * 0.5 * dy * dy;
            o[F_O] = dL_dalpha * e->G;
        } else {
            for (int q = F_MX; q <= F_O; ++q)
                o[q] = 0.0;
        }
        for (int ch = 0; ch < 3; ++ch)
            S[ch] += col[ch] * w;
        SE += w * E;
    }
}

static void add_fields(orc_grads *gr, int64_t i, const double *v, int absval)
{
#define ACC(dst, x) ((dst) += absval ? fabs(x) : (x))
    ACC(gr->dmean2d[2 * i], v[F_MX]);
    ACC(gr->dmean2d[2 * i + 1], v[F_MY]);
    ACC(gr->dconic[3 * i], v[F_A]);
    ACC(gr->dconic[3 * i + 1], v[F_B]);
    ACC(gr->dconic[3 * i + 2], v[F_C]);
    ACC(gr->dopacity[i], v[F_O]);
    ACC(gr->drgb[3 * i], v[F_R]);
    ACC(gr->drgb[3 * i + 1], v[F_G]);
    ACC(gr->drgb[3 * i + 2], v[F_BL]);
    if (gr->accum)
        ACC(gr->accum[i], v[F_W]);
    if (gr->ddepth)
        ACC(gr->ddepth[i], v[F_Z]);
#undef ACC
}

/* Accumulates (+=) into grads; the caller zeroes them.  slack (may be NULL)
 * receives, per splat and field, the sum over knife-edge decisions of
 * |alternative - normal| contribution.  accum_err (may be NULL) receives a
 * bound on the error of a float32 evaluation of the accumulated weight, per
 * blended pixel w (2 relT + 3 u n + mrel + 33 u) + 2^-32 with relT the
 * bound on the pixel's final T and n its blended splats: the backward
 * recovers T in front of a splat from T_final by one rounded 1 - alpha, one
 * reciprocal of at most 1 ulp (2 u) and one rounded product per later
 * splat (at most relT + 3 u n beyond T_final's own relT), w = alpha T adds
 * alpha's mrel and a rounding; the sum over the at most 32 pixels of a
 * block in float32 adds at most 31 u of the block's weight (32 u a pixel),
 * and the 32.32 fixed-point conversion at most 2^-33 a block (2^-32 a
 * pixel). */
int orc_backward(const orc_splats_d *s, const orc_frame *f, const double *dL_dimage,
                 orc_grads *grads, orc_grads *slack, double *accum_err)
{
    const int32_t W = f->W, H = f->H;
    const int32_t tiles_x = (W + ORC_TILE - 1) / ORC_TILE;
    const int32_t tiles_y = (H + ORC_TILE - 1) / ORC_TILE;
    const int64_t HW = (int64_t)W * H;
    const int64_t mlen = max_list(f, tiles_x * tiles_y);
    pix_run r, r2;
    r.rec = malloc(sizeof(blend_rec) * (size_t)mlen);
    r2.rec = malloc(sizeof(blend_rec) * (size_t)mlen);
    double *c1 = malloc(sizeof(double) * NF * (size_t)mlen);
    double *c2 = malloc(sizeof(double) * NF * (size_t)mlen);
    double *byp1 = calloc((size_t)mlen * NF, sizeof(double));
    double *byp2 = calloc((size_t)mlen * NF, sizeof(double));
    for (int32_t ty = 0; ty < tiles_y; ++ty)
        for (int32_t tx = 0; tx < tiles_x; ++tx) {
            const int32_t t = ty * tiles_x + tx;
            if (f->tile_mask && !f->tile_mask[t])
                continue;
            const uint32_t *list = f->vals + f->offs[t];
            const int64_t len = (int64_t)f->offs[t + 1] - (int64_t)f->offs[t];
            for (int32_t y = ty * ORC_TILE; y < (ty + 1) * ORC_TILE && y < H; ++y)
                for (int32_t x = tx * ORC_TILE; x < (tx + 1) * ORC_TILE && x < W; ++x) {
                    const int64_t p = (int64_t)y * W + x;
                    const double g[3] = {dL_dimage[p], dL_dimage[HW + p], dL_dimage[2 * HW + p]};
                    const double px = x + 0.5, py = y + 0.5;
                    const double gD = f->dL_ddist ? f->dL_ddist[p] : 0.0;
                    run_pixel(s, list, len, px, py, -1, 0, &r);
                    pixel_backward(s, list, &r, px, py, g, f->bg, gD, c1);
                    for (int64_t k = 0; k < r.n; ++k) {
                        const int64_t i = list[r.rec[k].pos];
                        add_fields(grads, i, c1 + NF * k, 0);
                        if (accum_err) {
                            const double relw = 2.0 * r.relT + r.rec[k].mrel +
                                                3.0 * U32 * (double)r.n + 33.0 * U32;
                            accum_err[i] += c1[NF * k + F_W] * relw + 1.0 / 4294967296.0;
                        }
                    }
                    if (!slack || r.n_amb == 0)
                        continue;
                    /* Contributions by list position, normal vs each alternative. */
                    const int na = r.n_amb < MAX_AMB ? r.n_amb : MAX_AMB;
                    for (int j = 0; j < na; ++j) {
                        run_pixel(s, list, len, px, py, r.amb_pos[j], r.amb_kind[j], &r2);
                        pixel_backward(s, list, &r2, px, py, g, f->bg, gD, c2);
                        memset(byp1, 0, sizeof(double) * NF * (size_t)len);
                        memset(byp2, 0, sizeof(double) * NF * (size_t)len);
                        for (int64_t k = 0; k < r.n; ++k)
                            memcpy(byp1 + NF * r.rec[k].pos, c1 + NF * k, sizeof(double) * NF);
                        for (int64_t k = 0; k < r2.n; ++k)
                            memcpy(byp2 + NF * r2.rec[k].pos, c2 + NF * k, sizeof(double) * NF);
                        for (int64_t q = 0; q < len; ++q) {
                            double d[NF];
                            for (int fld = 0; fld < NF; ++fld)
                                d[fld] = byp2[NF * q + fld] - byp1[NF * q + fld];
                            add_fields(slack, list[q], d, 1);
                        }
                    }
                }
        }
    free(r.rec);
    free(r2.rec);
    free(c1);
    free(c2);
    free(byp1);
    free(byp2);
    return 0;
}
