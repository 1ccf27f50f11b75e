/*
 * oracle.h -- plain CPU oracle for tile-based rasterization of projected 2D
 * Gaussian splats (forward compositing and its analytic backward).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this code: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant generator
 * with the CUDA library; the two meet only through the seeded inputs of
 * synth/.
 *
 * Sources (the pages name the model but print none of its equations):
 *   - "Spirula Studio ... 3D Gaussian splatting backward rasterization 19%
 *     faster" (wzjinhao.cn/news/70431), section "mechanism": the backward
 *     rasterizer works on the 2D screen-space path of splats.
 *   - "Phase 5 step 30b -- kernel-by-kernel timing" (otkrickey-splat.pages.dev),
 *     "hotspot ranking" and "conclusion": per-splat gradient of 9 fields
 *     (dmean2d x2, dconic x3, dopacity, dRGB x3), 16x16-pixel tiles, the
 *     emit_pairs / radix sort / extract_offsets / rasterize kernels.
 * Every constant and rule the pages leave open is the plainest reading of
 * front-to-back alpha compositing of 2D Gaussians; each is stated at its
 * point of use in oracle.c.
 *
 * Precision: the tile binning is a float32 decision (same arithmetic as the
 * CUDA side, IEEE + - * / sqrt only, no contraction: build with
 * -ffp-contract=off); compositing and gradients are double.
 */
#ifndef SS_ORACLE_H
#define SS_ORACLE_H
#include <stdint.h>

#define ORC_TILE 16

typedef struct {
    int64_t n;
    const float *mean2d;   /* [n][2] */
    const float *conic;    /* [n][3]  (a, b, c) of [[a, b], [b, c]] */
    const float *opacity;  /* [n]    */
    const float *rgb;      /* [n][3] */
    const float *depth;    /* [n]    */
} orc_splats_f;

typedef struct {
    int64_t n;
    const double *mean2d, *conic, *opacity, *rgb, *depth;
} orc_splats_d;

typedef struct {
    int32_t W, H;
    double bg[3];
    const uint32_t *vals;      /* splat index per sorted pair */
    const uint32_t *offs;      /* [tiles + 1] CSR ranges into vals */
    const uint8_t *tile_mask;  /* NULL: all tiles; else only tiles with mask != 0 */
    const double *dL_ddist;    /* [H][W] upstream gradient of the distortion image, or NULL */
} orc_frame;

typedef struct {               /* forward outputs; any pointer may be NULL */
    double *image;             /* [3][H][W] */
    double *T_final;           /* [H][W] */
    uint32_t *last;            /* [H][W] */
    double *median;            /* [H][W] */
    uint8_t *n_amb;            /* [H][W] ambiguous float32 decisions (knife edges) */
    double *max_w;             /* [n] max over pixels of the blend weight alpha T (+=max) */
    uint32_t *count;           /* [n] pixels that blended the splat (+=) */
    uint8_t *splat_amb;        /* [n] 1 if blended at a knife-edge pixel in any outcome */
    double *dist;              /* [H][W] depth distortion sum_{i<j} w_i w_j (z_i - z_j)^2 */
    double *dist_err;          /* [H][W] bound on the error of its float32 evaluation */
} orc_fwd_out;

/* One alternative outcome of a pixel: the result when one knife-edge
 * decision is taken the other way. */
typedef struct {
    int32_t pixel;             /* y * W + x */
    int32_t kind;              /* ORC_AMB_* */
    int32_t list_pos;          /* position in the tile's list */
    uint32_t last;
    double image[3];
    double T_final;
    double median;
    double dist;
} orc_alt;

enum { ORC_AMB_ALPHA = 1, ORC_AMB_TERM = 2, ORC_AMB_CLAMP = 3, ORC_AMB_MEDIAN = 4 };

typedef struct {               /* per-splat fields, all double */
    double *dmean2d;           /* [n][2] */
    double *dconic;            /* [n][3] */
    double *dopacity;          /* [n]    */
    double *drgb;              /* [n][3] */
    double *accum;             /* [n]    */
    double *ddepth;            /* [n] (only with dL_ddist; may be NULL) */
} orc_grads;

/* One blended splat of a traced pixel (orc_trace_pixel). */
typedef struct {
    int64_t pos;               /* position in the tile's list */
    double alpha, G;
    double T;                  /* transmittance before blending */
    double mrel;               /* bound on the relative error of a float32 alpha */
    double relT;               /* bound on the relative error of a float32 T before it */
    int32_t clamped, pad;
} orc_trace_rec;

#define ORC_MAX_AMB 8

void orc_constants(double out[4]);   /* alpha_min, alpha_max, T_eps, tile */
float orc_ln(float x);               /* natural log by the atanh series, float32 */

/* -1: splat culled (invalid); 0: valid, touches no tile; 1: rect in r[4] =
 * (x0, y0, x1, y1) inclusive tile coordinates. */
int orc_splat_rect(const orc_splats_f *s, int64_t i, int32_t W, int32_t H, int32_t r[4]);
int64_t orc_bin(const orc_splats_f *s, int32_t W, int32_t H, uint64_t *keys, uint32_t *vals,
                int64_t capacity, int64_t *culled);
void orc_sort(uint64_t *keys, uint32_t *vals, int64_t n);
int orc_offsets(const uint64_t *keys, int64_t n, int32_t n_tiles, uint32_t *offs);

int64_t orc_forward(const orc_splats_d *s, const orc_frame *f, orc_fwd_out *out,
                    orc_alt *alts, int64_t alt_capacity);

/* Error bounds of a float32 evaluation at one (pixel, splat), d = pixel -
 * mean: out[0] the relative margin of the alpha-floor decision, out[1] the
 * relative error bound of alpha (knife-edge model; see oracle.c). */
void orc_margins(double a, double b, double c, double dx, double dy, double o, double out[2]);
/* orc_margins over n (pixel, splat) pairs given as arrays. */
void orc_margins_n(int64_t n, const double *a, const double *b, const double *c,
                   const double *dx, const double *dy, const double *o, double *skip,
                   double *value);
/* One pixel's front-to-back compositing with its error bounds (test accessor). */
int64_t orc_trace_pixel(const orc_splats_d *s, const uint32_t *list, int64_t len, double px,
                        double py, orc_trace_rec *out, int64_t cap, double tail[4],
                        int32_t *amb);
int orc_backward(const orc_splats_d *s, const orc_frame *f, const double *dL_dimage,
                 orc_grads *grads, orc_grads *slack, double *accum_err);
#endif
