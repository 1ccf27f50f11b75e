/*
 * ss_project.h -- C ABI of libss.so, part 2: projection of 3D Gaussian splats
 * to the 2D splats that ss.h rasterizes, and its backward.
 *
 * The training step of "Phase 5 step 30b -- kernel-by-kernel timing"
 * (measurement table, hotspot ranking) runs a forward projection kernel
 * (project_soa) before the tile binning and its backward (project_backwards)
 * after the rasterizer's backward; the page puts most of the projection's
 * cost in the spherical-harmonic colour evaluation.  It prints no formula;
 * the model below is the plainest reading of projecting a 3D Gaussian through
 * a pinhole camera:
 *
 *   p_c = R p + t (R world-to-camera, row-major);  depth = p_c.z;
 *   mean2d = (fx x/z + cx, fy y/z + cy) in the rasterizer's pixel frame
 *     (pixel centres at +0.5);
 *   Sigma = R(q/|q|) diag(scale)^2 R(q/|q|)^T, q = (w, x, y, z);
 *   2D covariance = J R Sigma R^T J^T + blur I, J the Jacobian of
 *     (fx x/z, fy y/z) at p_c (local affine approximation, x/z not clamped);
 *   conic = (a, b, c) of its inverse [[a, b], [b, c]];
 *   rgb = max(0, sum_k sh[k] Y_k(d) + 0.5) per channel, d the unit vector
 *     from the camera centre -R^T t to the mean; Y_k the real spherical
 *     harmonics of degree <= 3, k = l^2 + l + m,
 *     Y_lm = N_lm P_l^(|m|)(z) Re((x + i y)^|m|) (m >= 0) or Im(...) (m < 0),
 *     N_lm = sqrt((2l+1)/(4 pi) (l-|m|)!/(l+|m|)!) (times sqrt 2 if m != 0),
 *     no Condon-Shortley phase;
 *   a splat with z <= near_z, a 2D covariance that is not positive definite,
 *     or a non-finite output is culled: all its outputs are 0 (so the
 *     rasterizer culls it on depth <= 0) and so are its gradients.
 *
 * Conventions are those of ss.h (caller-owned device memory, asynchronous on
 * `stream`, argument errors found on the host before anything is enqueued).
 */
#ifndef SS_PROJECT_H
#define SS_PROJECT_H

#include "ss.h"

#ifdef __cplusplus
extern "C" {
#endif

/* 3D splats, float32, device memory.  The SH coefficients are stored
 * coefficient-major, sh[(k * 3 + channel) * n + i], so that one warp's
 * loads of coefficient k are contiguous. */
typedef struct {
    const float *mean3;    /* [n][3] world position */
    const float *scale;    /* [n][3] standard deviation along each local axis */
    const float *quat;     /* [n][4] rotation (w, x, y, z), any nonzero norm; 16-byte aligned */
    const float *sh;       /* [K][3][n], K = (sh_degree + 1)^2 */
    int32_t n;             /* 0 <= n < 2^31; pointers may be NULL when n == 0 */
    int32_t sh_degree;     /* 0..3 */
} ss_splats3d;

/* Pinhole camera; a HOST struct, copied into the launch. */
typedef struct {
    float R[9];            /* world-to-camera rotation, row-major */
    float t[3];            /* world-to-camera translation */
    float fx, fy, cx, cy;  /* focal lengths and principal point, pixels */
    float near_z;          /* splats with camera z <= near_z are culled */
    float blur;            /* added to both diagonal entries of the 2D covariance, px^2 */
} ss_camera;

/* Per-splat gradients of the 3D parameters, float32, device memory, the
 * layouts of ss_splats3d (dquat 16-byte aligned, dsh coefficient-major). */
typedef struct {
    float *dmean3;         /* [n][3] */
    float *dscale;         /* [n][3] */
    float *dquat;          /* [n][4] with respect to the unnormalised q */
    float *dsh;            /* [K][3][n] */
} ss_grads3d;

/* Forward projection.  Outputs (device, overwritten, the layouts ss_splats
 * reads): mean2d [n][2] (8-byte aligned), conic [n][3], depth [n], rgb [n][3].
 * Opacity is not touched: the rasterizer takes the caller's opacity array.
 * Errors: SS_ERR_INVALID_ARG for a NULL pointer with n > 0, a degree outside
 * 0..3, a misaligned quat / mean2d, or a camera with a non-finite entry or
 * fx, fy <= 0. */
ss_status ss_project_fwd(const ss_splats3d *splats, const ss_camera *cam, float *mean2d,
                         float *conic, float *depth, float *rgb, ss_stream_t stream);

/* Backward of ss_project_fwd: the exact partial derivatives of
 *   L = sum_i dmean2d_i . mean2d_i + dconic_i . conic_i + drgb_i . rgb_i
 * with respect to mean3, scale, quat (unnormalised) and sh, for upstream
 * gradients in the forward outputs' layouts (dconic's b entry is the partial
 * with respect to the stored b, as ss_raster_bwd writes it).  The camera is
 * fixed; depth has no upstream gradient.  Every array of `grads` is
 * overwritten (0 for culled splats).  Errors as ss_project_fwd. */
ss_status ss_project_bwd(const ss_splats3d *splats, const ss_camera *cam, const float *dmean2d,
                         const float *dconic, const float *drgb, const ss_grads3d *grads,
                         ss_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SS_PROJECT_H */
