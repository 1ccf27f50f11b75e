/*
 * ss_ssim.h -- C ABI of libss.so, part 3: the L1 + SSIM training loss and its
 * gradient with respect to the rendered image, in one call.
 *
 * "Phase 5 step 30b -- kernel-by-kernel timing" trains with L1 + SSIM,
 * lambda = 0.20 and a K = 7 window (setup), and times the SSIM forward and
 * backward as one step, "ssim_fwd_bwd" (measurement table, hotspot ranking).
 * The page prints no formula; the model is the plainest reading of the
 * structural-similarity index of Wang et al. (2004) used as a loss:
 *
 *   window: the 7 x 7 Gaussian, outer product of the 1D window
 *     exp(-i^2 / (2 * 1.5^2)), i = -3..3, normalised to sum 1;
 *   per channel, "same"-size correlation with zero padding outside the
 *     image: mu_x = w * x, sigma_x^2 = w * x^2 - mu_x^2,
 *     sigma_xy = w * (x y) - mu_x mu_y (and likewise for y);
 *   SSIM(p) = (2 mu_x mu_y + C1)(2 sigma_xy + C2) /
 *             ((mu_x^2 + mu_y^2 + C1)(sigma_x^2 + sigma_y^2 + C2)),
 *     C1 = 0.01^2, C2 = 0.03^2;
 *   loss = (1 - lambda) mean |x - y| + lambda (1 - mean SSIM), means over
 *     every channel and pixel; x the rendered image, y the target;
 *   dL/dx with d|x - y|/dx = sign(x - y) (0 where x = y).
 *
 * Conventions are those of ss.h.
 */
#ifndef SS_SSIM_H
#define SS_SSIM_H

#include "ss.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of workspace ss_ssim_loss needs (one 16-byte partial sum per
 * 32 x 32 tile and channel, and a 16-byte slot for the completion counter);
 * 0 for sizes outside the limits below. */
size_t ss_ssim_workspace_bytes(int32_t C, int32_t H, int32_t W);

/* loss:    device float[3], overwritten with (loss, mean SSIM, mean |x - y|),
 *          summed in double in a fixed order (deterministic).
 * img, target: device float [C][H][W] (planar, as ss_raster_fwd writes).
 * dL_dimg: device float [C][H][W], overwritten; may be passed straight to
 *          ss_raster_bwd as its dL_dimage.
 * workspace: device, 16-byte aligned, >= ss_ssim_workspace_bytes (partial sums
 *          and a counter, which the call clears itself).
 * Errors: SS_ERR_UNSUPPORTED unless 1 <= C <= 64 and 1 <= H, W <= 32768;
 * SS_ERR_INVALID_ARG for a NULL pointer, lambda outside [0, 1], or a small
 * or misaligned workspace. */
ss_status ss_ssim_loss(const float *img, const float *target, int32_t C, int32_t H, int32_t W,
                       float lambda, float *loss, float *dL_dimg, void *workspace,
                       size_t workspace_bytes, ss_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SS_SSIM_H */
