/*
 * ss.h -- C ABI of libss.so, a GB300 (sm_103a) implementation of tile-based
 * differentiable rasterization of projected 2D Gaussian splats.
 *
 * The path has the kernels the pages time one after another in a training
 * step ("Phase 5 step 30b -- kernel-by-kernel timing", measurement table:
 * emit_pairs, radix_hist / radix_scatter, extract_offsets, rasterize_f32,
 * rasterize_backwards) and that the Spirula Studio write-up benchmarks as
 * "tile isect", "raster fwd" and "raster bwd" ("从 8.6 KB 到 4.2 KB ...",
 * section 亲手验证):
 *
 *   ss_bin_tiles   tile binning: one (key, value) pair per (splat, touched tile)
 *   ss_pair_count  the one device-to-host read: how many pairs were emitted
 *   ss_sort_pairs  radix sort of the pairs by (tile, depth) + per-tile ranges
 *   ss_raster_fwd  front-to-back compositing per pixel, from the splats
 *   ss_raster_bwd  back-to-front gradient of the 9 per-splat fields, from the
 *                  splats, the forward's T_final / last_contrib and dL/dimage
 *
 * ss_raster_fwd_records / ss_raster_bwd_records are the same two steps on
 * the per-splat records ss_bin_tiles writes, with the optional outputs
 * (weight statistics, distortion) and the forward's blend decisions passed
 * to the backward (blend_masks), which then need not re-evaluate them: the
 * form a training step uses.
 *
 * Conventions (every function):
 *   - Memory: the caller owns all memory.  Every pointer is a DEVICE pointer
 *     unless its name starts with h_ or the comment says host.  The library
 *     allocates nothing and keeps no state except a per-thread error string.
 *   - Streams: work is enqueued on `stream` (NULL = the legacy default stream)
 *     and returns before it runs, except ss_pair_count and ss_sort_status,
 *     which synchronize `stream`.
 *   - Errors: argument errors are found on the host before anything is
 *     enqueued and return SS_ERR_INVALID_ARG / SS_ERR_UNSUPPORTED with a
 *     message in ss_last_error(); a failed CUDA launch returns SS_ERR_CUDA.
 *     Nothing traps or asserts on the device.
 *   - Tiles are 16x16 pixels, tile id = ty * ceil(W/16) + tx, in row-major
 *     order; 1 <= W, H <= 32768.
 *   - Images are planar float32: image[c][y][x], c = 0..2.
 *   - The model (the pages name it but print no equation; these are the
 *     plainest readings of front-to-back alpha compositing of 2D Gaussians):
 *       pixel (x, y) is sampled at (x + 0.5, y + 0.5); d = pixel - mean;
 *       sigma = (a dx^2 + c dy^2) / 2 + b dx dy,  G = exp(-sigma);
 *       alpha = min(0.99, opacity G); splats with alpha < 1/255 are skipped;
 *       T starts at 1; a splat whose blend would take T below 1e-4 ends the
 *       pixel unblended; otherwise color += rgb alpha T and T *= (1 - alpha);
 *       image = color + T_final * bg.
 */
#ifndef SS_H
#define SS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the same pointer type); NULL is the legacy default stream. */
typedef struct CUstream_st *ss_stream_t;

typedef enum {
    SS_OK = 0,
    SS_ERR_INVALID_ARG = 1,  /* bad pointer, size or flag; nothing was enqueued */
    SS_ERR_CAPACITY = 2,     /* more pairs than the caller's capacity (ss_pair_count) */
    SS_ERR_CUDA = 3,         /* a CUDA call failed; message in ss_last_error() */
    SS_ERR_TIMEOUT = 4,      /* a bounded device wait gave up (ss_sort_status) */
    SS_ERR_UNSUPPORTED = 5,  /* a size beyond the documented limits */
    SS_ERR_DEVICE = 6        /* a device-side check failed (ss_sort_status) */
} ss_status;

/* flags of the ss_raster_* calls: optional outputs, each compiled
 * as its own kernel variant so that a disabled output costs no shared memory
 * or registers (the pattern of "从 8.6 KB 到 4.2 KB ...", section 最小改动:
 * optional per-pixel arrays sized by a compile-time constant). */
enum {
    SS_ACCUM_WEIGHT = 1u,  /* bwd: per-splat accumulated blend weight sum_p alpha T */
    SS_MEDIAN_DEPTH = 2u,  /* fwd: per-pixel depth of the last splat blended while T > 0.5 */
    SS_WEIGHT_STATS = 4u,  /* fwd: per-splat max blend weight and blending-pixel count
                              ("max wt" and, with the accumulated weight, the "Avg"
                              weight of the Spirula Studio write-up, 机制拆解 / 亲手验证) */
    SS_DISTORTION = 8u,    /* fwd: per-pixel depth distortion and its totals; bwd: its
                              gradient, including dL/ddepth (the write-up's distortion
                              option with per-pixel float4 totals, 最小改动) */
    SS_RECORDS_CLEARED = 16u  /* bwd only: the gradient records in the workspace were
                                 cleared by ss_raster_fwd_records (its bwd_workspace
                                 argument)
                                 and nothing wrote the workspace since; the backward
                                 then skips its own clearing pass */
};

/* Splats, structure of arrays, float32, device memory.  The pages' inputs:
 * per-splat 2D mean, conic (inverse 2D covariance), opacity, RGB and depth
 * ("Phase 5 step 30b", hotspot ranking: 9 gradient fields per splat). */
typedef struct {
    const float *mean2d;   /* [n][2] pixel coordinates */
    const float *conic;    /* [n][3] (a, b, c) of [[a, b], [b, c]] */
    const float *opacity;  /* [n] */
    const float *rgb;      /* [n][3] */
    const float *depth;    /* [n] > 0; sort key within a tile (front = small) */
    int32_t n;             /* 0 <= n < 2^31; pointers may be NULL when n == 0 */
} ss_splats;

/* Per-splat gradients of L, float32, device memory, same layouts as ss_splats.
 * db is the full partial derivative of L with respect to the stored b. */
typedef struct {
    float *dmean2d;        /* [n][2] */
    float *dconic;         /* [n][3] */
    float *dopacity;       /* [n] */
    float *drgb;           /* [n][3] */
    float *ddepth;         /* [n], only with SS_DISTORTION (else may be NULL) */
} ss_grads;

/* Version of this ABI (incremented on any change of a signature, or of the
 * meaning or size of an argument). */
int32_t ss_abi_version(void);

/* Host: the model's constants as the kernels use them:
 * out[0] = 1/255 (alpha floor), out[1] = 0.99 (alpha cap),
 * out[2] = 1e-4 (transmittance floor), out[3] = 16 (tile side). */
void ss_constants(float out[4]);

/* Host: message of the last failed call on this thread ("" if none).  The
 * string stays valid until the next ss_* call on the same thread. */
const char *ss_last_error(void);

/* Host: bytes of workspace that ss_sort_pairs (for n_pairs pairs on a W x H
 * image), ss_raster_bwd and ss_raster_bwd_records (for n_splats splats and
 * n_pairs pairs) need.  One buffer of this size serves all of them, in any
 * order on one stream.  Returns 0 if a size is out of range. */
size_t ss_workspace_bytes(int32_t n_splats, int64_t n_pairs, int32_t W, int32_t H);

/* Tile binning ("Phase 5 step 30b", emit_pairs: tile id computation and an
 * atomic counter).  For each splat that is not culled, one pair per tile of
 * the axis-aligned box of the ellipse where alpha >= 1/255 is possible,
 * {d : d^T conic d <= k}, k = 2 ln(255 opacity) widened by 2^-10 relative and
 * absolute, clipped to the image's tiles:
 *   keys[p] = tile << 32 | bits of depth (float32, > 0, so ordered as u32)
 *   vals[p] = splat index
 * A splat is culled (no pairs, counted) unless all its inputs are finite,
 * depth > 0, a > 0, c > 0, ac - b^2 > 0 and 1/255 <= opacity.
 * Pairs are written in no particular order (each CTA takes its slots from an
 * atomic counter); pairs beyond `capacity` are counted but not written.
 *   d_counters: device uint64[4], 8-byte aligned; set here, then
 *               [0] = pairs needed, [1] = culled splats,
 *               [2] / [3] = the smallest / largest float bits of the depth of
 *               a splat that has pairs (2^64 - 1 / 0 if no splat has any);
 *               ss_sort_pairs_dev reads [0], [2] and [3].
 *   keys, vals: device, `capacity` entries each (may be NULL if capacity 0).
 *   records: device, ss_record_bytes(n) bytes, 16-byte aligned; receives one
 *            64-byte record per splat (its position, base-2 exponent
 *            coefficients and threshold, opacity, depth, colour, index and a
 *            conservative pixel box), the form in which the rasterizers
 *            gather splats.  Opaque to the caller; valid while the splat
 *            inputs are unchanged.
 */
ss_status ss_bin_tiles(const ss_splats *splats, int32_t W, int32_t H, uint64_t *keys,
                       uint32_t *vals, int64_t capacity, uint64_t *d_counters, void *records,
                       ss_stream_t stream);

/* Host: bytes of the record buffer for n splats (64 n). */
size_t ss_record_bytes(int32_t n_splats);

/* Host: synchronizes `stream` and reads the counters of ss_bin_tiles.
 * *h_pairs = pairs needed, *h_culled = culled splats (either may be NULL).
 * Returns SS_ERR_CAPACITY if pairs needed > capacity (re-run ss_bin_tiles
 * with a capacity of at least *h_pairs). */
ss_status ss_pair_count(const uint64_t *d_counters, int64_t capacity, int64_t *h_pairs,
                        int64_t *h_culled, ss_stream_t stream);

/* Radix sort of the pairs by key, then by value within equal keys, in place
 * ("Phase 5 step 30b", radix_hist / radix_scatter; here a onesweep LSD sort
 * with decoupled look-back: one histogram pass, then one pass per 8-bit
 * digit of the 32 + ceil(log2 tiles) key bits), followed by the per-tile
 * ranges (extract_offsets):
 *   tile_offsets[t] = number of pairs whose tile is < t, t = 0..tiles;
 *   pairs of tile t are [tile_offsets[t], tile_offsets[t+1]), by ascending
 *   depth, ties by ascending splat index.
 *   keys, vals: device, n_pairs entries, sorted in place.
 *   tile_offsets: device uint32[tiles + 1].
 *   workspace: device, >= ss_workspace_bytes(0, n_pairs, W, H) bytes, 256-byte
 *   aligned; its contents need no initialisation.
 * 0 <= n_pairs < 2^32.  The look-back waits are bounded: a wait that gives up
 * records SS_ERR_TIMEOUT for ss_sort_status (the result is then invalid);
 * a key whose tile is >= tiles records SS_ERR_DEVICE. */
ss_status ss_sort_pairs(uint64_t *keys, uint32_t *vals, int64_t n_pairs, int32_t W, int32_t H,
                        uint32_t *tile_offsets, void *workspace, size_t workspace_bytes,
                        ss_stream_t stream);

/* ss_sort_pairs with the pair count read on the device: sorts
 * min(d_counters[0], capacity) pairs, where d_counters are the counters
 * ss_bin_tiles filled and capacity the size of keys / vals.  Nothing is read
 * back to the host, so bin -> sort -> forward -> backward can be enqueued
 * without a synchronisation (and captured in a CUDA graph); the grids are
 * sized for `capacity` and the surplus CTAs exit at once.  If the count
 * exceeded the capacity, ss_sort_status reports SS_ERR_CAPACITY (the first
 * `capacity` pairs were sorted; re-bin with a larger buffer).  The depth
 * range d_counters[2..3] lets the radix passes skip the depth bits that no
 * two pairs can differ in: the depth part is sorted as (bits - lo) on
 * max(16, ceil log2(hi - lo + 1)) bits, lo = d_counters[2] with its low 16
 * bits cleared (one 8-bit pass fewer for depths in [1, 100]); a key whose
 * depth bits are outside [lo, lo + 2^that) records SS_ERR_DEVICE.  The result
 * is the same order.  workspace: >= ss_workspace_bytes(0, capacity, W, H)
 * bytes. */
ss_status ss_sort_pairs_dev(uint64_t *keys, uint32_t *vals, const uint64_t *d_counters,
                            int64_t capacity, int32_t W, int32_t H, uint32_t *tile_offsets,
                            void *workspace, size_t workspace_bytes, ss_stream_t stream);

/* Host: synchronizes `stream` and returns SS_OK, SS_ERR_TIMEOUT,
 * SS_ERR_DEVICE or SS_ERR_CAPACITY for the last sort that used `workspace`. */
ss_status ss_sort_status(const void *workspace, ss_stream_t stream);

/* Forward rasterization ("Phase 5 step 30b", rasterize_f32) from the splats
 * themselves: as ss_raster_fwd_records (below), with each batch's records
 * computed from `splats` (the ones ss_bin_tiles would write, bit for bit)
 * and no blend masks, weight statistics or distortion (SS_WEIGHT_STATS and
 * SS_DISTORTION return SS_ERR_UNSUPPORTED; SS_MEDIAN_DEPTH is supported, the
 * other flags are ignored).
 *   splats: the splats ss_bin_tiles binned; vals, tile_offsets: the output of
 *   ss_sort_pairs for the same W, H.  Outputs as ss_raster_fwd_records. */
ss_status ss_raster_fwd(const ss_splats *splats, const uint32_t *vals, const uint32_t *tile_offsets,
                        int32_t W, int32_t H, const float *bg, uint32_t flags, float *image,
                        float *T_final, uint32_t *last_contrib, float *median_depth,
                        ss_stream_t stream);

/* Forward rasterization ("Phase 5 step 30b", rasterize_f32) on the records of
 * ss_bin_tiles: one CTA per 16x16 tile, one thread per pixel, the tile's
 * pairs staged in shared memory in batches; each pixel composites its tile's
 * splats front to back (model above).  Outputs (device, W x H each, planar):
 *   image[3][H][W]      color + T_final * bg
 *   T_final[H][W]       transmittance after the last blended splat (>= 1e-4)
 *   last_contrib[H][W]  1 + position in the tile's list of the last blended
 *                       splat, 0 if none (what the backward replays from)
 *   median_depth[H][W]  only with SS_MEDIAN_DEPTH (else may be NULL): depth
 *                       of the last splat blended while T > 0.5, 0 if none
 *   bg: HOST float[3] background, or NULL for black.
 *   distortion, dist_totals: only with SS_DISTORTION (else may be NULL):
 *                device float [H][W] and float4 [H][W] (16-byte aligned),
 *                overwritten with each pixel's depth distortion
 *                D = sum over pairs i < j of its blended splats of
 *                w_i w_j (z_i - z_j)^2 (w = alpha T, z = depth), and with the
 *                running totals (A = sum w, D1 = sum w z', D2 = sum w z'^2,
 *                z_ref), z' = z - z_ref, z_ref the first blended splat's depth,
 *                which the backward reads.
 *   max_weight, blend_count: only with SS_WEIGHT_STATS (else may be NULL):
 *                device float[n] / uint32[n], overwritten with, per splat, the
 *                maximum over pixels of alpha T and the number of pixels that
 *                blended it (average weight = accumulated weight / count).
 *   blend_masks: device uint32[8][n_pairs]; for each pair p the forward
 *                reached and each 8x4 pixel block b of p's tile
 *                (b = 2 (row / 4) + (column / 8) within the tile),
 *                blend_masks[b * n_pairs + p] has bit i set iff pixel
 *                (column 8 (b & 1) + (i & 7), row 4 (b >> 1) + (i >> 3)) blended
 *                the splat.  The backward replays exactly these decisions.
 *                Entries past the point where every pixel of a block stopped
 *                are left unwritten.
 *   records, n_splats: the records ss_bin_tiles wrote for these splats.
 *   vals, tile_offsets: the output of ss_sort_pairs for the same W, H.
 *   n_pairs: the stride of blend_masks and a bound on the pairs sorted: the
 *            pair count, or the capacity when the count stayed on the device
 *            (ss_sort_pairs_dev).  The backward must get the same value.
 *   bwd_workspace, bwd_workspace_bytes: optional (NULL: unused).  The
 *            workspace the following ss_raster_bwd_records gets (256-byte aligned,
 *            >= ss_workspace_bytes(n_splats, 0, W, H) bytes): the forward's
 *            CTAs then also clear the backward's per-splat gradient records
 *            in it (a few stores a thread, hidden under the compositing),
 *            and that ss_raster_bwd_records call, given SS_RECORDS_CLEARED, skips its
 *            separate clearing pass.  No call may write the workspace in
 *            between (ss_sort_pairs uses the same bytes).
 * Pair values >= n_splats are ignored. */
ss_status ss_raster_fwd_records(const void *records, int32_t n_splats, const uint32_t *vals,
                                const uint32_t *tile_offsets, int64_t n_pairs, int32_t W,
                                int32_t H, const float *bg, uint32_t flags, float *image,
                                float *T_final, uint32_t *last_contrib, float *median_depth,
                                uint32_t *blend_masks, float *max_weight, uint32_t *blend_count,
                                float *distortion, float *dist_totals, void *bwd_workspace,
                                size_t bwd_workspace_bytes, ss_stream_t stream);

/* Backward rasterization from the splats themselves ("Phase 5 step 30b",
 * rasterize_backwards; conclusion: each thread computes its own (pixel,
 * splat) term and the warp sums them before one atomic): the inputs are
 * the splats, their sorted pairs and tile ranges, the forward's T_final and
 * last_contrib and dL/dimage.  The records are built into the workspace
 * (those ss_bin_tiles would write), the forward's blend decisions are
 * re-evaluated from them (a pixel blended list position j iff j <
 * last_contrib and alpha >= 1/255, the forward's own test on the same
 * float32 values), and then the gradients follow as in
 * ss_raster_bwd_records.
 *   flags: SS_ACCUM_WEIGHT as there; SS_DISTORTION returns
 *   SS_ERR_UNSUPPORTED (its totals are an input of ss_raster_bwd_records);
 *   SS_RECORDS_CLEARED returns SS_ERR_INVALID_ARG; the rest are ignored.
 *   grads, accum_weight: as ss_raster_bwd_records (overwritten).
 *   workspace: 256-byte aligned, at least ss_workspace_bytes(n, n_pairs, W, H)
 *   bytes for n_pairs = tile_offsets[tiles] (the list length, known here
 *   only on the device): the blend masks take 32 bytes a pair after the
 *   records, and a list longer than the workspace holds makes
 *   ss_sort_status(workspace) return SS_ERR_CAPACITY (the gradients are then
 *   invalid); bits this call sets add to the status word of the last sort.
 *   bg: HOST float[3] or NULL (must match the forward call). */
ss_status ss_raster_bwd(const ss_splats *splats, const uint32_t *vals, const uint32_t *tile_offsets,
                        int32_t W, int32_t H, const float *bg, uint32_t flags,
                        const float *T_final, const uint32_t *last_contrib,
                        const float *dL_dimage, const ss_grads *grads, float *accum_weight,
                        void *workspace, size_t workspace_bytes, ss_stream_t stream);

/* Backward rasterization on the records of ss_bin_tiles ("从 8.6 KB 到 4.2 KB
 * ...", rasterize_bwd_2d on the 2D screen-space path; "Phase 5 step 30b",
 * rasterize_backwards: the 9-field per-splat gradient).  Each pixel walks its tile's list back to front from
 * last_contrib, recovering T before each blended splat as T / (1 - alpha),
 * and adds, for L = sum dL/dimage * image:
 *   dL/drgb += g w,  w = alpha T
 *   dL/dalpha = sum_c g_c (rgb_c T - (S_c + T_final bg_c) / (1 - alpha)),
 *     S = sum of rgb w over the splats blended after this one
 *   dL/dopacity += G dL/dalpha; dL/dsigma = -alpha dL/dalpha
 *   dL/dmean += dL/dsigma (-(a dx + b dy), -(b dx + c dy))
 *   dL/dconic += dL/dsigma (dx^2 / 2, dx dy, dy^2 / 2)
 * (through the 0.99 cap alpha has zero derivative).  The per-pixel terms of
 * a splat are summed over each 8x4 pixel block before any atomic
 * ("Phase 5 step 30b", conclusion: reduce within the warp, then one atomic
 * per warp instead of per thread); here the block's pixels store
 * (dL/dsigma, alpha T) in shared memory and are summed into moments from
 * which all fields follow, then added with four vector reductions per
 * (block, splat) into a per-splat record in the workspace.
 *   records, n_splats: the records ss_bin_tiles wrote for these splats.
 *   T_final, last_contrib, blend_masks: from ss_raster_fwd_records with the
 *   same inputs (the blend decisions are the forward's, not re-evaluated).
 *   blend_masks may be NULL: the decisions are then re-evaluated as in
 *   ss_raster_bwd, into the workspace, which must then hold
 *   ss_workspace_bytes(n_splats, n_pairs, W, H) bytes.
 *   dL_dimage: device float[3][H][W].
 *   dist_totals, dL_ddist: only with SS_DISTORTION (else may be NULL): the
 *   forward's totals and the upstream gradient of its distortion image,
 *   device float [H][W]; L then also has the term sum dL/ddist * D, which
 *   adds, with E_k = dD/dw_k = sum_j w_j (z_k - z_j)^2,
 *     dL/dalpha_k += dL/ddist (E_k T_k - sum_{i after k} w_i E_i / (1 - alpha_k))
 *     dL/ddepth_k  = dL/ddist 2 w_k sum_j w_j (z_k - z_j)   (grads->ddepth).
 *   grads: the four 2D arrays required (and ddepth with SS_DISTORTION);
 *   overwritten (zeroed here first).
 *   accum_weight: with SS_ACCUM_WEIGHT, device float[n] overwritten with
 *   sum over pixels of alpha T (summed exactly in 32.32 fixed point, so the
 *   result does not depend on the order of the atomics); else may be NULL.
 *   workspace: >= ss_workspace_bytes(n, 0, W, H) bytes (48 per splat + 256),
 *   256-byte aligned; required whenever n > 0.  Its gradient records are
 *   cleared here first, unless flags has SS_RECORDS_CLEARED (the forward
 *   cleared them; see ss_raster_fwd_records' bwd_workspace).
 *   bg: HOST float[3] or NULL (must match the forward call). */
ss_status ss_raster_bwd_records(const void *records, int32_t n_splats, const uint32_t *vals,
                                const uint32_t *tile_offsets, int64_t n_pairs, int32_t W,
                                int32_t H, const float *bg, uint32_t flags, const float *T_final,
                                const uint32_t *last_contrib, const uint32_t *blend_masks,
                                const float *dL_dimage, const float *dist_totals,
                                const float *dL_ddist, const ss_grads *grads,
                                float *accum_weight, void *workspace, size_t workspace_bytes,
                                ss_stream_t stream);

/* The backward pass for callers that cannot allocate (the pages have no
 * counterpart: this is a property of the library, not of the method).
 * Some callers may not call cudaMalloc and cannot provide a workspace: a
 * plugin inside an application that owns all device memory through its own
 * pool, or a real-time thread that must not risk the device-wide
 * synchronisation cudaMalloc / cudaFree can cause.  This entry point
 * computes exactly what ss_raster_bwd_records computes, with the same arguments
 * minus the workspace, and calls no allocator: the accumulated-weight
 * scratch (8 bytes per splat) is a fixed array inside the library,
 * 2,097,152 splats (16 MiB), which every GPU that loads the library holds
 * until the process exits.
 *   - n_splats > 2,097,152 returns SS_ERR_UNSUPPORTED (use ss_raster_bwd_records).
 *   - SS_DISTORTION returns SS_ERR_UNSUPPORTED (use ss_raster_bwd_records).
 *   - SS_RECORDS_CLEARED is accepted and ignored (this call keeps no
 *     gradient records; it always clears its outputs first).
 *   - The first call in a CUDA context on a device, made with that device
 *     current, looks up the array's device address (cudaGetSymbolAddress)
 *     and caches it under the context's id; a call in another context
 *     (another driver-API context, or the primary context re-created after
 *     cudaDeviceReset) looks it up again.  Make that first call before any
 *     stream capture: a first call on a capturing stream returns
 *     SS_ERR_UNSUPPORTED without touching the capture.
 *   - All calls share the array.  Each call clears the part it uses, but
 *     calls that overlap on the GPU (other streams, other host threads) race
 *     on it: serialise them. */
ss_status ss_raster_bwd_noalloc(const void *records, int32_t n_splats, const uint32_t *vals,
                                const uint32_t *tile_offsets, int64_t n_pairs, int32_t W,
                                int32_t H, const float *bg, uint32_t flags, const float *T_final,
                                const uint32_t *last_contrib, const uint32_t *blend_masks,
                                const float *dL_dimage, const ss_grads *grads,
                                float *accum_weight, ss_stream_t stream);

/* Device-side bounds checks (a build variant, not part of the method).  A
 * library built with -DSS_DEBUG_BOUNDS (gaussian_splatting_differentiable_gb300/
 * build.py --debug-bounds, libss_debug.so) checks, in its kernels, that tile
 * lists lie inside the pairs, that a last_contrib does not reach past its
 * tile's list, that gradient-record indices lie inside the splats and that
 * the sort's ranks and destinations lie inside their ranges; a failed check
 * sets a bit in a device error word and skips or clamps the access it
 * guards -- nothing traps.
 * ss_debug_bounds_enabled: 1 in that build, 0 in the normal one.
 * ss_debug_status: synchronizes `stream`, reads and clears the error word:
 * SS_OK, or SS_ERR_DEVICE with the failed checks' bits in the message (the
 * normal build never sets any). */
int32_t ss_debug_bounds_enabled(void);
ss_status ss_debug_status(ss_stream_t stream);

/* Per-kernel timing ("从 8.6 KB 到 4.2 KB ...", section 亲手验证: SS_PROFILE=1
 * gives per-kernel segment timings).  Off unless the environment has
 * SS_PROFILE=1 when the library loads or ss_profile_enable(1) is called.
 * When on, each kernel launch is bracketed by two CUDA events on its own
 * stream (host-side cost only; nothing is added to the kernels). */
void ss_profile_enable(int32_t on);

/* Host: waits for the events recorded since the last collect and writes one
 * line per kernel name, "name launches total_ms min_ms max_ms\n", into
 * buf[0..len) (NUL-terminated, truncated if short; buf may be NULL).
 * The records are consumed by the call, with or without a buffer.
 * Returns the full length of the text. */
int64_t ss_profile_collect(char *buf, size_t len);

/* Measurement helper, not part of the path: `rounds` rounds of float atomic
 * adds (red.global.add.f32), one per thread per round, into buf[0..n)
 * (device, n >= 1) with consecutive threads on consecutive addresses.  Timed
 * by the caller, it gives the L2 atomic throughput that bounds the backward
 * pass's gradient accumulation. */
ss_status ss_probe_red_f32(float *buf, int64_t n, int32_t rounds, ss_stream_t stream);

/* Test hook for failure detection, not part of the path: runs one onesweep
 * pass CTA whose look-back waits on a partition that never publishes, so
 * the bounded wait gives up (after roughly 0.2-0.5 s); ss_sort_status on the
 * same workspace then returns SS_ERR_TIMEOUT and the CUDA context stays
 * usable.  workspace: >= ss_workspace_bytes(0, 8192, 16, 16) bytes, 256-byte
 * aligned; its contents are overwritten. */
ss_status ss_test_sort_wait_timeout(void *workspace, size_t workspace_bytes, ss_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SS_H */
