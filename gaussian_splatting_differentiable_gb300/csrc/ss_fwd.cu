// Forward rasterization ("Phase 5 step 30b -- kernel-by-kernel timing",
// rasterize_f32; "从 8.6 KB 到 4.2 KB ...", raster fwd).
//
// One 256-thread CTA per 16x16 tile, one thread per pixel; warp w covers the
// 8x4 pixel block (8 (w & 1), 4 (w >> 1)) of the tile.  The tile's list is
// walked front to back in batches of 256 splats.  Each batch's 64-byte
// splat records are copied into shared memory with cp.async while the
// previous batch is composited (two buffers; the pair indices are read one
// batch further ahead), then each warp compacts the batch to the splats
// whose conservative box reaches its 8x4 block and each pixel composites
// that short list.  A pixel stops at the first splat whose blend would take
// T below 1e-4; the CTA stops once all its pixels have.  The median-depth
// output is a template variant, so the default variant does no median work.
//
// With SS_WEIGHT_STATS (the STATS variant) the warp also takes, per splat
// that any of its pixels blended, the maximum blend weight alpha T (a warp
// max of the float bits, which order like the values for w >= 0) and the
// number of blending pixels (the mask's popcount); the CTA's warps combine
// them in shared memory per batch entry, and when the batch is done one
// atomicMax and one atomicAdd per (tile, splat) go to the splat.
//
// With SS_DISTORTION (the DIST variant) each pixel also keeps running totals
// of its blended splats' weights and depths, A = sum w, D1 = sum w z',
// D2 = sum w z'^2, with z' = z - z_ref the depth relative to the first
// blended splat (the distortion does not change when every depth shifts, and
// the shift keeps the float32 terms small), and adds w (z'^2 A - 2 z' D1 + D2)
// -- the new splat's pairs with every splat in front -- to its depth
// distortion sum_{i<j} w_i w_j (z_i - z_j)^2.  It writes the distortion and
// the totals (A, D1, D2, z_ref), which the backward reads.
//
// The warp also records, for each pair it reached, which of its 32 pixels
// blended the splat (a ballot): blend_masks[b * n_pairs + p], b = warp.
// The backward reads these decisions instead of re-evaluating every
// (pixel, splat) of the list, and they are by construction exactly the
// forward's.
#include "ss_device.cuh"
#include "ss_internal.h"
#include "ss_profile.h"

namespace ss {

// Kept at 128 bytes: on sm_103a this kernel ran 8 % slower with a 136-byte
// parameter block than with a 128-byte one holding the same fields it reads
// (measured; the tile-column count is recomputed from W to stay inside).
struct FwdParams {
    const SplatRecord *recs;
    const uint32_t *vals;
    const uint32_t *offs;
    uint32_t *masks;   // [8][n_pairs]
    float *image;
    float *T_final;
    uint32_t *last;
    float *median;
    uint32_t *max_w_bits;  // [n] float bits of the max blend weight (STATS)
    uint32_t *count;       // [n] blending pixels (STATS)
    float *dist;           // [H][W] depth distortion (DIST)
    float4 *dist_totals;   // [H][W] (A, D1, D2, z_ref) (DIST)
    float4 *clear;         // the backward's gradient records to clear (3 n float4), or null
    uint32_t n_pairs;      // < 2^32 (checked on the host)
    int32_t n;
    uint16_t W, H;         // <= 32768 (checked on the host)
    float bg[3];
};
static_assert(sizeof(FwdParams) <= 128, "kernel parameters over 128 bytes run slower");

// The forward's body.  SOA: the splats come as the SoA inputs instead of
// the binning's records -- each batch's records are computed on the fly
// (record_of: the same bits the binning writes) and stored into shared
// memory -- and no blend masks are written (the entry point that takes the
// splats themselves has no mask buffer).
template <bool MEDIAN, bool STATS, bool DIST, bool SOA>
__device__ __forceinline__ void raster_fwd(const FwdParams &p, const SplatPtrs &soa) {
    __shared__ SplatGeo s_geo[2][256];
    __shared__ SplatGeo2 s_geo2[2][256];
    __shared__ SplatCol s_col[2][256];
    __shared__ SplatBox s_box[2][256];
    __shared__ uint8_t s_list[8][256];
    __shared__ uint32_t s_mask[8][256];
    // STATS: per-batch statistics of the batch's 256 entries (by buffer
    // parity), summed over the CTA's warps with shared atomics and sent to
    // the splats once per (tile, splat) when the batch is done.
    __shared__ uint32_t s_smax[STATS ? 2 : 1][STATS ? 256 : 1];
    __shared__ uint32_t s_scnt[STATS ? 2 : 1][STATS ? 256 : 1];

    const int tid = threadIdx.x;
    const int tile = blockIdx.x;
    const int ntx = (p.W + kTile - 1) / kTile;
    const int tx = tile % ntx, ty = tile / ntx;
    const int warp = tid >> 5, lane = tid & 31;
    const int bx = tx * kTile + ((warp & 1) << 3), by = ty * kTile + ((warp >> 1) << 2);
    const int x = bx + (lane & 7), y = by + (lane >> 3);
    const bool inside = x < p.W && y < p.H;
    const float px = float(x) + 0.5f, py = float(y) + 0.5f;
    const float wx0 = float(bx) + 0.5f, wx1 = wx0 + 7.0f;
    const float wy0 = float(by) + 0.5f, wy1 = wy0 + 3.0f;
    uint32_t start = p.offs[tile], end = p.offs[tile + 1];
    if (!SOA && SS_BAD(end < start || end > p.n_pairs, kDbgFwdList)) start = end = 0u;
    const uint32_t lt = lanemask_lt();

    if (STATS) {
        s_smax[0][tid] = 0u, s_smax[1][tid] = 0u;
        s_scnt[0][tid] = 0u, s_scnt[1][tid] = 0u;
    }
    // The backward's gradient records, cleared here when the caller asks (a
    // few 16-byte stores a thread, hidden under this kernel's arithmetic,
    // instead of a separate bandwidth-bound pass before the backward).
    if (p.clear) {
        const int64_t n4 = 3 * int64_t(p.n), stride = int64_t(gridDim.x) * 256;
        for (int64_t i = int64_t(tile) * 256 + tid; i < n4; i += stride)
            p.clear[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // STATS: thread t sends entry t of a finished batch (buffer b, nb entries)
    // and clears its slots; each thread reads only its own record slot, which
    // only its own prefetch overwrites afterwards.
    auto flush_stats = [&](int b, int nb) {
        if (STATS && tid < nb && s_scnt[b][tid]) {
            const uint32_t idx = s_col[b][tid].idx;
            atomicMax(p.max_w_bits + idx, s_smax[b][tid]);
            atomicAdd(p.count + idx, s_scnt[b][tid]);
            s_smax[b][tid] = 0u;
            s_scnt[b][tid] = 0u;
        }
    };
    int prev_nb = 0;

    float T = 1.0f, cr = 0.0f, cg = 0.0f, cb = 0.0f, med = 0.0f;
    float dA = 0.0f, dD1 = 0.0f, dD2 = 0.0f, dD = 0.0f, zref = 0.0f;
    uint32_t last = 0;
    bool done = !inside;

    const int nty = (p.H + kTile - 1) / kTile;
    // Record idx into slot t of buffer b: an asynchronous copy of the
    // binning's record, or (SOA) the record computed here.
    auto stage = [&](uint32_t idx, int b, int t) {
        if (SOA) {
            const SplatRecord r =
                idx < uint32_t(soa.n) ? record_of(soa, idx, ntx, nty) : invisible_record();
            s_geo[b][t] = r.geo;
            s_geo2[b][t] = r.geo2;
            s_col[b][t] = r.col;
            s_box[b][t] = r.box;
        } else {
            stage_record_async(p.recs, idx, p.n, s_geo[b], s_geo2[b], s_col[b], s_box[b], t);
        }
    };

    // Batch b covers list positions [start + 256 b, min(end, start + 256 (b + 1))).
    if (start < end) {
        if (uint32_t(tid) < end - start) stage(p.vals[start + tid], 0, tid);
        cp_async_commit();
    }
    uint32_t next_idx = start + 256u + uint32_t(tid) < end ? p.vals[start + 256u + tid] : 0u;
    int buf = 0;
    for (uint32_t base = start; base < end; base += 256, buf ^= 1) {
        cp_async_wait<0>();
        if (__syncthreads_count(!done) == 0) break;
        flush_stats(buf ^ 1, prev_nb);   // the previous batch, before its buffer is refilled
        // Prefetch the next batch into the other buffer (free: every thread
        // has passed the barrier, so nobody still reads the batch before).
        const uint32_t nbase = base + 256;
        if (nbase < end) {
            if (nbase + uint32_t(tid) < end) stage(next_idx, buf ^ 1, tid);
            cp_async_commit();
            next_idx = nbase + 256u + uint32_t(tid) < end ? p.vals[nbase + 256u + tid] : 0u;
        }
        const int nb = int(min(256u, end - base));
        prev_nb = nb;
        if (!__any_sync(0xffffffffu, !done)) continue;
        int cnt = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int j = q * 32 + lane;
            bool hit = false;
            if (j < nb) {
                const SplatBox b = s_box[buf][j];
                hit = b.x0 <= wx1 && b.x1 >= wx0 && b.y0 <= wy1 && b.y1 >= wy0;
            }
            const uint32_t m = __ballot_sync(0xffffffffu, hit);
            if (hit) s_list[warp][cnt + __popc(m & lt)] = uint8_t(j);
            cnt += __popc(m);
        }
        if (!SOA)
            for (int k = lane; k < nb; k += 32) s_mask[warp][k] = 0u;
        __syncwarp();
        for (int q = 0; q < cnt; ++q) {
            const int j = s_list[warp][q];
            const SplatGeo g = s_geo[buf][j];
            const SplatGeo2 g2 = s_geo2[buf][j];
            float dx, dy;
            const float e2 = eval_e2(g, g2.C, px, py, dx, dy);
            float oG;
            const float alpha = eval_alpha(g2.o, ex2_approx(e2), oG);
            const float Tn = __fmul_rn(T, __fsub_rn(1.0f, alpha));
            // skipped where alpha < 1/255 (e2 < thr; false for NaN too)
            const bool cand = !done && e2 >= g2.thr;
            const bool stop = cand && Tn < kTEps;
            const bool blend = cand && !stop;
            done = done || stop;
            // The evaluation runs on every lane and the decisions are
            // predicates (measured 7 % faster than branching on them).
            float wblend = 0.0f;
            if (blend) {
                const SplatCol c = s_col[buf][j];
                const float w = alpha * T;
                wblend = w;
                cr = fmaf(c.r, w, cr);
                cg = fmaf(c.g, w, cg);
                cb = fmaf(c.b, w, cb);
                if (MEDIAN && T > 0.5f) med = g2.depth;
                if (DIST) {
                    if (dA == 0.0f) zref = g2.depth;   // first blend: w > 0 always
                    const float z = g2.depth - zref;
                    dD = fmaf(w, fmaf(z, fmaf(z, dA, -2.0f * dD1), dD2), dD);
                    dA += w;
                    dD1 = fmaf(w, z, dD1);
                    dD2 = fmaf(w * z, z, dD2);
                }
                T = Tn;
                last = base - start + uint32_t(j) + 1u;
            }
            const uint32_t m = __ballot_sync(0xffffffffu, blend);
            if (!SOA && lane == 0) s_mask[warp][j] = m;
            if (STATS && m) {
                const uint32_t wmax = __reduce_max_sync(0xffffffffu, __float_as_uint(wblend));
                if (lane == 0) {
                    atomicMax(&s_smax[buf][j], wmax);
                    atomicAdd(&s_scnt[buf][j], uint32_t(__popc(m)));
                }
            }
            // No per-entry exit once every pixel of the warp is done (the
            // batch and CTA checks above end the work): the vote cost more
            // than the entries it saved (measured 0.496 vs 0.470 ms on the
            // 2M-splat scene, 0.520 vs 0.498 ms with the four dense blobs).
        }
        __syncwarp();
        if (!SOA) {
            uint32_t *gm = p.masks + size_t(warp) * size_t(p.n_pairs) + base;
            for (int k = lane; k < nb; k += 32)
                if (base + uint32_t(k) < p.n_pairs) gm[k] = s_mask[warp][k];
        }
    }
    cp_async_wait<0>();  // no copy may outlive the CTA
    if (STATS) {
        __syncthreads();                 // every warp is done with the last batch
        flush_stats(buf ^ 1, prev_nb);   // (the loop toggled buf past it)
    }
    if (inside) {
        const size_t HW = size_t(p.W) * p.H, pix = size_t(y) * p.W + x;
        p.image[pix] = fmaf(T, p.bg[0], cr);
        p.image[HW + pix] = fmaf(T, p.bg[1], cg);
        p.image[2 * HW + pix] = fmaf(T, p.bg[2], cb);
        p.T_final[pix] = T;
        p.last[pix] = last;
        if (MEDIAN) p.median[pix] = med;
        if (DIST) {
            p.dist[pix] = dD;
            p.dist_totals[pix] = make_float4(dA, dD1, dD2, zref);
        }
    }
}

// A minimum of CTAs a SM only where it measured faster: five for the plain
// variant (48 registers, ~3 µs at 2M splats), four for the distortion one
// (62 registers); the statistics and median variants ran slower bounded
// (0.585 vs 0.567 and 0.517 vs 0.513 ms) and keep the compiler's choice.
template <bool MEDIAN, bool STATS, bool DIST>
__global__ void __launch_bounds__(256, (!MEDIAN && !STATS && !DIST) ? 5 : (DIST && !STATS && !MEDIAN) ? 4 : 0)
k_raster_fwd(FwdParams p) {
    raster_fwd<MEDIAN, STATS, DIST, false>(p, SplatPtrs{});
}

// The forward from the SoA splats (ss_raster_fwd): records computed per
// batch, no blend masks.
template <bool MEDIAN>
__global__ void __launch_bounds__(256) k_raster_fwd_splats(FwdParams p, SplatPtrs s) {
    raster_fwd<MEDIAN, false, false, true>(p, s);
}

template <bool MEDIAN, bool STATS, bool DIST>
static void launch_fwd(const FwdParams &p, int grid, cudaStream_t st) {
    SS_LAUNCH("k_raster_fwd", st, (k_raster_fwd<MEDIAN, STATS, DIST><<<grid, 256, 0, st>>>(p)));
}

}  // namespace ss

using namespace ss;

extern "C" ss_status ss_raster_fwd_records(const void *records, int32_t n_splats,
                                           const uint32_t *vals, const uint32_t *tile_offsets,
                                           int64_t n_pairs, int32_t W, int32_t H, const float *bg,
                                           uint32_t flags, float *image, float *T_final,
                                           uint32_t *last_contrib, float *median_depth,
                                           uint32_t *blend_masks, float *max_weight,
                                           uint32_t *blend_count, float *distortion,
                                           float *dist_totals, void *bwd_workspace,
                                           size_t bwd_workspace_bytes, ss_stream_t stream) {
    clear_error();
    if (W < 1 || H < 1 || W > kMaxSide || H > kMaxSide)
        return fail(SS_ERR_UNSUPPORTED, "ss_raster_fwd_records: image %dx%d outside 1..%d", W, H, kMaxSide);
    if (flags & ~uint32_t(SS_ACCUM_WEIGHT | SS_MEDIAN_DEPTH | SS_WEIGHT_STATS | SS_DISTORTION))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd_records: unknown flag bits 0x%x", flags);
    const bool dist = flags & SS_DISTORTION;
    if (dist && (!distortion || !dist_totals))
        return fail(SS_ERR_INVALID_ARG,
                    "ss_raster_fwd_records: SS_DISTORTION set but distortion / dist_totals NULL");
    if (dist && (reinterpret_cast<uintptr_t>(dist_totals) & 15))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd_records: dist_totals not 16-byte aligned");
    const bool stats = flags & SS_WEIGHT_STATS;
    if (stats && n_splats > 0 && (!max_weight || !blend_count))
        return fail(SS_ERR_INVALID_ARG,
                    "ss_raster_fwd_records: SS_WEIGHT_STATS set but max_weight / blend_count NULL");
    if (n_splats < 0) return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd_records: n_splats < 0");
    if (n_splats > 0 && !records) return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd_records: records is NULL");
    if (reinterpret_cast<uintptr_t>(records) & 15)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd_records: records not 16-byte aligned");
    if (!vals || !tile_offsets) return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd_records: vals/offsets NULL");
    if (!image || !T_final || !last_contrib)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd_records: an output is NULL");
    if (n_pairs < 0 || n_pairs > int64_t(0xffffffffu))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd_records: n_pairs outside 0..2^32-1");
    if (n_pairs > 0 && !blend_masks)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd_records: blend_masks is NULL");
    const bool median = flags & SS_MEDIAN_DEPTH;
    if (median && !median_depth)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd_records: SS_MEDIAN_DEPTH set but median_depth NULL");
    if (bwd_workspace) {
        if (reinterpret_cast<uintptr_t>(bwd_workspace) & 255)
            return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd_records: bwd_workspace not 256-byte aligned");
        const size_t need = ws_layout(n_splats, 0, W, H).bwd_end;
        if (bwd_workspace_bytes < need)
            return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd_records: bwd_workspace %zu bytes < %zu needed",
                        bwd_workspace_bytes, need);
    }
    FwdParams p{};
    p.recs = static_cast<const SplatRecord *>(records);
    p.n = n_splats;
    p.vals = vals;
    p.offs = tile_offsets;
    p.W = uint16_t(W);
    p.H = uint16_t(H);
    for (int c = 0; c < 3; ++c) p.bg[c] = bg ? bg[c] : 0.0f;
    p.image = image;
    p.T_final = T_final;
    p.last = last_contrib;
    p.median = median_depth;
    p.masks = blend_masks;
    p.n_pairs = uint32_t(n_pairs);
    p.max_w_bits = reinterpret_cast<uint32_t *>(max_weight);
    p.count = blend_count;
    p.dist = distortion;
    p.dist_totals = reinterpret_cast<float4 *>(dist_totals);
    p.clear = bwd_workspace ? reinterpret_cast<float4 *>(static_cast<unsigned char *>(bwd_workspace) +
                                                         ws_layout(n_splats, 0, W, H).accum)
                            : nullptr;
    const int grid = tiles_x(W) * tiles_y(H);
    cudaStream_t st = (cudaStream_t)stream;
    if (stats && n_splats > 0) {
        ss_status s = check_cuda(cudaMemsetAsync(max_weight, 0, size_t(n_splats) * 4, st),
                                 "ss_raster_fwd_records: memset");
        if (s == SS_OK)
            s = check_cuda(cudaMemsetAsync(blend_count, 0, size_t(n_splats) * 4, st),
                           "ss_raster_fwd_records: memset");
        if (s != SS_OK) return s;
    }
    switch ((median ? 4 : 0) | (stats ? 2 : 0) | (dist ? 1 : 0)) {
        case 0: launch_fwd<false, false, false>(p, grid, st); break;
        case 1: launch_fwd<false, false, true>(p, grid, st); break;
        case 2: launch_fwd<false, true, false>(p, grid, st); break;
        case 3: launch_fwd<false, true, true>(p, grid, st); break;
        case 4: launch_fwd<true, false, false>(p, grid, st); break;
        case 5: launch_fwd<true, false, true>(p, grid, st); break;
        case 6: launch_fwd<true, true, false>(p, grid, st); break;
        default: launch_fwd<true, true, true>(p, grid, st); break;
    }
    return check_launch("ss_raster_fwd_records");
}

extern "C" ss_status ss_raster_fwd(const ss_splats *splats, const uint32_t *vals,
                                   const uint32_t *tile_offsets, int32_t W, int32_t H,
                                   const float *bg, uint32_t flags, float *image, float *T_final,
                                   uint32_t *last_contrib, float *median_depth,
                                   ss_stream_t stream) {
    clear_error();
    if (!splats) return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd: splats is NULL");
    if (W < 1 || H < 1 || W > kMaxSide || H > kMaxSide)
        return fail(SS_ERR_UNSUPPORTED, "ss_raster_fwd: image %dx%d outside 1..%d", W, H, kMaxSide);
    if (flags & ~uint32_t(SS_ACCUM_WEIGHT | SS_MEDIAN_DEPTH | SS_WEIGHT_STATS | SS_DISTORTION |
                          SS_RECORDS_CLEARED))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd: unknown flag bits 0x%x", flags);
    if (flags & (SS_WEIGHT_STATS | SS_DISTORTION))
        return fail(SS_ERR_UNSUPPORTED,
                    "ss_raster_fwd: the weight statistics and the distortion need their output "
                    "buffers: use ss_raster_fwd_records");
    const int32_t n = splats->n;
    if (n < 0) return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd: n < 0");
    if (n > 0 && (!splats->mean2d || !splats->conic || !splats->opacity || !splats->rgb ||
                  !splats->depth))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd: a splat array is NULL");
    if (n > 0 && (reinterpret_cast<uintptr_t>(splats->mean2d) & 7))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd: mean2d not 8-byte aligned");
    if (!vals || !tile_offsets) return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd: vals/offsets NULL");
    if (!image || !T_final || !last_contrib)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd: an output is NULL");
    const bool median = flags & SS_MEDIAN_DEPTH;
    if (median && !median_depth)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_fwd: SS_MEDIAN_DEPTH set but median_depth NULL");
    FwdParams p{};
    p.recs = nullptr;
    p.n = n;
    p.vals = vals;
    p.offs = tile_offsets;
    p.W = uint16_t(W);
    p.H = uint16_t(H);
    for (int c = 0; c < 3; ++c) p.bg[c] = bg ? bg[c] : 0.0f;
    p.image = image;
    p.T_final = T_final;
    p.last = last_contrib;
    p.median = median_depth;
    const SplatPtrs sp{splats->mean2d, splats->conic, splats->opacity, splats->rgb, splats->depth,
                       n};
    const int grid = tiles_x(W) * tiles_y(H);
    cudaStream_t st = (cudaStream_t)stream;
    if (median)
        SS_LAUNCH("k_raster_fwd_splats", st, (k_raster_fwd_splats<true><<<grid, 256, 0, st>>>(p, sp)));
    else
        SS_LAUNCH("k_raster_fwd_splats", st, (k_raster_fwd_splats<false><<<grid, 256, 0, st>>>(p, sp)));
    return check_launch("ss_raster_fwd");
}

namespace ss {
cudaError_t debug_word_fwd(uint32_t *out) { return read_and_clear_debug_word(out); }
}  // namespace ss
