// Backward rasterization ("从 8.6 KB 到 4.2 KB ...", rasterize_bwd_2d, the
// 2D screen-space backward; "Phase 5 step 30b -- kernel-by-kernel timing",
// rasterize_backwards: 52 % of the step, bound by per-pixel float atomics
// on the 9 gradient fields of every splat).
//
// Same CTA/tile and warp/8x4-block layout as the forward.  Each pixel starts
// from its forward state (T_final, last_contrib) and walks its tile's list
// back to front in batches of 256 staged splats, recovering the
// transmittance in front of each blended splat as T / (1 - alpha) and
// keeping the colour S of what lies behind it; the blend decision is the
// forward's own (same staging and exponent functions), so exactly the
// forward's splats are revisited.
//
// Reduction.  The pages' baseline issues 9 atomics per (pixel, splat); their
// proposed fix sums each field across the warp first and issues one atomic
// per warp ("Phase 5 step 30b", conclusion).  Here the warp's 10 fields
// (9 gradients + the accumulated weight) are reduced together by a
// reduce-scatter butterfly: at each of the 5 xor steps every lane keeps half
// of its remaining fields and trades the other half with its partner, so
// 5 + 3 + 2 + 1 + 1 = 12 shuffles (instead of 10 x 5 = 50) leave each field's
// warp total in one even lane; those 10 lanes then issue the warp's atomics
// as one instruction.  Warps where no pixel blends the splat skip all of it
// (a warp vote).  The accumulated weight is summed in 32.32 fixed point with
// 64-bit integer atomics, so it is exact and independent of atomic order.
#include "ss_device.cuh"
#include "ss_internal.h"
#include "ss_profile.h"

namespace ss {

struct BwdParams {
    SplatPtrs s;
    const uint32_t *vals;
    const uint32_t *offs;
    int32_t W, H, tiles_x;
    float bg[3];
    const float *T_final;
    const uint32_t *last;
    const float *dL;
    float *dmean2d, *dconic, *dopacity, *drgb;
    unsigned long long *accum;  // 32.32 fixed point
};

// One butterfly step of the reduce-scatter: N values, lanes with `hi` set
// keep the upper half, the others the lower half (zero-padded), each adding
// its partner's copy of the kept half.  Result in v[0 .. (N+1)/2).
template <int N>
__device__ __forceinline__ void rs_step(float *v, int off, bool hi) {
    constexpr int H = (N + 1) / 2;
#pragma unroll
    for (int k = 0; k < H; ++k) {
        const float lo_v = v[k];
        const float hi_v = (k + H < N) ? v[k + H] : 0.0f;
        const float send = hi ? lo_v : hi_v;
        const float recv = __shfl_xor_sync(0xffffffffu, send, off);
        v[k] = (hi ? hi_v : lo_v) + recv;
    }
}

// Field whose warp total lane `lane` holds after the reduce-scatter of 10
// values, or -1: field = 5 h16 + 3 h8 + 2 h4 + h2 (h* = lane bits), valid
// when 2 h4 + h2 < 3 and 3 h8 + 2 h4 + h2 < 5, and only even lanes.
__device__ __forceinline__ int rs_field(int lane) {
    if (lane & 1) return -1;
    const int h2 = (lane >> 1) & 1, h4 = (lane >> 2) & 1, h8 = (lane >> 3) & 1, h16 = (lane >> 4) & 1;
    const int b = 2 * h4 + h2;
    if (b >= 3) return -1;
    const int a = 3 * h8 + b;
    if (a >= 5) return -1;
    return 5 * h16 + a;
}

template <bool ACCUM>
__global__ void __launch_bounds__(256) k_raster_bwd(BwdParams p) {
    __shared__ SplatGeo s_geo[256];
    __shared__ SplatGeo2 s_geo2[256];
    __shared__ SplatCol s_col[256];
    __shared__ SplatBox s_box[256];
    __shared__ uint32_t s_idx[256];
    __shared__ uint8_t s_list[8][256];
    __shared__ uint32_t s_wmax[8];

    const int tile = blockIdx.x;
    const int tx = tile % p.tiles_x, ty = tile / p.tiles_x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bx = tx * kTile + ((warp & 1) << 3), by = ty * kTile + ((warp >> 1) << 2);
    const int x = bx + (lane & 7), y = by + (lane >> 3);
    const bool inside = x < p.W && y < p.H;
    const float px = float(x) + 0.5f, py = float(y) + 0.5f;
    const float wx0 = float(bx) + 0.5f, wx1 = wx0 + 7.0f;
    const float wy0 = float(by) + 0.5f, wy1 = wy0 + 3.0f;
    const uint32_t start = p.offs[tile], len = p.offs[tile + 1] - start;
    const uint32_t lt = lanemask_lt();

    const size_t HW = size_t(p.W) * p.H, pix = size_t(y) * p.W + x;
    uint32_t n_p = 0;
    float T = 1.0f, g0 = 0.0f, g1 = 0.0f, g2 = 0.0f;
    if (inside) {
        n_p = min(p.last[pix], len);  // a stale last_contrib cannot reach past the tile's pairs
        T = p.T_final[pix];
        g0 = p.dL[pix];
        g1 = p.dL[HW + pix];
        g2 = p.dL[2 * HW + pix];
    }
    const float Tb0 = T * p.bg[0], Tb1 = T * p.bg[1], Tb2 = T * p.bg[2];
    float S0 = 0.0f, S1 = 0.0f, S2 = 0.0f;

    const uint32_t wmax = __reduce_max_sync(0xffffffffu, n_p);
    if (lane == 0) s_wmax[warp] = wmax;
    __syncthreads();
    uint32_t bmax = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) bmax = max(bmax, s_wmax[w]);

    // Where this lane's reduced field goes.
    const int fld = rs_field(lane);
    float *fptr = nullptr;
    int fstride = 0;
    if (fld >= 0 && fld < 2) { fptr = p.dmean2d + fld; fstride = 2; }
    else if (fld >= 2 && fld < 5) { fptr = p.dconic + (fld - 2); fstride = 3; }
    else if (fld == 5) { fptr = p.dopacity; fstride = 1; }
    else if (fld >= 6 && fld < 9) { fptr = p.drgb + (fld - 6); fstride = 3; }
    const bool hi16 = lane & 16, hi8 = lane & 8, hi4 = lane & 4, hi2 = lane & 2;

    for (int32_t hi = int32_t(bmax); hi > 0; hi -= 256) {
        const int32_t lo = hi > 256 ? hi - 256 : 0;
        const int nb = hi - lo;
        __syncthreads();  // the previous batch is no longer read
        if (int(threadIdx.x) < nb) {
            const uint32_t idx = p.vals[start + uint32_t(lo) + threadIdx.x];
            s_idx[threadIdx.x] = idx;
            stage_splat(p.s, idx, s_geo[threadIdx.x], s_geo2[threadIdx.x], s_col[threadIdx.x],
                        s_box[threadIdx.x], nullptr);
        }
        __syncthreads();
        if (uint32_t(lo) >= wmax) continue;
        int cnt = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int j = q * 32 + lane;
            bool hit = false;
            if (j < nb && uint32_t(lo + j) < wmax) {
                const SplatBox b = s_box[j];
                hit = b.x0 <= wx1 && b.x1 >= wx0 && b.y0 <= wy1 && b.y1 >= wy0;
            }
            const uint32_t m = __ballot_sync(0xffffffffu, hit);
            if (hit) s_list[warp][cnt + __popc(m & lt)] = uint8_t(j);
            cnt += __popc(m);
        }
        __syncwarp();
        for (int q = cnt - 1; q >= 0; --q) {
            const int j = s_list[warp][q];
            const SplatGeo g = s_geo[j];
            const SplatGeo2 gg = s_geo2[j];
            float dx, dy;
            const float e2 = eval_e2(g, gg.C, px, py, dx, dy);
            const bool act = uint32_t(lo + j) < n_p && e2 >= gg.thr;
            if (!__any_sync(0xffffffffu, act)) continue;
            float v[10];
#pragma unroll
            for (int k = 0; k < 10; ++k) v[k] = 0.0f;
            if (act) {
                const SplatCol c = s_col[j];
                const float G = ex2_approx(e2);
                float oG;
                const float alpha = eval_alpha(c.o, G, oG);
                const float om = __fsub_rn(1.0f, alpha);
                const float inv = __frcp_rn(om);
                const float Ti = T * inv;          // T in front of this splat
                const float w = alpha * Ti;
                const float dLda = g0 * (c.r * Ti - (S0 + Tb0) * inv) +
                                   g1 * (c.g * Ti - (S1 + Tb1) * inv) +
                                   g2 * (c.b * Ti - (S2 + Tb2) * inv);
                v[6] = g0 * w;
                v[7] = g1 * w;
                v[8] = g2 * w;
                v[9] = w;
                if (oG <= kAlphaMax) {  // through the cap alpha is constant
                    const float dsig = -alpha * dLda;  // dL/dsigma
                    v[5] = G * dLda;                   // dL/dopacity
                    // a dx + b dy = -(2A dx + B dy) ln 2 (A, B, C are base-2 scaled)
                    const float s = dsig * kLn2;
                    v[0] = s * (2.0f * g.A * dx + g.B * dy);   // -dsig (a dx + b dy)
                    v[1] = s * (g.B * dx + 2.0f * gg.C * dy);  // -dsig (b dx + c dy)
                    v[2] = 0.5f * dsig * dx * dx;
                    v[3] = dsig * dx * dy;
                    v[4] = 0.5f * dsig * dy * dy;
                }
                S0 = fmaf(c.r, w, S0);
                S1 = fmaf(c.g, w, S1);
                S2 = fmaf(c.b, w, S2);
                T = Ti;
            }
            rs_step<10>(v, 16, hi16);
            rs_step<5>(v, 8, hi8);
            rs_step<3>(v, 4, hi4);
            rs_step<2>(v, 2, hi2);
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
            if (fld >= 0) {
                const uint32_t idx = s_idx[j];
                if (fld < 9) {
                    atomicAdd(fptr + size_t(fstride) * idx, v[0]);
                } else if (ACCUM) {
                    atomicAdd(p.accum + idx, (unsigned long long)__float2ull_rn(v[0] * 4294967296.0f));
                }
            }
        }
    }
}

__global__ void k_bwd_zero(BwdParams p, int64_t n, bool accum) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        p.dmean2d[2 * i] = 0.0f;
        p.dmean2d[2 * i + 1] = 0.0f;
        p.dconic[3 * i] = 0.0f;
        p.dconic[3 * i + 1] = 0.0f;
        p.dconic[3 * i + 2] = 0.0f;
        p.dopacity[i] = 0.0f;
        p.drgb[3 * i] = 0.0f;
        p.drgb[3 * i + 1] = 0.0f;
        p.drgb[3 * i + 2] = 0.0f;
        if (accum) p.accum[i] = 0ull;
    }
}

__global__ void k_accum_final(const unsigned long long *acc, float *out, int64_t n) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        out[i] = float(double(acc[i]) * (1.0 / 4294967296.0));
}

}  // namespace ss

using namespace ss;

extern "C" ss_status ss_raster_bwd(const ss_splats *splats, const uint32_t *vals,
                                   const uint32_t *tile_offsets, int32_t W, int32_t H,
                                   const float *bg, uint32_t flags, const float *T_final,
                                   const uint32_t *last_contrib, const float *dL_dimage,
                                   const ss_grads *grads, float *accum_weight, void *workspace,
                                   size_t workspace_bytes, ss_stream_t stream) {
    clear_error();
    if (!splats) return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd: splats is NULL");
    if (W < 1 || H < 1 || W > kMaxSide || H > kMaxSide)
        return fail(SS_ERR_UNSUPPORTED, "ss_raster_bwd: image %dx%d outside 1..%d", W, H, kMaxSide);
    if (flags & ~uint32_t(SS_ACCUM_WEIGHT | SS_MEDIAN_DEPTH))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd: unknown flag bits 0x%x", flags);
    const int32_t n = splats->n;
    if (n < 0) return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd: n < 0");
    if (n > 0 && (!splats->mean2d || !splats->conic || !splats->opacity || !splats->rgb ||
                  !splats->depth))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd: a splat array is NULL");
    if (!vals || !tile_offsets) return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd: vals/offsets NULL");
    if (!T_final || !last_contrib || !dL_dimage)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd: T_final/last_contrib/dL_dimage NULL");
    if (!grads || (n > 0 && (!grads->dmean2d || !grads->dconic || !grads->dopacity || !grads->drgb)))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd: a gradient array is NULL");
    const bool accum = flags & SS_ACCUM_WEIGHT;
    if (accum && n > 0 && !accum_weight)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd: SS_ACCUM_WEIGHT set but accum_weight NULL");
    if (n > 0 && (reinterpret_cast<uintptr_t>(splats->mean2d) & 7))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd: mean2d not 8-byte aligned");
    const WsLayout L = ws_layout(n, 0, W, H);
    if (accum && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd: workspace NULL or not 256-byte aligned");
    if (accum && workspace_bytes < L.bwd_end)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd: workspace %zu bytes < %zu needed",
                    workspace_bytes, L.bwd_end);
    if (n == 0) return SS_OK;

    BwdParams p{};
    p.s = SplatPtrs{splats->mean2d, splats->conic, splats->opacity, splats->rgb, splats->depth, n};
    p.vals = vals;
    p.offs = tile_offsets;
    p.W = W;
    p.H = H;
    p.tiles_x = tiles_x(W);
    for (int c = 0; c < 3; ++c) p.bg[c] = bg ? bg[c] : 0.0f;
    p.T_final = T_final;
    p.last = last_contrib;
    p.dL = dL_dimage;
    p.dmean2d = grads->dmean2d;
    p.dconic = grads->dconic;
    p.dopacity = grads->dopacity;
    p.drgb = grads->drgb;
    p.accum = accum ? reinterpret_cast<unsigned long long *>(static_cast<unsigned char *>(workspace) +
                                                              L.accum)
                    : nullptr;
    cudaStream_t st = (cudaStream_t)stream;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (int64_t(n) + 255) / 256;
    const int zgrid = int(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
    SS_LAUNCH("k_bwd_zero", st, k_bwd_zero<<<zgrid, 256, 0, st>>>(p, n, accum));
    const int grid = tiles_x(W) * tiles_y(H);
    if (accum)
        SS_LAUNCH("k_raster_bwd", st, k_raster_bwd<true><<<grid, 256, 0, st>>>(p));
    else
        SS_LAUNCH("k_raster_bwd", st, k_raster_bwd<false><<<grid, 256, 0, st>>>(p));
    if (accum)
        SS_LAUNCH("k_accum_final", st, k_accum_final<<<zgrid, 256, 0, st>>>(p.accum, accum_weight, n));
    return check_launch("ss_raster_bwd");
}

// ---------------------------------------------------------------------------
// ss_raster_bwd_noalloc: the backward pass for callers that cannot allocate.
//
// Some callers may not call cudaMalloc, and cannot hand the library a
// workspace either: plugins living inside an application that owns all
// device memory through its own pool, or real-time render threads that must
// not risk the device-wide synchronisation that cudaMalloc / cudaFree can
// cause.  For them the accumulated-weight scratch of the backward (one
// 32.32 fixed-point uint64 per splat) lives in the fixed array below
// instead of a caller workspace.  Every GPU that loads the library holds it
// (16 MiB) until the process exits.
//
// The array is shared by every call: each call clears the part it uses
// before accumulating, but two calls that run at the same time on the GPU
// (different streams, or different host threads) race on it and corrupt each
// other's accumulated weights.  Serialise them.
namespace ss {

constexpr int32_t kNoAllocMaxSplats = 1 << 21;  // 2,097,152 splats -> 16 MiB of scratch

static __device__ __align__(256) unsigned long long g_noalloc_accum[kNoAllocMaxSplats];

static unsigned long long *g_noalloc_ptr[64];  // device address of the array, per device

}  // namespace ss

extern "C" ss_status ss_raster_bwd_noalloc(const ss_splats *splats, const uint32_t *vals,
                                           const uint32_t *tile_offsets, int32_t W, int32_t H,
                                           const float *bg, uint32_t flags, const float *T_final,
                                           const uint32_t *last_contrib, const float *dL_dimage,
                                           const ss_grads *grads, float *accum_weight,
                                           ss_stream_t stream) {
    clear_error();
    if (!splats) return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: splats is NULL");
    if (W < 1 || H < 1 || W > kMaxSide || H > kMaxSide)
        return fail(SS_ERR_UNSUPPORTED, "ss_raster_bwd_noalloc: image %dx%d outside 1..%d", W, H,
                    kMaxSide);
    if (flags & ~uint32_t(SS_ACCUM_WEIGHT | SS_MEDIAN_DEPTH))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: unknown flag bits 0x%x", flags);
    const int32_t n = splats->n;
    if (n < 0) return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: n < 0");
    if (n > kNoAllocMaxSplats)
        return fail(SS_ERR_UNSUPPORTED,
                    "ss_raster_bwd_noalloc: %d splats exceed its fixed scratch of %d splats; "
                    "use ss_raster_bwd with a workspace",
                    n, kNoAllocMaxSplats);
    if (n > 0 && (!splats->mean2d || !splats->conic || !splats->opacity || !splats->rgb ||
                  !splats->depth))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: a splat array is NULL");
    if (!vals || !tile_offsets)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: vals/offsets NULL");
    if (!T_final || !last_contrib || !dL_dimage)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: T_final/last_contrib/dL_dimage NULL");
    if (!grads || (n > 0 && (!grads->dmean2d || !grads->dconic || !grads->dopacity || !grads->drgb)))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: a gradient array is NULL");
    const bool accum = flags & SS_ACCUM_WEIGHT;
    if (accum && n > 0 && !accum_weight)
        return fail(SS_ERR_INVALID_ARG,
                    "ss_raster_bwd_noalloc: SS_ACCUM_WEIGHT set but accum_weight NULL");
    if (n > 0 && (reinterpret_cast<uintptr_t>(splats->mean2d) & 7))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: mean2d not 8-byte aligned");
    if (n == 0) return SS_OK;

    int dev = 0, sms = 0;
    ss_status s = check_cuda(cudaGetDevice(&dev), "ss_raster_bwd_noalloc: cudaGetDevice");
    if (s != SS_OK) return s;
    if (dev < 0 || dev >= 64)
        return fail(SS_ERR_UNSUPPORTED, "ss_raster_bwd_noalloc: device %d >= 64", dev);
    if (accum && !g_noalloc_ptr[dev]) {
        // First call on this device (with this device current): look up the
        // array's device address once.
        void *ptr = nullptr;
        s = check_cuda(cudaGetSymbolAddress(&ptr, g_noalloc_accum),
                       "ss_raster_bwd_noalloc: cudaGetSymbolAddress");
        if (s != SS_OK) return s;
        g_noalloc_ptr[dev] = static_cast<unsigned long long *>(ptr);
    }

    BwdParams p{};
    p.s = SplatPtrs{splats->mean2d, splats->conic, splats->opacity, splats->rgb, splats->depth, n};
    p.vals = vals;
    p.offs = tile_offsets;
    p.W = W;
    p.H = H;
    p.tiles_x = tiles_x(W);
    for (int c = 0; c < 3; ++c) p.bg[c] = bg ? bg[c] : 0.0f;
    p.T_final = T_final;
    p.last = last_contrib;
    p.dL = dL_dimage;
    p.dmean2d = grads->dmean2d;
    p.dconic = grads->dconic;
    p.dopacity = grads->dopacity;
    p.drgb = grads->drgb;
    p.accum = accum ? g_noalloc_ptr[dev] : nullptr;
    cudaStream_t st = (cudaStream_t)stream;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (int64_t(n) + 255) / 256;
    const int zgrid = int(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
    // k_bwd_zero clears this call's part of the shared array before use.
    SS_LAUNCH("k_bwd_zero", st, k_bwd_zero<<<zgrid, 256, 0, st>>>(p, n, accum));
    const int grid = tiles_x(W) * tiles_y(H);
    if (accum)
        SS_LAUNCH("k_raster_bwd", st, k_raster_bwd<true><<<grid, 256, 0, st>>>(p));
    else
        SS_LAUNCH("k_raster_bwd", st, k_raster_bwd<false><<<grid, 256, 0, st>>>(p));
    if (accum)
        SS_LAUNCH("k_accum_final", st, k_accum_final<<<zgrid, 256, 0, st>>>(p.accum, accum_weight, n));
    return check_launch("ss_raster_bwd_noalloc");
}
