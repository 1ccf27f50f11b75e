// Backward rasterization ("从 8.6 KB 到 4.2 KB ...", rasterize_bwd_2d, the
// 2D screen-space backward; "Phase 5 step 30b -- kernel-by-kernel timing",
// rasterize_backwards: 52 % of the step, bound by per-pixel float atomics
// on the 9 gradient fields of every splat).
//
// Same CTA/tile and warp/8x4-block layout as the forward.  Each pixel starts
// from its forward state (T_final, last_contrib) and walks its tile's list
// back to front in batches of 256 staged 64-byte splat records (cp.async,
// double buffered), recovering the transmittance in front of each blended
// splat as T / (1 - alpha) and keeping dL/dimage . (colour behind + T_final
// bg) as one scalar.
//
// Reduction.  The pages' baseline issues 9 atomics per (pixel, splat); their
// proposed fix sums each field across the warp first and issues one atomic
// per warp ("Phase 5 step 30b", conclusion).  Summing 10 fields across 32
// lanes with shuffles costs ~46 instructions per (warp, splat), while only
// ~9 of the 32 pixels of a warp touch a given splat.  Here the sum is
// transposed instead: every field is linear in two per-pixel scalars,
//   q = dL/dsigma  and  w = alpha T  (the pixel's blend weight),
// so for each splat blended somewhere in the warp the 32 pixels write (q, w)
// into a shared-memory slot (zeros where the splat is not blended), and
// once 16 slots are full each lane pair takes one slot and sums its 32
// pixels with plain FMAs into ten moments:
//   Q = sum q, Qx = sum q dx, Qy = sum q dy, Qxx, Qxy, Qyy, W = sum w,
//   Wr, Wg, Wb = sum w dL/dimage_c,
// from which (a dx + b dy = -(2A dx + B dy) ln 2 with the base-2 scaled
// A, B, C of the staged splat)
//   dmean = ln2 (2A Qx + B Qy, B Qx + 2C Qy),  dconic = (Qxx/2, Qxy, Qyy/2),
//   dopacity = -Q / o  (G dL/dalpha = -q / o when alpha is not capped),
//   drgb = (Wr, Wg, Wb),  accumulated weight = W,
// and adds them, with four reductions per (warp, splat) (two
// red.global.add.v4.f32, one f32, one u64), into a 48-byte per-splat record
// that k_grad_final converts to the SoA outputs (the entry point for
// callers that cannot allocate adds the ten fields directly to the outputs
// instead).  The accumulated weight is added in 32.32 fixed point with
// 64-bit integer atomics, so it is exact and independent of atomic order.
//
// Distortion (the DIST variant).  The depth distortion's gradient has the
// colour's shape: with E = dD/dw = z'^2 A - 2 z' D1 + D2 from the forward's
// per-pixel totals (depths z' relative to the pixel's first blended splat),
// dD/dalpha = E T_front - (sum of w E over later splats) / (1 - alpha), so
// dL/ddist E joins dL/dimage . rgb in the per-splat scalar and in GR, and
// dL/ddepth = 2 dL/ddist w (z A - D1) sums, per warp and splat, to
// 2 (z Wa - Wd) with Wa = sum w dL/ddist A and Wd = sum w dL/ddist D1 --
// two more moments of the slot sums, added with the blue gradient as one
// 8-byte reduction into the record's spare tenth float.
//
// The blend decisions are the forward's: its per-(pair, 8x4 block) masks
// select the entries each warp handles and each pixel's bit, so nothing is
// re-evaluated; after a chunk of 16 selected entries each pixel walks only
// its own blended entries (independent trip counts per lane).
#include <atomic>
#include <mutex>

#include "ss_device.cuh"
#include "ss_internal.h"
#include "ss_profile.h"

namespace ss {

// 168 bytes.  Unlike the forward kernel (faster with its parameters packed
// into 128 bytes), this one measured 17 % slower in a 128-byte layout: ptxas
// then spilled under the 3-CTA register cap.
struct BwdParams {
    const SplatRecord *recs;
    int32_t n;
    int32_t accum_on;           // add the accumulated weight (SS_ACCUM_WEIGHT): a runtime
                                // switch, not a template variant -- the variant without it
                                // spilled under the 3-CTA register cap and ran 9 % slower
    const uint32_t *vals;
    const uint32_t *offs;
    const uint32_t *masks;  // [8][n_pairs] the forward's blend decisions
    int64_t n_pairs;
    int32_t W, H, tiles_x;
    float bg[3];
    const float *T_final;
    const uint32_t *last;
    const float *dL;
    float *dmean2d, *dconic, *dopacity, *drgb;
    float *ddepth;              // (DIST)
    const float4 *dist_totals;  // [H][W] (A, D1, D2, z_ref) from the forward (DIST)
    const float *dL_ddist;      // [H][W] (DIST)
    unsigned long long *accum;  // 32.32 fixed point (SoA mode)
    float *scratch;             // [n][12] per-splat gradient record (AoS mode)
};

// Per-splat gradient scratch record (AoS mode), 48 bytes, 16-byte aligned:
// [0..3] dmean x, dmean y, dconic a, dconic b; [4..7] dconic c, dopacity,
// drgb r, drgb g; [8] drgb b; [9] ddepth (DIST); [10..11] accumulated weight
// as a uint64 in 32.32 fixed point.
constexpr int kGradRec = 12;

__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void red_add_v2(float *addr, float a, float b) {
    asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(addr), "f"(a), "f"(b) : "memory");
}

constexpr int kSlots = 16;     // slots per warp
// A warp's list: up to 64 entries of a segment below up to kChunk - 1
// entries left over from the segments above (chunks are always full but
// for the batch's last).
constexpr int kListCap = 64 + 16;
constexpr int kChunk = 16;     // list entries evaluated together (<= kSlots)
constexpr int kSlotPad = 32;   // entries per slot row (one per pixel of the warp's block)
// Pixel p of slot row r is stored at column p ^ (2 (r & 7)): the replay's
// row writes are permutations, and the flush's 64-bit reads, where lane pair
// (r, h) takes pixels 2i + h, hit 32 distinct bank pairs.
__device__ __forceinline__ int slot_col(int row, int pix) { return pix ^ ((row & 7) << 1); }

// 32 x 32 bit transpose across the warp: on return, bit k of lane p's word
// is bit p of lane k's word on entry (five butterfly stages of shuffles).
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane) {
    constexpr uint32_t kMask[5] = {0x0000ffffu, 0x00ff00ffu, 0x0f0f0f0fu, 0x33333333u, 0x55555555u};
#pragma unroll
    for (int s = 0; s < 5; ++s) {
        const int j = 16 >> s;
        const uint32_t m = kMask[s];
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
        x = (lane & j) ? ((x & ~m) | ((y >> j) & m)) : ((x & m) | ((y & m) << j));
    }
    return x;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A list entry's replay data, gathered per chunk next to the chunk's other
// entries: the per-lane walk then reads 16 nearby records instead of 256.
struct __align__(16) ChunkEnt {
    SplatGeo g;   // mx, my, A, B
    float4 c1;    // C, o, r, g
    float4 c2;    // b, depth
};

// Per-warp slot storage.
struct __align__(16) SlotRec {
    float mx, my, A, B;   // staged geometry of the slot's splat
    float C, o;
    uint32_t idx;
    float depth;
};

template <bool AOS, bool DIST>
__device__ __forceinline__ void flush_slots(const BwdParams &p, int nslots, int lane, float wx0,
                                            float wy0, const float2 (*qw)[kSlotPad],
                                            const float4 *g, const float *gd1, const SlotRec *rec) {
    __syncwarp();
    // Every lane runs the sums (lanes of unused slots read stale, in-bounds
    // rows) so that the pair shuffles see the whole warp; only the atomics
    // are limited to the filled slots.
    const int slot = lane >> 1, half = lane & 1;
    {
        const SlotRec r = rec[slot];
        // Lane half h sums pixels 2i + h, i.e. column u = 2k + h (k = i & 3)
        // and row v = i >> 2 of the 8x4 block; k and v are constants of the
        // unrolled loop.  Raw moments in (k, v), then u = 2k + h and the
        // centring dx = u + ex, dy = v + ey.
        float M1 = 0.f, Mk = 0.f, Mkk = 0.f, Mv = 0.f, Mkv = 0.f, Mvv = 0.f;
        float Wt = 0.f, Wr = 0.f, Wg = 0.f, Wb = 0.f, Wa = 0.f, Wd = 0.f;
        const float2 *row = qw[slot];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int k = i & 3, v = i >> 2;
            const int pix = 2 * i + half;
            const float2 e = row[slot_col(slot, pix)];
            const float qi = e.x, wi = e.y;
            M1 += qi;
            if (k) {
                Mk = fmaf(float(k), qi, Mk);
                Mkk = fmaf(float(k * k), qi, Mkk);
            }
            if (v) {
                Mv = fmaf(float(v), qi, Mv);
                Mvv = fmaf(float(v * v), qi, Mvv);
                if (k) Mkv = fmaf(float(k * v), qi, Mkv);
            }
            const float4 gg = g[pix];
            Wt += wi;
            Wr = fmaf(wi, gg.x, Wr);
            Wg = fmaf(wi, gg.y, Wg);
            Wb = fmaf(wi, gg.z, Wb);
            if (DIST) {
                Wa = fmaf(wi, gg.w, Wa);
                Wd = fmaf(wi, gd1[pix], Wd);
            }
        }
        const float hf = float(half);
        const float Mu = fmaf(2.0f, Mk, hf * M1);
        const float Muu = fmaf(4.0f, Mkk, hf * fmaf(4.0f, Mk, M1));
        const float Muv = fmaf(2.0f, Mkv, hf * Mv);
        const float ex = __fsub_rn(wx0, r.mx), ey = __fsub_rn(wy0, r.my);
        float Q = M1;
        float Qx = fmaf(ex, M1, Mu);
        float Qy = fmaf(ey, M1, Mv);
        float Qxx = fmaf(ex, fmaf(ex, M1, 2.0f * Mu), Muu);
        float Qxy = fmaf(ex, fmaf(ey, M1, Mv), fmaf(ey, Mu, Muv));
        float Qyy = fmaf(ey, fmaf(ey, M1, 2.0f * Mv), Mvv);
        // Sum the two halves of the slot (lanes 2k and 2k+1).
        Q += __shfl_xor_sync(0xffffffffu, Q, 1, 2);
        Qx += __shfl_xor_sync(0xffffffffu, Qx, 1, 2);
        Qy += __shfl_xor_sync(0xffffffffu, Qy, 1, 2);
        Qxx += __shfl_xor_sync(0xffffffffu, Qxx, 1, 2);
        Qxy += __shfl_xor_sync(0xffffffffu, Qxy, 1, 2);
        Qyy += __shfl_xor_sync(0xffffffffu, Qyy, 1, 2);
        Wt += __shfl_xor_sync(0xffffffffu, Wt, 1, 2);
        Wr += __shfl_xor_sync(0xffffffffu, Wr, 1, 2);
        Wg += __shfl_xor_sync(0xffffffffu, Wg, 1, 2);
        Wb += __shfl_xor_sync(0xffffffffu, Wb, 1, 2);
        float dz = 0.0f;
        if (DIST) {
            Wa += __shfl_xor_sync(0xffffffffu, Wa, 1, 2);
            Wd += __shfl_xor_sync(0xffffffffu, Wd, 1, 2);
            dz = 2.0f * fmaf(r.depth, Wa, -Wd);
        }
        const size_t i = r.idx;
        const bool bad_idx = SS_BAD(slot < nslots && r.idx >= uint32_t(p.n), kDbgBwdSplat);
        const float dmx = kLn2 * (2.0f * r.A * Qx + r.B * Qy);
        const float dmy = kLn2 * (r.B * Qx + 2.0f * r.C * Qy);
        if (slot >= nslots || bad_idx) {
        } else if (AOS) {
            // Four reductions per (warp, splat) into one 48-byte record.
            float *g = p.scratch + kGradRec * i;
            if (half == 0) {
                red_add_v4(g, dmx, dmy, 0.5f * Qxx, Qxy);
            } else {
                red_add_v4(g + 4, 0.5f * Qyy, -Q / r.o, Wr, Wg);
                if (DIST)
                    red_add_v2(g + 8, Wb, dz);
                else
                    atomicAdd(g + 8, Wb);
                if (p.accum_on)
                    atomicAdd(reinterpret_cast<unsigned long long *>(g + 10),
                              (unsigned long long)__float2ull_rn(Wt * 4294967296.0f));
            }
        } else if (half == 0) {
            atomicAdd(p.dmean2d + 2 * i, dmx);
            atomicAdd(p.dmean2d + 2 * i + 1, dmy);
            atomicAdd(p.dconic + 3 * i, 0.5f * Qxx);
            atomicAdd(p.dconic + 3 * i + 1, Qxy);
            atomicAdd(p.dconic + 3 * i + 2, 0.5f * Qyy);
        } else {
            atomicAdd(p.dopacity + i, -Q / r.o);
            atomicAdd(p.drgb + 3 * i, Wr);
            atomicAdd(p.drgb + 3 * i + 1, Wg);
            atomicAdd(p.drgb + 3 * i + 2, Wb);
            if (p.accum_on) atomicAdd(p.accum + i, (unsigned long long)__float2ull_rn(Wt * 4294967296.0f));
        }
    }
    __syncwarp();
}

template <bool AOS, bool DIST>
__global__ void __launch_bounds__(256, 3) k_raster_bwd(BwdParams p) {
    __shared__ SplatGeo s_geo_[2][256];
    __shared__ SplatGeo2 s_geo2_[2][256];
    __shared__ SplatCol s_col_[2][256];
    __shared__ uint8_t s_list[8][kListCap];
    __shared__ uint32_t s_lmask[8][kListCap];
    __shared__ ChunkEnt s_ck[8][kChunk];
    __shared__ uint32_t s_wmax[8];
    __shared__ float4 s_g[8][32];
    __shared__ float s_gd1[DIST ? 8 : 1][32];
    __shared__ SlotRec s_rec[8][kSlots];
    // dynamic: (q, w) slots, [8 warps][kSlots][kSlotPad] float2
    extern __shared__ __align__(16) float2 s_dyn[];
    float2(*s_qw)[kSlots][kSlotPad] = reinterpret_cast<float2(*)[kSlots][kSlotPad]>(s_dyn);

    const int tile = blockIdx.x;
    const int tx = tile % p.tiles_x, ty = tile / p.tiles_x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bx = tx * kTile + ((warp & 1) << 3), by = ty * kTile + ((warp >> 1) << 2);
    const int x = bx + (lane & 7), y = by + (lane >> 3);
    const bool inside = x < p.W && y < p.H;
    const float px = float(x) + 0.5f, py = float(y) + 0.5f;
    const float wx0 = float(bx) + 0.5f, wy0 = float(by) + 0.5f;
    uint32_t start = p.offs[tile], len = p.offs[tile + 1] - start;
    if (SS_BAD(p.offs[tile + 1] < start || int64_t(start) + len > p.n_pairs, kDbgBwdList))
        start = len = 0u;
    const uint32_t lt = lanemask_lt();

    const size_t HW = size_t(p.W) * p.H, pix = size_t(y) * p.W + x;
    uint32_t n_p = 0;
    float T = 1.0f, g0 = 0.0f, g1 = 0.0f, g2 = 0.0f;
    if (inside) {
        n_p = p.last[pix];
        if (SS_BAD(n_p > len, kDbgBwdLast)) n_p = len;
        n_p = min(n_p, len);  // a stale last_contrib cannot reach past the tile's pairs
        T = p.T_final[pix];
        g0 = p.dL[pix];
        g1 = p.dL[HW + pix];
        g2 = p.dL[2 * HW + pix];
    }
    // DIST: the pixel's distortion gradient and the forward's totals
    float gD = 0.0f, dA = 0.0f, dD1 = 0.0f, dD2 = 0.0f, zref = 0.0f;
    if (DIST && inside) {
        gD = p.dL_ddist[pix];
        const float4 t = p.dist_totals[pix];
        dA = t.x, dD1 = t.y, dD2 = t.z, zref = t.w;
    }
    s_g[warp][lane] = make_float4(g0, g1, g2, gD * dA);
    if (DIST) s_gd1[warp][lane] = gD * fmaf(zref, dA, dD1);
    // GR = dL/dimage . (S + T_final bg), S the colour blended behind the
    // current splat: with it dL/dalpha = (T gc - GR) / (1 - alpha), where
    // gc = dL/dimage . rgb and T is the transmittance behind the splat, and
    // blending the splat adds w gc to GR.
    float GR = T * (g0 * p.bg[0] + g1 * p.bg[1] + g2 * p.bg[2]);

    const uint32_t wmax = __reduce_max_sync(0xffffffffu, n_p);
    if (lane == 0) s_wmax[warp] = wmax;
    __syncthreads();
    uint32_t bmax = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) bmax = max(bmax, s_wmax[w]);

    int nslots = 0;  // warp-uniform
    // Batches back to front: batch b covers positions [lo_b, hi_b) of the
    // tile's list, hi_b = bmax - 256 b, lo_b = max(0, hi_b - 256).  Its
    // records are copied into buffer b & 1 while batch b - 1 is processed.
    const int tid = threadIdx.x;
    if (bmax > 0) {
        const int32_t lo0 = bmax > 256u ? int32_t(bmax) - 256 : 0;
        if (tid < int32_t(bmax) - lo0) {
            const uint32_t idx = p.vals[start + uint32_t(lo0) + tid];
            stage_record3_async(p.recs, idx, p.n, s_geo_[0], s_geo2_[0], s_col_[0], tid);
        }
        cp_async_commit();
    }
    uint32_t next_idx = 0;
    {
        const int32_t hi1 = int32_t(bmax) - 256;
        const int32_t lo1 = hi1 > 256 ? hi1 - 256 : 0;
        if (hi1 > 0 && tid < hi1 - lo1) next_idx = p.vals[start + uint32_t(lo1) + tid];
    }
    int buf = 0;
    for (int32_t hi = int32_t(bmax); hi > 0; hi -= 256, buf ^= 1) {
        const int32_t lo = hi > 256 ? hi - 256 : 0;
        const int nb = hi - lo;
        cp_async_wait<0>();
        __syncthreads();  // batch staged everywhere; the other buffer is free
        {
            const int32_t nhi = hi - 256;  // prefetch the next batch (further to the front)
            if (nhi > 0) {
                const int32_t nlo = nhi > 256 ? nhi - 256 : 0;
                if (tid < nhi - nlo) {
                    stage_record3_async(p.recs, next_idx, p.n, s_geo_[buf ^ 1], s_geo2_[buf ^ 1],
                                        s_col_[buf ^ 1], tid);
                }
                cp_async_commit();
                const int32_t nnhi = nhi - 256;
                const int32_t nnlo = nnhi > 256 ? nnhi - 256 : 0;
                next_idx = (nnhi > 0 && tid < nnhi - nnlo) ? p.vals[start + uint32_t(nnlo) + tid] : 0u;
            }
        }
        const SplatGeo *s_geo = s_geo_[buf];
        const SplatGeo2 *s_geo2 = s_geo2_[buf];
        const SplatCol *s_col = s_col_[buf];
        if (uint32_t(lo) >= wmax) continue;
        // Positions [0, lim) of this batch may be blended in this warp's block.
        // They are taken in segments of 64, top segment first; each segment's
        // entries that the forward blended somewhere in the block are listed
        // with their masks (the next segment's masks load meanwhile) and then
        // processed back to front in chunks of kChunk.
        const int lim = min(nb, int(wmax) - lo);
        const uint32_t *gm = p.masks + size_t(warp) * size_t(p.n_pairs) + start + uint32_t(lo);
        const int64_t gbase = int64_t(start) + lo;
        int sg = (lim - 1) >> 6;
        uint32_t ma = 0, mb = 0;
        {
            const int j0 = 64 * sg + lane, j1 = j0 + 32;
            ma = (j0 < lim && gbase + j0 < p.n_pairs) ? gm[j0] : 0u;
            mb = (j1 < lim && gbase + j1 < p.n_pairs) ? gm[j1] : 0u;
        }
        // The listed entries of the batch, in ascending position, occupy
        // [kListCap - npend, kListCap) between segments: the ones left over
        // (fewer than kChunk) from the segments above.
        int npend = 0;
        for (; sg >= 0; --sg) {
            const uint32_t ca = ma, cb = mb;
            if (sg > 0) {
                const int j0 = 64 * (sg - 1) + lane, j1 = j0 + 32;
                ma = (j0 < lim && gbase + j0 < p.n_pairs) ? gm[j0] : 0u;
                mb = (j1 < lim && gbase + j1 < p.n_pairs) ? gm[j1] : 0u;
            }
            // This segment's entries go just below the left-over ones.
            const uint32_t b0 = __ballot_sync(0xffffffffu, ca != 0u);
            const uint32_t b1 = __ballot_sync(0xffffffffu, cb != 0u);
            const int cnt = __popc(b0) + __popc(b1);
            const int lbase = kListCap - npend - cnt;
            if (ca) {
                const int at = lbase + __popc(b0 & lt);
                s_list[warp][at] = uint8_t(64 * sg + lane);
                s_lmask[warp][at] = ca;
            }
            if (cb) {
                const int at = lbase + __popc(b0) + __popc(b1 & lt);
                s_list[warp][at] = uint8_t(64 * sg + 32 + lane);
                s_lmask[warp][at] = cb;
            }
            __syncwarp();
            const uint8_t *list = s_list[warp];
            const uint32_t *lmask = s_lmask[warp];
            // Full chunks from the top (the back of the list); the batch's
            // last segment also takes the rest.
            int have = npend + cnt, hq = kListCap;
            for (; have >= kChunk || (sg == 0 && have > 0); hq -= kChunk, have -= kChunk) {
                const int nq = have < kChunk ? have : kChunk;
                const int lq = hq - nq;
                // 1. This pixel's bit of each entry's mask: lane k holds entry
                //    k's mask, and the warp transposes the 32 x 32 bit matrix.
                const uint32_t mine0 = warp_transpose32(lane < nq ? lmask[lq + lane] : 0u, lane);
                // 2. One slot row per entry, zeroed (16 bytes a lane, two rows
                //    per store); lane k copies entry k's replay data next to
                //    the others' and records the splat for the flush.
                const int nrows = nq;
                if (nslots + nrows > kSlots) {
                    flush_slots<AOS, DIST>(p, nslots, lane, wx0, wy0, s_qw[warp],
                                                  s_g[warp], s_gd1[DIST ? warp : 0],
                                                  s_rec[warp]);
                    nslots = 0;
                }
                {
                    float4 *z = reinterpret_cast<float4 *>(&s_qw[warp][nslots][0]);
                    for (int i = lane; i < nrows * (kSlotPad / 2); i += 32)
                        z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (lane < nq) {
                    const int j = list[lq + lane];
                    const SplatGeo g = s_geo[j];
                    const SplatGeo2 g2 = s_geo2[j];
                    const SplatCol c = s_col[j];
                    s_ck[warp][lane] = ChunkEnt{g, make_float4(g2.C, g2.o, c.r, c.g),
                                                make_float4(c.b, g2.depth, 0.f, 0.f)};
                    s_rec[warp][nslots + lane] = SlotRec{g.mx, g.my, g.A, g.B, g2.C, g2.o, c.idx,
                                                         g2.depth};
                }
                __syncwarp();
                // 3. Each pixel walks only its own blended entries, back to front.
                uint32_t mine = mine0;
                while (mine) {
                    const int k = 31 - __clz(mine);
                    mine &= ~(1u << k);
                    const SplatGeo g = s_ck[warp][k].g;
                    const float4 c1 = s_ck[warp][k].c1;   // C, o, r, g
                    const float4 c2 = s_ck[warp][k].c2;   // b, depth
                    float dx, dy;
                    const float e2 = eval_e2(g, c1.x, px, py, dx, dy);
                    const float G = ex2_approx(e2);
                    float oG;
                    const float alpha = eval_alpha(c1.y, G, oG);
                    const float inv = rcp_approx(__fsub_rn(1.0f, alpha));
                    const float Ti = T * inv;  // T in front of this splat
                    const float wv = alpha * Ti;
                    float gc = fmaf(g0, c1.z, fmaf(g1, c1.w, g2 * c2.x));
                    if (DIST) {
                        const float z = c2.y - zref;
                        gc = fmaf(gD, fmaf(z, fmaf(z, dA, -2.0f * dD1), dD2), gc);
                    }
                    const float dLda = inv * fmaf(T, gc, -GR);
                    const float qv = oG <= kAlphaMax ? -alpha * dLda : 0.0f;  // capped: constant
                    GR = fmaf(wv, gc, GR);
                    T = Ti;
                    const int row = nslots + k;
                    s_qw[warp][row][slot_col(row, lane)] = make_float2(qv, wv);
                }
                __syncwarp();
                nslots += nrows;
            }
            // Move the left-over entries (below hq) up to the end of the list.
            have = have > 0 ? have : 0;
            if (hq != kListCap && have > 0) {
                uint8_t e = 0;
                uint32_t em = 0;
                if (lane < have) e = list[hq - have + lane], em = lmask[hq - have + lane];
                __syncwarp();
                if (lane < have) {
                    s_list[warp][kListCap - have + lane] = e;
                    s_lmask[warp][kListCap - have + lane] = em;
                }
                __syncwarp();
            }
            npend = have;
        }
    }
    cp_async_wait<0>();  // no copy may outlive the CTA
    if (nslots)
        flush_slots<AOS, DIST>(p, nslots, lane, wx0, wy0, s_qw[warp], s_g[warp],
                                      s_gd1[DIST ? warp : 0], s_rec[warp]);
}

constexpr int kBwdDynSmem = 2 * 8 * kSlots * kSlotPad * 4;

// k_raster_bwd's slot buffers are dynamic shared memory on top of ~25 KB of
// static arrays: raise its limit once per CUDA context.
static std::atomic<unsigned long long> g_bwd_smem_ctx[kMaxDevices];
static ss_status ensure_bwd_smem() {
    const void *fns[3] = {(const void *)k_raster_bwd<true, false>,
                          (const void *)k_raster_bwd<false, false>,
                          (const void *)k_raster_bwd<true, true>};
    return ensure_dyn_smem(g_bwd_smem_ctx, fns, 3, kBwdDynSmem, "backward");
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

// AoS mode: clear the per-splat gradient records (skipped when the forward
// cleared them: SS_RECORDS_CLEARED).
__global__ void k_grad_zero(float4 *scratch, int64_t n4) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride)
        scratch[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// AoS mode: gradient records -> the SoA outputs (and the weight to float).
__global__ void k_grad_final(BwdParams p, int64_t n, float *accum_out) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float4 *g = reinterpret_cast<const float4 *>(p.scratch + kGradRec * i);
        const float4 a = g[0], b = g[1], c = g[2];
        p.dmean2d[2 * i] = a.x;
        p.dmean2d[2 * i + 1] = a.y;
        p.dconic[3 * i] = a.z;
        p.dconic[3 * i + 1] = a.w;
        p.dconic[3 * i + 2] = b.x;
        p.dopacity[i] = b.y;
        p.drgb[3 * i] = b.z;
        p.drgb[3 * i + 1] = b.w;
        p.drgb[3 * i + 2] = c.x;
        if (p.ddepth) p.ddepth[i] = c.y;
        if (accum_out) {
            const unsigned long long w =
                *reinterpret_cast<const unsigned long long *>(p.scratch + kGradRec * i + 10);
            accum_out[i] = float(double(w) * (1.0 / 4294967296.0));
        }
    }
}

__global__ void k_accum_final(const unsigned long long *acc, float *out, int64_t n) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        out[i] = float(double(acc[i]) * (1.0 / 4294967296.0));
}

// Records of the splats from the SoA inputs: what the binning writes, bit
// for bit (record_of), for the backward that takes the splats themselves;
// the same pass clears each splat's 48-byte gradient record (clear[3 i ..]).
__global__ void k_make_records(SplatPtrs s, int32_t tiles_x, int32_t tiles_y, SplatRecord *out,
                               float4 *clear) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < s.n; i += stride) {
        const SplatRecord r = record_of(s, uint32_t(i), tiles_x, tiles_y);
        float4 *dst = reinterpret_cast<float4 *>(out + i);
        dst[0] = *reinterpret_cast<const float4 *>(&r.geo);
        dst[1] = *reinterpret_cast<const float4 *>(&r.geo2);
        dst[2] = *reinterpret_cast<const float4 *>(&r.col);
        dst[3] = *reinterpret_cast<const float4 *>(&r.box);
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        clear[3 * i] = z;
        clear[3 * i + 1] = z;
        clear[3 * i + 2] = z;
    }
}

struct MaskParams {
    const SplatRecord *recs;
    int32_t n;
    const uint32_t *vals;
    const uint32_t *offs;
    const uint32_t *last;
    int32_t W, H, tiles_x, tiles;
    uint32_t *masks;   // [8][stride]
    int64_t stride;
    uint32_t *status;  // the workspace's status word
};

// The forward's blend decisions, re-evaluated from the staged records for a
// backward given none: a pixel blended list position j of its tile iff
// j < last_contrib and e2 >= thr (the forward blends every splat it does
// not skip until it stops, and last_contrib is its last blend), with e2 the
// same eval_e2 of the same record bits.  One CTA per tile; batches of 256
// records are staged front to back with cp.async into two buffers (the next
// batch copies while this one is evaluated); each warp takes its 8x4 block,
// box-culls the batch and evaluates the rest, and writes the masks the
// backward reads, masks[warp][position].  A list longer than the mask rows
// (offsets[tiles] > stride) is recorded in the status word and its masks are
// not written past the rows.
__global__ void __launch_bounds__(256) k_blend_masks(MaskParams p) {
    __shared__ SplatGeo s_geo[2][256];
    __shared__ SplatGeo2 s_geo2[2][256];
    __shared__ SplatBox s_box[2][256];
    __shared__ uint32_t s_wmax[8];
    const int tile = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tx = tile % p.tiles_x, ty = tile / p.tiles_x;
    const int bx = tx * kTile + ((warp & 1) << 3), by = ty * kTile + ((warp >> 1) << 2);
    const int x = bx + (lane & 7), y = by + (lane >> 3);
    const bool inside = x < p.W && y < p.H;
    const float px = float(x) + 0.5f, py = float(y) + 0.5f;
    const float wx0 = float(bx) + 0.5f, wx1 = wx0 + 7.0f;
    const float wy0 = float(by) + 0.5f, wy1 = wy0 + 3.0f;
    uint32_t start = p.offs[tile], len = p.offs[tile + 1] - start;
    if (SS_BAD(p.offs[tile + 1] < start || int64_t(start) + len > p.stride, kDbgMaskList))
        start = len = 0u;
    if (tile == 0 && tid == 0 && int64_t(p.offs[p.tiles]) > p.stride)
        atomicOr(p.status, kDevErrCapacity);
    const uint32_t n_p = inside ? min(p.last[size_t(y) * p.W + x], len) : 0u;
    const uint32_t wmax = __reduce_max_sync(0xffffffffu, n_p);
    if (lane == 0) s_wmax[warp] = wmax;
    __syncthreads();
    uint32_t bmax = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) bmax = max(bmax, s_wmax[w]);

    // Record idx into slot t of buffer b (the invisible record past n).
    auto stage = [&](uint32_t idx, int b, int t) {
        if (idx < uint32_t(p.n)) {
            const SplatRecord *r = p.recs + idx;
            cp_async16(&s_geo[b][t], &r->geo);
            cp_async16(&s_geo2[b][t], &r->geo2);
            cp_async16(&s_box[b][t], &r->box);
        } else {
            const SplatRecord r = invisible_record();
            s_geo[b][t] = r.geo;
            s_geo2[b][t] = r.geo2;
            s_box[b][t] = r.box;
        }
    };
    // Batch b covers positions [256 b, min(bmax, 256 (b + 1))) of the list.
    if (bmax > 0) {
        if (uint32_t(tid) < bmax) stage(p.vals[start + tid], 0, tid);
        cp_async_commit();
    }
    uint32_t next_idx = 256u + uint32_t(tid) < bmax ? p.vals[start + 256u + tid] : 0u;
    int buf = 0;
    for (uint32_t base = 0; base < bmax; base += 256, buf ^= 1) {
        cp_async_wait<0>();
        __syncthreads();   // batch staged everywhere; nobody still reads the other buffer
        const uint32_t nbase = base + 256;
        if (nbase < bmax) {
            if (nbase + uint32_t(tid) < bmax) stage(next_idx, buf ^ 1, tid);
            cp_async_commit();
            next_idx = nbase + 256u + uint32_t(tid) < bmax ? p.vals[start + nbase + 256u + tid] : 0u;
        }
        const int nb = int(min(256u, bmax - base));
        if (base >= wmax) continue;   // warp-uniform: no pixel of this block reaches the batch
        const SplatGeo *geo = s_geo[buf];
        const SplatGeo2 *geo2 = s_geo2[buf];
        const SplatBox *box = s_box[buf];
        for (int q = 0; q < 8 && q * 32 < nb; ++q) {
            const int j = q * 32 + lane;
            bool hit = false;
            if (j < nb && base + uint32_t(j) < wmax) {
                const SplatBox b = box[j];
                hit = b.x0 <= wx1 && b.x1 >= wx0 && b.y0 <= wy1 && b.y1 >= wy0;
            }
            // The listed entries two at a time (independent evaluations; a
            // lone last one is evaluated twice): lane k keeps entry k's mask.
            uint32_t m = __ballot_sync(0xffffffffu, hit), mine = 0;
            while (m) {
                const int k0 = __ffs(m) - 1;
                m &= m - 1;
                const int k1 = m ? __ffs(m) - 1 : k0;
                m &= m - 1;
                const int j0 = q * 32 + k0, j1 = q * 32 + k1;
                float dx, dy;
                const float e0 = eval_e2(geo[j0], geo2[j0].C, px, py, dx, dy);
                const float e1 = eval_e2(geo[j1], geo2[j1].C, px, py, dx, dy);
                const uint32_t b0 = __ballot_sync(0xffffffffu,
                                                  base + uint32_t(j0) < n_p && e0 >= geo2[j0].thr);
                const uint32_t b1 = __ballot_sync(0xffffffffu,
                                                  base + uint32_t(j1) < n_p && e1 >= geo2[j1].thr);
                if (lane == k0) mine = b0;
                if (lane == k1) mine = b1;
            }
            if (j < nb) {
                const int64_t pos = int64_t(start) + base + j;
                if (pos < p.stride) p.masks[size_t(warp) * size_t(p.stride) + size_t(pos)] = mine;
            }
        }
    }
    cp_async_wait<0>();  // no copy may outlive the CTA
}

// The gradient launches shared by both backward entry points: clear the
// gradient records (unless the forward did), the rasterizer, the
// conversion to the caller's arrays.
static ss_status launch_bwd(const BwdParams &p, uint32_t flags, float *accum_weight,
                            cudaStream_t st, const char *name) {
    const bool accum = flags & SS_ACCUM_WEIGHT, dist = flags & SS_DISTORTION;
    ss_status es = ensure_bwd_smem();
    if (es != SS_OK) return es;
    int dev = 0, sms = 0;
    es = current_device(&dev, &sms, name);
    if (es != SS_OK) return es;
    const int64_t want = (int64_t(p.n) + 255) / 256;
    const int zgrid = int(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
    if (!(flags & SS_RECORDS_CLEARED))   // else ss_raster_fwd_records cleared them
        SS_LAUNCH("k_grad_zero", st,
                  k_grad_zero<<<zgrid, 256, 0, st>>>(reinterpret_cast<float4 *>(p.scratch),
                                                     3 * int64_t(p.n)));
    const int grid = tiles_x(p.W) * tiles_y(p.H);
    BwdParams q = p;
    q.accum_on = accum;
    if (dist)
        SS_LAUNCH("k_raster_bwd", st, (k_raster_bwd<true, true><<<grid, 256, kBwdDynSmem, st>>>(q)));
    else
        SS_LAUNCH("k_raster_bwd", st, (k_raster_bwd<true, false><<<grid, 256, kBwdDynSmem, st>>>(q)));
    SS_LAUNCH("k_grad_final", st,
              k_grad_final<<<zgrid, 256, 0, st>>>(p, p.n, accum ? accum_weight : nullptr));
    return check_launch(name);
}

// The blend masks of a backward given none (k_blend_masks) into rows of
// `stride` entries at `masks`.
static ss_status launch_masks(const SplatRecord *recs, int32_t n, const uint32_t *vals,
                              const uint32_t *offs, const uint32_t *last, int32_t W, int32_t H,
                              uint32_t *masks, int64_t stride, void *workspace, cudaStream_t st,
                              const char *name) {
    MaskParams m{};
    m.recs = recs;
    m.n = n;
    m.vals = vals;
    m.offs = offs;
    m.last = last;
    m.W = W;
    m.H = H;
    m.tiles_x = tiles_x(W);
    m.tiles = tiles_x(W) * tiles_y(H);
    m.masks = masks;
    m.stride = stride;
    m.status = static_cast<uint32_t *>(workspace);
    SS_LAUNCH("k_blend_masks", st, k_blend_masks<<<m.tiles, 256, 0, st>>>(m));
    return check_launch(name);
}

}  // namespace ss

using namespace ss;

extern "C" ss_status ss_raster_bwd_records(const void *records, int32_t n_splats,
                                           const uint32_t *vals, const uint32_t *tile_offsets,
                                           int64_t n_pairs, int32_t W, int32_t H, const float *bg,
                                           uint32_t flags, const float *T_final,
                                           const uint32_t *last_contrib,
                                           const uint32_t *blend_masks, const float *dL_dimage,
                                           const float *dist_totals, const float *dL_ddist,
                                           const ss_grads *grads, float *accum_weight,
                                           void *workspace, size_t workspace_bytes,
                                           ss_stream_t stream) {
    clear_error();
    const char *name = "ss_raster_bwd_records";
    if (W < 1 || H < 1 || W > kMaxSide || H > kMaxSide)
        return fail(SS_ERR_UNSUPPORTED, "%s: image %dx%d outside 1..%d", name, W, H, kMaxSide);
    if (flags & ~uint32_t(SS_ACCUM_WEIGHT | SS_MEDIAN_DEPTH | SS_WEIGHT_STATS | SS_DISTORTION |
                          SS_RECORDS_CLEARED))
        return fail(SS_ERR_INVALID_ARG, "%s: unknown flag bits 0x%x", name, flags);
    const bool dist = flags & SS_DISTORTION;
    if (dist && (!dist_totals || !dL_ddist))
        return fail(SS_ERR_INVALID_ARG, "%s: SS_DISTORTION set but dist_totals / dL_ddist NULL",
                    name);
    if (dist && (reinterpret_cast<uintptr_t>(dist_totals) & 15))
        return fail(SS_ERR_INVALID_ARG, "%s: dist_totals not 16-byte aligned", name);
    const int32_t n = n_splats;
    if (n < 0) return fail(SS_ERR_INVALID_ARG, "%s: n < 0", name);
    if (n > 0 && !records) return fail(SS_ERR_INVALID_ARG, "%s: records is NULL", name);
    if (reinterpret_cast<uintptr_t>(records) & 15)
        return fail(SS_ERR_INVALID_ARG, "%s: records not 16-byte aligned", name);
    if (!vals || !tile_offsets) return fail(SS_ERR_INVALID_ARG, "%s: vals/offsets NULL", name);
    if (!T_final || !last_contrib || !dL_dimage)
        return fail(SS_ERR_INVALID_ARG, "%s: T_final/last_contrib/dL_dimage NULL", name);
    if (n_pairs < 0 || n_pairs > int64_t(0xffffffffu))
        return fail(SS_ERR_INVALID_ARG, "%s: n_pairs outside 0..2^32-1", name);
    if (!grads || (n > 0 && (!grads->dmean2d || !grads->dconic || !grads->dopacity || !grads->drgb)))
        return fail(SS_ERR_INVALID_ARG, "%s: a gradient array is NULL", name);
    if (dist && n > 0 && !grads->ddepth)
        return fail(SS_ERR_INVALID_ARG, "%s: SS_DISTORTION set but grads->ddepth NULL", name);
    const bool accum = flags & SS_ACCUM_WEIGHT;
    if (accum && n > 0 && !accum_weight)
        return fail(SS_ERR_INVALID_ARG, "%s: SS_ACCUM_WEIGHT set but accum_weight NULL", name);
    const bool own_masks = !blend_masks && n_pairs > 0;
    const WsLayout L = ws_layout(n, own_masks ? n_pairs : 0, W, H);
    if (n > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)))
        return fail(SS_ERR_INVALID_ARG, "%s: workspace NULL or not 256-byte aligned", name);
    const size_t need = own_masks ? L.masks_end : L.bwd_end;
    if (n > 0 && workspace_bytes < need)
        return fail(SS_ERR_INVALID_ARG, "%s: workspace %zu bytes < %zu needed%s", name,
                    workspace_bytes, need, own_masks ? " (blend masks built here)" : "");
    if (n == 0) return SS_OK;

    cudaStream_t st = (cudaStream_t)stream;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    if (own_masks) {
        const ss_status ms = launch_masks(static_cast<const SplatRecord *>(records), n, vals,
                                          tile_offsets, last_contrib, W, H,
                                          reinterpret_cast<uint32_t *>(ws + L.masks), n_pairs,
                                          workspace, st, name);
        if (ms != SS_OK) return ms;
        blend_masks = reinterpret_cast<const uint32_t *>(ws + L.masks);
    }
    BwdParams p{};
    p.recs = static_cast<const SplatRecord *>(records);
    p.n = n;
    p.vals = vals;
    p.offs = tile_offsets;
    p.masks = blend_masks;
    p.n_pairs = n_pairs;
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
    p.ddepth = dist ? grads->ddepth : nullptr;
    p.dist_totals = reinterpret_cast<const float4 *>(dist_totals);
    p.dL_ddist = dL_ddist;
    p.accum = nullptr;
    p.scratch = reinterpret_cast<float *>(ws + L.accum);
    return launch_bwd(p, flags, accum_weight, st, name);
}

extern "C" ss_status ss_raster_bwd(const ss_splats *splats, const uint32_t *vals,
                                   const uint32_t *tile_offsets, int32_t W, int32_t H,
                                   const float *bg, uint32_t flags, const float *T_final,
                                   const uint32_t *last_contrib, const float *dL_dimage,
                                   const ss_grads *grads, float *accum_weight, void *workspace,
                                   size_t workspace_bytes, ss_stream_t stream) {
    clear_error();
    const char *name = "ss_raster_bwd";
    if (!splats) return fail(SS_ERR_INVALID_ARG, "%s: splats is NULL", name);
    if (W < 1 || H < 1 || W > kMaxSide || H > kMaxSide)
        return fail(SS_ERR_UNSUPPORTED, "%s: image %dx%d outside 1..%d", name, W, H, kMaxSide);
    if (flags & ~uint32_t(SS_ACCUM_WEIGHT | SS_MEDIAN_DEPTH | SS_WEIGHT_STATS | SS_DISTORTION |
                          SS_RECORDS_CLEARED))
        return fail(SS_ERR_INVALID_ARG, "%s: unknown flag bits 0x%x", name, flags);
    if (flags & SS_DISTORTION)
        return fail(SS_ERR_UNSUPPORTED,
                    "%s: the distortion's gradient needs its totals: use ss_raster_bwd_records",
                    name);
    if (flags & SS_RECORDS_CLEARED)
        return fail(SS_ERR_INVALID_ARG,
                    "%s: SS_RECORDS_CLEARED belongs to ss_raster_fwd_records' bwd_workspace", name);
    const int32_t n = splats->n;
    if (n < 0) return fail(SS_ERR_INVALID_ARG, "%s: n < 0", name);
    if (n > 0 && (!splats->mean2d || !splats->conic || !splats->opacity || !splats->rgb ||
                  !splats->depth))
        return fail(SS_ERR_INVALID_ARG, "%s: a splat array is NULL", name);
    if (n > 0 && (reinterpret_cast<uintptr_t>(splats->mean2d) & 7))
        return fail(SS_ERR_INVALID_ARG, "%s: mean2d not 8-byte aligned", name);
    if (!vals || !tile_offsets) return fail(SS_ERR_INVALID_ARG, "%s: vals/offsets NULL", name);
    if (!T_final || !last_contrib || !dL_dimage)
        return fail(SS_ERR_INVALID_ARG, "%s: T_final/last_contrib/dL_dimage NULL", name);
    if (!grads || (n > 0 && (!grads->dmean2d || !grads->dconic || !grads->dopacity || !grads->drgb)))
        return fail(SS_ERR_INVALID_ARG, "%s: a gradient array is NULL", name);
    const bool accum = flags & SS_ACCUM_WEIGHT;
    if (accum && n > 0 && !accum_weight)
        return fail(SS_ERR_INVALID_ARG, "%s: SS_ACCUM_WEIGHT set but accum_weight NULL", name);
    if (n == 0) return SS_OK;
    const WsLayout L = ws_layout(n, 0, W, H);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return fail(SS_ERR_INVALID_ARG, "%s: workspace NULL or not 256-byte aligned", name);
    if (workspace_bytes < L.masks + 32)
        return fail(SS_ERR_INVALID_ARG, "%s: workspace %zu bytes < %zu + 32 per pair needed", name,
                    workspace_bytes, L.masks);
    // Mask rows as long as the workspace allows; the list length is only on
    // the device (tile_offsets[tiles]): a longer one is reported through
    // the status word (ss_sort_status: SS_ERR_CAPACITY).
    const int64_t cap = int64_t((workspace_bytes - L.masks) / 32);
    const int64_t stride = cap < int64_t(0xffffffffu) ? cap : int64_t(0xffffffffu);

    cudaStream_t st = (cudaStream_t)stream;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    SplatRecord *recs = reinterpret_cast<SplatRecord *>(ws + L.recs);
    int dev = 0, sms = 0;
    ss_status s = current_device(&dev, &sms, name);
    if (s != SS_OK) return s;
    const SplatPtrs sp{splats->mean2d, splats->conic, splats->opacity, splats->rgb, splats->depth,
                       n};
    const int64_t want = (int64_t(n) + 255) / 256;
    const int rgrid = int(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
    SS_LAUNCH("k_make_records", st,
              k_make_records<<<rgrid, 256, 0, st>>>(sp, tiles_x(W), tiles_y(H), recs,
                                                    reinterpret_cast<float4 *>(ws + L.accum)));
    s = check_launch(name);
    if (s != SS_OK) return s;
    uint32_t *masks = reinterpret_cast<uint32_t *>(ws + L.masks);
    s = launch_masks(recs, n, vals, tile_offsets, last_contrib, W, H, masks, stride, workspace, st,
                     name);
    if (s != SS_OK) return s;
    BwdParams p{};
    p.recs = recs;
    p.n = n;
    p.vals = vals;
    p.offs = tile_offsets;
    p.masks = masks;
    p.n_pairs = stride;
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
    p.ddepth = nullptr;
    p.scratch = reinterpret_cast<float *>(ws + L.accum);
    // k_make_records cleared the gradient records
    return launch_bwd(p, (flags & SS_ACCUM_WEIGHT) | SS_RECORDS_CLEARED, accum_weight, st, name);
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

// The array's device address belongs to one CUDA context: it is looked up
// (cudaGetSymbolAddress, with the device current) on the first call in a
// context and cached per device under the context's process-unique id, so
// a call in another context of the same device -- a driver-API context the
// caller made current, or the primary context re-created after
// cudaDeviceReset -- looks it up again instead of using a stale address.
struct NoAllocSlot {
    unsigned long long ctx_id;   // 0: empty
    unsigned long long *ptr;
};
static std::mutex g_noalloc_mu;
static NoAllocSlot g_noalloc_slot[kMaxDevices];

// The array's address in the current context of device dev (cached; see
// above).  While `stream` is being captured only a cached address is used:
// the first call in a context is refused then, before any other CUDA call.
static ss_status noalloc_scratch(int dev, cudaStream_t stream, unsigned long long **out) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    ss_status s = check_cuda(cudaStreamIsCapturing(stream, &cs),
                             "ss_raster_bwd_noalloc: cudaStreamIsCapturing");
    if (s != SS_OK) return s;
    const bool capturing = cs != cudaStreamCaptureStatusNone;
    if (capturing && !context_id_ready())
        return fail(SS_ERR_UNSUPPORTED,
                    "ss_raster_bwd_noalloc: first call while the stream is being captured; make "
                    "one call on this device before capturing");
    unsigned long long id = 0;
    s = current_context_id(&id, "ss_raster_bwd_noalloc");
    if (s != SS_OK) return s;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (id != 0 && g_noalloc_slot[dev].ctx_id == id) {
            *out = g_noalloc_slot[dev].ptr;
            return SS_OK;
        }
    }
    if (capturing)
        return fail(SS_ERR_UNSUPPORTED,
                    "ss_raster_bwd_noalloc: first call in this context while the stream is being "
                    "captured; make one call on this device before capturing");
    void *ptr = nullptr;
    s = check_cuda(cudaGetSymbolAddress(&ptr, g_noalloc_accum),
                   "ss_raster_bwd_noalloc: cudaGetSymbolAddress");
    if (s != SS_OK) return s;
    s = current_context_id(&id, "ss_raster_bwd_noalloc");   // the lookup made the device's
                                                             // context current if it was not
    if (s != SS_OK) return s;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        g_noalloc_slot[dev] = NoAllocSlot{id, static_cast<unsigned long long *>(ptr)};
    }
    *out = static_cast<unsigned long long *>(ptr);
    return SS_OK;
}

}  // namespace ss

extern "C" ss_status ss_raster_bwd_noalloc(const void *records, int32_t n_splats,
                                   const uint32_t *vals,
                                           const uint32_t *tile_offsets, int64_t n_pairs,
                                           int32_t W, int32_t H,
                                           const float *bg, uint32_t flags, const float *T_final,
                                           const uint32_t *last_contrib,
                                           const uint32_t *blend_masks, const float *dL_dimage,
                                           const ss_grads *grads, float *accum_weight,
                                           ss_stream_t stream) {
    clear_error();
    if (W < 1 || H < 1 || W > kMaxSide || H > kMaxSide)
        return fail(SS_ERR_UNSUPPORTED, "ss_raster_bwd_noalloc: image %dx%d outside 1..%d", W, H,
                    kMaxSide);
    // SS_RECORDS_CLEARED is accepted and ignored: this call keeps no gradient
    // records and always clears its own outputs first.
    if (flags & ~uint32_t(SS_ACCUM_WEIGHT | SS_MEDIAN_DEPTH | SS_WEIGHT_STATS | SS_DISTORTION |
                          SS_RECORDS_CLEARED))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: unknown flag bits 0x%x", flags);
    if (flags & SS_DISTORTION)
        return fail(SS_ERR_UNSUPPORTED,
                    "ss_raster_bwd_noalloc: SS_DISTORTION needs ss_raster_bwd_records");
    const int32_t n = n_splats;
    if (n < 0) return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: n < 0");
    if (n > kNoAllocMaxSplats)
        return fail(SS_ERR_UNSUPPORTED,
                    "ss_raster_bwd_noalloc: %d splats exceed its fixed scratch of %d splats; "
                    "use ss_raster_bwd_records with a workspace",
                    n, kNoAllocMaxSplats);
    if (n > 0 && !records) return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: records is NULL");
    if (reinterpret_cast<uintptr_t>(records) & 15)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: records not 16-byte aligned");
    if (!vals || !tile_offsets)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: vals/offsets NULL");
    if (!T_final || !last_contrib || !dL_dimage)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: T_final/last_contrib/dL_dimage NULL");
    if (n_pairs < 0 || n_pairs > int64_t(0xffffffffu))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: n_pairs outside 0..2^32-1");
    if (n_pairs > 0 && !blend_masks)
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: blend_masks is NULL");
    if (!grads || (n > 0 && (!grads->dmean2d || !grads->dconic || !grads->dopacity || !grads->drgb)))
        return fail(SS_ERR_INVALID_ARG, "ss_raster_bwd_noalloc: a gradient array is NULL");
    const bool accum = flags & SS_ACCUM_WEIGHT;
    if (accum && n > 0 && !accum_weight)
        return fail(SS_ERR_INVALID_ARG,
                    "ss_raster_bwd_noalloc: SS_ACCUM_WEIGHT set but accum_weight NULL");
    if (n == 0) return SS_OK;

    int dev = 0, sms = 0;
    ss_status s = check_cuda(cudaGetDevice(&dev), "ss_raster_bwd_noalloc: cudaGetDevice");
    if (s != SS_OK) return s;
    if (dev < 0 || dev >= kMaxDevices)
        return fail(SS_ERR_UNSUPPORTED, "ss_raster_bwd_noalloc: device %d >= %d", dev, kMaxDevices);
    unsigned long long *scratch = nullptr;
    if (accum) {
        s = noalloc_scratch(dev, (cudaStream_t)stream, &scratch);
        if (s != SS_OK) return s;
    }

    BwdParams p{};
    p.recs = static_cast<const SplatRecord *>(records);
    p.n = n;
    p.vals = vals;
    p.offs = tile_offsets;
    p.masks = blend_masks;
    p.n_pairs = n_pairs;
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
    p.accum = scratch;
    cudaStream_t st = (cudaStream_t)stream;
    s = ensure_bwd_smem();
    if (s != SS_OK) return s;
    s = current_device(&dev, &sms, "ss_raster_bwd_noalloc: device query");
    if (s != SS_OK) return s;
    const int64_t want = (int64_t(n) + 255) / 256;
    const int zgrid = int(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
    // k_bwd_zero clears this call's part of the shared array before use.
    SS_LAUNCH("k_bwd_zero", st, k_bwd_zero<<<zgrid, 256, 0, st>>>(p, n, accum));
    const int grid = tiles_x(W) * tiles_y(H);
    p.accum_on = accum;
    SS_LAUNCH("k_raster_bwd", st, (k_raster_bwd<false, false><<<grid, 256, kBwdDynSmem, st>>>(p)));
    if (accum)
        SS_LAUNCH("k_accum_final", st, k_accum_final<<<zgrid, 256, 0, st>>>(p.accum, accum_weight, n));
    return check_launch("ss_raster_bwd_noalloc");
}

namespace ss {
cudaError_t debug_word_bwd(uint32_t *out) { return read_and_clear_debug_word(out); }
}  // namespace ss
