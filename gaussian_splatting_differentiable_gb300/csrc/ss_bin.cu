// Tile binning ("Phase 5 step 30b -- kernel-by-kernel timing", emit_pairs:
// tile id computation plus an atomic counter update).
//
// One thread per splat computes its tile rectangle; the CTA scans its pair
// counts (warp shuffles, then the eight warp totals) and one thread takes
// the CTA's slots with a single 64-bit atomic add, so the global counter
// sees one atomic per 256 splats rather than one per splat.  Each lane then writes its pairs into its slots.  The
// same thread also writes the splat's 64-byte record (derived exponent
// coefficients, threshold, colour, depth, cull box), which the forward and
// backward rasterizers gather by index instead of the five SoA inputs.
// The CTA also takes the smallest and largest depth bits of its splats that
// have pairs (warp reductions, one 64-bit atomic min and max per CTA): the
// device-count sort sorts only the depth bits in which the pairs can differ.
#include "ss_device.cuh"
#include "ss_internal.h"
#include "ss_profile.h"

namespace ss {

struct BinParams {
    SplatPtrs s;
    int32_t tiles_x, tiles_y;
    uint64_t *keys;
    uint32_t *vals;
    int64_t capacity;
    unsigned long long *counters;  // [0] pairs, [1] culled, [2] / [3] min / max depth bits
    SplatRecord *records;          // [n] 64-byte records for the rasterizers
};

// Six CTAs a SM (40 registers, one 4-byte spill): 0.068 -> 0.065 ms at 2M
// splats, measured against the compiler's own choice (42 registers).
__global__ void __launch_bounds__(256, 6) k_emit_pairs(BinParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    int x0 = 0, y0 = 0, x1 = -1, y1 = -1, st = 0;
    uint32_t dbits = 0;
    float rx = 0.0f, ry = 0.0f;
    if (i < p.s.n)
        st = splat_tile_rect(p.s, i, p.tiles_x, p.tiles_y, x0, y0, x1, y1, dbits, rx, ry);
    const uint32_t cnt = st > 0 ? uint32_t(x1 - x0 + 1) * uint32_t(y1 - y0 + 1) : 0u;
    if (i < p.s.n) {
        const SplatRecord r = st >= 0 ? make_record(p.s, uint32_t(i), rx, ry) : invisible_record();
        float4 *dst = reinterpret_cast<float4 *>(p.records + i);
        dst[0] = *reinterpret_cast<const float4 *>(&r.geo);
        dst[1] = *reinterpret_cast<const float4 *>(&r.geo2);
        dst[2] = *reinterpret_cast<const float4 *>(&r.col);
        dst[3] = *reinterpret_cast<const float4 *>(&r.box);
    }

    // Block-wide exclusive scan of the pair counts, then one 64-bit atomic
    // per CTA on the global counter (same-address atomics serialise in L2).
    __shared__ uint32_t s_wsum[8], s_wcull[8], s_wlo[8], s_whi[8];
    __shared__ unsigned long long s_base;
    const int warp = threadIdx.x >> 5;
    uint32_t inc = cnt;  // warp inclusive scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    const uint32_t culled = __ballot_sync(0xffffffffu, st < 0);
    const uint32_t wlo = __reduce_min_sync(0xffffffffu, cnt ? dbits : 0xffffffffu);
    const uint32_t whi = __reduce_max_sync(0xffffffffu, cnt ? dbits : 0u);
    if (lane == 31) s_wsum[warp] = inc;
    if (lane == 0) {
        s_wcull[warp] = __popc(culled);
        s_wlo[warp] = wlo;
        s_whi[warp] = whi;
    }
    __syncthreads();
    uint32_t before = 0;
    if (threadIdx.x == 0) {
        uint32_t tot = 0, tc = 0, lo = 0xffffffffu, hi = 0u;
        for (int w = 0; w < 8; ++w) {
            tot += s_wsum[w], tc += s_wcull[w];
            lo = min(lo, s_wlo[w]);
            hi = max(hi, s_whi[w]);
        }
        s_base = tot ? atomicAdd(p.counters, (unsigned long long)tot) : 0ull;
        if (tc) atomicAdd(p.counters + 1, (unsigned long long)tc);
        if (tot) {
            atomicMin(p.counters + 2, (unsigned long long)lo);
            atomicMax(p.counters + 3, (unsigned long long)hi);
        }
    }
    for (int w = 0; w < warp; ++w) before += s_wsum[w];
    __syncthreads();
    if (!cnt) return;

    unsigned long long pos = s_base + before + (inc - cnt);
    const unsigned long long cap = (unsigned long long)p.capacity;
    for (int ty = y0; ty <= y1; ++ty) {
        const uint64_t row = uint64_t(ty) * uint64_t(p.tiles_x);
        for (int tx = x0; tx <= x1; ++tx, ++pos) {
            if (pos < cap) {
                p.keys[pos] = ((row + uint64_t(tx)) << 32) | dbits;
                p.vals[pos] = uint32_t(i);
            }
        }
    }
}

}  // namespace ss

using namespace ss;

extern "C" ss_status ss_bin_tiles(const ss_splats *splats, int32_t W, int32_t H, uint64_t *keys,
                                  uint32_t *vals, int64_t capacity, uint64_t *d_counters,
                                  void *records, ss_stream_t stream) {
    clear_error();
    if (!splats) return fail(SS_ERR_INVALID_ARG, "ss_bin_tiles: splats is NULL");
    if (W < 1 || H < 1 || W > kMaxSide || H > kMaxSide)
        return fail(SS_ERR_UNSUPPORTED, "ss_bin_tiles: image %dx%d outside 1..%d", W, H, kMaxSide);
    if (splats->n < 0) return fail(SS_ERR_INVALID_ARG, "ss_bin_tiles: n < 0");
    if (splats->n > 0 && (!splats->mean2d || !splats->conic || !splats->opacity || !splats->rgb ||
                          !splats->depth))
        return fail(SS_ERR_INVALID_ARG, "ss_bin_tiles: a splat array is NULL");
    if (capacity < 0) return fail(SS_ERR_INVALID_ARG, "ss_bin_tiles: capacity < 0");
    if (capacity > 0 && (!keys || !vals))
        return fail(SS_ERR_INVALID_ARG, "ss_bin_tiles: keys/vals NULL with capacity > 0");
    if (!d_counters) return fail(SS_ERR_INVALID_ARG, "ss_bin_tiles: d_counters is NULL");
    if (splats->n > 0 && !records) return fail(SS_ERR_INVALID_ARG, "ss_bin_tiles: records is NULL");
    if (reinterpret_cast<uintptr_t>(records) & 15)
        return fail(SS_ERR_INVALID_ARG, "ss_bin_tiles: records not 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(d_counters) & 7) || (reinterpret_cast<uintptr_t>(keys) & 7) ||
        (splats->n > 0 && (reinterpret_cast<uintptr_t>(splats->mean2d) & 7)))
        return fail(SS_ERR_INVALID_ARG, "ss_bin_tiles: keys, counters and mean2d need 8-byte alignment");
    cudaStream_t st = (cudaStream_t)stream;
    ss_status s = check_cuda(cudaMemsetAsync(d_counters, 0, 32, st), "ss_bin_tiles: memset");
    if (s == SS_OK)  // [2] = the largest u64: no depth seen yet
        s = check_cuda(cudaMemsetAsync(d_counters + 2, 0xff, 8, st), "ss_bin_tiles: memset");
    if (s != SS_OK || splats->n == 0) return s;
    BinParams p{};
    p.s = SplatPtrs{splats->mean2d, splats->conic, splats->opacity, splats->rgb, splats->depth,
                    splats->n};
    p.tiles_x = tiles_x(W);
    p.tiles_y = tiles_y(H);
    p.keys = keys;
    p.vals = vals;
    p.capacity = capacity;
    p.counters = reinterpret_cast<unsigned long long *>(d_counters);
    p.records = static_cast<SplatRecord *>(records);
    const int grid = int((int64_t(splats->n) + 255) / 256);
    SS_LAUNCH("k_emit_pairs", st, k_emit_pairs<<<grid, 256, 0, st>>>(p));
    return check_launch("ss_bin_tiles: k_emit_pairs");
}

namespace ss {
cudaError_t debug_word_bin(uint32_t *out) { return read_and_clear_debug_word(out); }
}  // namespace ss
