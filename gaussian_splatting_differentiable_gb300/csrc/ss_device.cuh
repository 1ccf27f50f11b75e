// Device functions shared by the binning, forward and backward kernels.
//
// The forward and backward kernels must take the same per-(pixel, splat)
// decision "is this splat blended here", or the backward replay would walk a
// different list than the forward composited.  Both therefore stage splats
// and evaluate the Gaussian exponent through the functions below, written
// with explicit round-to-nearest intrinsics so that the compiler cannot
// contract or reassociate them differently in the two kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace ss {

constexpr float kAlphaMin = 1.0f / 255.0f;  // skip threshold on alpha
constexpr float kAlphaMax = 0.99f;          // alpha cap
constexpr float kTEps = 1e-4f;              // transmittance floor
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

// Binning ellipse margins: k widened by 2^-10 relative and absolute.
constexpr float kKRel = 1.0f + 1.0f / 1024.0f;
constexpr float kKAbs = 1.0f / 1024.0f;

// Device-side bounds checks of the SS_DEBUG_BOUNDS build.  A failed check
// sets its bit in this translation unit's debug word (ss_debug_status reads
// and clears the words of every unit) and the access it guards is skipped
// or clamped: nothing traps.  In the normal build SS_BAD(...) is the
// constant false and its condition is not evaluated.
enum : unsigned {
    kDbgSortScatter = 1u,   // a sort pass's destination outside the pairs
    kDbgSortRank = 2u,      // a sort pass's rank outside its partition
    kDbgFwdList = 4u,       // a forward tile list outside the pairs
    kDbgBwdList = 8u,       // a backward tile list outside the pairs
    kDbgBwdLast = 16u,      // a last_contrib beyond its tile's list
    kDbgBwdSplat = 32u,     // a gradient record index outside the splats
    kDbgMaskList = 64u      // a blend-mask tile list outside the mask rows
};
#ifdef SS_DEBUG_BOUNDS
static __device__ unsigned int g_debug_word;
#define SS_BAD(bad, bit) ((bad) ? (atomicOr(&::ss::g_debug_word, (bit)), true) : false)
// Host: ORs this unit's debug word into *out and clears it.
static inline cudaError_t read_and_clear_debug_word(uint32_t *out) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_debug_word, sizeof v);
    if (e != cudaSuccess) return e;
    *out |= v;
    if (v) {
        const unsigned z = 0;
        e = cudaMemcpyToSymbol(g_debug_word, &z, sizeof z);
    }
    return e;
}
#else
#define SS_BAD(bad, bit) false
static inline cudaError_t read_and_clear_debug_word(uint32_t *) { return cudaSuccess; }
#endif

struct SplatPtrs {
    const float *mean2d, *conic, *opacity, *rgb, *depth;
    int32_t n;
};

// 2^x, the hardware approximation (relative error about 2^-22 on [-8, 0]).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ln(x) for positive, finite, normal float32 x: x = m 2^e, m in [1, 2),
// ln x = e ln 2 + 2 atanh(t), t = (m - 1) / (m + 1), atanh by its Taylor
// series to t^15 (Horner).  Only IEEE-rounded + - * /, so the value is the
// same bits on any IEEE float32 machine: the binning must agree bit for bit
// with an independent CPU evaluation.
__device__ __forceinline__ float ln_series(float x) {
    const uint32_t u = __float_as_uint(x);
    const int e = int((u >> 23) & 0xffu) - 127;
    const float m = __uint_as_float((u & 0x007fffffu) | 0x3f800000u);
    const float t = __fdiv_rn(__fsub_rn(m, 1.0f), __fadd_rn(m, 1.0f));
    const float t2 = __fmul_rn(t, t);
    float p = 1.0f / 15.0f;
    p = __fadd_rn(__fmul_rn(p, t2), 1.0f / 13.0f);
    p = __fadd_rn(__fmul_rn(p, t2), 1.0f / 11.0f);
    p = __fadd_rn(__fmul_rn(p, t2), 1.0f / 9.0f);
    p = __fadd_rn(__fmul_rn(p, t2), 1.0f / 7.0f);
    p = __fadd_rn(__fmul_rn(p, t2), 1.0f / 5.0f);
    p = __fadd_rn(__fmul_rn(p, t2), 1.0f / 3.0f);
    p = __fadd_rn(__fmul_rn(p, t2), 1.0f);
    const float lnm = __fmul_rn(2.0f, __fmul_rn(t, p));
    return __fadd_rn(__fmul_rn(__int2float_rn(e), kLn2), lnm);
}

// Tile rectangle of splat i (inclusive tile coordinates).  Returns -1 if the
// splat is culled (non-finite input, depth <= 0, conic not positive
// definite, opacity < 1/255), 0 if it touches no tile of the image, else 1.
// The rectangle is the axis-aligned box of the ellipse where alpha >= 1/255
// is possible: {d : d^T Q d <= k}, k = 2 ln(255 o), half widths
// sqrt(k c / det) and sqrt(k a / det), Q = [[a, b], [b, c]].
__device__ __forceinline__ int splat_tile_rect(const SplatPtrs &s, int64_t i, int32_t tiles_x,
                                               int32_t tiles_y, int &x0, int &y0, int &x1,
                                               int &y1, uint32_t &depth_bits, float &rx_out,
                                               float &ry_out) {
    const float2 mu = reinterpret_cast<const float2 *>(s.mean2d)[i];
    const float a = s.conic[3 * i], b = s.conic[3 * i + 1], c = s.conic[3 * i + 2];
    const float o = s.opacity[i], d = s.depth[i];
    const float r = s.rgb[3 * i], g = s.rgb[3 * i + 1], bl = s.rgb[3 * i + 2];
    if (!isfinite(mu.x) || !isfinite(mu.y) || !isfinite(a) || !isfinite(b) || !isfinite(c) ||
        !isfinite(o) || !isfinite(d) || !isfinite(r) || !isfinite(g) || !isfinite(bl))
        return -1;
    if (!(d > 0.0f) || !(a > 0.0f) || !(c > 0.0f)) return -1;
    const float det = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, b));
    if (!(det > 0.0f)) return -1;
    if (!(o >= kAlphaMin)) return -1;
    const float x = __fmul_rn(255.0f, o);
    if (isinf(x)) return -1;
    float k = __fmul_rn(2.0f, ln_series(x));
    k = __fadd_rn(__fmul_rn(k, kKRel), kKAbs);
    const float rx = __fsqrt_rn(__fdiv_rn(__fmul_rn(k, c), det));
    const float ry = __fsqrt_rn(__fdiv_rn(__fmul_rn(k, a), det));
    if (rx != rx || ry != ry) return -1;
    rx_out = rx;
    ry_out = ry;
    float fx0 = floorf(__fmul_rn(__fsub_rn(mu.x, rx), 0.0625f));
    float fx1 = floorf(__fmul_rn(__fadd_rn(mu.x, rx), 0.0625f));
    float fy0 = floorf(__fmul_rn(__fsub_rn(mu.y, ry), 0.0625f));
    float fy1 = floorf(__fmul_rn(__fadd_rn(mu.y, ry), 0.0625f));
    fx0 = fmaxf(fx0, 0.0f);
    fy0 = fmaxf(fy0, 0.0f);
    fx1 = fminf(fx1, float(tiles_x - 1));
    fy1 = fminf(fy1, float(tiles_y - 1));
    depth_bits = __float_as_uint(d);
    if (fx0 > fx1 || fy0 > fy1) return 0;
    x0 = int(fx0);
    y0 = int(fy0);
    x1 = int(fx1);
    y1 = int(fy1);
    return 1;
}

// A splat as the rasterizers read it: one 64-byte record, written once by
// the binning kernel, gathered by index (two aligned 32-byte sectors) by
// the forward and backward kernels.  The exponent is handled in base 2:
// e2 = -sigma log2(e) = A dx^2 + B dx dy + C dy^2 with A = -a log2(e) / 2,
// B = -b log2(e), C = -c log2(e) / 2; the splat is skipped at a pixel iff
// e2 < thr = -log2(255 o)  (alpha < 1/255).
struct __align__(16) SplatGeo {
    float mx, my, A, B;
};
struct __align__(16) SplatGeo2 {
    float C, thr, o, depth;
};
struct __align__(16) SplatCol {
    float r, g, b;
    uint32_t idx;  // the splat's own index (the backward's atomic target)
};
// Conservative box of pixel centres where e2 >= thr can hold (the alpha
// ellipse's bounding box grown by 0.4 % + 0.01 px); used only to skip work.
struct __align__(16) SplatBox {
    float x0, x1, y0, y1;
};
struct __align__(16) SplatRecord {
    SplatGeo geo;
    SplatGeo2 geo2;
    SplatCol col;
    SplatBox box;
};
static_assert(sizeof(SplatRecord) == 64, "record is 64 bytes");

// The record of a splat that is never blended (culled or not a splat).
__device__ __forceinline__ SplatRecord invisible_record() {
    SplatRecord r;
    r.geo = SplatGeo{0.f, 0.f, 0.f, 0.f};
    r.geo2 = SplatGeo2{0.f, __int_as_float(0x7f800000), 0.f, 0.f};
    r.col = SplatCol{0.f, 0.f, 0.f, 0u};
    r.box = SplatBox{1.f, -1.f, 1.f, -1.f};
    return r;
}

// Record of splat idx from the SoA inputs; rx, ry: the half widths of its
// binning rectangle (the alpha ellipse's box, k already widened), which the
// cull box grows by 0.4 % + 0.01 px.
__device__ __forceinline__ SplatRecord make_record(const SplatPtrs &s, uint32_t idx, float rx,
                                                   float ry) {
    const float2 mu = reinterpret_cast<const float2 *>(s.mean2d)[idx];
    const float a = s.conic[3 * idx], b = s.conic[3 * idx + 1], c = s.conic[3 * idx + 2];
    const float o = s.opacity[idx];
    SplatRecord r;
    r.geo = SplatGeo{mu.x, mu.y, __fmul_rn(-0.5f * kLog2e, a), __fmul_rn(-kLog2e, b)};
    r.geo2 = SplatGeo2{__fmul_rn(-0.5f * kLog2e, c), -log2f(__fmul_rn(255.0f, o)), o, s.depth[idx]};
    r.col = SplatCol{s.rgb[3 * idx], s.rgb[3 * idx + 1], s.rgb[3 * idx + 2], idx};
    const float bx = rx * 1.004f + 0.01f, by = ry * 1.004f + 0.01f;
    r.box = SplatBox{mu.x - bx, mu.x + bx, mu.y - by, mu.y + by};
    return r;
}

// The record of splat idx computed from the SoA inputs, bit for bit what
// the binning writes (the culled get the invisible record).
__device__ __forceinline__ SplatRecord record_of(const SplatPtrs &s, uint32_t idx, int32_t tiles_x,
                                                 int32_t tiles_y) {
    int x0, y0, x1, y1;
    uint32_t dbits;
    float rx = 0.0f, ry = 0.0f;
    const int st = splat_tile_rect(s, idx, tiles_x, tiles_y, x0, y0, x1, y1, dbits, rx, ry);
    return st >= 0 ? make_record(s, idx, rx, ry) : invisible_record();
}

// 16-byte asynchronous global -> shared copy (cp.async, L2 only).
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The backward's staging: the record without its cull box (the forward's
// blend masks replace the box test there).
__device__ __forceinline__ void stage_record3_async(const SplatRecord *recs, uint32_t idx, int32_t n,
                                                    SplatGeo *geo, SplatGeo2 *geo2, SplatCol *col,
                                                    int t) {
    if (idx < uint32_t(n)) {
        const SplatRecord *r = recs + idx;
        cp_async16(&geo[t], &r->geo);
        cp_async16(&geo2[t], &r->geo2);
        cp_async16(&col[t], &r->col);
    } else {
        const SplatRecord r = invisible_record();
        geo[t] = r.geo;
        geo2[t] = r.geo2;
        col[t] = r.col;
    }
}

// Stage record `idx` (or the invisible record if idx >= n) into shared
// memory slot `t` of the four arrays with 16-byte asynchronous copies.
__device__ __forceinline__ void stage_record_async(const SplatRecord *recs, uint32_t idx, int32_t n,
                                                   SplatGeo *geo, SplatGeo2 *geo2, SplatCol *col,
                                                   SplatBox *box, int t) {
    if (idx < uint32_t(n)) {
        const SplatRecord *r = recs + idx;
        cp_async16(&geo[t], &r->geo);
        cp_async16(&geo2[t], &r->geo2);
        cp_async16(&col[t], &r->col);
        cp_async16(&box[t], &r->box);
    } else {
        const SplatRecord r = invisible_record();
        geo[t] = r.geo;
        geo2[t] = r.geo2;
        col[t] = r.col;
        box[t] = r.box;
    }
}

// Base-2 exponent of the splat's Gaussian at pixel centre (px, py); also
// returns d = pixel - mean.  Identical operations in forward and backward.
__device__ __forceinline__ float eval_e2(const SplatGeo &g, float C, float px, float py,
                                         float &dx, float &dy) {
    dx = __fsub_rn(px, g.mx);
    dy = __fsub_rn(py, g.my);
    const float t = __fmaf_rn(g.A, dx, __fmul_rn(g.B, dy));
    return __fmaf_rn(dx, t, __fmul_rn(__fmul_rn(C, dy), dy));
}

// alpha = min(0.99, o 2^e2), and the unclamped o G.
__device__ __forceinline__ float eval_alpha(float o, float G, float &oG) {
    oG = __fmul_rn(o, G);
    return fminf(kAlphaMax, oG);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

}  // namespace ss
