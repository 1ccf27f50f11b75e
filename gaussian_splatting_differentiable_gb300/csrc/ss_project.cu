// Projection of 3D Gaussian splats to the rasterizer's 2D splats, and its
// backward (the forward projection and "project_backwards" kernels of
// "Phase 5 step 30b -- kernel-by-kernel timing", measurement table; the model
// is stated in include/ss_project.h).
//
// Both kernels are per-splat maps with no reuse between splats, so they are
// bound by HBM: one thread per splat, every load and store of a warp covering
// contiguous memory.  The bulk of the bytes is the SH colour coefficients
// (48 floats a splat at degree 3), stored coefficient-major so that the
// warp's load of coefficient k is one contiguous 128-byte line per channel.
// The small AoS fields (mean3, scale, quat) are read as 3 / 3 / 4 consecutive
// floats per thread: a warp touches 384-512 contiguous bytes and L1 merges
// the three or four partial-sector loads.  The backward recomputes the
// forward's intermediates instead of storing them (a few hundred FLOPs
// against ~500 bytes of traffic a splat).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "ss_internal.h"
#include "ss_profile.h"
#include "ss_project.h"

namespace ss {
namespace {

struct ProjParams {
    const float *mean3, *scale, *quat, *sh;
    int n;
    float R[9], t[3], campos[3], fx, fy, cx, cy, near_z, blur;
    float *mean2d, *conic, *depth, *rgb;           // forward outputs
    const float *gmean2d, *gconic, *grgb;          // backward inputs
    float *dmean3, *dscale, *dquat, *dsh;          // backward outputs
};

// Real spherical harmonics of degree <= 3 written out as polynomials of the
// unit direction (x, y, z).  Each constant is N_lm times the integer factor
// of the polynomial P_l^(|m|)(z) Re/Im((x + iy)^|m|):
constexpr float kY00 = 0.28209479177387814f;  // sqrt(1 / (4 pi))
constexpr float kY1 = 0.4886025119029199f;    // sqrt(3 / (4 pi)):     y, z, x
constexpr float kY2a = 1.0925484305920792f;   // sqrt(15 / (4 pi)):    xy, yz, xz
constexpr float kY2b = 0.31539156525252005f;  // sqrt(5 / (16 pi)):    3z^2 - 1
constexpr float kY2c = 0.5462742152960396f;   // sqrt(15 / (16 pi)):   x^2 - y^2
constexpr float kY3a = 0.5900435899266435f;   // sqrt(35 / (32 pi)):   3x^2 y - y^3, x^3 - 3x y^2
constexpr float kY3b = 2.890611442640554f;    // sqrt(105 / (4 pi)):   xyz
constexpr float kY3c = 0.4570457994644658f;   // sqrt(21 / (32 pi)):   y (5z^2 - 1), x (5z^2 - 1)
constexpr float kY3d = 0.3731763325901154f;   // sqrt(7 / (16 pi)):    5z^3 - 3z
constexpr float kY3e = 1.445305721320277f;    // sqrt(105 / (16 pi)):  z (x^2 - y^2)

template <int DEG>
__device__ __forceinline__ void sh_eval(float x, float y, float z, float *Y) {
    Y[0] = kY00;
    if (DEG >= 1) {
        Y[1] = kY1 * y;
        Y[2] = kY1 * z;
        Y[3] = kY1 * x;
    }
    if (DEG >= 2) {
        const float xx = x * x, yy = y * y, zz = z * z;
        Y[4] = kY2a * x * y;
        Y[5] = kY2a * y * z;
        Y[6] = kY2b * (3.0f * zz - 1.0f);
        Y[7] = kY2a * x * z;
        Y[8] = kY2c * (xx - yy);
        if (DEG >= 3) {
            Y[9] = kY3a * y * (3.0f * xx - yy);
            Y[10] = kY3b * x * y * z;
            Y[11] = kY3c * y * (5.0f * zz - 1.0f);
            Y[12] = kY3d * z * (5.0f * zz - 3.0f);
            Y[13] = kY3c * x * (5.0f * zz - 1.0f);
            Y[14] = kY3e * z * (xx - yy);
            Y[15] = kY3a * x * (xx - 3.0f * yy);
        }
    }
}

// g += sum_k dY[k] grad Y_k, the gradient of the polynomials above in
// (x, y, z); the caller projects it onto the sphere's tangent plane.
template <int DEG>
__device__ __forceinline__ void sh_grad(float x, float y, float z, const float *dY, float &gx,
                                        float &gy, float &gz) {
    if (DEG >= 1) {
        gx = fmaf(kY1, dY[3], gx);
        gy = fmaf(kY1, dY[1], gy);
        gz = fmaf(kY1, dY[2], gz);
    }
    if (DEG >= 2) {
        gx += kY2a * (y * dY[4] + z * dY[7]) + 2.0f * kY2c * x * dY[8];
        gy += kY2a * (x * dY[4] + z * dY[5]) - 2.0f * kY2c * y * dY[8];
        gz += kY2a * (y * dY[5] + x * dY[7]) + 6.0f * kY2b * z * dY[6];
        if (DEG >= 3) {
            const float xx = x * x, yy = y * y, zz = z * z;
            const float t5 = 5.0f * zz - 1.0f;
            gx += kY3a * (6.0f * x * y * dY[9] + 3.0f * (xx - yy) * dY[15]) +
                  kY3b * y * z * dY[10] + kY3c * t5 * dY[13] + 2.0f * kY3e * x * z * dY[14];
            gy += kY3a * (3.0f * (xx - yy) * dY[9] - 6.0f * x * y * dY[15]) +
                  kY3b * x * z * dY[10] + kY3c * t5 * dY[11] - 2.0f * kY3e * y * z * dY[14];
            gz += kY3b * x * y * dY[10] + 10.0f * kY3c * z * (y * dY[11] + x * dY[13]) +
                  kY3d * (15.0f * zz - 3.0f) * dY[12] + kY3e * (xx - yy) * dY[14];
        }
    }
}

// Everything the forward computes for one splat except the colour.
struct Geo {
    float xc, yc, zc, iz;       // camera-space mean, 1/z
    float u[4], inv_qn;         // unit quaternion (w, x, y, z), 1/|q|
    float r[9];                 // splat rotation, row-major
    float s[3];
    float M[9];                 // r diag(s)
    float c3[6];                // 3D covariance 00 01 02 11 12 22
    float T[6];                 // J Rc, 2x3 row-major
    float U[6];                 // T c3
    float p, q, rr, det;        // 2D covariance [[p, q], [q, rr]] with blur
    float ca, cb, cc;           // conic
    float mx, my;               // mean2d
    float dx, dy, dz, inv_len;  // unit view direction, 1/|mean - campos|
    bool valid;
};

__device__ __forceinline__ float c3at(const float *c3, int i, int j) {
    // symmetric 3x3 stored 00 01 02 11 12 22
    const int a = i < j ? i : j, b = i < j ? j : i;
    return c3[a == 0 ? b : (a == 1 ? 2 + b : 5)];
}

__device__ __forceinline__ void geometry(const ProjParams &P, int i, Geo &g) {
    const float px = P.mean3[3 * i], py = P.mean3[3 * i + 1], pz = P.mean3[3 * i + 2];
    g.xc = fmaf(P.R[0], px, fmaf(P.R[1], py, fmaf(P.R[2], pz, P.t[0])));
    g.yc = fmaf(P.R[3], px, fmaf(P.R[4], py, fmaf(P.R[5], pz, P.t[1])));
    g.zc = fmaf(P.R[6], px, fmaf(P.R[7], py, fmaf(P.R[8], pz, P.t[2])));
    g.iz = 1.0f / g.zc;

    const float4 q = reinterpret_cast<const float4 *>(P.quat)[i];
    const float qn2 = q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w;
    g.inv_qn = 1.0f / sqrtf(qn2);
    const float w = q.x * g.inv_qn, x = q.y * g.inv_qn, y = q.z * g.inv_qn, z = q.w * g.inv_qn;
    g.u[0] = w, g.u[1] = x, g.u[2] = y, g.u[3] = z;
    g.r[0] = 1.0f - 2.0f * (y * y + z * z);
    g.r[1] = 2.0f * (x * y - w * z);
    g.r[2] = 2.0f * (x * z + w * y);
    g.r[3] = 2.0f * (x * y + w * z);
    g.r[4] = 1.0f - 2.0f * (x * x + z * z);
    g.r[5] = 2.0f * (y * z - w * x);
    g.r[6] = 2.0f * (x * z - w * y);
    g.r[7] = 2.0f * (y * z + w * x);
    g.r[8] = 1.0f - 2.0f * (x * x + y * y);
    g.s[0] = P.scale[3 * i], g.s[1] = P.scale[3 * i + 1], g.s[2] = P.scale[3 * i + 2];
#pragma unroll
    for (int a = 0; a < 3; ++a)
#pragma unroll
        for (int b = 0; b < 3; ++b) g.M[3 * a + b] = g.r[3 * a + b] * g.s[b];
    auto dot3 = [](const float *a, const float *b) { return a[0] * b[0] + a[1] * b[1] + a[2] * b[2]; };
    g.c3[0] = dot3(g.M, g.M);
    g.c3[1] = dot3(g.M, g.M + 3);
    g.c3[2] = dot3(g.M, g.M + 6);
    g.c3[3] = dot3(g.M + 3, g.M + 3);
    g.c3[4] = dot3(g.M + 3, g.M + 6);
    g.c3[5] = dot3(g.M + 6, g.M + 6);

    const float fxz = P.fx * g.iz, fyz = P.fy * g.iz;
    const float xz = g.xc * g.iz, yz = g.yc * g.iz;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        g.T[j] = fxz * (P.R[j] - xz * P.R[6 + j]);
        g.T[3 + j] = fyz * (P.R[3 + j] - yz * P.R[6 + j]);
    }
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int j = 0; j < 3; ++j)
            g.U[3 * a + j] = g.T[3 * a] * c3at(g.c3, 0, j) + g.T[3 * a + 1] * c3at(g.c3, 1, j) +
                             g.T[3 * a + 2] * c3at(g.c3, 2, j);
    g.p = dot3(g.U, g.T) + P.blur;
    g.q = dot3(g.U, g.T + 3);
    g.rr = dot3(g.U + 3, g.T + 3) + P.blur;
    g.det = g.p * g.rr - g.q * g.q;
    const float id = 1.0f / g.det;
    g.ca = g.rr * id;
    g.cb = -g.q * id;
    g.cc = g.p * id;
    g.mx = fmaf(P.fx, xz, P.cx);
    g.my = fmaf(P.fy, yz, P.cy);

    const float vx = px - P.campos[0], vy = py - P.campos[1], vz = pz - P.campos[2];
    g.inv_len = 1.0f / sqrtf(vx * vx + vy * vy + vz * vz);
    g.dx = vx * g.inv_len, g.dy = vy * g.inv_len, g.dz = vz * g.inv_len;

    g.valid = g.zc > P.near_z && g.det > 0.0f && isfinite(g.mx) && isfinite(g.my) &&
              isfinite(g.ca) && isfinite(g.cb) && isfinite(g.cc) && isfinite(g.inv_len);
}

template <int DEG>
__global__ void __launch_bounds__(256) k_project_fwd(ProjParams P) {
    constexpr int K = (DEG + 1) * (DEG + 1);
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= P.n) return;
    Geo g;
    geometry(P, i, g);
    float Y[K];
    sh_eval<DEG>(g.dx, g.dy, g.dz, Y);
    float col[3];
    const size_t n = size_t(P.n);
#pragma unroll
    for (int c = 0; c < 3; ++c) {
        float acc = 0.5f;
#pragma unroll
        for (int k = 0; k < K; ++k) acc = fmaf(__ldg(P.sh + (size_t(3 * k + c)) * n + i), Y[k], acc);
        col[c] = fmaxf(acc, 0.0f);
    }
    const bool ok = g.valid && isfinite(col[0]) && isfinite(col[1]) && isfinite(col[2]);
    reinterpret_cast<float2 *>(P.mean2d)[i] = ok ? make_float2(g.mx, g.my) : make_float2(0.f, 0.f);
    P.conic[3 * i] = ok ? g.ca : 0.0f;
    P.conic[3 * i + 1] = ok ? g.cb : 0.0f;
    P.conic[3 * i + 2] = ok ? g.cc : 0.0f;
    P.depth[i] = ok ? g.zc : 0.0f;
#pragma unroll
    for (int c = 0; c < 3; ++c) P.rgb[3 * i + c] = ok ? col[c] : 0.0f;
}

template <int DEG>
__global__ void __launch_bounds__(256) k_project_bwd(ProjParams P) {
    constexpr int K = (DEG + 1) * (DEG + 1);
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= P.n) return;
    const size_t n = size_t(P.n);
    // Colour first, from the view direction alone, so that the 48 SH
    // coefficients and the geometry's ~45 intermediates are never live
    // together (128 -> fewer registers, more warps per SM).  Its outputs are
    // written as if the splat were visible; a culled splat's are zeroed at
    // the end.
    float dm[3];
    bool col_ok;
    {
        const float px = P.mean3[3 * i], py = P.mean3[3 * i + 1], pz = P.mean3[3 * i + 2];
        const float vx = px - P.campos[0], vy = py - P.campos[1], vz = pz - P.campos[2];
        const float inv_len = 1.0f / sqrtf(vx * vx + vy * vy + vz * vz);
        const float ux = vx * inv_len, uy = vy * inv_len, uz = vz * inv_len;
        float Y[K];
        sh_eval<DEG>(ux, uy, uz, Y);
        float sh[K][3];
        float raw[3] = {0.5f, 0.5f, 0.5f};
#pragma unroll
        for (int k = 0; k < K; ++k)
#pragma unroll
            for (int c = 0; c < 3; ++c) {
                sh[k][c] = __ldg(P.sh + size_t(3 * k + c) * n + i);
                raw[c] = fmaf(sh[k][c], Y[k], raw[c]);
            }
        col_ok = isfinite(raw[0]) && isfinite(raw[1]) && isfinite(raw[2]) && isfinite(inv_len);
        // the clamp passes the gradient where raw >= 0
        float gcol[3];
#pragma unroll
        for (int c = 0; c < 3; ++c) gcol[c] = raw[c] >= 0.0f ? P.grgb[3 * i + c] : 0.0f;
        float dY[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            dY[k] = gcol[0] * sh[k][0] + gcol[1] * sh[k][1] + gcol[2] * sh[k][2];
#pragma unroll
            for (int c = 0; c < 3; ++c) P.dsh[size_t(3 * k + c) * n + i] = gcol[c] * Y[k];
        }
        float gdx = 0.0f, gdy = 0.0f, gdz = 0.0f;
        sh_grad<DEG>(ux, uy, uz, dY, gdx, gdy, gdz);
        const float dd = gdx * ux + gdy * uy + gdz * uz;
        dm[0] = (gdx - ux * dd) * inv_len;
        dm[1] = (gdy - uy * dd) * inv_len;
        dm[2] = (gdz - uz * dd) * inv_len;
    }
    Geo g;
    geometry(P, i, g);
    const bool ok = g.valid && col_ok;

    const float gu = ok ? P.gmean2d[2 * i] : 0.0f, gv = ok ? P.gmean2d[2 * i + 1] : 0.0f;
    const float ga = ok ? P.gconic[3 * i] : 0.0f, gb = ok ? P.gconic[3 * i + 1] : 0.0f,
                gc = ok ? P.gconic[3 * i + 2] : 0.0f;
    // conic = inverse(cov2): dL/dcov2 = -conic G conic, G = [[ga, gb/2], [gb/2, gc]]
    const float a = g.ca, b = g.cb, c = g.cc;
    const float G00 = -(a * a * ga + a * b * gb + b * b * gc);
    const float G01 = -(a * b * ga + 0.5f * (a * c + b * b) * gb + b * c * gc);
    const float G11 = -(b * b * ga + b * c * gb + c * c * gc);
    // cov2 = T c3 T^T: dT = 2 G T c3 = 2 G U;  dc3 = T^T G T
    float dT[6], W[6];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        dT[j] = 2.0f * (G00 * g.U[j] + G01 * g.U[3 + j]);
        dT[3 + j] = 2.0f * (G01 * g.U[j] + G11 * g.U[3 + j]);
        W[j] = G00 * g.T[j] + G01 * g.T[3 + j];          // (G T)[0][j]
        W[3 + j] = G01 * g.T[j] + G11 * g.T[3 + j];      // (G T)[1][j]
    }
    float dc3[9];
#pragma unroll
    for (int j = 0; j < 3; ++j)
#pragma unroll
        for (int k = 0; k < 3; ++k) dc3[3 * j + k] = g.T[j] * W[k] + g.T[3 + j] * W[3 + k];
    // c3 = M M^T: dM = 2 dc3 M;  M = r diag(s)
    float ds[3] = {0.0f, 0.0f, 0.0f}, dr[9];
#pragma unroll
    for (int a2 = 0; a2 < 3; ++a2)
#pragma unroll
        for (int b2 = 0; b2 < 3; ++b2) {
            const float dM = 2.0f * (dc3[3 * a2] * g.M[b2] + dc3[3 * a2 + 1] * g.M[3 + b2] +
                                     dc3[3 * a2 + 2] * g.M[6 + b2]);
            ds[b2] = fmaf(dM, g.r[3 * a2 + b2], ds[b2]);
            dr[3 * a2 + b2] = dM * g.s[b2];
        }
    // rotation of the unit quaternion u = (w, x, y, z)
    const float w = g.u[0], x = g.u[1], y = g.u[2], z = g.u[3];
    float du[4];
    du[0] = 2.0f * (-z * dr[1] + y * dr[2] + z * dr[3] - x * dr[5] - y * dr[6] + x * dr[7]);
    du[1] = 2.0f * (y * dr[1] + z * dr[2] + y * dr[3] - 2.0f * x * dr[4] - w * dr[5] + z * dr[6] +
                    w * dr[7] - 2.0f * x * dr[8]);
    du[2] = 2.0f * (-2.0f * y * dr[0] + x * dr[1] + w * dr[2] + x * dr[3] + z * dr[5] - w * dr[6] +
                    z * dr[7] - 2.0f * y * dr[8]);
    du[3] = 2.0f * (-2.0f * z * dr[0] - w * dr[1] + x * dr[2] + w * dr[3] - 2.0f * z * dr[4] +
                    y * dr[5] + x * dr[6] + y * dr[7]);
    const float ud = du[0] * w + du[1] * x + du[2] * y + du[3] * z;
    float4 dq;
    dq.x = (du[0] - w * ud) * g.inv_qn;
    dq.y = (du[1] - x * ud) * g.inv_qn;
    dq.z = (du[2] - y * ud) * g.inv_qn;
    dq.w = (du[3] - z * ud) * g.inv_qn;

    // T = J Rc; J = [[fx/z, 0, -fx x/z^2], [0, fy/z, -fy y/z^2]]
    float dJ00 = 0.0f, dJ02 = 0.0f, dJ11 = 0.0f, dJ12 = 0.0f;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        dJ00 = fmaf(dT[j], P.R[j], dJ00);
        dJ02 = fmaf(dT[j], P.R[6 + j], dJ02);
        dJ11 = fmaf(dT[3 + j], P.R[3 + j], dJ11);
        dJ12 = fmaf(dT[3 + j], P.R[6 + j], dJ12);
    }
    const float iz = g.iz, iz2 = iz * iz, iz3 = iz2 * iz;
    const float fx = P.fx, fy = P.fy;
    const float dxc = (gu - dJ02 * iz) * fx * iz;
    const float dyc = (gv - dJ12 * iz) * fy * iz;
    const float dzc = -(dJ00 * fx + dJ11 * fy) * iz2 +
                      2.0f * (dJ02 * fx * g.xc + dJ12 * fy * g.yc) * iz3 -
                      (gu * fx * g.xc + gv * fy * g.yc) * iz2;
#pragma unroll
    for (int j = 0; j < 3; ++j) dm[j] += P.R[j] * dxc + P.R[3 + j] * dyc + P.R[6 + j] * dzc;

#pragma unroll
    for (int j = 0; j < 3; ++j) {
        P.dmean3[3 * i + j] = ok ? dm[j] : 0.0f;
        P.dscale[3 * i + j] = ok ? ds[j] : 0.0f;
    }
    reinterpret_cast<float4 *>(P.dquat)[i] = ok ? dq : make_float4(0.f, 0.f, 0.f, 0.f);
    if (!ok)
#pragma unroll
        for (int k = 0; k < 3 * K; ++k) P.dsh[size_t(k) * n + i] = 0.0f;
}

ss_status fill_params(const char *fn, const ss_splats3d *s, const ss_camera *cam, ProjParams &P) {
    if (!s || !cam) return fail(SS_ERR_INVALID_ARG, "%s: splats or camera is NULL", fn);
    if (s->n < 0) return fail(SS_ERR_INVALID_ARG, "%s: n < 0", fn);
    if (s->sh_degree < 0 || s->sh_degree > 3)
        return fail(SS_ERR_INVALID_ARG, "%s: sh_degree %d outside 0..3", fn, s->sh_degree);
    if (s->n > 0 && (!s->mean3 || !s->scale || !s->quat || !s->sh))
        return fail(SS_ERR_INVALID_ARG, "%s: a splat array is NULL", fn);
    if (reinterpret_cast<uintptr_t>(s->quat) & 15)
        return fail(SS_ERR_INVALID_ARG, "%s: quat not 16-byte aligned", fn);
    const float *cv = &cam->R[0];
    for (size_t k = 0; k < sizeof(ss_camera) / sizeof(float); ++k)
        if (!std::isfinite(cv[k])) return fail(SS_ERR_INVALID_ARG, "%s: camera entry %zu not finite", fn, k);
    if (!(cam->fx > 0.0f) || !(cam->fy > 0.0f))
        return fail(SS_ERR_INVALID_ARG, "%s: fx, fy must be > 0", fn);
    P = ProjParams{};
    P.mean3 = s->mean3, P.scale = s->scale, P.quat = s->quat, P.sh = s->sh;
    P.n = s->n;
    for (int k = 0; k < 9; ++k) P.R[k] = cam->R[k];
    for (int k = 0; k < 3; ++k) {
        P.t[k] = cam->t[k];
        // camera centre -R^T t, in double then rounded once
        P.campos[k] = float(-(double(cam->R[k]) * cam->t[0] + double(cam->R[3 + k]) * cam->t[1] +
                              double(cam->R[6 + k]) * cam->t[2]));
    }
    P.fx = cam->fx, P.fy = cam->fy, P.cx = cam->cx, P.cy = cam->cy;
    P.near_z = cam->near_z, P.blur = cam->blur;
    return SS_OK;
}

}  // namespace
}  // namespace ss

using namespace ss;

extern "C" ss_status ss_project_fwd(const ss_splats3d *splats, const ss_camera *cam,
                                    float *mean2d, float *conic, float *depth, float *rgb,
                                    ss_stream_t stream) {
    clear_error();
    ProjParams P;
    ss_status st = fill_params("ss_project_fwd", splats, cam, P);
    if (st != SS_OK) return st;
    if (P.n == 0) return SS_OK;
    if (!mean2d || !conic || !depth || !rgb)
        return fail(SS_ERR_INVALID_ARG, "ss_project_fwd: an output is NULL");
    if (reinterpret_cast<uintptr_t>(mean2d) & 7)
        return fail(SS_ERR_INVALID_ARG, "ss_project_fwd: mean2d not 8-byte aligned");
    P.mean2d = mean2d, P.conic = conic, P.depth = depth, P.rgb = rgb;
    cudaStream_t s = (cudaStream_t)stream;
    const int grid = (P.n + 255) / 256;
    switch (splats->sh_degree) {
        case 0: SS_LAUNCH("k_project_fwd", s, k_project_fwd<0><<<grid, 256, 0, s>>>(P)); break;
        case 1: SS_LAUNCH("k_project_fwd", s, k_project_fwd<1><<<grid, 256, 0, s>>>(P)); break;
        case 2: SS_LAUNCH("k_project_fwd", s, k_project_fwd<2><<<grid, 256, 0, s>>>(P)); break;
        default: SS_LAUNCH("k_project_fwd", s, k_project_fwd<3><<<grid, 256, 0, s>>>(P)); break;
    }
    return check_launch("ss_project_fwd");
}

extern "C" ss_status ss_project_bwd(const ss_splats3d *splats, const ss_camera *cam,
                                    const float *dmean2d, const float *dconic, const float *drgb,
                                    const ss_grads3d *grads, ss_stream_t stream) {
    clear_error();
    ProjParams P;
    ss_status st = fill_params("ss_project_bwd", splats, cam, P);
    if (st != SS_OK) return st;
    if (P.n == 0) return SS_OK;
    if (!dmean2d || !dconic || !drgb)
        return fail(SS_ERR_INVALID_ARG, "ss_project_bwd: an upstream gradient is NULL");
    if (!grads || !grads->dmean3 || !grads->dscale || !grads->dquat || !grads->dsh)
        return fail(SS_ERR_INVALID_ARG, "ss_project_bwd: a gradient output is NULL");
    if (reinterpret_cast<uintptr_t>(grads->dquat) & 15)
        return fail(SS_ERR_INVALID_ARG, "ss_project_bwd: dquat not 16-byte aligned");
    P.gmean2d = dmean2d, P.gconic = dconic, P.grgb = drgb;
    P.dmean3 = grads->dmean3, P.dscale = grads->dscale, P.dquat = grads->dquat,
    P.dsh = grads->dsh;
    cudaStream_t s = (cudaStream_t)stream;
    const int grid = (P.n + 255) / 256;
    switch (splats->sh_degree) {
        case 0: SS_LAUNCH("k_project_bwd", s, k_project_bwd<0><<<grid, 256, 0, s>>>(P)); break;
        case 1: SS_LAUNCH("k_project_bwd", s, k_project_bwd<1><<<grid, 256, 0, s>>>(P)); break;
        case 2: SS_LAUNCH("k_project_bwd", s, k_project_bwd<2><<<grid, 256, 0, s>>>(P)); break;
        default: SS_LAUNCH("k_project_bwd", s, k_project_bwd<3><<<grid, 256, 0, s>>>(P)); break;
    }
    return check_launch("ss_project_bwd");
}
