// L1 + SSIM training loss and its gradient with respect to the rendered
// image in one pass ("ssim_fwd_bwd" of "Phase 5 step 30b -- kernel-by-kernel
// timing": SSIM forward and backward in one command buffer; lambda = 0.20,
// K = 7 window).  The model is stated in include/ss_ssim.h.
//
// The gradient is a correlation of the SSIM map's three adjoint maps
// (d SSIM / d mu_x, d SSIM / d E[x^2], d SSIM / d E[xy]) with the window, so
// the pixel at q needs the statistics of every p within 3 px, which need the
// images within 6 px.  One CTA owns a 32 x 32 output tile of one channel and
// does everything for it in shared memory: it loads the 44 x 44 input
// region (zero outside the image), forms the five window moments on the
// 38 x 38 region by two 1D passes, evaluates SSIM and the adjoint maps there
// (0 outside the image), correlates them back by two more 1D passes and
// writes dL/dimage.  HBM traffic is the two input images once (plus the
// halo, which neighbouring CTAs read from L2) and the gradient once: 12 bytes
// a pixel and channel.  Per-CTA partial sums of SSIM and |x - y| go to the
// workspace in double; the last CTA to finish (a ticket counter) adds them
// in block order, so the loss is deterministic.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "ss_internal.h"
#include "ss_profile.h"
#include "ss_ssim.h"

namespace ss {
namespace {

constexpr int kT = 32;               // output tile side
constexpr int kR = 3;                // window radius
constexpr int kW = 2 * kR + 1;       // window taps
constexpr int kIn = kT + 4 * kR;     // 44: input region side
constexpr int kMom = kT + 2 * kR;    // 38: statistics / adjoint region side
constexpr int kThreads = 256;
constexpr float kC1 = 0.01f * 0.01f;
constexpr float kC2 = 0.03f * 0.03f;

struct SsimParams {
    const float *img, *tgt;
    float *grad;
    double2 *partial;    // [blocks] (sum SSIM, sum |x - y|)
    unsigned int *ticket;
    float *out;          // (loss, mean SSIM, mean |x - y|)
    int C, H, W, n_blocks;
    float g[kW];
    float cs;            // dL/dSSIM(p) = -lambda / N
    float cl;            // dL/d|x - y| = (1 - lambda) / N
    float lambda;
    double inv_n;
};

// The input region is dead once the horizontal pass has read it, so the
// adjoint maps take its place (~51 KB in all: four CTAs per SM instead of
// three); the gradient phase reads its pixel's x and y again from L2.
struct SsimSmem {
    union {
        struct {
            float x[kIn][kIn];
            float y[kIn][kIn];
        } in;
        float a[3][kMom][kMom];  // adjoint maps on the moment region
    } u;
    float h[5][kIn][kMom];   // horizontal pass: moments, then the adjoint maps
    double red[2][kThreads / 32];
    int last;
};

__global__ void __launch_bounds__(kThreads) k_ssim(SsimParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SsimSmem &s = *reinterpret_cast<SsimSmem *>(smem_raw);
    const int tid = threadIdx.x;
    const int tx = blockIdx.x, ty = blockIdx.y, c = blockIdx.z;
    const int x0 = tx * kT, y0 = ty * kT;
    const size_t plane = size_t(p.H) * p.W;
    const float *img = p.img + c * plane, *tgt = p.tgt + c * plane;

    // A: the input region, zero outside the image; every load of a thread is
    // issued before its first shared store (one memory latency, not eight)
    constexpr int kLoads = (kIn * kIn + kThreads - 1) / kThreads;
    float lx[kLoads], ly[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
        const int k = tid + u * kThreads;
        const int r = k / kIn, q = k % kIn;
        const int gy = y0 - 2 * kR + r, gx = x0 - 2 * kR + q;
        const bool in = k < kIn * kIn && gy >= 0 && gy < p.H && gx >= 0 && gx < p.W;
        const size_t o = size_t(gy) * p.W + gx;
        lx[u] = in ? __ldg(img + o) : 0.0f;
        ly[u] = in ? __ldg(tgt + o) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
        const int k = tid + u * kThreads;
        if (k < kIn * kIn) {
            const int r = k / kIn, q = k % kIn;
            s.u.in.x[r][q] = lx[u];
            s.u.in.y[r][q] = ly[u];
        }
    }
    __syncthreads();

    // Each thread computes two neighbouring outputs of a 1D pass (they share
    // six of their eight window inputs, which it reads once).

    // B: horizontal window sums of x, y, x^2, y^2, xy (pairs along a row)
    for (int k = tid; k < kIn * (kMom / 2); k += kThreads) {
        const int r = k / (kMom / 2), q = 2 * (k % (kMom / 2));
        float xa[kW + 1], ya[kW + 1];
#pragma unroll
        for (int j = 0; j <= kW; ++j) xa[j] = s.u.in.x[r][q + j], ya[j] = s.u.in.y[r][q + j];
#pragma unroll
        for (int o = 0; o < 2; ++o) {
            float m0 = 0.f, m1 = 0.f, m2 = 0.f, m3 = 0.f, m4 = 0.f;
#pragma unroll
            for (int j = 0; j < kW; ++j) {
                const float a = xa[o + j], b = ya[o + j], w = p.g[j];
                const float wa = w * a, wb = w * b;
                m0 += wa;
                m1 += wb;
                m2 = fmaf(wa, a, m2);
                m3 = fmaf(wb, b, m3);
                m4 = fmaf(wa, b, m4);
            }
            s.h[0][r][q + o] = m0, s.h[1][r][q + o] = m1, s.h[2][r][q + o] = m2,
            s.h[3][r][q + o] = m3, s.h[4][r][q + o] = m4;
        }
    }
    __syncthreads();

    // C: vertical sums -> statistics, SSIM and the adjoint maps (pairs down a column)
    double ssim_sum = 0.0;
    for (int k = tid; k < (kMom / 2) * kMom; k += kThreads) {
        const int q = k % kMom, r0 = 2 * (k / kMom);
        float v[5][kW + 1];
#pragma unroll
        for (int t = 0; t < 5; ++t)
#pragma unroll
            for (int j = 0; j <= kW; ++j) v[t][j] = s.h[t][r0 + j][q];
        const int gx = x0 - kR + q;
        const bool col_in = gx >= 0 && gx < p.W, col_mid = q >= kR && q < kR + kT;
#pragma unroll
        for (int o = 0; o < 2; ++o) {
            const int r = r0 + o;
            float m[5];
#pragma unroll
            for (int t = 0; t < 5; ++t) {
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < kW; ++j) acc = fmaf(p.g[j], v[t][o + j], acc);
                m[t] = acc;
            }
            const int gy = y0 - kR + r;
            const bool in = col_in && gy >= 0 && gy < p.H;
            const float mx = m[0], my = m[1];
            const float A1 = 2.0f * mx * my + kC1;
            const float A2 = 2.0f * (m[4] - mx * my) + kC2;
            const float B1 = mx * mx + my * my + kC1;
            const float B2 = (m[2] - mx * mx) + (m[3] - my * my) + kC2;
            // the hardware reciprocal (about 1 ulp; the loss sums in double
            // and the gradient's tolerance are far coarser)
            const float iA1 = __fdividef(1.0f, A1), iA2 = __fdividef(1.0f, A2);
            const float iB1 = __fdividef(1.0f, B1), iB2 = __fdividef(1.0f, B2);
            const float S = A1 * A2 * iB1 * iB2;
            const float cS = in ? p.cs * S : 0.0f;
            s.u.a[0][r][q] = cS * 2.0f * (my * (iA1 - iA2) - mx * (iB1 - iB2));   // d/d mu_x
            s.u.a[1][r][q] = -cS * iB2;                                            // d/d E[x^2]
            s.u.a[2][r][q] = 2.0f * cS * iA2;                                      // d/d E[xy]
            if (in && col_mid && r >= kR && r < kR + kT) ssim_sum += S;
        }
    }
    __syncthreads();

    // D: horizontal correlation of the adjoint maps (reuses h; pairs along a row)
    for (int k = tid; k < kMom * (kT / 2); k += kThreads) {
        const int r = k / (kT / 2), q = 2 * (k % (kT / 2));
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            float v[kW + 1];
#pragma unroll
            for (int j = 0; j <= kW; ++j) v[j] = s.u.a[t][r][q + j];
            float v0 = 0.f, v1 = 0.f;
#pragma unroll
            for (int j = 0; j < kW; ++j) {
                v0 = fmaf(p.g[j], v[j], v0);
                v1 = fmaf(p.g[j], v[j + 1], v1);
            }
            s.h[t][r][q] = v0, s.h[t][r][q + 1] = v1;
        }
    }
    __syncthreads();

    // E: vertical correlation and the gradient (pairs down a column)
    double l1_sum = 0.0;
    float *grad = p.grad + c * plane;
    for (int k = tid; k < (kT / 2) * kT; k += kThreads) {
        const int q = k % kT, r0 = 2 * (k / kT);
        const int gx = x0 + q;
        float acc[3][2];
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            float v[kW + 1];
#pragma unroll
            for (int j = 0; j <= kW; ++j) v[j] = s.h[t][r0 + j][q];
            float v0 = 0.f, v1 = 0.f;
#pragma unroll
            for (int j = 0; j < kW; ++j) {
                v0 = fmaf(p.g[j], v[j], v0);
                v1 = fmaf(p.g[j], v[j + 1], v1);
            }
            acc[t][0] = v0, acc[t][1] = v1;
        }
#pragma unroll
        for (int o = 0; o < 2; ++o) {
            const int r = r0 + o, gy = y0 + r;
            if (gy >= p.H || gx >= p.W) continue;
            const size_t off = size_t(gy) * p.W + gx;
            const float xv = __ldg(img + off), yv = __ldg(tgt + off);
            const float d = xv - yv;
            const float sg = d > 0.0f ? 1.0f : (d < 0.0f ? -1.0f : 0.0f);
            grad[off] =
                acc[0][o] + 2.0f * xv * acc[1][o] + yv * acc[2][o] + p.cl * sg;
            l1_sum += fabsf(d);
        }
    }

    // per-CTA partial sums in double, then the last CTA adds them in order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ssim_sum += __shfl_xor_sync(0xffffffffu, ssim_sum, o);
        l1_sum += __shfl_xor_sync(0xffffffffu, l1_sum, o);
    }
    if ((tid & 31) == 0) s.red[0][tid >> 5] = ssim_sum, s.red[1][tid >> 5] = l1_sum;
    __syncthreads();
    if (tid == 0) {
        double a = 0.0, b = 0.0;
        for (int w = 0; w < kThreads / 32; ++w) a += s.red[0][w], b += s.red[1][w];
        const int blk = (c * gridDim.y + ty) * gridDim.x + tx;
        p.partial[blk] = make_double2(a, b);
        __threadfence();
        s.last = atomicAdd(p.ticket, 1u) == unsigned(p.n_blocks - 1);
    }
    __syncthreads();
    if (!s.last) return;
    __threadfence();
    double a = 0.0, b = 0.0;
    for (int k = tid; k < p.n_blocks; k += kThreads) {
        const double2 v = __ldcg(p.partial + k);
        a += v.x, b += v.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    __syncthreads();
    if ((tid & 31) == 0) s.red[0][tid >> 5] = a, s.red[1][tid >> 5] = b;
    __syncthreads();
    if (tid == 0) {
        double sa = 0.0, sb = 0.0;
        for (int w = 0; w < kThreads / 32; ++w) sa += s.red[0][w], sb += s.red[1][w];
        const double ssim = sa * p.inv_n, l1 = sb * p.inv_n;
        p.out[0] = float((1.0 - p.lambda) * l1 + p.lambda * (1.0 - ssim));
        p.out[1] = float(ssim);
        p.out[2] = float(l1);
        *p.ticket = 0u;
    }
}

int64_t ssim_blocks(int32_t C, int32_t H, int32_t W) {
    return int64_t((W + kT - 1) / kT) * ((H + kT - 1) / kT) * C;
}

}  // namespace
}  // namespace ss

using namespace ss;

extern "C" size_t ss_ssim_workspace_bytes(int32_t C, int32_t H, int32_t W) {
    if (C < 1 || H < 1 || W < 1 || H > kMaxSide || W > kMaxSide || C > 64) return 0;
    return size_t(ssim_blocks(C, H, W)) * sizeof(double2) + 16;   // partials + ticket
}

extern "C" ss_status ss_ssim_loss(const float *img, const float *target, int32_t C, int32_t H,
                                  int32_t W, float lambda, float *loss, float *dL_dimg,
                                  void *workspace, size_t workspace_bytes, ss_stream_t stream) {
    clear_error();
    if (C < 1 || C > 64 || H < 1 || W < 1 || H > kMaxSide || W > kMaxSide)
        return fail(SS_ERR_UNSUPPORTED, "ss_ssim_loss: image %dx%dx%d outside 1..64 x 1..%d x 1..%d",
                    C, H, W, kMaxSide, kMaxSide);
    if (!img || !target || !loss || !dL_dimg || !workspace)
        return fail(SS_ERR_INVALID_ARG, "ss_ssim_loss: a pointer is NULL");
    if (!(lambda >= 0.0f && lambda <= 1.0f))
        return fail(SS_ERR_INVALID_ARG, "ss_ssim_loss: lambda outside [0, 1]");
    if (reinterpret_cast<uintptr_t>(workspace) & 15)
        return fail(SS_ERR_INVALID_ARG, "ss_ssim_loss: workspace not 16-byte aligned");
    const size_t need = ss_ssim_workspace_bytes(C, H, W);
    if (workspace_bytes < need)
        return fail(SS_ERR_INVALID_ARG, "ss_ssim_loss: workspace %zu bytes < %zu", workspace_bytes,
                    need);
    static std::atomic<unsigned long long> smem_ctx[kMaxDevices];   // see ensure_dyn_smem
    const void *fn = (const void *)k_ssim;
    ss_status st = ensure_dyn_smem(smem_ctx, &fn, 1, int(sizeof(SsimSmem)), "ss_ssim_loss");
    if (st != SS_OK) return st;
    SsimParams p{};
    p.img = img, p.tgt = target, p.grad = dL_dimg;
    p.partial = static_cast<double2 *>(workspace);
    p.n_blocks = int(ssim_blocks(C, H, W));
    p.ticket = reinterpret_cast<unsigned int *>(p.partial + p.n_blocks);
    p.out = loss;
    p.lambda = lambda;
    p.C = C, p.H = H, p.W = W;
    // the 1D window exp(-i^2 / (2 sigma^2)), sigma = 1.5, normalised in double
    double g[2 * kR + 1], gs = 0.0;
    for (int i = -kR; i <= kR; ++i) gs += (g[i + kR] = std::exp(-double(i * i) / (2.0 * 1.5 * 1.5)));
    for (int i = 0; i <= 2 * kR; ++i) p.g[i] = float(g[i] / gs);
    const double n = double(C) * H * W;
    p.cs = float(-double(lambda) / n);
    p.cl = float((1.0 - double(lambda)) / n);
    p.inv_n = 1.0 / n;
    cudaStream_t s = (cudaStream_t)stream;
    st = check_cuda(cudaMemsetAsync(p.ticket, 0, sizeof(unsigned int), s), "ss_ssim_loss: memset");
    if (st != SS_OK) return st;
    const dim3 grid((W + kT - 1) / kT, (H + kT - 1) / kT, C);
    SS_LAUNCH("k_ssim", s, k_ssim<<<grid, kThreads, sizeof(SsimSmem), s>>>(p));
    return check_launch("ss_ssim_loss");
}
