// Shared pieces of the C ABI: error strings, constants, workspace sizing,
// the pair-count read-back, the sort status read-back and the atomic probe.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "ss_device.cuh"
#include "ss_internal.h"
#include "ss_profile.h"

namespace ss {

static thread_local char g_err[512];

ss_status fail(ss_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

void clear_error() { g_err[0] = 0; }

ss_status check_cuda(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return SS_OK;
    return fail(SS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

ss_status check_launch(const char *what) { return check_cuda(cudaGetLastError(), what); }

// The driver's cuCtxGetCurrent and cuCtxGetId, found through the runtime
// (the library links no driver library, so that it loads where no driver
// is installed).
using CtxGetCurrentFn = int (*)(void **);
using CtxGetIdFn = int (*)(void *, unsigned long long *);

static std::atomic<CtxGetCurrentFn> g_get_current{nullptr};
static std::atomic<CtxGetIdFn> g_get_id{nullptr};

bool context_id_ready() { return g_get_id.load(std::memory_order_acquire) != nullptr; }

ss_status current_context_id(unsigned long long *id, const char *what) {
    CtxGetCurrentFn fc = g_get_current.load(std::memory_order_acquire);
    CtxGetIdFn fi = g_get_id.load(std::memory_order_acquire);
    if (!fc || !fi) {
        void *pc = nullptr, *pi = nullptr;
        cudaDriverEntryPointQueryResult qc = cudaDriverEntryPointSymbolNotFound, qi = qc;
        ss_status s = check_cuda(
            cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &pc, 12000, cudaEnableDefault, &qc),
            what);
        if (s != SS_OK) return s;
        s = check_cuda(
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &pi, 12000, cudaEnableDefault, &qi),
            what);
        if (s != SS_OK) return s;
        if (qc != cudaDriverEntryPointSuccess || qi != cudaDriverEntryPointSuccess || !pc || !pi)
            return fail(SS_ERR_CUDA, "%s: the driver has no cuCtxGetCurrent / cuCtxGetId", what);
        fc = reinterpret_cast<CtxGetCurrentFn>(pc);
        fi = reinterpret_cast<CtxGetIdFn>(pi);
        g_get_current.store(fc, std::memory_order_release);
        g_get_id.store(fi, std::memory_order_release);
    }
    void *ctx = nullptr;
    if (fc(&ctx) != 0) return fail(SS_ERR_CUDA, "%s: cuCtxGetCurrent failed", what);
    *id = 0;
    if (ctx && fi(ctx, id) != 0)
        return fail(SS_ERR_CUDA, "%s: cuCtxGetId failed", what);
    return SS_OK;
}

ss_status ensure_dyn_smem(std::atomic<unsigned long long> *cache, const void *const *fns, int n,
                          int bytes, const char *what) {
    int dev = 0;
    ss_status s = current_device(&dev, nullptr, what);
    if (s != SS_OK) return s;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    unsigned long long id = 0;
    s = current_context_id(&id, what);
    if (s != SS_OK) return s;
    if (cached && id != 0 && cache[dev].load(std::memory_order_acquire) == id) return SS_OK;
    for (int f = 0; f < n; ++f) {
        s = check_cuda(cudaFuncSetAttribute(fns[f], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            bytes),
                       what);
        if (s != SS_OK) return s;
    }
    s = current_context_id(&id, what);   // the first CUDA call made the device's context current
    if (s != SS_OK) return s;
    if (cached) cache[dev].store(id, std::memory_order_release);
    return SS_OK;
}

ss_status current_device(int *dev, int *sms, const char *what) {
    ss_status s = check_cuda(cudaGetDevice(dev), what);
    if (s == SS_OK && sms)
        s = check_cuda(cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev), what);
    return s;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(int32_t n_splats, int64_t n_pairs, int32_t W, int32_t H) {
    WsLayout L{};
    const int64_t tiles = int64_t(tiles_x(W)) * tiles_y(H);
    L.ndig = sort_digits(tiles);
    L.nparts = (n_pairs + kSortPart - 1) / kSortPart;
    size_t off = 0;
    L.status_word = off;
    off += 256;
    L.hist = off;
    off = align256(off + size_t(L.ndig) * 256 * 4);
    L.gofs = off;
    off = align256(off + size_t(L.ndig) * 256 * 4);
    L.tickets = off;              // [0, 8) pass tickets, [8] long tie runs, [9] largest value, [10] histogram CTAs done
    off = align256(off + 16 * 4);
    L.lookback = off;
    off = align256(off + size_t(L.ndig) * size_t(L.nparts) * 256 * 8);
    L.zero_end = off;
    L.alt_keys = off;
    off = align256(off + size_t(n_pairs) * 8);
    L.alt_vals = off;
    off = align256(off + size_t(n_pairs) * 4);
    L.ties = off;                 // uint2 (start, length) of runs of > 32 equal keys
    off = align256(off + size_t(n_pairs / 33 + 1) * 8);
    L.pack_words = off;           // uint64 [n_pairs]: the packed passes' third buffer
    off = align256(off + size_t(n_pairs) * 8);
    L.sort_end = off;
    L.accum = 256;  // after the status word; the sort's regions are dead by then
    L.bwd_end = align256(L.accum + size_t(n_splats) * 48);  // 48-byte gradient record per splat
    // The backward without the forward's blend masks (or without records)
    // builds them here, after its gradient records.
    L.recs = L.bwd_end;
    L.masks = align256(L.recs + size_t(n_splats) * 64);
    L.masks_end = align256(L.masks + size_t(n_pairs) * 32);
    L.total = L.sort_end > L.masks_end ? L.sort_end : L.masks_end;
    return L;
}

// Measurement probe: rounds of red.global.add.f32, consecutive threads on
// consecutive addresses, grid-stride over n.
__global__ void k_probe_red(float *buf, int64_t n, int32_t rounds) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int32_t r = 0; r < rounds; ++r)
        for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
            atomicAdd(buf + i, 1.0f);
}

}  // namespace ss

using namespace ss;

extern "C" {

int32_t ss_abi_version(void) { return 8; }

size_t ss_record_bytes(int32_t n_splats) { return n_splats < 0 ? 0 : size_t(n_splats) * 64; }

void ss_constants(float out[4]) {
    out[0] = kAlphaMin;
    out[1] = kAlphaMax;
    out[2] = kTEps;
    out[3] = float(kTile);
}

const char *ss_last_error(void) { return g_err; }

size_t ss_workspace_bytes(int32_t n_splats, int64_t n_pairs, int32_t W, int32_t H) {
    if (n_splats < 0 || n_pairs < 0 || n_pairs > int64_t(0xffffffffu) || W < 1 || H < 1 ||
        W > kMaxSide || H > kMaxSide)
        return 0;
    return ws_layout(n_splats, n_pairs, W, H).total;
}

ss_status ss_pair_count(const uint64_t *d_counters, int64_t capacity, int64_t *h_pairs,
                        int64_t *h_culled, ss_stream_t stream) {
    clear_error();
    if (!d_counters) return fail(SS_ERR_INVALID_ARG, "ss_pair_count: d_counters is NULL");
    if (capacity < 0) return fail(SS_ERR_INVALID_ARG, "ss_pair_count: capacity < 0");
    unsigned long long h[2] = {0, 0};
    ss_status st = check_cuda(
        cudaMemcpyAsync(h, d_counters, sizeof h, cudaMemcpyDeviceToHost, (cudaStream_t)stream),
        "ss_pair_count: cudaMemcpyAsync");
    if (st != SS_OK) return st;
    st = check_cuda(cudaStreamSynchronize((cudaStream_t)stream), "ss_pair_count: synchronize");
    if (st != SS_OK) return st;
    if (h_pairs) *h_pairs = int64_t(h[0]);
    if (h_culled) *h_culled = int64_t(h[1]);
    if (int64_t(h[0]) > capacity)
        return fail(SS_ERR_CAPACITY, "ss_pair_count: %lld pairs needed, capacity %lld",
                    (long long)h[0], (long long)capacity);
    return SS_OK;
}

ss_status ss_sort_status(const void *workspace, ss_stream_t stream) {
    clear_error();
    if (!workspace) return fail(SS_ERR_INVALID_ARG, "ss_sort_status: workspace is NULL");
    uint32_t word = 0;
    ss_status st = check_cuda(cudaMemcpyAsync(&word, workspace, 4, cudaMemcpyDeviceToHost,
                                              (cudaStream_t)stream),
                              "ss_sort_status: cudaMemcpyAsync");
    if (st != SS_OK) return st;
    st = check_cuda(cudaStreamSynchronize((cudaStream_t)stream), "ss_sort_status: synchronize");
    if (st != SS_OK) return st;
    if (word & kDevErrTimeout)
        return fail(SS_ERR_TIMEOUT, "ss_sort_pairs: a look-back wait gave up (status 0x%x)", word);
    if (word & kDevErrCapacity)
        return fail(SS_ERR_CAPACITY,
                    "ss_sort_pairs_dev: more pairs than the capacity; the first capacity were "
                    "sorted (status 0x%x)", word);
    if (word & kDevErrKeyRange)
        return fail(SS_ERR_DEVICE, "ss_sort_pairs: a key's tile id is >= the tile count (status 0x%x)",
                    word);
    return SS_OK;
}

int32_t ss_debug_bounds_enabled(void) {
#ifdef SS_DEBUG_BOUNDS
    return 1;
#else
    return 0;
#endif
}

ss_status ss_debug_status(ss_stream_t stream) {
    clear_error();
    ss_status st = check_cuda(cudaStreamSynchronize((cudaStream_t)stream),
                              "ss_debug_status: synchronize");
    if (st != SS_OK) return st;
    uint32_t w = 0;
    cudaError_t (*const readers[4])(uint32_t *) = {debug_word_bin, debug_word_sort,
                                                   debug_word_fwd, debug_word_bwd};
    for (int k = 0; k < 4 && st == SS_OK; ++k)
        st = check_cuda(readers[k](&w), "ss_debug_status: reading a debug word");
    if (st != SS_OK) return st;
    if (w)
        return fail(SS_ERR_DEVICE,
                    "device bounds checks failed: 0x%x (1 sort destination, 2 sort rank, 4 forward "
                    "list, 8 backward list, 16 last_contrib past its list, 32 splat index, 64 "
                    "mask list)", w);
    return SS_OK;
}

ss_status ss_probe_red_f32(float *buf, int64_t n, int32_t rounds, ss_stream_t stream) {
    clear_error();
    if (!buf || n < 1 || rounds < 0)
        return fail(SS_ERR_INVALID_ARG, "ss_probe_red_f32: bad buffer, size or rounds");
    int dev = 0, sms = 0;
    ss_status s = current_device(&dev, &sms, "ss_probe_red_f32: device query");
    if (s != SS_OK) return s;
    const int64_t want = (n + 255) / 256;
    const int grid = int(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
    SS_LAUNCH("k_probe_red", (cudaStream_t)stream,
              k_probe_red<<<grid, 256, 0, (cudaStream_t)stream>>>(buf, n, rounds));
    return check_launch("ss_probe_red_f32");
}

}  // extern "C"
