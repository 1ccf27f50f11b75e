// Host-side internals of libss.so: error reporting, size limits, workspace
// layout.  Not part of the ABI.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>

#include "ss.h"

namespace ss {

constexpr int kTile = 16;
constexpr int32_t kMaxSide = 32768;   // fits the forward's 16-bit image sides
constexpr int kSortThreads = 256;
constexpr int kSortKeysPerThread = 16;
constexpr int kSortPart = kSortThreads * kSortKeysPerThread;  // keys per onesweep partition
static_assert(kSortPart <= 65536, "k_sort_pass keeps two 16-bit ranks in a register");

// Records `st` and a printf-style message as this thread's last error.
ss_status fail(ss_status st, const char *fmt, ...);
// Clears this thread's last error (start of every ABI call).
void clear_error();
// SS_OK, or SS_ERR_CUDA with the pending launch error's text.
ss_status check_launch(const char *what);
// SS_ERR_CUDA with the text of `e` if e != cudaSuccess.
ss_status check_cuda(cudaError_t e, const char *what);
// The current device and its SM count (an error status if either query fails).
ss_status current_device(int *dev, int *sms, const char *what);
// The current CUDA context's process-unique id in *id (0 if no context is
// current yet), through the driver's cuCtxGetCurrent / cuCtxGetId; the first
// call resolves those two functions.
ss_status current_context_id(unsigned long long *id, const char *what);
// True once current_context_id has resolved the driver functions.
bool context_id_ready();
// Per-device caches of per-context settings cover devices [0, kMaxDevices).
constexpr int kMaxDevices = 64;
// Raises the dynamic shared-memory limit of the kernels fns[0, n) to
// `bytes`, once per CUDA context: cache[dev] holds the id of the context in
// which that was done, so a new context on the device (the primary context
// re-created after cudaDeviceReset, or a driver-API context made current)
// sets it again.  Devices past kMaxDevices set it on every call.
ss_status ensure_dyn_smem(std::atomic<unsigned long long> *cache, const void *const *fns, int n,
                          int bytes, const char *what);

inline int32_t tiles_x(int32_t W) { return (W + kTile - 1) / kTile; }
inline int32_t tiles_y(int32_t H) { return (H + kTile - 1) / kTile; }

// Bits of a tile id for `tiles` tiles (ceil log2).
inline int tile_bits(int64_t tiles) {
    int b = 0;
    while (b < 32 && (int64_t(1) << b) < tiles) ++b;
    return b;
}

// Number of 8-bit digits in a (tile << 32 | depth bits) key for `tiles` tiles.
inline int sort_digits(int64_t tiles) { return (32 + tile_bits(tiles) + 7) / 8; }

// Workspace layout.  The first 256 bytes hold the device status word of the
// last sort; the rest is shared by ss_sort_pairs and the backward calls.
struct WsLayout {
    size_t status_word;   // uint32, offset 0
    size_t hist;          // uint32 [ndig][256] digit counts
    size_t gofs;          // uint32 [ndig][256] exclusive digit starts
    size_t tickets;       // uint32 [16]: partition tickets per pass, [8] long-run count,
                          // [9] largest value (packed-pass decision), [10] histogram CTAs done
    size_t lookback;      // uint64 [ndig][nparts][256] onesweep look-back words
    size_t zero_end;      // [0, zero_end) is cleared before each sort
    size_t alt_keys;      // uint64 [n_pairs] ping-pong buffer
    size_t alt_vals;      // uint32 [n_pairs]
    size_t ties;          // uint2 [n_pairs / 33 + 1] long runs of equal keys
    size_t pack_words;    // uint64 [n_pairs] third buffer of the packed passes
    size_t sort_end;
    size_t accum;         // backward per-splat gradient records, 48 bytes each
    size_t bwd_end;
    size_t recs;          // 64-byte splat records built by the backward from the splats
    size_t masks;         // uint32 [8][n_pairs] blend masks re-evaluated by the backward
    size_t masks_end;
    size_t total;
    int ndig;
    int64_t nparts;
};

WsLayout ws_layout(int32_t n_splats, int64_t n_pairs, int32_t W, int32_t H);

// The SS_DEBUG_BOUNDS debug words of the kernel translation units (each
// ORs its word into *out and clears it; no-ops in the normal build).
cudaError_t debug_word_bin(uint32_t *out);
cudaError_t debug_word_sort(uint32_t *out);
cudaError_t debug_word_fwd(uint32_t *out);
cudaError_t debug_word_bwd(uint32_t *out);

// Device status bits written by the sort kernels.
enum : uint32_t { kDevErrTimeout = 1u, kDevErrKeyRange = 2u, kDevErrCapacity = 4u };

}  // namespace ss
