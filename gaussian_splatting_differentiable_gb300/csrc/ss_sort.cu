// Sort of the (tile << 32 | depth bits, splat index) pairs and per-tile
// ranges ("Phase 5 step 30b -- kernel-by-kernel timing": radix_hist,
// radix_scatter -- 16 passes there -- and extract_offsets).
//
// Here an LSD radix sort in the onesweep style (Adinets & Merrill, "Onesweep:
// A Faster Least Significant Digit Radix Sort for GPUs", 2022):
//   k_sort_hist   one read of all keys builds the histograms of every 8-bit
//                 digit at once; its last CTA scans them into digit starts;
//   k_sort_pass   one launch per digit: each CTA takes the next partition of
//                 4096 keys by an atomic ticket (so a CTA only ever waits on
//                 CTAs that are already running), ranks its keys with warp
//                 match + per-warp histograms (stable), publishes its digit
//                 counts, and finds its global offsets by decoupled look-back
//                 over earlier partitions; every wait is bounded and reports
//                 a timeout through the workspace status word instead of
//                 spinning forever;
//   k_sort_final  equal keys (same tile, same depth) come out in emission
//                 order, which the atomic counter of the binning makes
//                 arbitrary: each run of equal keys is re-sorted by splat
//                 index (by its first thread when it is short; runs longer
//                 than 32 go to a list), and the tile boundaries give the
//                 CSR offsets;
//   k_sort_ties   one CTA per long run: a stable radix sort of its indices
//                 in global memory (no quadratic insertion sort, whatever
//                 the number of equal depths).
// Packed words: when the sorted key bits (below) and the bits of the largest
// value fit in 64 together, the passes move one word per pair, (mapped key
// << value bits) | value, instead of a 64-bit key and a 32-bit value (16
// instead of 24 bytes a pair and a pass, and one less shared-memory array);
// k_sort_hist finds the largest value, every kernel takes the same decision
// from it, and k_sort_final unpacks the words into the caller's buffers.
// Only 32 + ceil(log2 tiles) key bits are sorted -- and with the depth range
// that the binning recorded (the device-count sort), only the depth bits in
// which two pairs can differ: each kernel maps a key to
// (tile << db) | (depth bits - lo) on db + ceil(log2 tiles) bits and takes
// its digits from that; passes past the last digit return at once, and the
// final kernels find the sorted data by the parity of the passes run.
#include <atomic>

#include "ss_device.cuh"
#include "ss_internal.h"
#include "ss_profile.h"

namespace ss {

constexpr uint64_t kFlagAgg = 1ull << 62;
constexpr uint64_t kFlagInc = 2ull << 62;
constexpr uint64_t kValMask = (1ull << 62) - 1;
constexpr uint32_t kSpinLimit = 1u << 21;  // x ~100 ns backoff: about 0.2 s per wait

__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// The sorted key bits: identity (lo = 0, db = 32, nd = ndig) unless dr holds
// a recorded depth-bit range [dr[0], dr[1]]; then lo = dr[0] with its low 16
// bits cleared, db = max(16, bits of dr[1] - lo) and nd = the 8-bit digits of
// the db + tile_bits bit key.  Packed mode: when the mapped key and the
// largest value (*vmax, vb bits) fit in 64 bits together, the passes move one
// word (mapped key << vb | value) per pair instead of a key and a value.
struct KeyMap {
    uint32_t lo;
    int db, nd, vb;
    bool packed;
};

__device__ __forceinline__ KeyMap key_map(const unsigned long long *dr, int tile_bits, int ndig,
                                          const uint32_t *vmax) {
    KeyMap m{0u, 32, ndig, 32, false};
    if (dr) {
        const unsigned long long lo64 = dr[0], hi64 = dr[1];
        if (lo64 <= hi64 && hi64 <= 0xffffffffull) {
            m.lo = uint32_t(lo64) & 0xffff0000u;
            m.db = max(16, 32 - __clz(int(uint32_t(hi64) - m.lo)));
            m.nd = min(ndig, (m.db + tile_bits + 7) / 8);
        }
    }
    if (vmax) {
        m.vb = 32 - __clz(int(*vmax));
        m.packed = m.db + tile_bits + m.vb <= 64 && m.nd >= 2;
    }
    return m;
}

// The key as sorted: (tile << db) | (depth bits - lo); the identity map
// returns the key itself.
__device__ __forceinline__ uint64_t mapped_key(uint64_t key, const KeyMap &m) {
    return ((key >> 32) << m.db) | uint64_t(uint32_t(key) - m.lo);
}

// Packed mode: the word of a pair, and the key and value it holds.
__device__ __forceinline__ uint64_t pack_word(uint64_t key, uint32_t val, const KeyMap &m) {
    return (mapped_key(key, m) << m.vb) | val;
}

__device__ __forceinline__ uint64_t unpack_key(uint64_t w, const KeyMap &m) {
    const uint64_t mk = w >> m.vb;
    const uint32_t dbits = uint32_t(mk & ((1ull << m.db) - 1ull)) + m.lo;
    return ((mk >> m.db) << 32) | dbits;
}

__device__ __forceinline__ uint32_t unpack_val(uint64_t w, const KeyMap &m) {
    return uint32_t(w & ((1ull << m.vb) - 1ull));
}

// Packed mode: the word buffer pass d < nd - 1 writes.  Pass 0 reads the
// caller's keys and values, and the last pass writes them back unpacked, so
// the pass before the last always lands in the alternate key buffer `ak`;
// the ones before alternate with the caller's key buffer, and `zk` serves
// pass 0 when it is not the one before the last and would otherwise write
// the keys it reads.
__device__ __forceinline__ uint64_t *packed_dest(int d, int nd, uint64_t *keys, uint64_t *ak,
                                                 uint64_t *zk) {
    return ((nd - 2 - d) & 1) == 0 ? ak : (d == 0 ? zk : keys);
}

// Number of pairs to sort: n_max, or the device count *dn clamped to n_max.
__device__ __forceinline__ int64_t pair_count(const unsigned long long *dn, int64_t n_max) {
    if (!dn) return n_max;
    const unsigned long long c = *dn;
    return c < (unsigned long long)n_max ? int64_t(c) : n_max;
}

// Exclusive scan of one value per thread over a 256-thread block.
__device__ __forceinline__ uint32_t block_excl_scan256(uint32_t v, uint32_t *s_warp,
                                                       uint32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t t = s_warp[w];
        before += w < warp ? t : 0u;
        all += t;
    }
    __syncthreads();
    if (total) *total = all;
    return before + inc - v;
}

// Also finds the largest value (*vmax, zeroed before), which decides
// whether the passes run packed.
__global__ void __launch_bounds__(256) k_sort_hist(const uint64_t *__restrict__ keys,
                                                   const uint32_t *__restrict__ vals, int64_t n_max,
                                                   const unsigned long long *dn,
                                                   const unsigned long long *dr, int tile_bits,
                                                   int ndig, uint32_t *__restrict__ hist,
                                                   uint32_t *__restrict__ gofs, uint32_t *done,
                                                   uint32_t *vmax, uint32_t *err) {
    __shared__ uint32_t s_h[8][256];
    const int64_t n = pair_count(dn, n_max);
    const KeyMap m = key_map(dr, tile_bits, ndig, nullptr);
    for (int k = threadIdx.x; k < 8 * 256; k += 256) (&s_h[0][0])[k] = 0;
    __syncthreads();
    const int64_t stride = int64_t(gridDim.x) * 256;
    bool bad = false;
    auto count = [&](uint64_t k) {
        bad |= m.db < 32 && ((uint32_t(k) - m.lo) >> m.db) != 0u;   // depth outside the range
        const uint64_t v = mapped_key(k, m);
        for (int d = 0; d < m.nd; ++d) atomicAdd(&s_h[d][(v >> (8 * d)) & 255u], 1u);
    };
    // four keys in flight a thread (their loads issued together), then the rest
    uint32_t vm = 0;
    int64_t i = int64_t(blockIdx.x) * 256 + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        uint64_t k4[4];
        uint32_t v4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            k4[u] = keys[i + u * stride];
            v4[u] = vals[i + u * stride];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            count(k4[u]);
            vm = max(vm, v4[u]);
        }
    }
    for (; i < n; i += stride) {
        count(keys[i]);
        vm = max(vm, vals[i]);
    }
    if (bad) atomicOr(err, kDevErrKeyRange);
    vm = __reduce_max_sync(0xffffffffu, vm);
    if ((threadIdx.x & 31) == 0 && vm) atomicMax(vmax, vm);
    __syncthreads();
    for (int k = threadIdx.x; k < ndig * 256; k += 256) {
        const uint32_t v = (&s_h[0][0])[k];
        if (v) atomicAdd(hist + k, v);
    }
    // The last CTA to finish turns the histograms into exclusive digit
    // starts (the counts of every CTA are in L2 once it sees the count).
    __shared__ uint32_t s_last, s_warp[8];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int d = 0; d < ndig; ++d)
        gofs[d * 256 + threadIdx.x] =
            block_excl_scan256(__ldcg(hist + d * 256 + threadIdx.x), s_warp, nullptr);
}

struct PassParams {
    const uint64_t *kin;
    const uint32_t *vin;
    uint64_t *kout;
    uint32_t *vout;
    int64_t n;
    int shift;
    const uint32_t *gofs;  // [256] exclusive starts of this digit
    uint64_t *lookback;    // [nparts][256]
    uint32_t *ticket;
    uint32_t *err;
    const unsigned long long *dn;  // device pair count (clamped to n), or null
    const unsigned long long *dr;  // device depth-bit range [lo, hi], or null (identity map)
    int tile_bits, ndig;
    // packed mode (null vmax: never packed)
    const uint32_t *vmax;  // largest value, from k_sort_hist
    uint64_t *keys;        // the caller's key buffer
    uint32_t *vals;        // the caller's value buffer (the last pass's output)
    uint64_t *ak;          // alternate key buffer
    uint64_t *zk;          // third word buffer (pass 0 of an even pass count)
};

// One onesweep pass over one partition; PACKED moves words (mapped key << vb
// | value), otherwise keys and values.
template <bool PACKED>
__device__ __forceinline__ void sort_pass_body(const PassParams &p, const KeyMap &km, int64_t part,
                                               uint32_t (*s_whist)[256], uint32_t *s_lstart,
                                               uint32_t *s_gbase, uint32_t *s_warp,
                                               uint64_t *s_keys, uint32_t *s_vals) {
    constexpr int KPT = kSortKeysPerThread;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t base = part * kSortPart;
    const int64_t n = p.n;
    const int64_t wbase = base + warp * (KPT * 32);
    const int d = p.shift / 8;
    const uint64_t *win = nullptr;
    uint64_t *wout = nullptr;
    const bool last = d == km.nd - 1;   // packed: writes unpacked keys and values
    if (PACKED) {
        if (!last) wout = packed_dest(d, km.nd, p.keys, p.ak, p.zk);
        if (d > 0) win = packed_dest(d - 1, km.nd, p.keys, p.ak, p.zk);
    }
    const int dsh = PACKED ? km.vb + p.shift : p.shift;
    auto digit = [&](uint64_t k) -> uint32_t {
        return PACKED ? uint32_t(k >> dsh) & 255u : uint32_t(mapped_key(k, km) >> dsh) & 255u;
    };

    uint64_t key[KPT];
    uint32_t val[KPT];
    uint32_t rank2[KPT / 2];   // ranks (< kSortPart <= 2^16), two to a register
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
        const int64_t idx = wbase + j * 32 + lane;
        const bool ok = idx < n;
        if (PACKED) {
            key[j] = !ok ? ~0ull : (d == 0 ? pack_word(p.kin[idx], p.vin[idx], km) : win[idx]);
            val[j] = 0u;
        } else {
            key[j] = ok ? p.kin[idx] : ~0ull;
            val[j] = ok ? p.vin[idx] : 0u;
        }
    }
    // Stable rank within the warp: keys in order (j, lane).
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
        const int64_t idx = wbase + j * 32 + lane;
        const bool ok = idx < n;
        const uint32_t dig = ok ? digit(key[j]) : 256u + lane;
        const uint32_t peers = __match_any_sync(0xffffffffu, dig);
        const uint32_t before = __popc(peers & lt);
        uint32_t cur = 0;
        if (ok) cur = s_whist[warp][dig];
        if (j & 1)
            rank2[j >> 1] |= (cur + before) << 16;
        else
            rank2[j >> 1] = cur + before;
        __syncwarp();
        if (ok && before == 0) s_whist[warp][dig] = cur + __popc(peers);
        __syncwarp();
    }
    __syncthreads();

    // Per digit (thread = digit): warp-exclusive offsets and partition total.
    const int dg = tid;
    uint32_t total = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t c = s_whist[w][dg];
        s_whist[w][dg] = total;
        total += c;
    }
    uint64_t *my = p.lookback + part * 256 + dg;
    st_relaxed(my, (part == 0 ? kFlagInc : kFlagAgg) | uint64_t(total));

    s_lstart[dg] = block_excl_scan256(total, s_warp, nullptr);

    // Decoupled look-back: sum the counts of digit dg in earlier partitions.
    uint64_t excl = 0;
    if (part > 0) {
        int64_t q = part - 1;
        uint32_t spins = 0;
        while (true) {
            const uint64_t sw = ld_relaxed(p.lookback + q * 256 + dg);
            const uint64_t flag = sw & ~kValMask;
            if (flag == 0) {
                if (++spins > kSpinLimit) {
                    atomicOr(p.err, kDevErrTimeout);
                    break;
                }
                if (spins > 32) __nanosleep(100);
                continue;
            }
            excl += sw & kValMask;
            if (flag == kFlagInc || q == 0) break;
            --q;
            spins = 0;
        }
        st_relaxed(my, kFlagInc | (excl + total));
    }
    s_gbase[dg] = p.gofs[dg] + uint32_t(excl);
    __syncthreads();

    // Scatter into shared memory in (digit, rank) order, then out.
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
        const int64_t idx = wbase + j * 32 + lane;
        if (idx < n) {
            const uint32_t dig = digit(key[j]);
            const uint32_t rank = (j & 1) ? rank2[j >> 1] >> 16 : rank2[j >> 1] & 0xffffu;
            const uint32_t pos = s_lstart[dig] + s_whist[warp][dig] + rank;
            if (SS_BAD(pos >= uint32_t(kSortPart), kDbgSortRank)) continue;
            s_keys[pos] = key[j];
            if (!PACKED) s_vals[pos] = val[j];
        }
    }
    __syncthreads();
    const int64_t left = n - base;
    const int cnt = int(left < kSortPart ? left : kSortPart);
    for (int i = tid; i < cnt; i += 256) {
        const uint64_t k = s_keys[i];
        const uint32_t dig = digit(k);
        const uint32_t g = s_gbase[dig] + uint32_t(i) - s_lstart[dig];
        if (SS_BAD(int64_t(g) >= n, kDbgSortScatter)) continue;
        if (PACKED && !last) {
            wout[g] = k;
        } else if (PACKED) {
            p.keys[g] = unpack_key(k, km);
            p.vals[g] = unpack_val(k, km);
        } else {
            p.kout[g] = k;
            p.vout[g] = s_vals[i];
        }
    }
}

__global__ void __launch_bounds__(256, 3) k_sort_pass(PassParams p) {
    __shared__ uint32_t s_whist[8][256];  // per-warp digit counts, then warp-exclusive offsets
    __shared__ uint32_t s_lstart[256];    // digit start within the partition
    __shared__ uint32_t s_gbase[256];     // global start of the partition's keys of each digit
    __shared__ uint32_t s_warp[8];
    __shared__ uint32_t s_part;
    extern __shared__ __align__(16) unsigned char s_dyn[];
    uint64_t *s_keys = reinterpret_cast<uint64_t *>(s_dyn);
    uint32_t *s_vals = reinterpret_cast<uint32_t *>(s_dyn + kSortPart * 8);

    const int tid = threadIdx.x;
    const KeyMap km = key_map(p.dr, p.tile_bits, p.ndig, p.vmax);
    if (p.shift / 8 >= km.nd) return;   // past the last digit of the mapped key
    if (p.dn) p.n = pair_count(p.dn, p.n);   // the device count, clamped to the capacity
    // Persistent: each CTA takes partitions by ticket until none is left (a
    // CTA only ever waits on partitions that running CTAs have taken).
    for (;;) {
        if (tid == 0) s_part = atomicAdd(p.ticket, 1u);
        for (int k = tid; k < 8 * 256; k += 256) (&s_whist[0][0])[k] = 0;
        __syncthreads();
        const int64_t part = s_part;
        if (part * kSortPart >= p.n) return;
        if (km.packed)
            sort_pass_body<true>(p, km, part, s_whist, s_lstart, s_gbase, s_warp, s_keys, s_vals);
        else
            sort_pass_body<false>(p, km, part, s_whist, s_lstart, s_gbase, s_warp, s_keys,
                                  s_vals);
        __syncthreads();   // the shared arrays are reused by the next partition
    }
}

// Ties and offsets.  For element i of the sorted keys:
//  - tile boundaries: offs[t] = i for every tile t in (tile(i-1), tile(i)],
//    and offs[t] = n for t > tile(n-1);
//  - a run of equal keys starting at i is re-sorted by value (insertion sort
//    by the run's first thread; runs are a few elements);
//  - when src != dst the element is copied (run members by the run head).
constexpr int kTieInsert = 32;   // longest run of equal keys sorted by insertion

constexpr int kFinalPer = 4;   // consecutive sorted elements per k_sort_final thread (measured: 1, 4, 8, 16)

__global__ void __launch_bounds__(256) k_sort_final(uint64_t *dk, uint32_t *dv, uint64_t *ak,
                                                    uint32_t *av, int64_t n_max,
                                                    const unsigned long long *dn,
                                                    const unsigned long long *dr, int tile_bits,
                                                    int ndig, const uint32_t *vmax, int64_t tiles,
                                                    uint32_t *offs, uint32_t *err,
                                                    uint32_t *tie_count, uint2 *ties) {
    // Unpacked, the passes ping-pong between (dk, dv) and (ak, av): after nd
    // of them the sorted data is in (ak, av) iff nd is odd.  Packed, the last
    // pass wrote it unpacked to (dk, dv).
    const KeyMap km = key_map(dr, tile_bits, ndig, vmax);
    const bool alt = !km.packed && (km.nd & 1);
    const uint64_t *sk = alt ? ak : dk;
    const uint32_t *sv = alt ? av : dv;
    const bool copy = alt;
    const int64_t t0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t n = pair_count(dn, n_max);
    if (t0 == 0 && dn && *dn > (unsigned long long)n_max) atomicOr(err, kDevErrCapacity);
    if (n == 0 && t0 == 0)
        for (int64_t u = 0; u <= tiles; ++u) offs[u] = 0u;
    // Elements [i0, i0 + kFinalPer), with their neighbours: all loads issued
    // together (one element a thread left the kernel waiting on memory).
    const int64_t i0 = t0 * kFinalPer;
    if (i0 >= n) return;
    uint64_t kk[kFinalPer + 2];
#pragma unroll
    for (int j = 0; j < kFinalPer + 2; ++j) {
        const int64_t idx = i0 - 1 + j;
        kk[j] = idx >= 0 && idx < n ? sk[idx] : 0ull;
    }
#pragma unroll
    for (int j = 0; j < kFinalPer; ++j) {
        const int64_t i = i0 + j;
        if (i >= n) continue;
        const uint64_t key = kk[j + 1];
        int64_t t = int64_t(key >> 32);
        if (t >= tiles) {
            atomicOr(err, kDevErrKeyRange);
            t = tiles;
        }
        int64_t tp = -1;
        if (i > 0) {
            tp = int64_t(kk[j] >> 32);
            if (tp > tiles) tp = tiles;
        }
        for (int64_t u = tp + 1; u <= t; ++u) offs[u] = uint32_t(i);
        if (i == n - 1)
            for (int64_t u = t + 1; u <= tiles; ++u) offs[u] = uint32_t(n);

        const bool member = i > 0 && kk[j] == key;
        if (member) continue;
        const bool head = i + 1 < n && kk[j + 2] == key;
        if (!head) {
            if (copy) {
                dk[i] = key;
                dv[i] = sv[i];
            }
            continue;
        }
        int64_t e = i + 1;
        while (e < n && sk[e] == key && e - i <= kTieInsert) ++e;
        if (e - i > kTieInsert) {   // a long run: k_sort_ties sorts (and copies) it
            while (e < n && sk[e] == key) ++e;
            ties[atomicAdd(tie_count, 1u)] = make_uint2(uint32_t(i), uint32_t(e - i));
            continue;
        }
        // insertion sort of sv[i..e) by value, written to dv[i..e)
        for (int64_t a = i; a < e; ++a) {
            const uint32_t v = sv[a];
            int64_t b = a;
            while (b > i && dv[b - 1] > v) {
                dv[b] = dv[b - 1];
                --b;
            }
            dv[b] = v;
            if (copy) dk[a] = key;
        }
    }
}

// Stable LSD radix sort of one range in global memory by one CTA, over the
// 64-bit key (depth bits << 32 | splat index): 8 passes of 8 bits (passes
// whose digit is the same for the whole range are skipped -- for a run of
// equal keys, all four depth digits), each a histogram, a scan and a stable
// scatter in chunks of 256 elements.  Data ping-pongs between the range in
// buffer a and in buffer b; the result is written to (dk, dv) with tile bits
// `tile`.
__device__ void segment_sort_global(uint64_t *ak, uint32_t *av, uint64_t *bk, uint32_t *bv,
                                    uint64_t *dk, uint32_t *dv, int64_t lo, int len, uint64_t tile,
                                    uint32_t *s_cnt, uint32_t *s_wc, uint32_t *s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t lt = lanemask_lt();
    uint64_t *ck[2] = {ak + lo, bk + lo};
    uint32_t *cv[2] = {av + lo, bv + lo};
    int cur = 0;
    // composite key of element e in buffer c: (key & 0xffffffff) << 32 | val
    for (int pass = 0; pass < 8; ++pass) {
        const int sh = 8 * pass;
        for (int d = tid; d < 256; d += 256) s_cnt[d] = 0;
        __syncthreads();
        for (int e = tid; e < len; e += 256) {
            const uint64_t c = (ck[cur][e] << 32) | cv[cur][e];
            atomicAdd(&s_cnt[uint32_t(c >> sh) & 255u], 1u);
        }
        __syncthreads();
        const uint32_t mine = s_cnt[tid];
        const uint32_t uniform = __syncthreads_or(mine == uint32_t(len));
        if (uniform) continue;   // every element has the same digit: nothing moves
        uint32_t run = block_excl_scan256(mine, s_warp, nullptr);   // running output offset of digit tid
        const int nxt = cur ^ 1;
        for (int base = 0; base < len; base += 256) {
            const int e = base + tid;
            const bool ok = e < len;
            uint64_t kk = 0;
            uint32_t vv = 0, dig = 256u + uint32_t(lane);
            if (ok) {
                kk = ck[cur][e];
                vv = cv[cur][e];
                dig = uint32_t(((kk << 32) | vv) >> sh) & 255u;
            }
            const uint32_t peers = __match_any_sync(0xffffffffu, dig);
            const uint32_t before = __popc(peers & lt);
            for (int k = tid; k < 8 * 256; k += 256) s_wc[k] = 0;
            __syncthreads();
            if (ok && before == 0) s_wc[warp * 256 + dig] = __popc(peers);
            __syncthreads();
            // thread d: exclusive prefix over warps of digit d, chunk total
            uint32_t tot = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const uint32_t c = s_wc[w * 256 + tid];
                s_wc[w * 256 + tid] = tot;
                tot += c;
            }
            s_cnt[tid] = run;
            __syncthreads();
            if (ok) {
                const uint32_t pos = s_cnt[dig] + s_wc[warp * 256 + dig] + before;
                ck[nxt][pos] = kk;
                cv[nxt][pos] = vv;
            }
            run += tot;
            __syncthreads();
        }
        cur = nxt;
        __syncthreads();
    }
    for (int e = tid; e < len; e += 256) {
        const uint64_t kk = ck[cur][e];
        dk[lo + e] = (tile << 32) | (kk & 0xffffffffull);
        dv[lo + e] = cv[cur][e];
    }
}

// One CTA per long run of equal keys (grid-stride over the list that
// k_sort_final filled): the run's indices in ascending order.  (ok, ov) is
// the other buffer, scratch for the radix passes.
__global__ void __launch_bounds__(256) k_sort_ties(uint64_t *dk, uint32_t *dv, uint64_t *ak,
                                                   uint32_t *av, const unsigned long long *dr,
                                                   int tile_bits, int ndig, const uint32_t *vmax,
                                                   const uint32_t *tie_count, const uint2 *ties) {
    __shared__ uint32_t s_wc[8 * 256];
    __shared__ uint32_t s_cnt[256];
    __shared__ uint32_t s_warp[8];
    // source: the passes' last output buffer (packed: the caller's, which
    // the last pass wrote unpacked); scratch: the other one
    const KeyMap km = key_map(dr, tile_bits, ndig, vmax);
    const bool alt = !km.packed && (km.nd & 1);
    uint64_t *sk = alt ? ak : dk, *ok_ = alt ? dk : ak;
    uint32_t *sv = alt ? av : dv, *ov = alt ? dv : av;
    const uint32_t nt = *tie_count;
    for (uint32_t r = blockIdx.x; r < nt; r += gridDim.x) {
        const uint2 run = ties[r];
        segment_sort_global(sk, sv, ok_, ov, dk, dv, int64_t(run.x), int(run.y),
                            sk[run.x] >> 32, s_cnt, s_wc, s_warp);
        __syncthreads();
    }
}

static std::atomic<unsigned long long> g_pass_smem_ctx[kMaxDevices];

// k_sort_pass needs 48 KB of dynamic shared memory (32 KB when packed) on
// top of its static arrays: raise its limit once per CUDA context.
static ss_status ensure_pass_smem(int dyn) {
    const void *fn = (const void *)k_sort_pass;
    return ensure_dyn_smem(g_pass_smem_ctx, &fn, 1, dyn, "ss_sort_pairs");
}

__global__ void k_set_u32(uint32_t *p, uint32_t v) { *p = v; }

// Sort of n_max pairs, or of the device count *dn (clamped to n_max) when dn
// is not null: grids are then sized for n_max and surplus CTAs leave.
static ss_status sort_impl(const char *who, uint64_t *keys, uint32_t *vals, int64_t n_max,
                           const unsigned long long *dn, int32_t W, int32_t H,
                           uint32_t *tile_offsets, void *workspace, size_t workspace_bytes,
                           cudaStream_t st) {
    if (W < 1 || H < 1 || W > kMaxSide || H > kMaxSide)
        return fail(SS_ERR_UNSUPPORTED, "%s: image %dx%d outside 1..%d", who, W, H, kMaxSide);
    if (n_max < 0) return fail(SS_ERR_INVALID_ARG, "%s: pair count < 0", who);
    if (n_max > int64_t(0xffffffffu))
        return fail(SS_ERR_UNSUPPORTED, "%s: %lld pairs >= 2^32", who, (long long)n_max);
    if (!tile_offsets) return fail(SS_ERR_INVALID_ARG, "%s: tile_offsets is NULL", who);
    if (n_max > 0 && (!keys || !vals)) return fail(SS_ERR_INVALID_ARG, "%s: keys/vals NULL", who);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return fail(SS_ERR_INVALID_ARG, "%s: workspace NULL or not 256-byte aligned", who);
    if ((reinterpret_cast<uintptr_t>(keys) & 7) || (reinterpret_cast<uintptr_t>(dn) & 7))
        return fail(SS_ERR_INVALID_ARG, "%s: keys / counters not 8-byte aligned", who);
    const WsLayout L = ws_layout(0, n_max, W, H);
    if (workspace_bytes < L.sort_end)
        return fail(SS_ERR_INVALID_ARG, "%s: workspace %zu bytes < %zu needed", who,
                    workspace_bytes, L.sort_end);
    const int64_t tiles = int64_t(tiles_x(W)) * tiles_y(H);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    uint32_t *err = reinterpret_cast<uint32_t *>(ws + L.status_word);
    ss_status s = check_cuda(cudaMemsetAsync(ws, 0, L.zero_end, st), "sort: memset");
    if (s != SS_OK) return s;
    if (n_max == 0)
        return check_cuda(cudaMemsetAsync(tile_offsets, 0, size_t(tiles + 1) * 4, st),
                          "sort: memset offsets");

    int dev = 0, sms = 0;
    s = current_device(&dev, &sms, "ss_sort_pairs: device query");
    if (s != SS_OK) return s;
    const int dyn = kSortPart * 12;
    s = ensure_pass_smem(dyn);
    if (s != SS_OK) return s;

    uint32_t *hist = reinterpret_cast<uint32_t *>(ws + L.hist);
    uint32_t *gofs = reinterpret_cast<uint32_t *>(ws + L.gofs);
    uint32_t *tickets = reinterpret_cast<uint32_t *>(ws + L.tickets);
    uint64_t *lookback = reinterpret_cast<uint64_t *>(ws + L.lookback);
    uint64_t *ak = reinterpret_cast<uint64_t *>(ws + L.alt_keys);
    uint32_t *av = reinterpret_cast<uint32_t *>(ws + L.alt_vals);
    uint64_t *zk = reinterpret_cast<uint64_t *>(ws + L.pack_words);
    uint32_t *vmax = tickets + 9;   // largest value (cleared with the tickets)

    const int64_t blocks = (n_max + 255) / 256;
    const int hgrid = int(blocks < int64_t(sms) * 4 ? blocks : int64_t(sms) * 4);
    const unsigned long long *dr = dn ? dn + 2 : nullptr;   // depth-bit range from the binning
    const int tbits = tile_bits(tiles);
    SS_LAUNCH("k_sort_hist", st,
              k_sort_hist<<<hgrid, 256, 0, st>>>(keys, vals, n_max, dn, dr, tbits, L.ndig, hist,
                                                 gofs, tickets + 10, vmax, err));
    uint64_t *bk[2] = {keys, ak};
    uint32_t *bv[2] = {vals, av};
    // persistent pass CTAs: as many as fit on the GPU at once (3 a SM)
    const int pgrid = int(L.nparts < int64_t(sms) * 3 ? L.nparts : int64_t(sms) * 3);
    for (int d = 0; d < L.ndig; ++d) {
        PassParams p{};
        p.kin = bk[d & 1];
        p.vin = bv[d & 1];
        p.kout = bk[(d + 1) & 1];
        p.vout = bv[(d + 1) & 1];
        p.n = n_max;
        p.shift = 8 * d;
        p.gofs = gofs + 256 * d;
        p.lookback = lookback + size_t(d) * size_t(L.nparts) * 256;
        p.ticket = tickets + d;
        p.err = err;
        p.dn = dn;
        p.dr = dr;
        p.tile_bits = tbits;
        p.ndig = L.ndig;
        p.vmax = vmax;
        p.keys = keys;
        p.vals = vals;
        p.ak = ak;
        p.zk = zk;
        SS_LAUNCH("k_sort_pass", st, k_sort_pass<<<pgrid, 256, dyn, st>>>(p));
    }
    uint32_t *tie_count = tickets + 8;
    uint2 *ties = reinterpret_cast<uint2 *>(ws + L.ties);
    const int64_t fblocks = (n_max + 256 * kFinalPer - 1) / (256 * kFinalPer);
    SS_LAUNCH("k_sort_final", st,
              k_sort_final<<<int(fblocks), 256, 0, st>>>(keys, vals, ak, av, n_max, dn, dr, tbits,
                                                        L.ndig, vmax, tiles, tile_offsets, err,
                                                        tie_count, ties));
    const int64_t max_runs = n_max / (kTieInsert + 1) + 1;
    const int tgrid = int(max_runs < int64_t(sms) * 2 ? max_runs : int64_t(sms) * 2);
    SS_LAUNCH("k_sort_ties", st,
              k_sort_ties<<<tgrid, 256, 0, st>>>(keys, vals, ak, av, dr, tbits, L.ndig, vmax,
                                                 tie_count, ties));
    return check_launch(who);
}

}  // namespace ss

using namespace ss;

extern "C" ss_status ss_sort_pairs(uint64_t *keys, uint32_t *vals, int64_t n_pairs, int32_t W,
                                   int32_t H, uint32_t *tile_offsets, void *workspace,
                                   size_t workspace_bytes, ss_stream_t stream) {
    clear_error();
    return sort_impl("ss_sort_pairs", keys, vals, n_pairs, nullptr, W, H, tile_offsets, workspace,
                     workspace_bytes, (cudaStream_t)stream);
}

extern "C" ss_status ss_sort_pairs_dev(uint64_t *keys, uint32_t *vals, const uint64_t *d_counters,
                                       int64_t capacity, int32_t W, int32_t H,
                                       uint32_t *tile_offsets, void *workspace,
                                       size_t workspace_bytes, ss_stream_t stream) {
    clear_error();
    if (!d_counters) return fail(SS_ERR_INVALID_ARG, "ss_sort_pairs_dev: d_counters is NULL");
    return sort_impl("ss_sort_pairs_dev", keys, vals, capacity,
                     reinterpret_cast<const unsigned long long *>(d_counters), W, H, tile_offsets,
                     workspace, workspace_bytes, (cudaStream_t)stream);
}

// Test hook: one onesweep pass CTA that holds partition 1 of a 2-partition
// problem whose partition 0 never publishes, so its look-back wait runs out
// (a flag that nothing sets).  All of its reads and writes stay inside the
// workspace: keys are the zeroed ping-pong buffer, every key has digit 0 and
// lands in the first partition's range.
extern "C" ss_status ss_test_sort_wait_timeout(void *workspace, size_t workspace_bytes,
                                               ss_stream_t stream) {
    clear_error();
    const int64_t n = 2 * kSortPart;
    const WsLayout L = ws_layout(0, n, kTile, kTile);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return fail(SS_ERR_INVALID_ARG, "ss_test_sort_wait_timeout: workspace NULL or unaligned");
    if (workspace_bytes < L.sort_end)
        return fail(SS_ERR_INVALID_ARG, "ss_test_sort_wait_timeout: workspace %zu bytes < %zu",
                    workspace_bytes, L.sort_end);
    cudaStream_t st = (cudaStream_t)stream;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    ss_status s = check_cuda(cudaMemsetAsync(ws, 0, L.sort_end, st), "memset");
    if (s != SS_OK) return s;
    s = ensure_pass_smem(kSortPart * 12);
    if (s != SS_OK) return s;
    uint32_t *tickets = reinterpret_cast<uint32_t *>(ws + L.tickets);
    SS_LAUNCH("k_set_u32", st, k_set_u32<<<1, 1, 0, st>>>(tickets, 1u));
    PassParams p{};
    p.kin = reinterpret_cast<const uint64_t *>(ws + L.alt_keys);
    p.vin = reinterpret_cast<const uint32_t *>(ws + L.alt_vals);
    p.kout = reinterpret_cast<uint64_t *>(ws + L.alt_keys);
    p.vout = reinterpret_cast<uint32_t *>(ws + L.alt_vals);
    p.n = n;
    p.shift = 0;
    p.gofs = reinterpret_cast<const uint32_t *>(ws + L.gofs);
    p.lookback = reinterpret_cast<uint64_t *>(ws + L.lookback);
    p.ticket = tickets;
    p.err = reinterpret_cast<uint32_t *>(ws + L.status_word);
    p.ndig = L.ndig;   // no depth range: the identity map, pass 0 active
    SS_LAUNCH("k_sort_pass", st, k_sort_pass<<<1, 256, kSortPart * 12, st>>>(p));
    return check_launch("ss_test_sort_wait_timeout");
}

namespace ss {
cudaError_t debug_word_sort(uint32_t *out) { return read_and_clear_debug_word(out); }
}  // namespace ss
