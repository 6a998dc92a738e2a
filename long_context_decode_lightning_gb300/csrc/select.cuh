// K3 / K4: exact per-query selection over fp32 scores.
//
// Both the top-k of a score row and the candidate pool (a top-n_keep over
// block maxima, ids then sorted ascending) are "the k best items by (key desc,
// index asc)" with key = order_key(value). One routine serves both:
//
//   * items of a query that fit in shared memory (<= SEL_CAP) are loaded once
//     and selected in shared memory by a 4-pass 8-bit radix select, with
//     per-warp histograms;
//   * longer rows first go through a 4096-bin histogram of the top 12 key bits
//     (many CTAs per query, shared-memory atomics merged into a global
//     histogram) and a collect pass that keeps only items in or above the bin
//     that holds the k-th key; the survivors (about k plus one bin) are then
//     selected in shared memory;
//   * if the survivors overflow their buffer (heavily tied inputs), the same
//     select runs directly over the row in global memory.
// Ties at the threshold key are broken by index with a second radix select
// over ~index among the tied items, so the result is exact in every case.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace hsi {

constexpr int SEL_THREADS = 1024;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr int SEL_CAP = 16384;      // items held in shared memory by one CTA
constexpr int SEL_MAXK = 4096;      // largest k (top-k) or n_keep (pool)
constexpr int HIST_BINS = 4096;     // top 12 bits of the key
constexpr int SEL_B2 = 2048;        // second-level bins of the kept keys (select_small_hist)
constexpr int SCAN_THREADS = 512;
#ifndef HSI_SCAN_CHUNK
#define HSI_SCAN_CHUNK 8192
#endif
constexpr int SCAN_CHUNK = HSI_SCAN_CHUNK;  // items per CTA in the histogram / collect passes

constexpr uint32_t KEY_POS_INF = 0xFF800000u;  // order_key(+inf)
constexpr uint32_t KEY_NEG_INF = 0x007FFFFFu;  // order_key(-inf)

enum : int { SEL_TOPK = 0, SEL_POOL = 1 };

struct SelParams {
    // items: item i of query b is src[b*ld + i], i < n_items(b)
    const float* src;
    int64_t ld;
    const int32_t* n_src;  // [B]; n_items(b) = ceil(n_src[b] / div)
    int64_t max_src;       // the caller's bound on n_src[b]; a larger value is clamped and reported
    int32_t div;
    int32_t B;
    int32_t k;
    int32_t mode;  // SEL_TOPK or SEL_POOL (pin the last item to +inf, drop -inf items)
    // workspace
    uint32_t* hist;      // [B][HIST_BINS]
    uint32_t* cand_cnt;  // [B]
    uint32_t* cand_key;  // [B][cap]
    uint32_t* cand_idx;  // [B][cap]
    uint32_t* thr;       // [B] bin (top 12 key bits) holding the k-th key
    int32_t cap;
    // optional: [B] counters of histogram CTAs done (zero at the start); the
    // last CTA of a query computes its threshold bin, so no threshold pass runs
    uint32_t* done;
    // optional (TOPK mode): the maxima of the row's blocks of 8 items,
    // blk_max[b * ld_bmax + j] = max of items 8j .. 8j+7 (the visible ones); the
    // collect pass then reads only the blocks whose maximum reaches the
    // threshold bin (a block below it holds no survivor)
    const float* blk_max;
    int64_t ld_bmax;
    // rows of at most SEL_CAP items whose histogram is already in `hist` (TOPK
    // mode): the final kernel takes the threshold bin from it and loads only
    // the items at or above that bin
    int32_t hist_small;
    // top-k outputs
    const int32_t* block_ids;
    int64_t ld_blocks;
    int32_t block_size;
    int32_t* out_idx;
    float* out_val;
    // pool outputs (block size = div)
    int32_t* blk_out;  // [B][k]
    int32_t* n_kept;
    int32_t* n_pool;
    uint32_t* bits;
    int64_t ld_bits;
};

// n_src[b] within [0, max_src]: a length past the caller's bound (which sized
// the rows and buffers) is reported as a device-side argument error and
// clamped, so that no pass reads or writes past a row.
__device__ __forceinline__ int64_t sel_len(const SelParams& p, int b) {
    int64_t n = p.n_src[b];
    if (n > p.max_src) {
        raise_error(DEVERR_ARG);
        n = p.max_src;
    }
    return n < 0 ? 0 : n;
}

__device__ __forceinline__ int64_t sel_items(const SelParams& p, int b) {
    const int64_t n = sel_len(p, b);
    return (n + p.div - 1) / p.div;
}

// Key of item i of value v (n = item count); `ok`: whether it is eligible.
__device__ __forceinline__ uint32_t sel_key_of(const SelParams& p, float v, int64_t i, int64_t n, bool& ok) {
    uint32_t key = order_key(v);
    if (p.mode == SEL_POOL) {
        if (i == n - 1) key = KEY_POS_INF;  // the block of the newest position
        ok = key != KEY_NEG_INF;
    } else {
        ok = true;
    }
    return key;
}

// Key of item i (n = item count); `ok` says whether the item is eligible.
__device__ __forceinline__ uint32_t sel_key(const SelParams& p, int b, int64_t i, int64_t n, bool& ok) {
    uint32_t key = order_key(p.src[(int64_t)b * p.ld + i]);
    if (p.mode == SEL_POOL) {
        if (i == n - 1) key = KEY_POS_INF;  // the block of the newest position
        ok = key != KEY_NEG_INF;
    } else {
        ok = true;
    }
    return key;
}

// Zeroes n16 16-byte words, in stream order (after the previous kernel) like
// every kernel here, so that the next kernel's launch can still overlap it.
__global__ void __launch_bounds__(256) zero_kernel(uint4* p, int64_t n16) {
    griddep_wait();
    griddep_launch_dependents();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x)
        p[i] = make_uint4(0u, 0u, 0u, 0u);
}

// ------------------------------------------------------------ scan passes --

// Four consecutive items of a row starting at `base` (< hi): keys and eligibility.
__device__ __forceinline__ void sel_key4(const SelParams& p, int b, const float* row, bool vec, int64_t base,
                                         int64_t hi, int64_t n, uint32_t (&key)[4], bool (&ok)[4]) {
    float v[4];
    if (vec && base + 3 < hi) {
        const float4 f = *reinterpret_cast<const float4*>(row + base);
        v[0] = f.x, v[1] = f.y, v[2] = f.z, v[3] = f.w;
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = base + i < hi ? row[base + i] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t idx = base + i;
        key[i] = order_key(v[i]);
        ok[i] = idx < hi;
        if (p.mode == SEL_POOL) {
            if (idx == n - 1) key[i] = KEY_POS_INF;  // the block of the newest position
            ok[i] = ok[i] && key[i] != KEY_NEG_INF;
        }
    }
}

// The items [lo, hi) of a row that one scan CTA covers, SCAN_ROUNDS groups of
// 4 consecutive items per thread (group r at lo + 4 (r SCAN_THREADS + thread)),
// all loads issued before any is used: keys and eligibility bits (bit 4r+i).
constexpr int SCAN_ROUNDS = SCAN_CHUNK / (4 * SCAN_THREADS);
__device__ __forceinline__ void load_chunk(const SelParams& p, int b, const float* row, bool vec, int64_t lo,
                                           int64_t hi, int64_t n, uint32_t (&key)[SCAN_ROUNDS][4], uint32_t& okm) {
    static_assert(SCAN_ROUNDS * 4 <= 32, "eligibility bits");
    okm = 0;
    if (vec && lo + SCAN_CHUNK <= hi) {  // a whole chunk (uniform per CTA): unconditional 16-byte loads
        float4 f[SCAN_ROUNDS];
#pragma unroll
        for (int r = 0; r < SCAN_ROUNDS; ++r)
            f[r] = *reinterpret_cast<const float4*>(row + lo + 4 * ((int64_t)r * SCAN_THREADS + threadIdx.x));
#pragma unroll
        for (int r = 0; r < SCAN_ROUNDS; ++r) {
            const int64_t base = lo + 4 * ((int64_t)r * SCAN_THREADS + threadIdx.x);
            const float v[4] = {f[r].x, f[r].y, f[r].z, f[r].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                bool ok;
                key[r][i] = sel_key_of(p, v[i], base + i, n, ok);
                okm |= (ok ? 1u : 0u) << (4 * r + i);
            }
        }
        return;
    }
#pragma unroll
    for (int r = 0; r < SCAN_ROUNDS; ++r) {
        const int64_t base = lo + 4 * ((int64_t)r * SCAN_THREADS + threadIdx.x);
        bool ok[4] = {false, false, false, false};
        if (base < hi) sel_key4(p, b, row, vec, base, hi, n, key[r], ok);
#pragma unroll
        for (int i = 0; i < 4; ++i) okm |= (ok[i] ? 1u : 0u) << (4 * r + i);
    }
}

// The largest bin t such that the items in bins >= t number at least k (0 if
// there are fewer than k items). Whole block; SCAN_THREADS * 8 == HIST_BINS.
__device__ uint32_t threshold_bin(const uint32_t* gh, int k, uint32_t* scratch /*SCAN_THREADS+1*/) {
    static_assert(SCAN_THREADS * 8 == HIST_BINS, "bins per thread");
    const int t = threadIdx.x;
    uint32_t c[8];
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        c[i] = __ldcg(gh + t * 8 + i);  // counts other CTAs added in L2
        s += c[i];
    }
    scratch[t] = s;
    __syncthreads();
    // suffix sums over threads, from the top (Hillis-Steele on the reversed order)
    for (int off = 1; off < SCAN_THREADS; off <<= 1) {
        const uint32_t add = (t + off < SCAN_THREADS) ? scratch[t + off] : 0u;
        __syncthreads();
        scratch[t] += add;
        __syncthreads();
    }
    const uint32_t incl = scratch[t];      // items in bins >= t*8
    const uint32_t excl = incl - s;        // items in bins >= t*8 + 8
    __syncthreads();
    if (t == 0) scratch[SCAN_THREADS] = 0;
    __syncthreads();
    if (excl < (uint32_t)k && incl >= (uint32_t)k) {
        uint32_t run = excl;
        for (int i = 7; i >= 0; --i) {
            run += c[i];
            if (run >= (uint32_t)k) {
                scratch[SCAN_THREADS] = (uint32_t)(t * 8 + i);
                break;
            }
        }
    }
    __syncthreads();
    return scratch[SCAN_THREADS];
}

__global__ void __launch_bounds__(SCAN_THREADS) sel_hist_kernel(SelParams p) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ uint32_t sh[HIST_BINS];
    const int b = blockIdx.y;
    const int64_t n = sel_items(p, b);
    const int64_t lo = (int64_t)blockIdx.x * SCAN_CHUNK;
    if (lo >= n) return;
    const int64_t hi = min(n, lo + SCAN_CHUNK);
    for (int i = threadIdx.x; i < HIST_BINS; i += SCAN_THREADS) sh[i] = 0;
    __syncthreads();
    const float* row = p.src + (int64_t)b * p.ld;
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    uint32_t key[SCAN_ROUNDS][4], okm;
    load_chunk(p, b, row, vec, lo, hi, n, key, okm);
#pragma unroll
    for (int r = 0; r < SCAN_ROUNDS; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (okm >> (4 * r + i) & 1u) atomicAdd(&sh[key[r][i] >> 20], 1u);
    __syncthreads();
    uint32_t* gh = p.hist + (int64_t)b * HIST_BINS;
    for (int i = threadIdx.x; i < HIST_BINS; i += SCAN_THREADS)
        if (sh[i]) atomicAdd(&gh[i], sh[i]);
    if (!p.done) return;
    // the query's last CTA to finish computes its threshold bin
    __shared__ int last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t chunks = (uint32_t)((n + SCAN_CHUNK - 1) / SCAN_CHUNK);
        last = atomicAdd(p.done + b, 1u) == chunks - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    const uint32_t thr = threshold_bin(gh, p.k, sh);  // sh: scratch now
    if (threadIdx.x == 0) {
        p.thr[b] = thr;
        p.cand_cnt[b] = 0u;  // the collect pass counts from zero
    }
}

// One CTA per query: the threshold bin from the merged histogram.
__global__ void __launch_bounds__(SCAN_THREADS) sel_thresh_kernel(SelParams p) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ uint32_t scratch[SCAN_THREADS + 1];
    const int b = blockIdx.x;
    const uint32_t thr = threshold_bin(p.hist + (int64_t)b * HIST_BINS, p.k, scratch);
    if (threadIdx.x == 0) {
        p.thr[b] = thr;
        p.cand_cnt[b] = 0u;  // the collect pass, launched after this one, counts from zero
    }
}

__global__ void __launch_bounds__(SCAN_THREADS) sel_collect_kernel(SelParams p) {
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.y;
    const int64_t n = sel_items(p, b);
    const int64_t lo = (int64_t)blockIdx.x * SCAN_CHUNK;
    if (lo >= n) return;
    const int64_t hi = min(n, lo + SCAN_CHUNK);
    const uint32_t thr = p.thr[b];
    const int lane = threadIdx.x & 31;
    uint32_t* cnt = p.cand_cnt + b;
    uint32_t* ck = p.cand_key + (int64_t)b * p.cap;
    uint32_t* ci = p.cand_idx + (int64_t)b * p.cap;
    const float* row = p.src + (int64_t)b * p.ld;
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    uint32_t keys[SCAN_ROUNDS][4], okm;
    load_chunk(p, b, row, vec, lo, hi, n, keys, okm);
    // survivors of this thread (bit 4r+i), then one global reservation per warp
    // for the whole chunk: its latency is paid once, not once per round
    uint32_t sm = 0;
#pragma unroll
    for (int r = 0; r < SCAN_ROUNDS; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if ((okm >> (4 * r + i) & 1u) && (keys[r][i] >> 20) >= thr) sm |= 1u << (4 * r + i);
    // one reservation in the query's list per CTA (per warp, the CTAs of all
    // queries crowded the few cache lines of the counters)
    __shared__ uint32_t wsum[SCAN_THREADS / 32 + 1];
    const int warp = threadIdx.x >> 5;
    const uint32_t c = (uint32_t)__popc(sm);
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t run = 0;
        for (int w = 0; w < SCAN_THREADS / 32; ++w) {
            const uint32_t x = wsum[w];
            wsum[w] = run;
            run += x;
        }
        wsum[SCAN_THREADS / 32] = run ? atomicAdd(cnt, run) : 0u;
    }
    __syncthreads();
    if (c == 0) return;
    uint32_t at = wsum[SCAN_THREADS / 32] + wsum[warp] + incl - c;
#pragma unroll
    for (int r = 0; r < SCAN_ROUNDS; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (sm >> (4 * r + i) & 1u) {
                if (at < (uint32_t)p.cap) {
                    ck[at] = keys[r][i];
                    ci[at] = (uint32_t)(lo + 4 * ((int64_t)r * SCAN_THREADS + threadIdx.x) + i);
                }
                ++at;
            }
}

// The collect pass guided by block maxima (TOPK mode, blk_max given): a CTA
// covers SCAN_CHUNK blocks of 8 items; it reads their maxima (an eighth of
// the items' bytes) and only the items of blocks whose maximum's bin reaches
// the threshold, which are few (about one block per survivor).
__global__ void __launch_bounds__(SCAN_THREADS) sel_collect_blocks_kernel(SelParams p) {
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.y;
    const int64_t n = sel_items(p, b);
    const int64_t nb = (n + 7) / 8;
    const int64_t lo = (int64_t)blockIdx.x * SCAN_CHUNK;  // in blocks
    if (lo >= nb) return;
    const int64_t hi = min(nb, lo + SCAN_CHUNK);
    const uint32_t thr = p.thr[b];
    const int lane = threadIdx.x & 31;
    const float* bm = p.blk_max + (int64_t)b * p.ld_bmax;
    const float* row = p.src + (int64_t)b * p.ld;
    const bool bvec = (reinterpret_cast<uintptr_t>(bm) & 15) == 0;
    // the block maxima (as plain TOPK keys: blocks are never pinned or dropped)
    uint32_t key[SCAN_ROUNDS][4], okm;
    load_chunk(p, b, bm, bvec, lo, hi, nb, key, okm);  // TOPK mode: every block below hi counts
    uint32_t hit = 0;
#pragma unroll
    for (int r = 0; r < SCAN_ROUNDS; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if ((okm >> (4 * r + i) & 1u) && (key[r][i] >> 20) >= thr) hit |= 1u << (4 * r + i);
    // survivors of the hit blocks (few): counted, then written after one
    // reservation per warp; compact loops over the hit bits (this code runs for
    // few lanes, and unrolled copies of it cost instruction fetches)
    const bool rvec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    auto block_mask = [&](int64_t blk) -> uint32_t {  // survivors among the block's items
        const int64_t j0 = 8 * blk;
        float v[8];
        if (rvec && j0 + 7 < n) {
            const float4 a = *reinterpret_cast<const float4*>(row + j0);
            const float4 c4 = *reinterpret_cast<const float4*>(row + j0 + 4);
            v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = c4.x, v[5] = c4.y, v[6] = c4.z, v[7] = c4.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = j0 + e < n ? row[j0 + e] : __uint_as_float(0xFF800000u);
        }
        uint32_t m = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (j0 + e < n && (order_key(v[e]) >> 20) >= thr) m |= 1u << e;
        return m;
    };
    auto block_of = [&](int q) -> int64_t { return lo + 4 * ((int64_t)(q >> 2) * SCAN_THREADS + threadIdx.x) + (q & 3); };
    uint32_t c = 0;
#pragma unroll 1
    for (uint32_t h = hit; h; h &= h - 1) c += (uint32_t)__popc(block_mask(block_of(__ffs(h) - 1)));
    // one reservation in the query's list per CTA
    __shared__ uint32_t wsum[SCAN_THREADS / 32 + 1];
    const int warp = threadIdx.x >> 5;
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t run = 0;
        for (int w = 0; w < SCAN_THREADS / 32; ++w) {
            const uint32_t x = wsum[w];
            wsum[w] = run;
            run += x;
        }
        wsum[SCAN_THREADS / 32] = run ? atomicAdd(p.cand_cnt + b, run) : 0u;
    }
    __syncthreads();
    if (c == 0) return;
    uint32_t at = wsum[SCAN_THREADS / 32] + wsum[warp] + incl - c;
    uint32_t* ck = p.cand_key + (int64_t)b * p.cap;
    uint32_t* ci = p.cand_idx + (int64_t)b * p.cap;
#pragma unroll 1
    for (uint32_t h = hit; h; h &= h - 1) {
        const int64_t blk = block_of(__ffs(h) - 1);
        uint32_t m = block_mask(blk);
#pragma unroll 1
        for (; m; m &= m - 1) {
            const int64_t jj = 8 * blk + (__ffs(m) - 1);
            if (at < (uint32_t)p.cap) {
                ck[at] = order_key(row[jj]);
                ci[at] = (uint32_t)jj;
            }
            ++at;
        }
    }
}

// -------------------------------------------------------- block select --

struct SelSmem {
    uint32_t whist[SEL_WARPS][256];
    uint32_t hsum[256];
    unsigned long long win[SEL_MAXK];
    uint64_t bar;  // completion of the bulk copies of a row (select_small_fast)
    int abort;
    uint32_t bcast[8];
    alignas(16) uint32_t keys[SEL_CAP];
    alignas(16) uint32_t idx[SEL_CAP];
#ifdef HSI_TRACE
    long long t_last;
#endif
};

// Phase timing of the final selection (only with -DHSI_TRACE): thread 0 adds
// the cycles since the previous mark to trace slot `slot`.
#ifdef HSI_TRACE
#define SEL_MARK(s, slot)                                                                  \
    do {                                                                                   \
        if (threadIdx.x == 0) {                                                            \
            const long long now_ = clock64();                                              \
            atomicAdd(&g_hsi_trace[slot], (unsigned long long)(now_ - (s).t_last));        \
            (s).t_last = now_;                                                             \
        }                                                                                  \
    } while (0)
#else
#define SEL_MARK(s, slot) \
    do {                  \
    } while (0)
#endif

// Counts of the routes select_small_fast leaves by (only with -DHSI_TRACE).
#ifdef HSI_TRACE
#define SEL_COUNT(slot)                                        \
    do {                                                       \
        if (threadIdx.x == 0) atomicAdd(&g_hsi_trace[slot], 1ull); \
    } while (0)
#else
#define SEL_COUNT(slot) \
    do {                \
    } while (0)
#endif

// Sources of items for the block select.
struct SmemSrc {  // keys and indices in shared memory
    const uint32_t* keys;
    const uint32_t* ids;
    int64_t n;
    __device__ uint32_t key(int64_t j, bool& ok) const {
        ok = true;
        return keys[j];
    }
    __device__ uint32_t idx(int64_t j) const { return ids[j]; }
};
struct GlobalSrc {  // survivor keys and indices in global memory
    const uint32_t* keys;
    const uint32_t* ids;
    int64_t n;
    __device__ uint32_t key(int64_t j, bool& ok) const {
        ok = true;
        return keys[j];
    }
    __device__ uint32_t idx(int64_t j) const { return ids[j]; }
};
struct RowSrc {  // the row in global memory
    const SelParams* p;
    int b;
    int64_t n;
    __device__ uint32_t key(int64_t j, bool& ok) const { return sel_key(*p, b, j, n, ok); }
    __device__ uint32_t idx(int64_t j) const { return (uint32_t)j; }
};

// One radix pass: histogram of bits [shift, shift+8) over eligible items whose
// (selector & mask) == prefix, then the digit holding the `need`-th largest.
// sel = 0 selects on the key, sel = 1 on ~index among items with key == T.
// Returns the digit; *above = items with a larger digit; *at = items at it;
// *total = all counted items.
// rel: a window of 256 consecutive values of the key's top 16 bits instead,
// digit = (key >> 16) - prefix for keys above `prefix`, 0 for the rest (every
// key lies at or below prefix + 255; mask and shift are unused).
template <class Src>
__device__ uint32_t radix_pass(const Src& src, SelSmem& s, int sel, uint32_t T, uint32_t prefix, uint32_t mask,
                               int shift, uint32_t need, uint32_t* above, uint32_t* at, uint32_t* total,
                               bool rel = false) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < SEL_WARPS * 256; i += SEL_THREADS) (&s.whist[0][0])[i] = 0;
    __syncthreads();
    for (int64_t j0 = 0; j0 < src.n; j0 += SEL_THREADS) {  // uniform trip count per warp
        const int64_t j = j0 + tid;
        uint32_t bin = 0xFFFFFFFFu;
        if (j < src.n) {
            bool ok;
            const uint32_t key = src.key(j, ok);
            if (ok && (sel == 0 || key == T)) {
                const uint32_t v = sel == 0 ? key : ~src.idx(j);
                if (rel) {
                    const uint32_t hv = v >> 16;
                    bin = hv > prefix ? min(hv - prefix, 255u) : 0u;
                } else if ((v & mask) == prefix) {
                    bin = (v >> shift) & 255u;
                }
            }
        }
        if (bin != 0xFFFFFFFFu) atomicAdd(&s.whist[warp][bin], 1u);
    }
    __syncthreads();
    if (tid < 256) {
        uint32_t t = 0;
#pragma unroll 8
        for (int w = 0; w < SEL_WARPS; ++w) t += s.whist[w][tid];
        s.hsum[tid] = t;
    }
    __syncthreads();
    if (warp == 0) {
        uint32_t c[8], sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            c[i] = s.hsum[lane * 8 + i];
            sum += c[i];
        }
        // inclusive suffix over lanes (lane 31 holds the top bins)
        uint32_t suf = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t o = __shfl_down_sync(0xFFFFFFFFu, suf, off);
            if (lane + off < 32) suf += o;
        }
        const uint32_t tot = __shfl_sync(0xFFFFFFFFu, suf, 0);
        const uint32_t excl = suf - sum;
        if (lane == 0) {
            s.bcast[0] = 0;
            s.bcast[1] = 0;
            s.bcast[2] = 0;
            s.bcast[3] = tot;
        }
        __syncwarp();
        if (excl < need && suf >= need) {
            uint32_t run = excl;
            for (int i = 7; i >= 0; --i) {
                if (run + c[i] >= need) {
                    s.bcast[0] = (uint32_t)(lane * 8 + i);
                    s.bcast[1] = run;
                    s.bcast[2] = c[i];
                    break;
                }
                run += c[i];
            }
        }
    }
    __syncthreads();
    const uint32_t d = s.bcast[0];
    *above = s.bcast[1];
    *at = s.bcast[2];
    *total = s.bcast[3];
    __syncthreads();
    return d;
}

// Slot of this lane's item in a shared-memory list counted by *counter, one
// atomic per warp (every lane of the warp calls it; `take` says whether the
// lane has an item).
__device__ __forceinline__ uint32_t warp_append(bool take, uint32_t* counter) {
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, take);
    const int lane = threadIdx.x & 31;
    if (!m) return 0u;
    const int leader = __ffs(m) - 1;
    uint32_t base = 0;
    if (lane == leader) base = atomicAdd(counter, (uint32_t)__popc(m));
    base = __shfl_sync(0xFFFFFFFFu, base, leader);
    return base + (uint32_t)__popc(m & ((1u << lane) - 1u));
}

// The largest eligible key of src below +inf (0 if none); *any_inf: whether
// some eligible key is +inf or above (the pool's pinned block).
template <class Src>
__device__ uint32_t max_key(const Src& src, SelSmem& s, bool* any_inf) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t mx = 0;
    bool inf = false;
    for (int64_t j = threadIdx.x; j < src.n; j += SEL_THREADS) {
        bool ok;
        const uint32_t key = src.key(j, ok);
        if (ok) {
            if (key >= KEY_POS_INF) inf = true;
            else mx = max(mx, key);
        }
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 0) s.hsum[warp] = mx;
    *any_inf = __syncthreads_or(inf);
    if (warp == 0) {
        const uint32_t v = __reduce_max_sync(0xFFFFFFFFu, lane < SEL_WARPS ? s.hsum[lane] : 0u);
        if (lane == 0) s.bcast[7] = v;
    }
    __syncthreads();
    const uint32_t r = s.bcast[7];
    __syncthreads();
    return r;
}

// Sort s.win[0 .. count) descending: a bitonic network over m = the next
// power of two >= max(count, 8). In each round every one of m/8 threads owns
// the 8 elements whose indices differ only in three bits and applies up to
// three consecutive compare-exchange layers of the network to them in
// registers, so one barrier among those threads covers three layers (18
// rounds for m = 512 instead of 45 block-wide steps). Padding elements are 0,
// below every real entry.
__device__ void sort_desc(SelSmem& s, int count) {
    int m = 8;
    while (m < count) m <<= 1;
    for (int i = count + threadIdx.x; i < m; i += SEL_THREADS) s.win[i] = 0ull;
    __syncthreads();
    const int groups = m >> 3;
    const int nthr = groups < 32 ? 32 : groups;  // whole warps meet at the named barrier
    const int tid = threadIdx.x;
    if (tid < nthr) {
        for (int size = 2; size <= m; size <<= 1) {
            for (int S = size >> 1; S > 0;) {
                const int nst = S >= 4 ? 3 : (S == 2 ? 2 : 1);  // layers this round: strides S, S/2, S/4
                // owned index bits p0 > p1 > p2 (element bits 2, 1, 0)
                const int p0 = S >= 4 ? 31 - __clz(S) : 2, p1 = p0 - 1, p2 = p0 - 2;
                if (tid < groups) {
                    uint32_t t = (uint32_t)tid;  // tid with zero bits inserted at p2, p1, p0
                    t = ((t >> p2) << (p2 + 1)) | (t & ((1u << p2) - 1u));
                    t = ((t >> p1) << (p1 + 1)) | (t & ((1u << p1) - 1u));
                    t = ((t >> p0) << (p0 + 1)) | (t & ((1u << p0) - 1u));
                    uint32_t idx[8];
                    unsigned long long r[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        idx[e] = t | ((e & 4) ? 1u << p0 : 0u) | ((e & 2) ? 1u << p1 : 0u) | ((e & 1) ? 1u << p2 : 0u);
                        r[e] = s.win[idx[e]];
                    }
                    auto cx = [&](int lo, int hi) {  // lo/hi: element slots, literal at every call
                        const bool desc = (idx[lo] & (uint32_t)size) == 0;
                        if ((r[lo] < r[hi]) == desc) {
                            const unsigned long long x = r[lo];
                            r[lo] = r[hi];
                            r[hi] = x;
                        }
                    };
                    for (int l = 0; l < nst; ++l) {
                        const int eb = (S >= 4 ? 2 : (S == 2 ? 1 : 0)) - l;  // element bit of stride S >> l
                        if (eb == 2) {
                            cx(0, 4), cx(1, 5), cx(2, 6), cx(3, 7);
                        } else if (eb == 1) {
                            cx(0, 2), cx(1, 3), cx(4, 6), cx(5, 7);
                        } else {
                            cx(0, 1), cx(2, 3), cx(4, 5), cx(6, 7);
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) s.win[idx[e]] = r[e];
                }
                asm volatile("bar.sync 1, %0;" ::"r"(nthr) : "memory");
                S >>= nst;
            }
        }
    }
    __syncthreads();
}

// Exclusive prefix over the block of one count per thread; *total: the sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t c, SelSmem& s, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s.hsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t v = lane < SEL_WARPS ? s.hsum[lane] : 0u;
        uint32_t wi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += t;
        }
        if (lane < SEL_WARPS) s.hsum[lane] = wi - v;
        if (lane == 31) s.bcast[7] = wi;
    }
    __syncthreads();
    const uint32_t r = s.hsum[warp] + incl - c;
    *total = s.bcast[7];
    __syncthreads();
    return r;
}

// Sort s.win[0 .. count) descending for count <= 16 * 32: each warp sorts a run
// of 32 in registers (shuffles), then every element's place is its place in
// its run plus, for every other run, the number of that run's elements above
// it (a binary search). Entries are distinct and nonzero.
__device__ void sort_desc_runs(SelSmem& s, int count) {
    unsigned long long* run = reinterpret_cast<unsigned long long*>(s.keys);  // free once the winners are out
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int W = (count + 31) / 32;
    if (warp < W) {
        unsigned long long v = tid < count ? s.win[tid] : 0ull;  // 0 pads, below every entry
#pragma unroll
        for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
            for (int st = size >> 1; st > 0; st >>= 1) {
                const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, st);
                const bool lo = (lane & st) == 0, desc = size == 32 || (lane & size) == 0;
                const unsigned long long mx = v > w ? v : w, mn = v > w ? w : v;
                v = (lo == desc) ? mx : mn;
            }
        run[tid] = v;
    }
    __syncthreads();
    if (tid < count) {  // the real entries of a run come first
        const unsigned long long v = run[tid];
        uint32_t place = (uint32_t)lane;
        for (int q = 0; q < W; ++q) {
            if (q == warp) continue;
            const unsigned long long* R = run + q * 32;
            int pos = 0;
#pragma unroll
            for (int st = 32; st >= 1; st >>= 1)
                if (pos + st <= 32 && R[pos + st - 1] > v) pos += st;
            place += (uint32_t)pos;
        }
        s.win[place] = v;
    }
    __syncthreads();
}

constexpr int64_t SEL_BITMAP_IDS = SEL_MAXK * 64;  // ids a bitmap over s.win can hold

// Once the k-th largest key is known to have the high bits `prefix` (the bits
// set in `mask`, those above bit first_shift + 8), with above0 items above it:
// the remaining radix passes, the tie split at the k-th key and the gather of
// the winners into s.win, sorted descending: (key << 32 | ~idx) for top-k
// (id_range 0), or ~idx for a pool of ids below id_range (ascending ids).
// A pool whose ids fit SEL_BITMAP_IDS is put in order through a bitmap of the
// winners instead of a sort. Items of src whose masked high bits are below
// prefix may be absent.
template <class Src>
__device__ int select_finish(const Src& src, SelSmem& s, int k, int64_t id_range, bool take_all, uint32_t prefix,
                             uint32_t mask, int first_shift, uint32_t above0) {
    const bool ids_only = id_range > 0;
    const bool bitmap = ids_only && id_range <= SEL_BITMAP_IDS;
    uint32_t above, at = 0, total;
    uint32_t T = 0, T2 = 0;
    bool tie_split = false;
    if (!take_all) {
        uint32_t need = (uint32_t)k - above0;
        for (int shift = first_shift;; shift -= 8) {
            if (shift < 0) shift = 0;  // the last digit may overlap bits already fixed
            const uint32_t d = radix_pass(src, s, 0, 0, prefix, mask, shift, need, &above, &at, &total);
            need -= above;
            prefix |= d << shift;
            mask |= 0xFFu << shift;
            if (shift == 0) break;
        }
        SEL_MARK(s, 27);
        T = prefix;             // the k-th largest key
        tie_split = at > need;  // more items equal T than places left
        if (tie_split) {
            uint32_t p2 = 0, m2 = 0, need2 = need;
            for (int shift = 24; shift >= 0; shift -= 8) {
                const uint32_t d = radix_pass(src, s, 1, T, p2, m2, shift, need2, &above, &at, &total);
                need2 -= above;
                p2 |= d << shift;
                m2 |= 0xFFu << shift;
            }
            T2 = p2;  // ~index of the last tied item taken
        }
        SEL_MARK(s, 28);
    }
    if (threadIdx.x == 0) s.bcast[4] = 0;
    uint32_t* bits = reinterpret_cast<uint32_t*>(s.win);
    const int words = (int)((id_range + 31) / 32);
    if (bitmap)
        for (int i = threadIdx.x; i < words; i += SEL_THREADS) bits[i] = 0u;
    __syncthreads();
    for (int64_t j0 = 0; j0 < src.n; j0 += SEL_THREADS) {  // uniform trip count per warp
        const int64_t j = j0 + threadIdx.x;
        bool take = false;
        uint32_t key = 0;
        if (j < src.n) {
            bool ok;
            key = src.key(j, ok);
            if (ok) {
                if (take_all) take = true;
                else if (key != T) take = key > T;
                else take = !tie_split || (~src.idx(j)) >= T2;
            }
        }
        if (bitmap) {
            if (take) {
                const uint32_t id = src.idx(j);
                if (id < (uint64_t)id_range) atomicOr(&bits[id >> 5], 1u << (id & 31));
                else raise_error(DEVERR_ARG);  // never an id of this row: left out
            }
            continue;
        }
        const uint32_t pos = warp_append(take, &s.bcast[4]);
        if (take) {
            const uint32_t ni = ~src.idx(j);
            s.win[pos] = ids_only ? (unsigned long long)ni : (((unsigned long long)key << 32) | ni);
        }
    }
    __syncthreads();
    SEL_MARK(s, 29);
    if (bitmap) {
        // the set bits in id order: each thread takes a run of consecutive words
        constexpr int WPT = (int)(SEL_BITMAP_IDS / 32 / SEL_THREADS);
        uint32_t wv[WPT], c = 0;
#pragma unroll
        for (int i = 0; i < WPT; ++i) {
            const int wd = threadIdx.x * WPT + i;
            wv[i] = wd < words ? bits[wd] : 0u;
            c += (uint32_t)__popc(wv[i]);
        }
        uint32_t count;
        uint32_t pos = block_excl_scan(c, s, &count);  // its barriers also end the reads of the bitmap
#pragma unroll
        for (int i = 0; i < WPT; ++i) {
            const uint32_t base = (uint32_t)(threadIdx.x * WPT + i) * 32u;
            while (wv[i]) {
                const uint32_t id = base + (uint32_t)(__ffs(wv[i]) - 1);
                wv[i] &= wv[i] - 1u;
                s.win[pos++] = (unsigned long long)(~id);
            }
        }
        __syncthreads();
        SEL_MARK(s, 30);
        return (int)count;
    }
    const int count = (int)s.bcast[4];
    __syncthreads();
    if (count <= 16 * 32) sort_desc_runs(s, count);
    else sort_desc(s, count);
    SEL_MARK(s, 30);
    return count;
}

// The k best eligible items of src (see select_finish). The first radix pass
// looks at a window of 256 consecutive values of the keys' top 16 bits that
// ends at the largest key: scores cluster, so the window spreads them over
// many digits where the top byte would put nearly all in one; when the k-th
// key lies below the window, a pass on the top byte is taken instead. Then
// the items that can still win are packed into s.keys / s.idx when they fit,
// so the later passes run over those only. IN_SMEM: src itself lives in
// s.keys / s.idx (then it always fits; the items go through registers so
// none is overwritten before it is read).
template <bool IN_SMEM, class Src>
__device__ int block_select(const Src& src, SelSmem& s, int k, int64_t id_range) {
    uint32_t above, at, total;
    bool any_inf;
    const uint32_t top = max_key(src, s, &any_inf) >> 16;
    const uint32_t base = top > 255u ? top - 255u : 0u;
    // keys above the window (+inf) land in digit 255 with the window's top value
    uint32_t d0 = radix_pass(src, s, 0, 0, base, 0, 16, (uint32_t)k, &above, &at, &total, true);
    SEL_MARK(s, 25);
    if (total <= (uint32_t)k) return select_finish(src, s, k, id_range, true, 0, 0, 0, 0);
    uint32_t prefix, mask;
    int shift;
    if ((d0 > 0 || base == 0) && (d0 < 255 || !any_inf)) {  // digit d0 is exactly the value base + d0
        prefix = (base + d0) << 16;
        mask = 0xFFFF0000u;
        shift = 8;
    } else {
        d0 = radix_pass(src, s, 0, 0, 0, 0, 24, (uint32_t)k, &above, &at, &total);
        prefix = d0 << 24;
        mask = 0xFF000000u;
        shift = 16;
    }
    if (threadIdx.x == 0) s.bcast[6] = 0;
    if (IN_SMEM) {
        // in place, a chunk of 4 items per thread at a time: a chunk is read into
        // registers before any of it is overwritten, and the packed list never
        // reaches past the chunks already read
        constexpr int PER = 4, CHUNK = PER * SEL_THREADS;
        for (int64_t c0 = 0; c0 < src.n; c0 += CHUNK) {
            uint32_t kk[PER], ii[PER];
            bool keep[PER];
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int64_t j = c0 + threadIdx.x + (int64_t)i * SEL_THREADS;
                keep[i] = false;
                if (j < src.n) {
                    bool ok;
                    kk[i] = src.key(j, ok);
                    ii[i] = src.idx(j);
                    keep[i] = ok && (kk[i] & mask) >= prefix;
                }
            }
            // places by a block scan of the per-thread counts (its barriers also
            // end the chunk's reads)
            uint32_t mine = 0;
#pragma unroll
            for (int i = 0; i < PER; ++i) mine += keep[i] ? 1u : 0u;
            uint32_t kept;
            const uint32_t excl = block_excl_scan(mine, s, &kept);
            uint32_t pos = s.bcast[6] + excl;  // read after the scan's barriers
#pragma unroll
            for (int i = 0; i < PER; ++i)
                if (keep[i]) {
                    s.keys[pos] = kk[i];
                    s.idx[pos] = ii[i];
                    ++pos;
                }
            __syncthreads();  // everyone has read s.bcast[6]
            if (threadIdx.x == 0) s.bcast[6] += kept;
        }
    } else {
        if (above + at > (uint32_t)SEL_CAP) return select_finish(src, s, k, id_range, false, prefix, mask, shift, above);
        __syncthreads();
        for (int64_t j0 = 0; j0 < src.n; j0 += SEL_THREADS) {  // uniform trip count per warp
            const int64_t j = j0 + threadIdx.x;
            bool keep = false;
            uint32_t key = 0;
            if (j < src.n) {
                bool ok;
                key = src.key(j, ok);
                keep = ok && (key & mask) >= prefix;
            }
            const uint32_t pos = warp_append(keep, &s.bcast[6]);
            if (keep) {
                s.keys[pos] = key;
                s.idx[pos] = src.idx(j);
            }
        }
    }
    __syncthreads();
    SEL_MARK(s, 26);
    SmemSrc packed{s.keys, s.idx, (int64_t)s.bcast[6]};
    return select_finish(packed, s, k, id_range, false, prefix, mask, shift, above);
}

// The dynamic shared memory of the selection kernels, reached from any
// function through the shared-memory symbol itself (so that every access is a
// shared-memory access, also in functions that are not inlined).
__device__ __forceinline__ SelSmem& sel_smem() {
    extern __shared__ __align__(16) unsigned char sel_smem_raw[];
    return *reinterpret_cast<SelSmem*>(sel_smem_raw);
}

// The k best of a row of n <= SEL_CAP items (either mode): every item loaded
// into shared memory, then the block select. Returns the winners' count.
__device__ __noinline__ int select_row_smem(const SelParams& p, int b, int64_t n, int64_t id_range) {
    SelSmem& s = sel_smem();
    constexpr int PER = SEL_CAP / SEL_THREADS;
    const float* row = p.src + (int64_t)b * p.ld;
    float v[PER];
    uint32_t key[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {  // clamped index: every load issued unconditionally
        const int64_t j = (int64_t)i * SEL_THREADS + threadIdx.x;
        v[i] = n > 0 ? row[j < n ? j : n - 1] : 0.f;
    }
    __syncthreads();  // the caller's reads of shared memory are done
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int64_t j = (int64_t)i * SEL_THREADS + threadIdx.x;
        bool ok;
        key[i] = sel_key_of(p, v[i], j, n, ok);
        if (!ok || j >= n) key[i] = 0u;  // key 0 is never a real key (it is a NaN pattern)
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int64_t j = (int64_t)i * SEL_THREADS + threadIdx.x;
        if (j < n) {
            s.keys[j] = key[i];
            s.idx[j] = (uint32_t)j;
        }
    }
    __syncthreads();
    struct Filt : SmemSrc {
        __device__ uint32_t key(int64_t j, bool& ok) const {
            ok = keys[j] != 0u;
            return keys[j];
        }
    };
    Filt src;
    src.keys = s.keys;
    src.ids = s.idx;
    src.n = n;
    SEL_MARK(s, 24);
    return block_select<true>(src, s, p.k, id_range);
}

// The radix route of select_small (TOPK mode, n <= SEL_CAP items, T = the bin
// of the k-th key and `above` = the items in higher bins in s.bcast[0..1]):
// the items of bins >= T packed into s.keys / s.idx, then radix passes over
// the remaining 20 key bits. `in_smem`: the row is in s.keys.
__device__ __noinline__ int select_small_radix(const SelParams& p, int b, int64_t n, bool in_smem) {
    SelSmem& s = sel_smem();
    const int t = threadIdx.x;
    const uint32_t T = s.bcast[0], above = s.bcast[1];
    constexpr int PER = SEL_CAP / SEL_THREADS;
    const float* row = in_smem ? reinterpret_cast<const float*>(s.keys) : p.src + (int64_t)b * p.ld;
    uint32_t key[PER];
    bool keep[PER];
    float v[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {  // clamped index: every load issued unconditionally
        const int64_t j = (int64_t)i * SEL_THREADS + t;
        v[i] = row[j < n ? j : n - 1];
    }
    uint32_t mine = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int64_t j = (int64_t)i * SEL_THREADS + t;
        bool ok;
        key[i] = sel_key_of(p, v[i], j, n, ok);
        keep[i] = ok && j < n && (key[i] >> 20) >= T;
        mine += keep[i] ? 1u : 0u;
    }
    // places by a block scan of the per-thread counts (its barriers also end
    // every read of the row in shared memory)
    uint32_t kept;
    uint32_t pos = block_excl_scan(mine, s, &kept);
    SEL_MARK(s, 25);
#pragma unroll
    for (int i = 0; i < PER; ++i)
        if (keep[i]) {
            s.keys[pos] = key[i];
            s.idx[pos] = (uint32_t)(i * SEL_THREADS + t);
            ++pos;
        }
    if (t == 0) s.bcast[6] = kept;
    __syncthreads();
    SEL_MARK(s, 26);
    SmemSrc packed{s.keys, s.idx, (int64_t)s.bcast[6]};
    return select_finish(packed, s, p.k, 0, false, T << 20, 0xFFF00000u, 12, above);
}

enum : int { SMALL_WHOLE_ROW = -1, SMALL_RADIX = -2 };

// Top-k of a row of n <= SEL_CAP items (TOPK mode) whose 4096-bin histogram
// of the keys' top 12 bits is at hist (complete: every item counted). The bin
// T holding the k-th key comes from the histogram; only the items at or above
// it are kept. Returns the number of winners placed in s.win in order, or
// SMALL_WHOLE_ROW (the row holds fewer than k items) or SMALL_RADIX (the kept
// items are many or heavily tied: T and the items above bin T are left in
// s.bcast[0..1] for select_small_radix).
//
// When the row (and its block ids) start on 16-byte boundaries they come into
// shared memory by bulk copies, issued first so that they land while the
// histogram is scanned (*in_smem then says that s.keys holds the row, and
// *ids_in_smem that s.idx holds the block ids for the output). When the kept
// items are few (at most two per thread), they are ordered without radix
// passes or a sort: compared as floats against bin T's least value, they go
// into one list; a second histogram of SEL_B2 bins spans the kept keys' range
// (from bin T's least key to the largest key), its scan gives every bin's
// first rank (the items in the bins above it), each item goes to a slot of
// its bin's range, and its rank within the bin is the number of the bin's
// items that beat it. More than 256 items in one second-level bin (heavy
// ties) take the radix route instead.
__device__ __forceinline__ int select_small_fast(const SelParams& p, int b, int64_t n, const uint32_t* hist,
                                                 SelSmem& s, bool* in_smem, bool* ids_in_smem) {
    static_assert(HIST_BINS == 4 * SEL_THREADS, "four bins per thread");
    static_assert(3 * SEL_B2 + SEL_WARPS <= SEL_WARPS * 256, "second-level bins, offsets and counters fit in s.whist");
    static_assert(SEL_B2 == 2 * SEL_THREADS && SEL_MAXK - 2 * SEL_THREADS >= 2048,
                  "two bins per thread; the candidate lists past the k <= 2048 winners");
    static_assert(SEL_CAP == 16 * SEL_THREADS, "four float4 of the row per thread");
    const int t = threadIdx.x;
    const float* row = p.src + (int64_t)b * p.ld;
    const int64_t nb = p.block_ids ? (n + p.block_size - 1) / p.block_size : 0;
    const bool bulk = n > 0 && ((reinterpret_cast<uintptr_t>(p.src) & 15) | (p.ld & 3)) == 0;
    const bool bulk_ids = bulk && nb > 0 && ((reinterpret_cast<uintptr_t>(p.block_ids) & 15) | (p.ld_blocks & 3)) == 0 &&
                          nb <= p.ld_blocks && ((nb + 3) & ~3ll) <= SEL_CAP;
    *in_smem = bulk;
    *ids_in_smem = false;
    if (t == 0) {
        s.abort = 0;
        s.bcast[6] = 0;
        if (bulk) {
            const uint32_t bytes = (uint32_t)(((n + 3) & ~3ll) * 4);  // within the row: ld is a multiple of 4
            const uint32_t id_bytes = bulk_ids ? (uint32_t)(((nb + 3) & ~3ll) * 4) : 0u;
            mbar_init(&s.bar, 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(&s.bar, bytes + id_bytes);
            for (uint32_t o = 0; o < bytes; o += 16384u)
                bulk_g2s(reinterpret_cast<uint8_t*>(s.keys) + o, reinterpret_cast<const uint8_t*>(row) + o,
                         min(16384u, bytes - o), &s.bar);
            if (id_bytes) bulk_g2s(s.idx, p.block_ids + (int64_t)b * p.ld_blocks, id_bytes, &s.bar);
        }
    }
    uint32_t c[4], sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        c[i] = hist[4 * t + i];
        sum += c[i];
    }
    uint32_t total;
    const uint32_t below = block_excl_scan(sum, s, &total);  // items in bins under this thread's
    const uint32_t k = (uint32_t)p.k;
    SEL_MARK(s, 28);
    const uint32_t above_t = total - below - sum;  // items in bins over this thread's
    if (total >= k && above_t < k && above_t + sum >= k) {
        uint32_t run = above_t;
        for (int i = 3; i >= 0; --i) {
            if (run + c[i] >= k) {
                s.bcast[0] = (uint32_t)(4 * t + i);
                s.bcast[1] = run;
                s.bcast[2] = c[i];
                break;
            }
            run += c[i];
        }
    }
    // the row has landed (every thread waits; a wait that runs out aborts all)
    const bool ok = !bulk || wait_bounded(&s.bar, 0, &s.abort);
    if (!__syncthreads_and(ok)) {
        if (t == 0) wait_drain(&s.bar, 0);  // nothing may still be writing shared memory at exit
        __syncthreads();
        *in_smem = false;
        return 0;
    }
    SEL_MARK(s, 24);
    if (total < k) {
        SEL_COUNT(21);
        return SMALL_WHOLE_ROW;
    }
    const uint32_t T = s.bcast[0], above = s.bcast[1], at_T = s.bcast[2];
    const uint32_t kept_all = above + at_T;
    constexpr int KPT = 2;                        // kept items per thread
    constexpr int SMALL_CAP = KPT * SEL_THREADS;  // kept items ranked without radix passes
    static_assert(SEL_CAP / 8 <= 4096 && 8192 + 2 * SMALL_CAP <= SEL_CAP,
                  "block ids, the kept list and the grouped list share s.idx");
    if (!bulk || kept_all > (uint32_t)SMALL_CAP) {
        SEL_COUNT(bulk ? 22 : 21);
        return SMALL_RADIX;
    }

    uint32_t* h2 = &s.whist[0][0];  // second-level bins of the kept keys
    uint32_t* start2 = h2 + SEL_B2;
    uint32_t* fill2 = start2 + SEL_B2;
    uint32_t* wmax = fill2 + SEL_B2;                                                  // [SEL_WARPS]
    unsigned long long* clist = reinterpret_cast<unsigned long long*>(s.idx + 4096);  // the kept items, in no order
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(s.idx + 8192);   // the kept items, grouped by bin
    const int lane = t & 31, warp = t >> 5;
    const uint32_t base = T << 20;
    const float fT = key_to_float(base);  // the least value whose key lies in bin T or above
    // the kept items into one list: item j = 4 (i SEL_THREADS + t) + e, a ballot
    // per item slot, one reservation per warp
    float4 q[4];
    const float4* r4 = reinterpret_cast<const float4*>(s.keys);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = r4[i * SEL_THREADS + t];
    uint32_t bal[16], nw = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t j0 = 4 * ((int64_t)i * SEL_THREADS + t);
        const float e4[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            bal[4 * i + e] = __ballot_sync(0xFFFFFFFFu, j0 + e < n && e4[e] >= fT);
            nw += (uint32_t)__popc(bal[4 * i + e]);
        }
    }
    uint32_t wpos = 0;
    if (lane == 0 && nw) wpos = atomicAdd(&s.bcast[6], nw);
    wpos = __shfl_sync(0xFFFFFFFFu, wpos, 0);
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t j0 = 4u * (uint32_t)(i * SEL_THREADS + t);
        const float e4[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t m = bal[4 * i + e];
            if ((m >> lane) & 1u) {
                const uint32_t pos = wpos + (uint32_t)__popc(m & lt);
                if (pos < (uint32_t)SMALL_CAP)
                    clist[pos] = ((unsigned long long)order_key(e4[e]) << 32) | (uint32_t)~(j0 + (uint32_t)e);
            }
            wpos += (uint32_t)__popc(m);
        }
    }
    h2[2 * t] = 0u;
    h2[2 * t + 1] = 0u;
    __syncthreads();
    SEL_MARK(s, 27);
    const uint32_t cnt = s.bcast[6];
    if (cnt != kept_all) {  // the histogram does not describe the row (uniform)
        SEL_COUNT(21);
        return SMALL_RADIX;
    }
    // SEL_B2 bins over [T << 20, largest kept key], fine enough that few items share one
    bool mine[KPT];
    unsigned long long me[KPT];
    uint32_t key[KPT], x[KPT], mx = 0;
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
        const uint32_t j = (uint32_t)(t + i * SEL_THREADS);
        mine[i] = j < cnt;
        me[i] = mine[i] ? clist[j] : 0ull;
        key[i] = (uint32_t)(me[i] >> 32);
        if (mine[i]) mx = max(mx, key[i]);
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 0) wmax[warp] = mx;
    __syncthreads();
    const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, wmax[lane]);
    const uint32_t range = top - base;
    const int sh2 = range >= (uint32_t)SEL_B2 ? 32 - __clz((int)(range / SEL_B2)) : 0;  // range >> sh2 < SEL_B2
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
        x[i] = mine[i] ? (key[i] - base) >> sh2 : 0u;
        if (mine[i]) atomicAdd(&h2[x[i]], 1u);
    }
    __syncthreads();
    const uint32_t c0 = h2[2 * t], c1 = h2[2 * t + 1];
    uint32_t tot2;
    const uint32_t below2 = block_excl_scan(c0 + c1, s, &tot2);  // items in bins under 2t
    start2[2 * t] = tot2 - below2 - c0;  // items in the bins above
    start2[2 * t + 1] = tot2 - below2 - c0 - c1;
    fill2[2 * t] = 0u;
    fill2[2 * t + 1] = 0u;
    const uint32_t wc = __reduce_max_sync(0xFFFFFFFFu, max(c0, c1));
    if (lane == 0) wmax[warp] = wc;
    __syncthreads();
    SEL_MARK(s, 26);
    // a crowded bin costs its items one comparison per item of the bin: heavy
    // ties (more than 256 in one bin) take the radix passes (uniform)
    if (__reduce_max_sync(0xFFFFFFFFu, wmax[lane]) > 256u) {
        __syncthreads();  // every read of the bins is done before the radix passes reuse them
        SEL_COUNT(23);
        return SMALL_RADIX;
    }
#pragma unroll
    for (int i = 0; i < KPT; ++i)
        if (mine[i]) cand[start2[x[i]] + atomicAdd(&fill2[x[i]], 1u)] = me[i];
    __syncthreads();
    SEL_MARK(s, 25);
#pragma unroll
    for (int i = 0; i < KPT; ++i)
        if (mine[i]) {  // rank: the items of the bins above, then those of its own bin that beat it
            const uint32_t lo = start2[x[i]], hi = lo + fill2[x[i]];
            uint32_t r = lo;
            for (uint32_t c = lo; c < hi; ++c) r += cand[c] > me[i] ? 1u : 0u;
            if (r < k) s.win[r] = me[i];
        }
    __syncthreads();
    SEL_MARK(s, 30);
    *ids_in_smem = bulk_ids;
    return (int)k;
}

// Top-k outputs of query b from the `count` winners in s.win (key << 32 |
// ~local index), padded with -1 / -inf; local indices mapped through the block
// ids when given (from s.idx when ids_in_smem).
__device__ __forceinline__ void write_topk(const SelParams& p, int b, int count, const SelSmem& s, bool ids_in_smem) {
    int32_t* oi = p.out_idx + (int64_t)b * p.k;
    float* ov = p.out_val + (int64_t)b * p.k;
    for (int t = threadIdx.x; t < p.k; t += SEL_THREADS) {
        if (t < count) {
            const unsigned long long w = s.win[t];
            int64_t i = (int64_t)(uint32_t)~(uint32_t)(w & 0xFFFFFFFFull);
            if (p.block_ids) {
                const int64_t blk = ids_in_smem ? (int64_t)(int32_t)s.idx[i / p.block_size]
                                                : p.block_ids[(int64_t)b * p.ld_blocks + i / p.block_size];
                i = blk * p.block_size + i % p.block_size;
            }
            oi[t] = (int32_t)i;
            ov[t] = key_to_float((uint32_t)(w >> 32));
        } else {
            oi[t] = -1;
            ov[t] = __uint_as_float(0xFF800000u);
        }
    }
}

// Top-k of rows of at most SEL_CAP items whose histograms are complete
// (hist_small, TOPK mode): the Reindex layers' selection inside the pool.
__global__ void __launch_bounds__(SEL_THREADS, 1) sel_small_kernel(SelParams p) {
    griddep_wait();
    griddep_launch_dependents();
    SelSmem& s = sel_smem();
    const int b = blockIdx.x;
    const int64_t n = sel_items(p, b);
#ifdef HSI_TRACE
    if (threadIdx.x == 0) s.t_last = clock64();
#endif
    bool in_smem = false, ids_in_smem = false;
    int count = select_small_fast(p, b, n, p.hist + (int64_t)b * HIST_BINS, s, &in_smem, &ids_in_smem);
    if (count == SMALL_RADIX) count = select_small_radix(p, b, n, in_smem);
    else if (count == SMALL_WHOLE_ROW) count = select_row_smem(p, b, n, 0);
    write_topk(p, b, count, s, ids_in_smem);
    SEL_MARK(s, 31);
}

// Pool outputs of query b from the `count` winners in s.win (block ids in the
// low words, ~id): the ids in ascending order (s.win holds them so), -1
// padded; the visible-position count; the position bit table when given.
__device__ __noinline__ void write_pool(const SelParams& p, int b, int count) {
    SelSmem& s = sel_smem();
    const int bs = p.div;
    const int64_t n_vis = sel_len(p, b);
    const int64_t nb = (n_vis + bs - 1) / bs;
    int32_t* bo = p.blk_out + (int64_t)b * p.k;
    for (int t = threadIdx.x; t < p.k; t += SEL_THREADS)
        bo[t] = t < count ? (int32_t)(uint32_t)~(uint32_t)(s.win[t] & 0xFFFFFFFFull) : -1;
    if (threadIdx.x == 0) {
        p.n_kept[b] = count;
        // every kept block holds bs visible positions but the newest, which may hold fewer
        const int64_t last = count ? (int64_t)(uint32_t)~(uint32_t)(s.win[count - 1] & 0xFFFFFFFFull) : -1;
        p.n_pool[b] = (int32_t)((int64_t)bs * count - (last == nb - 1 ? (int64_t)bs * nb - n_vis : 0));
    }
    uint32_t* bits = p.bits ? p.bits + (int64_t)b * p.ld_bits : nullptr;
    if (!bits) return;
    const int64_t words = (n_vis + 31) / 32;
    if (bs == 8 && nb <= 32 * (int64_t)SEL_CAP) {
        // the kept blocks into a bitmap (s.keys), then every word of the table
        // at once: word w holds blocks 4w .. 4w+3, 8 bits each
        uint32_t* bm = s.keys;
        const int64_t bw = (nb + 31) / 32;
        for (int64_t w = threadIdx.x; w < bw; w += SEL_THREADS) bm[w] = 0u;
        __syncthreads();
        for (int t = threadIdx.x; t < count; t += SEL_THREADS) {
            const uint32_t id = ~(uint32_t)(s.win[t] & 0xFFFFFFFFull);
            atomicOr(&bm[id >> 5], 1u << (id & 31));
        }
        __syncthreads();
        write_pos_bits8(bits, bm, n_vis, threadIdx.x, SEL_THREADS);
        return;
    }
    for (int64_t wd = threadIdx.x; wd < words; wd += SEL_THREADS) bits[wd] = 0u;
    __syncthreads();
    for (int t = threadIdx.x; t < count; t += SEL_THREADS) {
        const int64_t blk = (int64_t)(uint32_t)~(uint32_t)(s.win[t] & 0xFFFFFFFFull);
        const int64_t a = blk * bs, e = min(n_vis, a + bs);
        for (int64_t pos = a; pos < e;) {
            const int64_t wd = pos >> 5;
            const int64_t we = min(e, (wd + 1) << 5);
            const int lo = (int)(pos & 31), cnt = (int)(we - pos);
            const uint32_t m = (cnt == 32) ? 0xFFFFFFFFu : (((1u << cnt) - 1u) << lo);
            atomicOr(&bits[wd], m);
            pos = we;
        }
    }
}

__global__ void __launch_bounds__(SEL_THREADS, 1) sel_final_kernel(SelParams p) {
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelSmem& s = *reinterpret_cast<SelSmem*>(smem_raw);
    const int b = blockIdx.x;
    const int64_t n = sel_items(p, b);
    int count;
    const int64_t id_range = p.mode == SEL_POOL ? n : 0;  // pool: block ids below n
#ifdef HSI_TRACE
    if (threadIdx.x == 0) s.t_last = clock64();
#endif
    if (n <= SEL_CAP) {
        count = select_row_smem(p, b, n, id_range);
    } else {
        const uint32_t c = p.cand_cnt[b];
        const uint32_t* ck = p.cand_key + (int64_t)b * p.cap;
        const uint32_t* ci = p.cand_idx + (int64_t)b * p.cap;
        if (c <= (uint32_t)SEL_CAP) {  // the survivors fit: select in shared memory
            for (uint32_t j = threadIdx.x; j < c; j += SEL_THREADS) {
                s.keys[j] = ck[j];
                s.idx[j] = ci[j];
            }
            __syncthreads();
            SmemSrc src{s.keys, s.idx, (int64_t)c};
            count = block_select<true>(src, s, p.k, id_range);
        } else if (c <= (uint32_t)p.cap) {  // all survivors kept: select over them in L2
            GlobalSrc src{ck, ci, (int64_t)c};
            count = block_select<false>(src, s, p.k, id_range);
        } else {  // survivors overflowed (heavy ties): select over the whole row
            RowSrc src{&p, b, n};
            count = block_select<false>(src, s, p.k, id_range);
        }
    }
    if (p.mode == SEL_TOPK) {
        write_topk(p, b, count, s, false);
    } else {
        write_pool(p, b, count);
    }
    SEL_MARK(s, 31);
}

// Pool rows of more than SEL_CAP blocks by the general route: the candidates
// of the collect pass (or the whole row when they overflowed) through the
// block select, then the pool outputs. Every thread of the block calls it.
__device__ __noinline__ void pool_generic(const SelParams& p, int b) {
    SelSmem& s = sel_smem();
    const int64_t n = sel_items(p, b);
    const uint32_t c = p.cand_cnt[b];
    const uint32_t* ck = p.cand_key + (int64_t)b * p.cap;
    const uint32_t* ci = p.cand_idx + (int64_t)b * p.cap;
    __syncthreads();  // the caller's reads of shared memory are done
    int count;
    if (c <= (uint32_t)SEL_CAP) {
        for (uint32_t j = threadIdx.x; j < c; j += SEL_THREADS) {
            s.keys[j] = ck[j];
            s.idx[j] = ci[j];
        }
        __syncthreads();
        SmemSrc src{s.keys, s.idx, (int64_t)c};
        count = block_select<true>(src, s, p.k, n);
    } else if (c <= (uint32_t)p.cap) {
        GlobalSrc src{ck, ci, (int64_t)c};
        count = block_select<false>(src, s, p.k, n);
    } else {
        RowSrc src{&p, b, n};
        count = block_select<false>(src, s, p.k, n);
    }
    write_pool(p, b, count);
}

constexpr int POOL_B2 = 2 * SEL_THREADS;  // second-level bins of the candidates' keys
constexpr int POOL_TIED_CAP = 2048;       // candidates of the threshold's second-level bin, ranked

// The candidate pool of rows of more than SEL_CAP blocks of 8 (SEL_POOL),
// after the threshold bin T (p.thr) and the collect pass (p.cand_*: every
// block whose maximum's key reaches bin T, the pinned newest block at key
// +inf). The candidates go into shared memory; a second histogram of POOL_B2
// bins spans their finite keys (from bin T's least key to the largest); its
// scan gives the bin T2 of the last place: the candidates at +inf and above
// T2 win, those in T2 are ranked among themselves (key, then lower id). The
// winners' bitmap gives the ids in ascending order, the pooled position count
// and the position bit table. Overflowing lists, more candidates at +inf than
// places and heavy ties in T2 take the general route.
__global__ void __launch_bounds__(SEL_THREADS, 1) pool_final_kernel(SelParams p) {
    static_assert(POOL_B2 + 2 * POOL_TIED_CAP + 2 * SEL_WARPS <= SEL_WARPS * 256, "bins, tied list, reductions in s.whist");
    static_assert(SEL_BITMAP_IDS / 64 <= SEL_MAXK, "the block bitmap fits in s.win");
    griddep_wait();
    griddep_launch_dependents();
    SelSmem& s = sel_smem();
    const int b = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t n_vis = sel_len(p, b);
    const int64_t nb = (n_vis + 7) / 8;
    const uint32_t c = p.cand_cnt[b];
    if (p.div != 8 || c > (uint32_t)SEL_CAP || nb > SEL_BITMAP_IDS) {
        pool_generic(p, b);
        return;
    }
    const uint32_t base = p.thr[b] << 20;
    const uint32_t* ck = p.cand_key + (int64_t)b * p.cap;
    const uint32_t* ci = p.cand_idx + (int64_t)b * p.cap;
    uint32_t* h2 = &s.whist[0][0];
    unsigned long long* tied = reinterpret_cast<unsigned long long*>(h2 + POOL_B2);
    uint32_t* wred = h2 + POOL_B2 + 2 * POOL_TIED_CAP;  // [2][SEL_WARPS]
    uint32_t* bm = reinterpret_cast<uint32_t*>(s.win);   // block bitmap
    const int words = (int)((nb + 31) / 32);
    uint32_t mx = 0, ninf = 0;
    for (uint32_t j = t; j < c; j += SEL_THREADS) {
        const uint32_t key = ck[j];
        s.keys[j] = key;
        s.idx[j] = ci[j];
        if (key >= KEY_POS_INF) ++ninf;
        else mx = max(mx, key);
    }
    h2[2 * t] = 0u;
    h2[2 * t + 1] = 0u;
    for (int w = t; w < words; w += SEL_THREADS) bm[w] = 0u;
    if (t == 0) s.bcast[6] = 0u;
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    ninf = __reduce_add_sync(0xFFFFFFFFu, ninf);
    if (lane == 0) {
        wred[warp] = mx;
        wred[SEL_WARPS + warp] = ninf;
    }
    __syncthreads();
    const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, wred[lane]);
    const uint32_t n_inf = __reduce_add_sync(0xFFFFFFFFu, wred[SEL_WARPS + lane]);
    const uint32_t k = (uint32_t)p.k;
    if (n_inf >= k && c > k) {  // more +inf keys than places (uniform)
        pool_generic(p, b);
        return;
    }
    const uint32_t kk = k > n_inf ? k - n_inf : 0u;  // places for the finite keys
    const uint32_t range = top > base ? top - base : 0u;
    const int sh2 = range >= (uint32_t)POOL_B2 ? 32 - __clz((int)(range / POOL_B2)) : 0;  // range >> sh2 < POOL_B2
    for (uint32_t j = t; j < c; j += SEL_THREADS) {
        const uint32_t key = s.keys[j];
        if (key < KEY_POS_INF) atomicAdd(&h2[min(key > base ? (key - base) >> sh2 : 0u, (uint32_t)(POOL_B2 - 1))], 1u);
    }
    __syncthreads();
    const uint32_t c0 = h2[2 * t], c1 = h2[2 * t + 1];
    uint32_t fin;
    const uint32_t below = block_excl_scan(c0 + c1, s, &fin);  // finite candidates in bins under 2t
    const bool take_all = fin <= kk;
    const uint32_t over = fin - below - c0 - c1;  // in the bins above 2t + 1
    if (!take_all && over < kk && over + c0 + c1 >= kk) {
        if (over + c1 >= kk) {
            s.bcast[2] = (uint32_t)(2 * t + 1);
            s.bcast[3] = over;
            s.bcast[4] = c1;
        } else {
            s.bcast[2] = (uint32_t)(2 * t);
            s.bcast[3] = over + c1;
            s.bcast[4] = c0;
        }
    }
    __syncthreads();
    const uint32_t T2 = take_all ? 0u : s.bcast[2], above = take_all ? 0u : s.bcast[3];
    if (!take_all && s.bcast[4] > (uint32_t)POOL_TIED_CAP) {  // heavy ties (uniform)
        pool_generic(p, b);
        return;
    }
    for (uint32_t j0 = 0; j0 < c; j0 += SEL_THREADS) {  // uniform trip count per warp
        const uint32_t j = j0 + (uint32_t)t;
        bool tie = false;
        uint32_t key = 0, id = 0;
        if (j < c) {
            key = s.keys[j];
            id = s.idx[j];
            bool win = key >= KEY_POS_INF || take_all;
            if (!win) {
                const uint32_t bin = min(key > base ? (key - base) >> sh2 : 0u, (uint32_t)(POOL_B2 - 1));
                win = bin > T2;
                tie = bin == T2;
            }
            if (win) {
                if (id < (uint32_t)nb) atomicOr(&bm[id >> 5], 1u << (id & 31));
                else raise_error(DEVERR_ARG);  // never a block of this row
            }
        }
        const uint32_t pos = warp_append(tie, &s.bcast[6]);
        if (tie && pos < (uint32_t)POOL_TIED_CAP) tied[pos] = ((unsigned long long)key << 32) | (uint32_t)~id;
    }
    __syncthreads();
    if (!take_all) {  // the tied candidates: the first (kk - above) by key, then lower id
        const uint32_t nt = min(s.bcast[6], (uint32_t)POOL_TIED_CAP);
        const uint32_t want = kk > above ? kk - above : 0u;
        for (uint32_t j = t; j < nt; j += SEL_THREADS) {
            const unsigned long long me = tied[j];
            uint32_t r = 0;
            for (uint32_t i = 0; i < nt; ++i) r += tied[i] > me ? 1u : 0u;
            const uint32_t id = ~(uint32_t)(me & 0xFFFFFFFFull);
            if (r < want && id < (uint32_t)nb) atomicOr(&bm[id >> 5], 1u << (id & 31));
        }
        __syncthreads();
    }
    // outputs: the ids in ascending order (each thread a run of consecutive words)
    constexpr int WPT = (int)(SEL_BITMAP_IDS / 32 / SEL_THREADS);
    uint32_t wv[WPT], mine = 0;
#pragma unroll
    for (int i = 0; i < WPT; ++i) {
        const int wd = t * WPT + i;
        wv[i] = wd < words ? bm[wd] : 0u;
        mine += (uint32_t)__popc(wv[i]);
    }
    uint32_t kept;
    uint32_t pos = block_excl_scan(mine, s, &kept);
    int32_t* bo = p.blk_out + (int64_t)b * p.k;
#pragma unroll
    for (int i = 0; i < WPT; ++i) {
        const uint32_t wbase = (uint32_t)(t * WPT + i) * 32u;
        uint32_t w = wv[i];
        while (w) {
            const uint32_t id = wbase + (uint32_t)(__ffs(w) - 1);
            w &= w - 1u;
            if (pos < k) bo[pos] = (int32_t)id;
            ++pos;
        }
    }
    for (uint32_t j = kept + (uint32_t)t; j < k; j += SEL_THREADS) bo[j] = -1;
    if (t == 0) {
        const bool last = nb > 0 && ((bm[(nb - 1) >> 5] >> ((nb - 1) & 31)) & 1u);
        p.n_kept[b] = (int32_t)min(kept, k);
        // every kept block holds 8 visible positions but the newest, which may hold fewer
        p.n_pool[b] = (int32_t)(8 * (int64_t)kept - (last ? 8 * nb - n_vis : 0));
    }
    if (p.bits) write_pos_bits8(p.bits + (int64_t)b * p.ld_bits, bm, n_vis, t, SEL_THREADS);
}

// A visible length within [0, max_n], the caller's bound that sized the rows;
// a larger value is clamped and reported as a device-side argument error.
__device__ __forceinline__ int64_t clamp_len(int64_t n, int64_t max_n) {
    if (n > max_n) {
        raise_error(DEVERR_ARG);
        n = max_n;
    }
    return n < 0 ? 0 : n;
}

// Block maxima of a score row: bmax[b][j] = max of scores[b][j*bs .. j*bs+bs)
// over visible positions (< n_visible[b]), for j < ceil(n_visible[b]/bs).
__global__ void block_max_kernel(const float* scores, int64_t ld, const int32_t* n_vis, int64_t max_n, int32_t bs,
                                 float* bmax, int64_t ldb) {
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.y;
    const int64_t n = clamp_len(n_vis[b], max_n);
    const int64_t nblk = (n + bs - 1) / bs;
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= nblk) return;
    const float* row = scores + (int64_t)b * ld;
    float m = __uint_as_float(0xFF800000u);
    const int64_t a = j * bs, e = min(n, a + bs);
    for (int64_t i = a; i < e; ++i) m = fmaxf(m, row[i]);
    bmax[(int64_t)b * ldb + j] = m;
}

// The pages' masked Reindex form, for comparison with the pooled layers: a
// score of query b at a visible position s (< n_visible[b]) whose pool bit
// (bit s%32 of bits[b][s/32]) is clear becomes -inf. One thread per position
// (a warp shares one bit word), grid = (ceil(max_visible / 256), B).
__global__ void __launch_bounds__(256) mask_scores_kernel(float* __restrict__ scores, int64_t ld,
                                                          const int32_t* __restrict__ n_vis, int64_t max_n,
                                                          const uint32_t* __restrict__ bits, int64_t ld_bits) {
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.y;
    const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t n = n_vis[b];
    if (blockIdx.x == 0 && threadIdx.x == 0 && n > max_n) raise_error(DEVERR_ARG);
    if (s >= min(n, max_n)) return;
    const uint32_t m = __ldg(bits + (int64_t)b * ld_bits + (s >> 5));
    if (!((m >> (s & 31)) & 1u)) scores[(int64_t)b * ld + s] = __uint_as_float(0xFF800000u);
}

}  // namespace hsi
