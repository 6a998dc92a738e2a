// Selection for many rows of moderate length, one CTA per query: the
// candidate pool and the top-k of a chunked-prefill layer from its block
// maxima, without a pass over the full score rows.
//
// For query b with n = n_visible[b] positions and nblk = ceil(n / 8) blocks
// (block value = max of its visible scores, the newest block pinned at +inf):
//   * the pool keeps the first min(n_keep, nblk) blocks by (value desc, block
//     index asc) whose value is > -inf;
//   * the top-k positions lie inside the first k blocks of that order without
//     the pin (a position outside them is outranked by the maximum of each of
//     k blocks ranked ahead of its own block), so inside the first k + 1
//     blocks of the pinned order; only those blocks' scores are read, and the
//     exact top-k by (score desc, position asc) is taken among them.
// Both block ranks come from one 4096-bin histogram of the order keys' top 12
// bits over the row of block maxima; the blocks at or above the lower of the
// two threshold bins are staged in shared memory (about n_keep plus one bin),
// and exact selection finishes there: radix passes over the remaining key
// bits, then over the index among items tied at the threshold key. A row
// whose staged blocks overflow the buffer (heavy ties) runs the same passes
// over the row in global memory instead.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace hsi {

constexpr int RS_THREADS = 256;
constexpr int RS_WARPS = RS_THREADS / 32;
constexpr int RS_CAP = 3072;             // staged items: blocks after the 12-bit filter, then candidate positions
constexpr int RS_MAX_BLOCKS = 65536;     // blocks per row (n_visible <= 524288)
constexpr int RS_MAXK = 2048;            // largest k
constexpr uint32_t RS_ALL = 0xFFFFFFFFu;  // index cutoff that takes every tied item
constexpr uint32_t RS_KEY_POS_INF = 0xFF800000u;  // order key of +inf (the pinned newest block)
constexpr uint32_t RS_KEY_NEG_INF = 0x007FFFFFu;  // order key of -inf (a block the pool drops)

struct RowSelParams {
    const float* bmax;  // [B][ldb] maxima of blocks of 8 visible scores
    int64_t ldb;
    const float* scores;  // [B][ld]
    int64_t ld;
    const int32_t* n_vis;  // [B]
    int64_t max_vis;       // the caller's bound on n_vis[b]
    int32_t B;
    int32_t k;  // top-k size, 1 .. RS_MAXK
    int32_t* out_idx;
    float* out_val;
    int32_t n_keep;  // pool size in blocks (0: no pool)
    int32_t* blk_out;
    int32_t* n_kept;
    int32_t* n_pool;
    uint32_t* bits;  // may be NULL
    int64_t ld_bits;
};

struct RowSelSmem {
    union {
        uint32_t hist[4096];
        unsigned long long win[RS_MAXK];  // winners of the top-k, sorted in place
    };
    uint32_t ckey[RS_CAP];
    uint32_t cidx[RS_CAP];
    union {
        uint32_t bitmap[RS_MAX_BLOCKS / 32];  // kept blocks of the pool
        int32_t cblk[RS_MAXK + 1];            // candidate blocks of the top-k
    };
    uint32_t scan[2 * RS_WARPS];
    uint32_t bc[8];
    uint32_t count;
};

// Item sources: n items, item j's order key (and whether it is eligible) and index.
struct RsBlockRow {  // the row of block maxima in global memory, all but the newest block
    const float* row;
    int64_t n;
    __device__ uint32_t key(int64_t j, bool& ok) const {
        ok = true;
        return order_key(row[j]);
    }
    __device__ uint32_t idx(int64_t j) const { return (uint32_t)j; }
};
struct RsStaged {  // items staged in shared memory
    const uint32_t* keys;
    const uint32_t* ids;
    int64_t n;
    __device__ uint32_t key(int64_t j, bool& ok) const {
        ok = true;
        return keys[j];
    }
    __device__ uint32_t idx(int64_t j) const { return ids[j]; }
};
struct RsCandScores {  // the 8 positions of each candidate block, scores in global memory
    const float* row;
    const int32_t* blocks;
    int64_t n;  // 8 x candidate blocks
    int64_t n_vis;
    uint32_t lo;  // positions whose key is below lo are not eligible
    __device__ uint32_t key(int64_t j, bool& ok) const {
        const int64_t pos = (int64_t)blocks[j >> 3] * 8 + (j & 7);
        ok = pos < n_vis;
        const uint32_t k = ok ? order_key(row[pos]) : 0u;
        ok = ok && k >= lo;
        return k;
    }
    __device__ uint32_t idx(int64_t j) const { return (uint32_t)((int64_t)blocks[j >> 3] * 8 + (j & 7)); }
};

// Whole block: exclusive scan of one value per thread, from the top thread
// down (from_top) or from thread 0 up; *total gets the sum over the block.
__device__ __forceinline__ uint32_t rs_scan(uint32_t v, bool from_top, RowSelSmem& s, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t inc = v;
    if (from_top) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, inc, o);
            if (lane + o < 32) inc += t;
        }
        if (lane == 0) s.scan[warp] = inc;
    } else {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += t;
        }
        if (lane == 31) s.scan[warp] = inc;
    }
    __syncthreads();
    uint32_t off = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < RS_WARPS; ++w) {
        const uint32_t c = s.scan[w];
        tot += c;
        if (from_top ? w > warp : w < warp) off += c;
    }
    __syncthreads();  // s.scan may be reused at once
    *total = tot;
    return off + inc - v;
}

// Whole block: counts of the bins of s.hist (nbins = 256 or 4096). Finds the
// bin holding the r-th item counted from the top bin (desc) or from bin 0
// (asc), r >= 1 and at most the total. Returns the bin; *before = items in
// the bins ahead of it in that direction; *at = items in it.
__device__ uint32_t rs_find(RowSelSmem& s, int nbins, uint32_t r, bool desc, uint32_t* before, uint32_t* at) {
    const int per = nbins / RS_THREADS;  // 1 or 16 bins per thread, thread t owning [t per, t per + per)
    const int t = threadIdx.x;
    uint32_t c = 0;
    for (int i = 0; i < per; ++i) c += s.hist[t * per + i];
    uint32_t tot;
    const uint32_t ex = rs_scan(c, desc, s, &tot);
    if (ex < r && ex + c >= r) {
        uint32_t run = ex;
        for (int i = 0; i < per; ++i) {
            const int bin = desc ? t * per + per - 1 - i : t * per + i;
            const uint32_t h = s.hist[bin];
            if (run + h >= r) {
                s.bc[0] = (uint32_t)bin;
                s.bc[1] = run;
                s.bc[2] = h;
                break;
            }
            run += h;
        }
    }
    __syncthreads();
    const uint32_t d = s.bc[0];
    *before = s.bc[1];
    *at = s.bc[2];
    __syncthreads();
    return d;
}

// Whole block: histogram into s.hist[0 .. nbins) of digit(j) over the items
// of src for which it is >= 0.
template <class Src, class Digit>
__device__ void rs_hist(const Src& src, RowSelSmem& s, int nbins, Digit digit) {
    for (int i = threadIdx.x; i < nbins; i += RS_THREADS) s.hist[i] = 0u;
    __syncthreads();
    for (int64_t j = threadIdx.x; j < src.n; j += RS_THREADS) {
        const int d = digit(j);
        if (d >= 0) atomicAdd(&s.hist[d], 1u);
    }
    __syncthreads();
}

struct RsCut {
    uint32_t key;  // the r-th item's key
    uint32_t idx;  // the largest index taken among items with that key (RS_ALL: all of them)
};

// Whole block: the r-th eligible item of src in (key desc, index asc) order,
// given that its key's top `bits` bits are `pfx` and `above` eligible items
// have a larger top-`bits` prefix. The first r items are exactly those with
// key > cut.key, or key == cut.key and index <= cut.idx. idx_bits bounds the
// indices (every index < 2^idx_bits).
template <class Src>
__device__ RsCut rs_select(const Src& src, RowSelSmem& s, uint32_t r, uint32_t pfx, int bits, uint32_t above,
                           int idx_bits) {
    uint32_t at = 0;
    while (bits < 32) {
        const int w = bits == 0 ? 12 : min(8, 32 - bits);
        const int shift = 32 - bits - w;
        const int nb = 1 << w;
        const uint32_t P = pfx;
        const int B = bits;
        rs_hist(src, s, nb < RS_THREADS ? RS_THREADS : nb, [&](int64_t j) -> int {
            bool ok;
            const uint32_t key = src.key(j, ok);
            if (!ok || (B > 0 && (key >> (32 - B)) != P)) return -1;
            return (int)((key >> shift) & (uint32_t)(nb - 1));
        });
        uint32_t before;
        const uint32_t d = rs_find(s, nb < RS_THREADS ? RS_THREADS : nb, r - above, true, &before, &at);
        above += before;
        pfx = (bits == 0 ? 0u : pfx << w) | d;
        bits += w;
    }
    const uint32_t need = r - above;  // 1 .. at
    if (need == at) return {pfx, RS_ALL};
    // the need-th smallest index among the items tied at key pfx
    const uint32_t T = pfx;
    uint32_t ipfx = 0, below = 0;
    int ib = 0;  // index bits resolved from the top of idx_bits
    while (ib < idx_bits) {
        const int w = min(8, idx_bits - ib);
        const int shift = idx_bits - ib - w;
        const uint32_t P = ipfx;
        const int IB = ib;
        rs_hist(src, s, RS_THREADS, [&](int64_t j) -> int {
            bool ok;
            if (src.key(j, ok) != T || !ok) return -1;
            const uint32_t i = src.idx(j);
            if (IB > 0 && (i >> (shift + w)) != P) return -1;
            return (int)((i >> shift) & ((1u << w) - 1u));
        });
        uint32_t bf, a2;
        const uint32_t d = rs_find(s, RS_THREADS, need - below, false, &bf, &a2);
        below += bf;
        ipfx = (ipfx << w) | d;
        ib += w;
    }
    return {T, ipfx};
}

__device__ __forceinline__ bool rs_taken(uint32_t key, uint32_t idx, RsCut c) {
    return key > c.key || (key == c.key && idx <= c.idx);
}

__device__ __forceinline__ int rs_bits_for(int64_t n) {  // bits holding every index < n
    return n <= 1 ? 1 : 64 - __clzll((unsigned long long)(n - 1));
}

// Slot of this thread's first item in a shared-memory list counted by
// *counter, for the items it marks in `take` (one bit each; its items follow
// consecutively): one warp scan and one atomic per warp. Every lane of the
// warp calls it.
__device__ __forceinline__ uint32_t rs_append_mask(uint32_t take, uint32_t* counter) {
    const int lane = threadIdx.x & 31;
    const uint32_t c = (uint32_t)__popc(take);
    uint32_t inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += t;
    }
    uint32_t base = 0;
    if (lane == 31 && inc) base = atomicAdd(counter, inc);
    base = __shfl_sync(0xFFFFFFFFu, base, 31);
    return base + inc - c;
}

// A bitonic compare-exchange of element e (value x) with its partner e ^ str
// (value y) inside merges of `size`: the final order is descending.
__device__ __forceinline__ unsigned long long rs_cmpx(unsigned long long x, unsigned long long y, int e, int str,
                                                      int size) {
    const bool keep_max = ((e & size) == 0) == ((e & str) == 0);
    return keep_max ? (x > y ? x : y) : (x < y ? x : y);
}

// Whole block: sort s.win[0 .. 512) descending (entries past count must be
// 0, below every real entry). Thread t holds elements t and t + 256 in
// registers: partners 256 apart are in the same thread, partners 1 .. 16
// apart in the same warp (shuffles), only strides 32 .. 128 go through
// shared memory.
__device__ void rs_sort512(RowSelSmem& s) {
    const int t = threadIdx.x;
    unsigned long long x[2] = {s.win[t], s.win[t + 256]};
    __syncthreads();
    for (int size = 2; size <= 512; size <<= 1) {
        for (int str = size >> 1; str > 0; str >>= 1) {
            if (str == 256) {
                const unsigned long long a = rs_cmpx(x[0], x[1], t, 256, size);
                x[1] = rs_cmpx(x[1], x[0], t + 256, 256, size);
                x[0] = a;
            } else if (str < 32) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const unsigned long long y = __shfl_xor_sync(0xFFFFFFFFu, x[r], str);
                    x[r] = rs_cmpx(x[r], y, t + 256 * r, str, size);
                }
            } else {
                s.win[t] = x[0];
                s.win[t + 256] = x[1];
                __syncthreads();
#pragma unroll
                for (int r = 0; r < 2; ++r) x[r] = rs_cmpx(x[r], s.win[(t + 256 * r) ^ str], t + 256 * r, str, size);
                __syncthreads();
            }
        }
    }
    s.win[t] = x[0];
    s.win[t + 256] = x[1];
    __syncthreads();
}

// Whole block: sort s.win[0 .. count) descending (bitonic network over the
// next power of two; padding entries are 0, below every real entry).
__device__ void rs_sort_desc(RowSelSmem& s, int count) {
    int m = 2;
    while (m < count) m <<= 1;
    for (int i = count + threadIdx.x; i < m; i += RS_THREADS) s.win[i] = 0ull;
    __syncthreads();
    for (int size = 2; size <= m; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < m / 2; i += RS_THREADS) {
                const int lo = 2 * i - (i & (stride - 1));  // i with a 0 inserted at bit log2(stride)
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const unsigned long long a = s.win[lo], c = s.win[hi];
                if (desc ? a < c : a > c) {
                    s.win[lo] = c;
                    s.win[hi] = a;
                }
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(RS_THREADS) rowsel_kernel(RowSelParams p) {
    extern __shared__ __align__(16) uint8_t rs_smem_raw[];
    RowSelSmem& s = *reinterpret_cast<RowSelSmem*>(rs_smem_raw);
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    int64_t n_vis = p.n_vis[b];
    if (n_vis > p.max_vis) {
        if (tid == 0) raise_error(DEVERR_ARG);
        n_vis = p.max_vis;
    }
    if (n_vis < 0) n_vis = 0;
    const int64_t nblk = (n_vis + 7) / 8;
    const RsBlockRow rowsrc{p.bmax + (int64_t)b * p.ldb, nblk > 0 ? nblk - 1 : 0};

    // The newest block is pinned first in both orders, so it is taken apart:
    // the selections run over the other nu = nblk - 1 blocks for ranks r - 1.
    const int64_t nu = nblk > 0 ? nblk - 1 : 0;
    const uint32_t r_pool = (uint32_t)min((int64_t)p.n_keep, nblk);
    const uint32_t r_cand = (uint32_t)min((int64_t)p.k + 1, nblk);
    const uint32_t rp = r_pool > 0 ? r_pool - 1 : 0, rc = r_cand > 0 ? r_cand - 1 : 0;
    constexpr int U = 8;  // 16-byte loads per thread issued before any is used
    const float4* row4 = reinterpret_cast<const float4*>(rowsrc.row);
    const int64_t n4 = (nu + 3) / 4;
    // fn(bit, j, key) for the 32 unpinned blocks of this thread in round q0
    auto round = [&](int64_t q0, auto fn) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t q = q0 + u * RS_THREADS + tid;
            v[u] = q < n4 ? row4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t j0 = 4 * (q0 + u * RS_THREADS + tid);
            const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) fn(4 * u + e, j0 + e, j0 + e < nu, order_key(f[e]));
        }
    };
    // 1. the largest key M of the unpinned blocks
    uint32_t mx = 0;
    for (int64_t q0 = 0; q0 < n4; q0 += (int64_t)U * RS_THREADS)
        round(q0, [&](int, int64_t, bool in, uint32_t key) {
            if (in) mx = max(mx, key);
        });
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if ((tid & 31) == 0) s.scan[tid >> 5] = mx;
    if (tid == 0) s.count = 0;
    __syncthreads();
    uint32_t M = 0;
#pragma unroll
    for (int w = 0; w < RS_WARPS; ++w) M = max(M, s.scan[w]);
    __syncthreads();
    // 2. histogram of the keys relative to M: bin (M >> sh) - (key >> sh), 4096
    // bins from the top (scores cluster: relative bins of 1/2048 octave spread
    // the top ranks where bins of the keys' top 12 bits would not); bins capped
    // at 4095. If a rank falls in the capped bin, again with sh = 20, where no
    // bin is capped.
    uint32_t tb_pool = 0, ab_pool = 0, tb_cand = 0, ab_cand = 0, at;
    int sh = 12;
    for (int attempt = 0; attempt < 2 && (rp > 0 || rc > 0); ++attempt) {
        for (int i = tid; i < 4096; i += RS_THREADS) s.hist[i] = 0u;
        __syncthreads();
        const uint32_t Ms = M >> sh;
        for (int64_t q0 = 0; q0 < n4; q0 += (int64_t)U * RS_THREADS)
            round(q0, [&](int, int64_t, bool in, uint32_t key) {
                if (in) atomicAdd(&s.hist[min(Ms - (key >> sh), 4095u)], 1u);
            });
        __syncthreads();
        if (rp > 0) tb_pool = rs_find(s, 4096, rp, false, &ab_pool, &at);
        if (rc > 0) tb_cand = rs_find(s, 4096, rc, false, &ab_cand, &at);
        if (sh == 20 || ((rp == 0 || tb_pool < 4095) && (rc == 0 || tb_cand < 4095))) break;
        sh = 20;
    }
    const uint32_t Ms = M >> sh;
    const uint32_t hi_bin = max(rp > 0 ? tb_pool : 0u, rc > 0 ? tb_cand : 0u);
    // 3. stage the blocks in bins 0 .. hi_bin (the row is read again, from L2)
    if (rp > 0 || rc > 0) {
        for (int64_t q0 = 0; q0 < n4; q0 += (int64_t)U * RS_THREADS) {
            uint32_t keys[4 * U];
            uint32_t take = 0;
            round(q0, [&](int bit, int64_t, bool in, uint32_t key) {
                keys[bit] = key;
                if (in && Ms - (key >> sh) <= hi_bin) take |= 1u << bit;
            });
            uint32_t slot = rs_append_mask(take, &s.count);
#pragma unroll
            for (int i = 0; i < 4 * U; ++i) {
                if ((take >> i) & 1u) {
                    if (slot < RS_CAP) {
                        s.ckey[slot] = keys[i];
                        s.cidx[slot] = (uint32_t)(4 * (q0 + (i / 4) * RS_THREADS + tid) + (i % 4));
                    }
                    ++slot;
                }
            }
        }
    }
    __syncthreads();
    const uint32_t staged = s.count;
    const bool fits = staged <= RS_CAP;
    const int blk_bits = rs_bits_for(nblk);
    const RsStaged stsrc{s.ckey, s.cidx, (int64_t)staged};
    constexpr RsCut none{0xFFFFFFFFu, 0u};  // no unpinned block taken (order keys never reach it)
    RsCut c_pool = none, c_cand = none;
    if (rp > 0)
        c_pool = fits ? rs_select(stsrc, s, rp, Ms - tb_pool, 32 - sh, ab_pool, blk_bits)
                      : rs_select(rowsrc, s, rp, Ms - tb_pool, 32 - sh, ab_pool, blk_bits);
    if (rc > 0)
        c_cand = fits ? rs_select(stsrc, s, rc, Ms - tb_cand, 32 - sh, ab_cand, blk_bits)
                      : rs_select(rowsrc, s, rc, Ms - tb_cand, 32 - sh, ab_cand, blk_bits);
    const int64_t nsrc = fits ? (int64_t)staged : nu;  // unpinned blocks the pool and the candidates come from

    // 4. the pool: kept blocks (dropping -inf ones) as a bitmap, then their ids
    // ascending, the visible-position count and the boolean table
    if (p.n_keep > 0) {
        const int64_t words = (nblk + 31) / 32;
        // the boolean table reads blocks 4w .. 4w+3 for its words w < ceil(n_vis / 32)
        const int64_t zwords = max(words, ((n_vis + 31) / 32 + 7) / 8);
        for (int64_t w = tid; w < zwords; w += RS_THREADS) s.bitmap[w] = 0u;
        __syncthreads();
        if (tid == 0 && r_pool > 0) atomicOr(&s.bitmap[(nblk - 1) >> 5], 1u << ((nblk - 1) & 31));  // pinned
        for (int64_t j = tid; j < nsrc; j += RS_THREADS) {
            bool ok;
            const uint32_t key = fits ? s.ckey[j] : rowsrc.key(j, ok);
            const uint32_t id = fits ? s.cidx[j] : (uint32_t)j;
            if (rs_taken(key, id, c_pool) && key != RS_KEY_NEG_INF) atomicOr(&s.bitmap[id >> 5], 1u << (id & 31));
        }
        __syncthreads();
        // ids ascending: thread t owns words [t per, t per + per)
        const int per = (int)((words + RS_THREADS - 1) / RS_THREADS);
        uint32_t mine = 0;
        for (int i = 0; i < per; ++i) {
            const int64_t w = (int64_t)tid * per + i;
            if (w < words) mine += __popc(s.bitmap[w]);
        }
        uint32_t kept;
        uint32_t rank = rs_scan(mine, false, s, &kept);
        int32_t* bo = p.blk_out + (int64_t)b * p.n_keep;
        for (int i = 0; i < per; ++i) {
            const int64_t w = (int64_t)tid * per + i;
            if (w >= words) break;
            uint32_t m = s.bitmap[w];
            while (m) {
                const int bit = __ffs(m) - 1;
                m &= m - 1;
                if (rank < (uint32_t)p.n_keep) bo[rank] = (int32_t)(w * 32 + bit);
                ++rank;
            }
        }
        for (int64_t t = kept + tid; t < p.n_keep; t += RS_THREADS) bo[t] = -1;
        if (tid == 0) {
            p.n_kept[b] = (int32_t)kept;
            // the newest block is pinned, so it is kept; its positions past n_vis are not in the pool
            p.n_pool[b] = (int32_t)(kept ? (int64_t)kept * 8 - (nblk * 8 - n_vis) : 0);
        }
        if (p.bits) write_pos_bits8(p.bits + (int64_t)b * p.ld_bits, s.bitmap, n_vis, tid, RS_THREADS);
        __syncthreads();  // the bitmap is reused for the candidate blocks
    }

    // 5. the top-k among the candidate blocks' positions
    if (p.k > 0) {
        if (tid == 0) {
            s.count = r_cand > 0 ? 1u : 0u;
            if (r_cand > 0) s.cblk[0] = (int32_t)(nblk - 1);  // the pinned block
        }
        __syncthreads();
        for (int64_t j0 = 0; j0 < nsrc; j0 += 8 * RS_THREADS) {
            uint32_t take = 0, id[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t j = j0 + u * RS_THREADS + tid;
                bool ok = false;
                uint32_t key = 0;
                id[u] = 0;
                if (j < nsrc) {
                    key = fits ? s.ckey[j] : rowsrc.key(j, ok);
                    id[u] = fits ? s.cidx[j] : (uint32_t)j;
                    if (rs_taken(key, id[u], c_cand)) take |= 1u << u;
                }
            }
            uint32_t slot = rs_append_mask(take, &s.count);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if ((take >> u) & 1u) {
                    if (slot <= (uint32_t)RS_MAXK) s.cblk[slot] = (int32_t)id[u];
                    ++slot;
                }
        }
        __syncthreads();
        const int64_t ncb = min((int64_t)s.count, (int64_t)RS_MAXK + 1);
        __syncthreads();
        // Every top-k position has a score at or above the k-th largest block
        // maximum, which is at least the key of the last candidate block (the
        // (k+1)-th of the pinned order) when there are more than k blocks; only
        // the candidate positions at or above that key are staged. With k + 1
        // blocks or fewer every visible position is a candidate.
        const uint32_t lo = r_cand == (uint32_t)p.k + 1 ? c_cand.key : 0u;
        const float* row = p.scores + (int64_t)b * p.ld;
        if (tid == 0) s.count = 0;
        __syncthreads();
        for (int64_t c0 = 0; c0 < ncb; c0 += 2 * RS_THREADS) {  // two blocks (16 positions) per thread per round
            float v[16];
            int64_t base[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int64_t ci = c0 + u * RS_THREADS + tid;
                base[u] = ci < ncb ? (int64_t)s.cblk[ci] * 8 : -1;
#pragma unroll
                for (int e = 0; e < 8; ++e) v[8 * u + e] = base[u] >= 0 && base[u] + e < n_vis ? row[base[u] + e] : 0.f;
            }
            uint32_t take = 0;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (base[i / 8] >= 0 && base[i / 8] + (i % 8) < n_vis && order_key(v[i]) >= lo) take |= 1u << i;
            uint32_t slot = rs_append_mask(take, &s.count);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if ((take >> i) & 1u) {
                    if (slot < RS_CAP) {
                        s.ckey[slot] = order_key(v[i]);
                        s.cidx[slot] = (uint32_t)(base[i / 8] + (i % 8));
                    }
                    ++slot;
                }
        }
        __syncthreads();
        const uint32_t staged2 = s.count;
        const bool fits2 = staged2 <= RS_CAP;
        const RsCandScores gsrc{row, s.cblk, ncb * 8, n_vis, lo};
        const uint32_t kk = (uint32_t)min((int64_t)p.k, n_vis);  // all of them lie among the staged positions
        const RsStaged st2{s.ckey, s.cidx, (int64_t)staged2};
        const int pos_bits = rs_bits_for(n_vis);
        RsCut c{0u, 0u};
        if (kk > 0) c = fits2 ? rs_select(st2, s, kk, 0u, 0, 0u, pos_bits) : rs_select(gsrc, s, kk, 0u, 0, 0u, pos_bits);
        // winners, then sorted by (key desc, position asc)
        if (tid == 0) s.count = 0;
        __syncthreads();
        const int64_t n2 = fits2 ? (int64_t)staged2 : ncb * 8;
        for (int64_t j0 = 0; j0 < n2; j0 += 8 * RS_THREADS) {
            uint32_t take = 0;
            unsigned long long w8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t j = j0 + u * RS_THREADS + tid;
                bool ok = false;
                uint32_t key = 0, id = 0;
                if (j < n2) {
                    if (fits2) {
                        ok = true;
                        key = s.ckey[j];
                        id = s.cidx[j];
                    } else {
                        key = gsrc.key(j, ok);
                        id = gsrc.idx(j);
                    }
                }
                if (ok && kk > 0 && rs_taken(key, id, c)) take |= 1u << u;
                w8[u] = ((unsigned long long)key << 32) | (uint32_t)~id;
            }
            uint32_t slot = rs_append_mask(take, &s.count);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if ((take >> u) & 1u) {
                    if (slot < (uint32_t)RS_MAXK) s.win[slot] = w8[u];
                    ++slot;
                }
        }
        __syncthreads();
        const int cnt = (int)min(s.count, kk);
        if (cnt <= 512) {
            for (int i = cnt + tid; i < 512; i += RS_THREADS) s.win[i] = 0ull;
            __syncthreads();
            rs_sort512(s);
        } else {
            rs_sort_desc(s, cnt);
        }
        int32_t* oi = p.out_idx + (int64_t)b * p.k;
        float* ov = p.out_val + (int64_t)b * p.k;
        for (int t = tid; t < p.k; t += RS_THREADS) {
            if (t < cnt) {
                const unsigned long long w = s.win[t];
                oi[t] = (int32_t)(uint32_t)~(uint32_t)(w & 0xFFFFFFFFull);
                ov[t] = key_to_float((uint32_t)(w >> 32));
            } else {
                oi[t] = -1;
                ov[t] = __uint_as_float(0xFF800000u);
            }
        }
    }
}

}  // namespace hsi
