// K2 / K5: lightning-indexer scoring on the tensor cores.
//
//   I = (g_q g_k / 128) * sum_j w_j * ReLU(q_j . k)
//
// One unit = UT tiles of 128 keys (16 NVFP4 block records of 8 keys each) x
// one query group (NQ queries x 32 heads). Per tile the contraction
// D[key][head] = K_tile . Q^T is tcgen05.mma kind::mxf4nvf4 with
// per-16-element E4M3 scales (M = 128, N = 32 NQ, K = 128 as two K = 64
// steps), accumulated in fp32 in Tensor Memory. The epilogue reads D from TMEM
// (one key per thread), applies ReLU and the head weights and writes one fp32
// score per key, so per-head logits never leave the SM.
//
// Warp roles in a persistent CTA (one per SM):
//   producer     full scan (warp 0): one bulk copy (TMA engine) per unit of its
//                16 UT consecutive records (36 KB for UT = 4; below ~18 KB the
//                per-copy rate, not HBM, limits a bulk-copy stream) into a
//                ring of shared-memory stages, and of the group's q records
//                into one of two q slots. Pool gather (warps 0..3): 16-byte
//                cp.async copies, four threads per pooled 576-byte record (one
//                bulk copy per record is slower: the engine takes ~77 cycles
//                per copy); the block ids come IDS_AHEAD units ahead by bulk
//                copy.
//   MMA warp     one thread issues every MMA and commit; the warp owns TMEM.
//   scale warps  a warpgroup that writes each unit's (and each q group's) E4M3
//                scales from the records in shared memory straight into TMEM
//                (tcgen05.st, one 32-lane quarter per warp) in the layout the
//                block-scaled MMA reads, so no copy instruction occupies the
//                tensor pipe. In a gather with pool_out, its first thread also
//                bulk-stores each landed unit into the compacted pool.
//   epilogue     groups of four warps (one per TMEM quarter): two for single
//                queries, three for 4-query tiles, one for the gather; group e
//                takes the units u with u % groups == e, and frees each tile of
//                an accumulator set as soon as it holds it in registers.
// The block records are used in place as the MMA operands: a record is eight
// rows of four 8x16-byte core matrices (K-major, no swizzle, core matrices
// 128 B apart along K, records 576 B apart along M/N).
//
// Record formats (template parameter FMT): NVFP4 records are 576 bytes (codes,
// then per row eight E4M3 scales of 16 elements; one fp32 tensor scale per
// query and per cache); MXFP4 records are 544 bytes (codes, then per row four
// E8M0 scales of 32 elements; no tensor scale) and take the MMA's
// scale_vec::2X form with UE8M0 scales.
//
// Work: units of all queries are numbered in order (query group, then key
// range) and each CTA takes one contiguous range, so it reloads q only when
// the group changes. Every wait is bounded; on a timeout the CTA records the
// error, drains its copies and MMAs, frees TMEM and returns.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace hsi {

constexpr int REC = 576;  // NVFP4 record bytes
enum : int { FMT_NVFP4 = 0, FMT_MXFP4 = 1 };
template <int FMT>
__host__ __device__ constexpr int rec_bytes() {
    return FMT == FMT_MXFP4 ? 544 : 576;
}
constexpr int TILE_KEYS = 128;
constexpr int IDS_AHEAD = 8;  // gather: units of block ids prefetched ahead

struct ScoreParams {
    const uint8_t* q_rec;
    const float* g_q;
    const float* w;
    const uint8_t* k_rec;
    const float* g_k;
    const int64_t* k_off;  // first record of query b's keys; NULL: b * k_stride
    int64_t k_stride;
    const int32_t* n_vis;
    int32_t max_vis;  // the caller's bound on n_vis[b]; a larger value is clamped and reported
    int32_t B;
    int32_t ngroups;
    // full scan
    float* scores;
    int64_t ld;
    float* bmax;
    int64_t ldb;
    // optional (a scan of pooled records laid out contiguously): keys in
    // [n_vis[b], 8 min(pad_blocks[b], n_keep)) are written as -inf
    const int32_t* pad_blocks;
    // optional (single-query groups): 4096-bin histogram of the top 12 bits of
    // the order keys of the scores, [B][4096], added to
    uint32_t* key_hist;
    // optional (single-query groups, with bmax): the same histogram of the
    // block maxima, [B][4096], added to
    uint32_t* bmax_hist;
    // pool gather
    const int32_t* block_ids;
    const int32_t* n_kept;
    int32_t n_keep;  // multiple of 16 UT
    float* pool_scores;
    int64_t ld_pool;
    // optional: the gathered records of each unit are also written here, query
    // b's pool slots at pool_out[(b n_keep + slot / 8) 576 ..] (the layout of a
    // compacted pool), records past n_kept[b] not written
    uint8_t* pool_out;
};

template <int NQ, bool GATHER, int STAGES, int UT, int FMT>
struct ScoreCfg {
    static constexpr int REC = rec_bytes<FMT>();
    static constexpr int N = 32 * NQ;
    static constexpr int UNIT_RECS = 16 * UT;
    static constexpr int UNIT_KEYS = TILE_KEYS * UT;
    // accumulator sets (one set = UT tiles)
    static constexpr int NACC = (NQ == 1 && UT <= 2) ? 4 : NQ > 1 ? 3 : 2;
    static constexpr int Q_BYTES = NQ * 4 * REC;
    static constexpr int STAGE_BYTES = UNIT_RECS * REC;
    static constexpr int QSLOT_BYTES = ((Q_BYTES + 127) / 128) * 128;
    // gather: producer warps of 16-byte async copies (TPR threads per pooled block)
#ifndef HSI_GATHER_PROD_WARPS
#define HSI_GATHER_PROD_WARPS 4
#endif
    static constexpr int PROD_WARPS = GATHER ? HSI_GATHER_PROD_WARPS : 1;
    static constexpr int TPR = GATHER ? 32 * PROD_WARPS / UNIT_RECS : 1;  // gather: producer threads per record
    // MMA-issuing warps (one thread each), taking alternate units: a single
    // thread's issue sequence (waits, descriptors, MMAs, commit) per unit is
    // longer than the tensor work of a 4-query tile
#ifndef HSI_DECODE_ISSUERS
#define HSI_DECODE_ISSUERS 2
#endif
    static constexpr int MMA_ISSUERS = GATHER ? 1 : NQ > 1 ? 2 : HSI_DECODE_ISSUERS;
    static constexpr int MMA_WARP = PROD_WARPS;
    static constexpr int FIRST_SF_WARP = PROD_WARPS + MMA_ISSUERS;
    static constexpr int FIRST_EPI_WARP = FIRST_SF_WARP + 4;
    // single queries: two groups taking alternate units; multi-query tiles: one
    // group per query, every group reading its query's 32 columns of every tile
    static constexpr int EPI_GROUPS = GATHER ? 1 : NQ > 1 ? NQ : 2;
    // warps that read a tile before the MMAs may overwrite it
    static constexpr int ACC_READERS = NQ > 1 ? 4 * NQ : 4;
    static constexpr int THREADS = 32 * (FIRST_EPI_WARP + 4 * EPI_GROUPS);
#ifndef HSI_COPY_AHEAD
#define HSI_COPY_AHEAD 4
#endif
    static constexpr int COPY_AHEAD = HSI_COPY_AHEAD;  // gather: units of async copies in flight per producer thread
    // TMEM columns: accumulators, one SFA set per stage (UT tiles x 2 chunks x 4),
    // one SFB set per q slot (2 chunks x 4)
    static constexpr int COL_ACC = 0;
    static constexpr int COL_SFA = NACC * UT * N;
    static constexpr int COL_SFB = COL_SFA + STAGES * UT * 8;
    static constexpr int COLS_USED = COL_SFB + 16;
    static constexpr int TMEM_COLS = COLS_USED <= 32 ? 32 : COLS_USED <= 64 ? 64 : COLS_USED <= 128 ? 128
                                     : COLS_USED <= 256 ? 256 : 512;
    static constexpr int OFF_STAGES = 0;
    static constexpr int OFF_QSLOTS = STAGES * STAGE_BYTES;
    static constexpr int OFF_IDS = OFF_QSLOTS + 2 * QSLOT_BYTES;
    static constexpr int IDS_BYTES = GATHER ? IDS_AHEAD * UNIT_RECS * 4 : 0;
    // histogram slots for the first HIST_SLOTS queries of the CTA's range: the
    // scores' keys, then the block maxima's
    static constexpr int HIST_SLOTS = NQ == 1 ? 2 : 0;
    static constexpr int OFF_HIST = OFF_IDS + IDS_BYTES;
    static constexpr int HIST_BYTES = 2 * HIST_SLOTS * 4096 * 4;
    static constexpr int OFF_BARS = OFF_HIST + HIST_BYTES;
    // full, sfready, empty per stage; acc_full per accumulator set, acc_empty per
    // tile of a set (the epilogue frees each tile as soon as it has read it);
    // q_full, q_ready, q_empty per slot; ids_full, ids_free per id slot; drain
    static constexpr int NBARS = 3 * STAGES + NACC * (1 + UT) + 6 + (GATHER ? 2 * IDS_AHEAD : 0) + 1;
    static constexpr int SMEM_BYTES = OFF_BARS + NBARS * 8 + 64 + 1024;  // + alignment slack
    static_assert(NQ <= 4, "B scale rows fit one 128-row layout");
    static_assert(COLS_USED <= 512, "TMEM");
    static_assert(NQ > 1 || NACC % EPI_GROUPS == 0, "accumulator sets split evenly between epilogue groups");
    static_assert(!GATHER || (NQ == 1 && UNIT_RECS == 32 && TPR * UNIT_RECS == 32 * PROD_WARPS),
                  "gather: single queries, units of 32 records, whole producer warps per record group");
    static_assert(!GATHER || COPY_AHEAD < STAGES, "gather: copies in flight fit the ring");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

struct ScoreShared {  // small control block after the barriers
    uint32_t tmem_base;
    int abort;
    int g0;
    int t0;
    long long count;
};


// Whole block (at most 1024 threads): this CTA's first unit (g0, t0) and unit
// count. part_smem holds at least 65 entries.
template <class TilesFn>
__device__ void schedule_range(int ngroups, TilesFn tiles, ScoreShared* sh, long long* part_smem) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (ngroups + nt - 1) / nt;
    const int ga = min(ngroups, tid * per), gb = min(ngroups, ga + per);
    long long mine = 0;
    for (int g = ga; g < gb; ++g) mine += tiles(g);
    // exclusive prefix of the per-thread counts: warp scans, then a scan of warp totals
    const int lane = tid & 31, wid = tid >> 5, nw = (nt + 31) >> 5;
    long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) part_smem[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        long long wt = lane < nw ? part_smem[lane] : 0, wincl = wt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long v = __shfl_up_sync(0xFFFFFFFFu, wincl, o);
            if (lane >= o) wincl += v;
        }
        if (lane < nw) part_smem[32 + lane] = wincl - wt;  // exclusive warp offsets
        if (lane == 31) part_smem[64] = wincl;              // total
        if (lane == 0) {
            sh->count = 0;
            sh->g0 = ngroups;
            sh->t0 = 0;
        }
    }
    __syncthreads();
    const long long base = part_smem[32 + wid] + incl - mine;
    const long long total = part_smem[64];
    const long long lo = total * blockIdx.x / gridDim.x;
    const long long hi = total * (blockIdx.x + 1) / gridDim.x;
    if (lo < hi && mine > 0 && lo >= base && lo < base + mine) {
        long long run = base;
        for (int g = ga; g < gb; ++g) {
            const long long n = tiles(g);
            if (lo < run + n) {
                sh->g0 = g;
                sh->t0 = (int)(lo - run);
                sh->count = hi - lo;
                break;
            }
            run += n;
        }
    }
    __syncthreads();
}

__device__ __forceinline__ bool wait_role(uint64_t* bar, uint32_t parity, ScoreShared* sh) {
    return wait_bounded(bar, parity, (volatile int*)&sh->abort);
}

// Trace slots: which role waited on what (only with -DHSI_TRACE).
enum : int {
    TR_PROD_QEMPTY = 0, TR_PROD_EMPTY, TR_PROD_IDS, TR_SF_QFULL, TR_SF_FULL, TR_MMA_QREADY, TR_MMA_SFREADY,
    TR_MMA_ACCEMPTY, TR_EPI_ACCFULL, TR_MMA_ISSUE, TR_SF_WORK, TR_EPI_WORK, TR_PROD_ISSUE, TR_PROD_LAND,
    TR_PROD_TOTAL = 16, TR_SF_TOTAL, TR_MMA_TOTAL, TR_EPI_TOTAL, TR_UNITS
};

#ifdef HSI_TRACE
#define HSI_TSTART(v) const long long v = clock64()
#define HSI_TEND(v, slot) tr.add(slot, (unsigned long long)(clock64() - v))
#else
#define HSI_TSTART(v)
#define HSI_TEND(v, slot)
#endif

// Whole warp: wait, then agree, so that a warp leaves its loop as one (its
// .sync.aligned tcgen05 instructions and __syncwarp need every lane).
__device__ __forceinline__ bool wait_traced(uint64_t* bar, uint32_t parity, ScoreShared* sh, WaitTrace& tr,
                                            int slot) {
#ifdef HSI_TRACE
    // (try_wait itself blocks for a while, so time the whole wait)
    const long long t0 = clock64();
    const bool ok = wait_role(bar, parity, sh);
    tr.add(slot, (unsigned long long)(clock64() - t0));
#else
    (void)tr;
    (void)slot;
    const bool ok = wait_role(bar, parity, sh);
#endif
    return __all_sync(0xFFFFFFFFu, ok);
}

// Single-thread variant of wait_traced (no warp vote).
__device__ __forceinline__ bool wait_one(uint64_t* bar, uint32_t parity, ScoreShared* sh, WaitTrace& tr, int slot) {
#ifdef HSI_TRACE
    const long long t0 = clock64();
    const bool ok = wait_role(bar, parity, sh);
    tr.add(slot, (unsigned long long)(clock64() - t0));
    return ok;
#else
    (void)tr;
    (void)slot;
    return wait_role(bar, parity, sh);
#endif
}

// n_vis[b] within [0, max_vis] (the bound that sized the score rows and the
// caches); `report`: record a larger value as a device-side argument error.
__device__ __forceinline__ int vis_of(const ScoreParams& p, int b, bool report = false) {
    int n = p.n_vis[b];
    if (n > p.max_vis) {
        if (report) raise_error(DEVERR_ARG);
        n = p.max_vis;
    }
    return n < 0 ? 0 : n;
}

template <int NQ, bool GATHER, int UT>
__device__ __forceinline__ int group_units(const ScoreParams& p, int g) {
    if (GATHER) {
        const int nk = p.n_kept[g];
        return nk <= 0 ? 0 : (min(nk, p.n_keep) + 16 * UT - 1) / (16 * UT);
    } else {
        int m = 0;
#pragma unroll
        for (int i = 0; i < NQ; ++i) m = max(m, vis_of(p, g * NQ + i));
        return (m + TILE_KEYS * UT - 1) / (TILE_KEYS * UT);
    }
}

// Walks the units (group, unit in group) of this CTA's range in order.
template <int NQ, bool GATHER, int UT>
struct UnitIter {
    int g, t, nunits;
    __device__ void init(const ScoreParams& p, const ScoreShared* sh) {
        g = sh->g0;
        t = sh->t0;
        nunits = sh->count > 0 ? group_units<NQ, GATHER, UT>(p, g) : 0;
    }
    __device__ void next(const ScoreParams& p) {
        if (++t == nunits) {
            t = 0;
            do {
                ++g;
            } while (g < p.ngroups && (nunits = group_units<NQ, GATHER, UT>(p, g)) == 0);
        }
    }
};

// Position in a ring of n slots and the phase parity of the current lap.
struct Ring {
    int i = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next(int n) {
        if (++i == n) {
            i = 0;
            ph ^= 1u;
        }
    }
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The scales of rows r, r+32, r+64, r+96 of records at `recs` (nrows valid
// rows) in the layout of one 32-lane TMEM quarter: column c holds row r+32c,
// columns 0-3 the first 64 values (K step 0), columns 4-7 the last 64. NVFP4:
// a word holds the step's four E4M3 scales. MXFP4: the step's two E8M0 scales
// in bytes 0 and 1 (the row's scale word, rotated by 16 bits for step 1).
template <int FMT>
__device__ __forceinline__ void sf_quarter(const uint8_t* recs, int nrows, int r, uint32_t (&v)[8]) {
    constexpr int RB = rec_bytes<FMT>();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int m = r + 32 * c;
        if constexpr (FMT == FMT_MXFP4) {
            uint32_t x = 0u;
            if (m < nrows) x = *reinterpret_cast<const uint32_t*>(recs + (m >> 3) * RB + 512 + (m & 7) * 4);
            v[c] = x;
            v[4 + c] = __funnelshift_l(x, x, 16);
        } else {
            uint2 x = make_uint2(0u, 0u);
            if (m < nrows) x = *reinterpret_cast<const uint2*>(recs + (m >> 3) * RB + 512 + (m & 7) * 8);
            v[c] = x.x;
            v[4 + c] = x.y;
        }
    }
}

// The weighted ReLU head sum of one key, sum_j w_j * max(x_j, 0) over the 32
// heads, evaluated as ((s0 + s1) + (s2 + s3)) where s_r is the fma chain over
// the heads j = r (mod 4) in increasing j. The chains run in pairs, (s0, s1)
// and (s2, s3), as packed f32x2 fmas (w2[i] = w_2i, w_2i+1): 32 max and 16
// fma instructions per key instead of 32 + 32, bit for bit the same result.
__device__ __forceinline__ float head_sum(const float (&x)[32], const uint64_t (&w2)[16]) {
    uint64_t a = f2_pack(0.f, 0.f), b = a;
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        a = f2_fma(w2[j >> 1], f2_pack(fmaxf(x[j], 0.f), fmaxf(x[j + 1], 0.f)), a);
        b = f2_fma(w2[(j >> 1) + 1], f2_pack(fmaxf(x[j + 2], 0.f), fmaxf(x[j + 3], 0.f)), b);
    }
    float s0, s1, s2, s3;
    f2_unpack(a, s0, s1);
    f2_unpack(b, s2, s3);
    return (s0 + s1) + (s2 + s3);
}

// The same sum in two halves of 16 heads (h = 0: heads 0 .. 15, h = 1: heads
// 16 .. 31), carrying the chains (a = (s0, s1), b = (s2, s3)) from one half to
// the next: head_sum_final after both gives bit for bit head_sum's result.
__device__ __forceinline__ void head_sum_half(const uint32_t (&r)[16], const uint64_t (&w2)[16], int h, uint64_t& a,
                                              uint64_t& b) {
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
        const int jw = (16 * h + j) >> 1;
        a = f2_fma(w2[jw], f2_pack(fmaxf(__uint_as_float(r[j]), 0.f), fmaxf(__uint_as_float(r[j + 1]), 0.f)), a);
        b = f2_fma(w2[jw + 1], f2_pack(fmaxf(__uint_as_float(r[j + 2]), 0.f), fmaxf(__uint_as_float(r[j + 3]), 0.f)),
                   b);
    }
}
__device__ __forceinline__ float head_sum_final(uint64_t a, uint64_t b) {
    float s0, s1, s2, s3;
    f2_unpack(a, s0, s1);
    f2_unpack(b, s2, s3);
    return (s0 + s1) + (s2 + s3);
}

template <int NQ, bool GATHER, int STAGES, int UT, int FMT>
__global__ void __launch_bounds__(ScoreCfg<NQ, GATHER, STAGES, UT, FMT>::THREADS, 1) score_kernel(ScoreParams p) {
    using C = ScoreCfg<NQ, GATHER, STAGES, UT, FMT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem + C::OFF_STAGES;
    uint8_t* qslots = smem + C::OFF_QSLOTS;
    int32_t* ids_ring = reinterpret_cast<int32_t*>(smem + C::OFF_IDS);
    uint32_t* hist_s = reinterpret_cast<uint32_t*>(smem + C::OFF_HIST);  // [2][slot][4096]
    const bool fuse_hist = C::HIST_SLOTS > 0 && p.key_hist;
    const bool fuse_bhist = C::HIST_SLOTS > 0 && p.bmax_hist && p.bmax;
    if (fuse_hist || fuse_bhist)
        for (int i = threadIdx.x; i < C::HIST_BYTES / 4; i += blockDim.x) hist_s[i] = 0u;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
    uint64_t* full = bars;
    uint64_t* sfready = full + STAGES;
    uint64_t* empty = sfready + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint64_t* acc_empty = acc_full + C::NACC;
    uint64_t* q_full = acc_empty + C::NACC * UT;
    uint64_t* q_ready = q_full + 2;
    uint64_t* q_empty = q_ready + 2;
    uint64_t* ids_full = q_empty + 2;
    uint64_t* ids_free = ids_full + (GATHER ? IDS_AHEAD : 0);
    uint64_t* drain = ids_free + (GATHER ? IDS_AHEAD : 0);
    ScoreShared* sh = reinterpret_cast<ScoreShared*>(bars + C::NBARS);
    __shared__ long long part[65];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#ifdef HSI_TRACE
    if (threadIdx.x == 0 && blockIdx.x < 1024) g_hsi_marks[blockIdx.x][0] = globaltimer_ns();
#endif

    if (warp == 0) {
        for (int s = lane; s < STAGES; s += 32) {
            mbar_init(&full[s], GATHER ? C::PROD_WARPS : 1);
            mbar_init(&sfready[s], 4);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NACC; ++i) mbar_init(&acc_full[i], 1);
        for (int i = 0; i < C::NACC * UT; ++i) mbar_init(&acc_empty[i], C::ACC_READERS);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_ready[i], 4);
            mbar_init(&q_empty[i], C::MMA_ISSUERS);
        }
        if (GATHER)
            for (int i = 0; i < IDS_AHEAD; ++i) {
                mbar_init(&ids_full[i], 1);
                mbar_init(&ids_free[i], C::PROD_WARPS);
            }
        mbar_init(drain, C::MMA_ISSUERS);
        sh->abort = 0;
        fence_mbar_init();
    }
    // everything above touches only this CTA's shared memory; inputs come next
    griddep_wait();
    griddep_launch_dependents();
    if (warp == C::MMA_WARP) tmem_alloc(&sh->tmem_base, C::TMEM_COLS);
    schedule_range(p.ngroups, [&](int g) { return group_units<NQ, GATHER, UT>(p, g); }, sh, part);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    const long long count = sh->count;
    WaitTrace tr;
#ifdef HSI_TRACE
    const long long t_start = clock64();
    if (threadIdx.x == 0 && blockIdx.x < 1024) g_hsi_marks[blockIdx.x][1] = globaltimer_ns();
#endif

    if (warp < C::PROD_WARPS) {
        // ------------------------------------------------------------ producer
        // warp 0 lane 0 also loads each group's q records and (gather) the
        // block ids, IDS_AHEAD units ahead.
        UnitIter<NQ, GATHER, UT> it;
        it.init(p, sh);
        UnitIter<NQ, GATHER, UT> ahead;  // gather: the unit whose block ids are fetched next
        ahead.init(p, sh);
        long long fetched = 0;  // kept identical in every lane of warp 0
        const bool leader = threadIdx.x == 0;
        auto fetch_ids = [&]() {  // warp 0: lane 0 bulk-copies the block ids of unit `fetched`
            const int slot = (int)(fetched % IDS_AHEAD);
            if (lane == 0) {
                mbar_arrive_expect_tx(&ids_full[slot], C::UNIT_RECS * 4);
                bulk_g2s(ids_ring + slot * C::UNIT_RECS,
                         p.block_ids + (int64_t)ahead.g * p.n_keep + (int64_t)ahead.t * C::UNIT_RECS,
                         C::UNIT_RECS * 4, &ids_full[slot]);
            }
            ahead.next(p);
            ++fetched;
        };
        if (GATHER && warp == 0)
            while (fetched < count && fetched < IDS_AHEAD - 1) fetch_ids();
        int cur_g = -1, gc = -1;
        int64_t k_base = 0;    // first record of the group's cache
        int64_t nrec_all = 0;  // records holding visible keys
        int nk = 0;            // gather: kept blocks
        long long issued_units = 0;
        int last_q_gc[2] = {-1, -1};
        Ring st;
        for (long long u = 0; u < count; ++u) {
            const int g = it.g, t = it.t;
            if (g != cur_g) {
                cur_g = g;
                ++gc;
                const int b0 = g * NQ;
                k_base = p.k_off ? p.k_off[b0] : (int64_t)b0 * p.k_stride;
                int maxv = 0;
#pragma unroll
                for (int i = 0; i < NQ; ++i) maxv = max(maxv, vis_of(p, b0 + i));
                nrec_all = (maxv + 7) / 8;
                if (GATHER) nk = min(p.n_kept[b0], p.n_keep);
                const int slot = gc & 1;
                if (warp == 0) {
                    if (!wait_traced(&q_empty[slot], ((gc >> 1) & 1) ^ 1, sh, tr, TR_PROD_QEMPTY)) break;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&q_full[slot], C::Q_BYTES);
                        bulk_g2s(qslots + slot * C::QSLOT_BYTES, p.q_rec + (int64_t)g * NQ * 4 * C::REC, C::Q_BYTES,
                                 &q_full[slot]);
                    }
                    last_q_gc[slot] = gc;
                }
            }
            if (GATHER) {
                const int islot = (int)(u % IDS_AHEAD);
                if (!wait_traced(&ids_full[islot], (uint32_t)((u / IDS_AHEAD) & 1), sh, tr, TR_PROD_IDS)) break;
            }
            if (!wait_traced(&empty[st.i], st.ph ^ 1u, sh, tr, TR_PROD_EMPTY)) break;
            HSI_TSTART(t_prod);
            uint8_t* dst = stages + st.i * C::STAGE_BYTES;
            if (!GATHER) {
                const int nrec = (int)min((int64_t)C::UNIT_RECS, nrec_all - (int64_t)t * C::UNIT_RECS);
                const bool skip = u == 0 && *(volatile int*)&g_hsi_skip_first_copy;  // diagnostics only
                if (lane == 0 && !skip) {
                    mbar_arrive_expect_tx(&full[st.i], (uint32_t)(nrec * C::REC));
                    bulk_g2s(dst, p.k_rec + (k_base + (int64_t)t * C::UNIT_RECS) * C::REC, (uint32_t)(nrec * C::REC),
                             &full[st.i]);
                }
            } else {
                // TPR threads per pooled block, 36 chunks of 16 bytes per NVFP4 record
                // (34 per MXFP4 one) shared among them
                const int islot = (int)(u % IDS_AHEAD);
                const int blk = threadIdx.x / C::TPR, prt = threadIdx.x % C::TPR;
                const int j = t * C::UNIT_RECS + blk;
                const int64_t id = ids_ring[islot * C::UNIT_RECS + blk];
                __syncwarp();
                if (lane == 0) mbar_arrive(&ids_free[islot]);
                const bool ok = j < nk && id >= 0 && id < nrec_all;
                if (j < nk && !ok && prt == 0) raise_error(DEVERR_ARG);
                if (ok) {
                    const uint8_t* src = p.k_rec + (k_base + id) * C::REC;
                    uint8_t* d = dst + blk * C::REC;
                    constexpr int CH = C::REC / 16;
#pragma unroll
                    for (int c = 0; c < (CH + C::TPR - 1) / C::TPR; ++c)
                        if (c * C::TPR + prt < CH)
                            cp_async16(d + (c * C::TPR + prt) * 16, src + (c * C::TPR + prt) * 16);
                }
                cp_async_commit();
                // refill the id slot of the previous unit once every producer warp has read it
                if (warp == 0 && fetched < count) {
                    if (u >= 1) {
                        const int prev = (int)((u - 1) % IDS_AHEAD);
                        if (!wait_traced(&ids_free[prev], (uint32_t)(((u - 1) / IDS_AHEAD) & 1), sh, tr,
                                         TR_PROD_IDS))
                            break;
                        fence_proxy_async_smem();  // the slot's reads precede the copy that refills it
                    }
                    fetch_ids();
                }
                // the unit COPY_AHEAD back has landed: publish it
                if (u >= C::COPY_AHEAD) {
                    HSI_TSTART(t_land);
                    cp_async_wait<C::COPY_AHEAD>();
                    HSI_TEND(t_land, TR_PROD_LAND);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full[(st.i + STAGES - C::COPY_AHEAD) % STAGES]);
                }
            }
            issued_units = u + 1;
            HSI_TEND(t_prod, TR_PROD_ISSUE);
            st.next(STAGES);
            it.next(p);
        }
        if (GATHER) {
            // publish the units still in flight, then nothing is left pending
            cp_async_wait<0>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                for (long long v = issued_units > C::COPY_AHEAD ? issued_units - C::COPY_AHEAD : 0; v < issued_units;
                     ++v)
                    mbar_arrive(&full[(int)(v % STAGES)]);
        }
        // drain: every bulk copy issued must have landed before the CTA exits
        if (leader) {
            if (!GATHER)
                for (long long v = issued_units > STAGES ? issued_units - STAGES : 0; v < issued_units; ++v)
                    wait_drain(&full[(int)(v % STAGES)], (uint32_t)((v / STAGES) & 1));
            for (int slot = 0; slot < 2; ++slot)
                if (last_q_gc[slot] >= 0) wait_drain(&q_full[slot], (uint32_t)((last_q_gc[slot] >> 1) & 1));
            if (GATHER)
                for (long long v = fetched > IDS_AHEAD ? fetched - IDS_AHEAD : 0; v < fetched; ++v)
                    wait_drain(&ids_full[(int)(v % IDS_AHEAD)], (uint32_t)((v / IDS_AHEAD) & 1));
        }
    } else if (warp < C::MMA_WARP + C::MMA_ISSUERS) {
        // ----------------------------------------------------------------- MMA
        // lane 0 of each MMA warp issues the MMAs and commits of every
        // MMA_ISSUERS-th unit; the rest of the warp waits at the end
        const int issuer = warp - C::MMA_WARP;
        if (lane == 0) {
            UnitIter<NQ, GATHER, UT> it;
            it.init(p, sh);
            int cur_g = -1, gc = -1;
            constexpr uint32_t idesc = FMT == FMT_MXFP4 ? idesc_mxf4(128, C::N) : idesc_nvf4(128, C::N);
            Ring st, ac;
            for (long long u = 0; u < count; ++u) {
                if (it.g != cur_g) {
                    // the old q slot is free once this thread's MMAs on it finish (every
                    // issuer commits, whether it issued on the slot or not)
                    if (cur_g >= 0) tc_commit(&q_empty[gc & 1]);
                    cur_g = it.g;
                    ++gc;
                    if (!wait_one(&q_ready[gc & 1], (gc >> 1) & 1, sh, tr, TR_MMA_QREADY)) break;
                }
                if (C::MMA_ISSUERS > 1 && (int)(u % C::MMA_ISSUERS) != issuer) {  // another issuer's unit
                    st.next(STAGES);
                    ac.next(C::NACC);
                    it.next(p);
                    continue;
                }
                if (!wait_one(&sfready[st.i], st.ph, sh, tr, TR_MMA_SFREADY)) break;
                HSI_TSTART(t_issue);
                bool stop = false;
                const uint32_t a0 = smem_u32(stages + st.i * C::STAGE_BYTES);
                const uint32_t b0 = smem_u32(qslots + (gc & 1) * C::QSLOT_BYTES);
                const uint32_t sfb = tmem + C::COL_SFB + (gc & 1) * 8;
#pragma unroll
                for (int sub = 0; sub < UT; ++sub) {
                    // the epilogue has read this tile of the set's previous unit
                    if (!wait_one(&acc_empty[ac.i * UT + sub], ac.ph ^ 1u, sh, tr, TR_MMA_ACCEMPTY)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + C::COL_ACC + (ac.i * UT + sub) * C::N;
                    const uint32_t sfa = tmem + C::COL_SFA + (st.i * UT + sub) * 8;
                    const uint32_t at = a0 + sub * 16 * C::REC;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint64_t ad = smem_desc(at + kk * 256, 128, C::REC);
                        const uint64_t bd = smem_desc(b0 + kk * 256, 128, C::REC);
                        if constexpr (FMT == FMT_MXFP4) mma_mxf4(d, ad, bd, idesc, sfa + kk * 4, sfb + kk * 4, kk);
                        else mma_nvf4(d, ad, bd, idesc, sfa + kk * 4, sfb + kk * 4, kk);
                    }
                }
                if (stop) break;
                // one commit: the epilogue that sees it also frees the stage
                tc_commit(&acc_full[ac.i]);
                HSI_TEND(t_issue, TR_MMA_ISSUE);
                st.next(STAGES);
                ac.next(C::NACC);
                it.next(p);
            }
            // drain: every MMA into TMEM done before the allocation is freed
            tc_commit(drain);
            wait_drain(drain, 0);
        }
        __syncwarp();
    } else if (warp < C::FIRST_EPI_WARP) {
        // ---------------------------------------------------- scale warpgroup
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        UnitIter<NQ, GATHER, UT> it;
        it.init(p, sh);
        int cur_g = -1, gc = -1;
        Ring st;
        for (long long u = 0; u < count; ++u) {
            if (it.g != cur_g) {
                cur_g = it.g;
                ++gc;
                const int slot = gc & 1;
                if (!wait_traced(&q_full[slot], (gc >> 1) & 1, sh, tr, TR_SF_QFULL)) break;
                uint32_t v[8];
                sf_quarter<FMT>(qslots + slot * C::QSLOT_BYTES, C::N, lane, v);
                tmem_st8_wait(tmem + lane_base + C::COL_SFB + slot * 8, v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_ready[slot]);
            }
            if (!wait_traced(&full[st.i], st.ph, sh, tr, TR_SF_FULL)) break;
            const uint8_t* st_recs = stages + st.i * C::STAGE_BYTES;
            HSI_TSTART(t_sf);
            if (GATHER && p.pool_out && warp == C::FIRST_SF_WARP && lane == 0) {
                // the landed unit also goes to the compacted pool; its shared source
                // is read before this warp releases the stage's scales (so before
                // the stage can be refilled)
                const int nk = min(p.n_kept[it.g], p.n_keep);
                const int nrec = min(C::UNIT_RECS, nk - it.t * C::UNIT_RECS);
                if (nrec > 0) {
                    bulk_s2g(p.pool_out + ((int64_t)it.g * p.n_keep + (int64_t)it.t * C::UNIT_RECS) * C::REC, st_recs,
                             (uint32_t)(nrec * C::REC));
                    bulk_commit();
                    bulk_wait_read_all();
                }
            }
#pragma unroll
            for (int sub = 0; sub < UT; ++sub) {
                uint32_t v[8];
                sf_quarter<FMT>(st_recs + sub * 16 * C::REC, TILE_KEYS, lane, v);
                tmem_st8_wait(tmem + lane_base + C::COL_SFA + (st.i * UT + sub) * 8, v);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sfready[st.i]);
            HSI_TEND(t_sf, TR_SF_WORK);
            st.next(STAGES);
            it.next(p);
        }
        if (GATHER && p.pool_out && warp == C::FIRST_SF_WARP && lane == 0) bulk_wait_all();
    } else {
        // ------------------------------------------------------------ epilogue
        const int grp = (warp - C::FIRST_EPI_WARP) >> 2;
        const int quarter = warp & 3;
        const bool group_leader = (warp - C::FIRST_EPI_WARP) % 4 == 0 && lane == 0;
        const int row = quarter * 32 + lane;  // key within a 128-key tile
        UnitIter<NQ, GATHER, UT> it;
        it.init(p, sh);
        const int b_first = sh->g0 * NQ;
        // histogram bins of query b: shared-memory slot, or global past the slots
        auto hist_of = [&](int b) -> uint32_t* {
            const int slot = b - b_first;
            if (slot >= 0 && slot < C::HIST_SLOTS) return hist_s + slot * 4096;
            return p.key_hist + (int64_t)b * 4096;
        };
        auto bhist_of = [&](int b) -> uint32_t* {
            const int slot = b - b_first;
            if (slot >= 0 && slot < C::HIST_SLOTS) return hist_s + (C::HIST_SLOTS + slot) * 4096;
            return p.bmax_hist + (int64_t)b * 4096;
        };
        // the scaled head weights of this warp's query, in f32x2 pairs
        uint64_t w2[16];
        auto load_w = [&](int b) {
            // the 2^-7 of the two unnormalised rotations; NVFP4 also its tensor scales
            const float sc = (FMT == FMT_MXFP4 ? 1.0f : p.g_q[b] * p.g_k[b]) * 0.0078125f;
            const float4* wv = reinterpret_cast<const float4*>(p.w + (int64_t)b * 32);
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
                const float4 v = __ldg(wv + j4);
                w2[2 * j4] = f2_pack(v.x * sc, v.y * sc);
                w2[2 * j4 + 1] = f2_pack(v.z * sc, v.w * sc);
            }
        };
        // one key's score: written, its 8-key block maximum, its histogram bin
        auto emit = [&](int b, int key, int nv, int npad, float sc) {
            const bool vis = key < nv;
            if (p.scores) {  // (block maxima only without a score row)
                if (vis) p.scores[(int64_t)b * p.ld + key] = sc;
                else if (key < npad) p.scores[(int64_t)b * p.ld + key] = __uint_as_float(0xFF800000u);
            }
            if (fuse_hist && vis) atomicAdd(hist_of(b) + (order_key(sc) >> 20), 1u);
            if (p.bmax) {
                float m = vis ? sc : __uint_as_float(0xFF800000u);
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
                if ((lane & 7) == 0 && vis) {
                    p.bmax[(int64_t)b * p.ldb + key / 8] = m;
                    if (fuse_bhist) atomicAdd(bhist_of(b) + (order_key(m) >> 20), 1u);
                }
            }
        };
        int cur_g = -1;
        Ring st, ac;
        if constexpr (NQ > 1) {
            // one group per query: every group takes every unit, reads its query's
            // 32 columns of each tile and frees the tile once all groups hold it,
            // so a tile stays allocated for one TMEM load, not a whole epilogue
            int nv = 0, npad = 0, b = 0;
            for (long long u = 0; u < count; ++u) {
                const int g = it.g, t = it.t;
                if (g != cur_g) {
                    cur_g = g;
                    b = g * NQ + grp;
                    nv = vis_of(p, b, lane == 0);
                    npad = p.pad_blocks ? 8 * min(p.pad_blocks[b], p.n_keep) : 0;
                    load_w(b);
                }
                if (!wait_traced(&acc_full[ac.i], ac.ph, sh, tr, TR_EPI_ACCFULL)) break;
                HSI_TSTART(t_epi);
                tc_fence_after();
                if (grp == 0 && group_leader) mbar_arrive(&empty[st.i]);  // the MMAs have read the stage
#pragma unroll
                for (int sub = 0; sub < UT; ++sub) {
                    float x[32];
                    tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + C::COL_ACC + (ac.i * UT + sub) * C::N + grp * 32,
                              x);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_empty[ac.i * UT + sub]);
                    emit(b, (t * UT + sub) * TILE_KEYS + row, nv, npad, head_sum(x, w2));
                }
                HSI_TEND(t_epi, TR_EPI_WORK);
                st.next(STAGES);
                ac.next(C::NACC);
                it.next(p);
            }
        } else {
        int nv = 0, npad = 0;
        int nk = 0;
        int turn = 0;
        for (long long u = 0; u < count; ++u) {
            if (turn != grp) {
                if (++turn == C::EPI_GROUPS) turn = 0;
                st.next(STAGES);
                ac.next(C::NACC);
                it.next(p);
                continue;
            }
            if (++turn == C::EPI_GROUPS) turn = 0;
            const int g = it.g, t = it.t;
            if (g != cur_g) {
                cur_g = g;
                nv = vis_of(p, g, lane == 0);
                npad = p.pad_blocks ? 8 * min(p.pad_blocks[g], p.n_keep) : 0;
                load_w(g);
                if (GATHER) nk = min(p.n_kept[g], p.n_keep);
            }
            // gather: the positions of this thread's slots, loaded before the wait
            int64_t pos[UT];
#pragma unroll
            for (int sub = 0; sub < UT; ++sub) {
                pos[sub] = -1;
                const int slot_i = (t * UT + sub) * TILE_KEYS + row;
                if (GATHER && (slot_i >> 3) < nk)
                    pos[sub] = (int64_t)__ldg(p.block_ids + (int64_t)g * p.n_keep + (slot_i >> 3)) * 8 + (slot_i & 7);
            }
            if (!wait_traced(&acc_full[ac.i], ac.ph, sh, tr, TR_EPI_ACCFULL)) break;
            HSI_TSTART(t_epi);
            tc_fence_after();
            if (group_leader) mbar_arrive(&empty[st.i]);  // the MMAs have read the stage
#pragma unroll
            for (int sub = 0; sub < UT; ++sub) {
                const int key = (t * UT + sub) * TILE_KEYS + row;  // key (full scan) or pool slot (gather)
                float x[32];
                tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + C::COL_ACC + (ac.i * UT + sub) * C::N, x);
                // the tile is in registers: the MMA may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[ac.i * UT + sub]);
                const float sc = head_sum(x, w2);
                if (!GATHER) {
                    emit(g, key, nv, npad, sc);
                } else if (pos[sub] >= 0) {
                    const bool vis = pos[sub] < nv;
                    p.pool_scores[(int64_t)g * p.ld_pool + key] = vis ? sc : __uint_as_float(0xFF800000u);
                    if (fuse_hist && vis) {  // the pool slot's key, for the selection inside the pool
                        const uint32_t bin = order_key(sc) >> 20;
                        const int slot = g - b_first;
                        if (slot >= 0 && slot < C::HIST_SLOTS) atomicAdd(hist_s + slot * 4096 + bin, 1u);
                        else atomicAdd(p.key_hist + (int64_t)g * 4096 + bin, 1u);
                    }
                }
            }
            HSI_TEND(t_epi, TR_EPI_WORK);
            st.next(STAGES);
            ac.next(C::NACC);
            it.next(p);
        }
        }
    }
#ifdef HSI_TRACE
    if (lane == 0 && (warp == 0 || warp == C::MMA_WARP || warp == C::FIRST_SF_WARP || warp == C::FIRST_EPI_WARP)) {
        const int slot = warp == 0 ? TR_PROD_TOTAL
                         : warp == C::MMA_WARP ? TR_MMA_TOTAL
                         : warp == C::FIRST_SF_WARP ? TR_SF_TOTAL
                                                    : TR_EPI_TOTAL;
        tr.add(slot, (unsigned long long)(clock64() - t_start));
        if (warp == 0) tr.add(TR_UNITS, (unsigned long long)count);
        tr.flush();
        if (warp == 0 && blockIdx.x < 1024) g_hsi_marks[blockIdx.x][2] = globaltimer_ns();
    }
#endif
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::MMA_WARP) tmem_dealloc(tmem, C::TMEM_COLS);
    if constexpr (C::HIST_SLOTS > 0)
    if (fuse_hist || fuse_bhist) {  // merge the shared-memory slots into the global histograms
        const int b_first = sh->g0 * NQ;
        for (int i = threadIdx.x; i < 2 * C::HIST_SLOTS * 4096; i += blockDim.x) {
            const uint32_t v = hist_s[i];
            const bool bm = i >= C::HIST_SLOTS * 4096;
            const int b = b_first + (i / 4096) % C::HIST_SLOTS;
            uint32_t* gh = bm ? p.bmax_hist : p.key_hist;
            if (v && b < p.B && gh) atomicAdd(gh + (int64_t)b * 4096 + (i & 4095), v);
        }
    }
#ifdef HSI_TRACE
    if (threadIdx.x == 0 && blockIdx.x < 1024) g_hsi_marks[blockIdx.x][3] = globaltimer_ns();
#endif
}

}  // namespace hsi
