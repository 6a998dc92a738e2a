// Chunked-prefill scoring with the key cache held in shared memory.
//
// In a chunked prefill every query of the layer scores the same cache: query
// t sees its first n_visible[t] keys. Streaming the cache past the queries
// (one 9 KB key tile per 4 queries, as the decode scan does) makes the copy
// engine and the per-tile bookkeeping the limit. Here each CTA instead keeps
// one contiguous chunk of the cache resident (up to PF_KT_MAX tiles of 128
// keys) and streams the queries past it, four at a time: per 128 keys x 4
// queries of work only 1 / (tiles in the chunk) of a 9.7 KB query slot is
// copied and its scales staged, and the MMAs, commits and epilogue are as in
// the 4-query tiles of the scoring kernel:
//
//   I = (g_q g_k / 128) * sum_j w_j * ReLU(q_j . k)
//
// per tile (128 keys x 4 queries x 32 heads) two tcgen05.mma kind::mxf4nvf4
// of M = 128, N = 128, K = 64 into one of three TMEM accumulator sets, the
// key scales of the resident chunk staged once in TMEM, each query group's
// scales per group.
//
// Warp roles (one CTA per SM, persistent over chunks):
//   producer     warp 0: the chunk's key tiles (bulk copies), then per query
//                group its four query records, head weights and tensor
//                scales into a ring of query slots;
//   MMA          two warps, one thread each, taking alternate tiles;
//   scale warps  a warpgroup writing the chunk's key scales and each slot's
//                query scales into TMEM (one 32-lane quarter per warp);
//   epilogue     4 / PF_QPW groups of four warps, each group scoring PF_QPW of
//                the four queries of every tile (its columns of a tile loaded
//                from TMEM one query at a time, the tile freed after the last);
//                ReLU and the head weights fused, scores and 8-key block
//                maxima written.
// Every wait is bounded; on a timeout the CTA records the error, drains what
// it has in flight, frees TMEM and returns.
#pragma once
#include <cstdint>

#include "score.cuh"

namespace hsi {

constexpr int PF_KT_MAX = 8;   // key tiles of 128 held per CTA
constexpr int PF_QSLOTS = 4;   // query-group slots in flight
constexpr int PF_NACC = 3;     // accumulator sets of 128 columns
constexpr int PF_ISSUERS = 2;  // MMA-issuing warps
constexpr int PF_MAX_GROUPS = 8192;  // query groups of 4 (the per-group length table lives in shared memory)
// queries of a group each epilogue warp scores (4 / PF_QPW groups of four
// warps): its per-tile bookkeeping is shared by PF_QPW queries
#ifndef HSI_PF_QPW
#define HSI_PF_QPW 1
#endif
constexpr int PF_QPW = HSI_PF_QPW;

struct PrefillParams {
    const uint8_t* q_rec;  // [B * 4] records
    const float* g_q;      // [B] (NVFP4), 16-byte aligned
    const float* w;        // [B][32], 16-byte aligned
    const uint8_t* k_rec;  // the cache's records start at k_rec + k_off[0] records
    const float* g_k;      // [B] (NVFP4), 16-byte aligned
    const int64_t* k_off;
    const int32_t* n_vis;  // [B]
    int32_t max_vis;
    int32_t B;        // multiple of 4
    int32_t ngroups;  // B / 4
    float* scores;    // [B][ld]
    int64_t ld;
    float* bmax;  // [B][ldb] or NULL
    int64_t ldb;
};

template <int FMT>
struct PfCfg {
    static constexpr int REC = rec_bytes<FMT>();
    static constexpr int TILE_BYTES = 16 * REC;
    static constexpr int Q_BYTES = 16 * REC;  // four queries x four records
    // a query slot: the records, then w [4][32], g_q [4], g_k [4]
    static constexpr int SLOT_W = Q_BYTES, SLOT_GQ = SLOT_W + 512, SLOT_GK = SLOT_GQ + 16;
    static constexpr int SLOT_BYTES = ((SLOT_GK + 16 + 127) / 128) * 128;
    static constexpr int SLOT_COPY = SLOT_GK + 16 - Q_BYTES;  // bytes of w, g_q, g_k
    static constexpr int N = 128;
    static constexpr int MMA_WARP = 1;
    static constexpr int FIRST_SF_WARP = MMA_WARP + PF_ISSUERS;
    static constexpr int FIRST_EPI_WARP = FIRST_SF_WARP + 4;
    static constexpr int EPI_WARPS = 4 * (4 / PF_QPW);
    static constexpr int THREADS = 32 * (FIRST_EPI_WARP + EPI_WARPS);
    static constexpr int COL_ACC = 0;
    static constexpr int COL_SFA = PF_NACC * N;
    static constexpr int COL_SFB = COL_SFA + PF_KT_MAX * 8;
    static constexpr int TMEM_COLS = 512;
    static_assert(COL_SFB + PF_QSLOTS * 8 <= TMEM_COLS, "TMEM");
    static constexpr int OFF_K = 0;
    static constexpr int OFF_Q = PF_KT_MAX * TILE_BYTES;
    static constexpr int OFF_GMAX = OFF_Q + PF_QSLOTS * SLOT_BYTES;  // then ngroups int32, then the barriers
    // kfull, kready, kempty; qfull, qready, qempty per slot; acc_full, acc_empty per set; drain
    static constexpr int NBARS = 3 + 3 * PF_QSLOTS + 2 * PF_NACC + 1;
    static constexpr size_t smem_bytes(int ngroups) {
        return (size_t)OFF_GMAX + (((size_t)ngroups * 4 + 15) / 16) * 16 + NBARS * 8 + sizeof(ScoreShared) + 1024 +
               64;
    }
};

// The units of one CTA: its chunks of the cache (tile ranges), and in each
// chunk the query groups that see any of it, each group taking the chunk's
// tiles that hold a key it sees. Every role walks the same sequence.
struct PfWalk {
    int t_lo, t_hi;  // the chunk's tiles
    int g;           // query group
    int nt;          // tiles of the chunk this group needs
    int nchunks, ntiles;
    const int32_t* gmax;  // per group: the largest n_visible of its queries
    int ngroups;
    __device__ bool set_chunk(int c) {
        const int64_t id = (int64_t)c * gridDim.x + blockIdx.x;
        if (id >= nchunks) return false;
        t_lo = (int)((int64_t)ntiles * id / nchunks);
        t_hi = (int)((int64_t)ntiles * (id + 1) / nchunks);
        g = -1;
        return true;
    }
    // tiles of this chunk group g needs
    __device__ int tiles_for(int gg) const {
        const int need = (gmax[gg] + TILE_KEYS - 1) / TILE_KEYS - t_lo;
        return max(0, min(need, t_hi - t_lo));
    }
    // advance to the next group of this chunk that needs a tile; false at the chunk's end
    __device__ bool next_group() {
        while (++g < ngroups) {
            nt = tiles_for(g);
            if (nt > 0) return true;
        }
        return false;
    }
};

template <int FMT>
__global__ void __launch_bounds__(PfCfg<FMT>::THREADS, 1) prefill_kernel(PrefillParams p, int ntiles, int nchunks) {
    using C = PfCfg<FMT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ktiles = smem + C::OFF_K;
    uint8_t* qslots = smem + C::OFF_Q;
    int32_t* gmax = reinterpret_cast<int32_t*>(smem + C::OFF_GMAX);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_GMAX + ((p.ngroups * 4 + 15) / 16) * 16);
    uint64_t* kfull = bars;
    uint64_t* kready = kfull + 1;
    uint64_t* kempty = kready + 1;
    uint64_t* qfull = kempty + 1;
    uint64_t* qready = qfull + PF_QSLOTS;
    uint64_t* qempty = qready + PF_QSLOTS;
    uint64_t* acc_full = qempty + PF_QSLOTS;
    uint64_t* acc_empty = acc_full + PF_NACC;
    uint64_t* drain = acc_empty + PF_NACC;
    ScoreShared* sh = reinterpret_cast<ScoreShared*>(drain + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // stale shared memory under a partial last tile is multiplied but never
    // written out; zero it once so that it holds no NaN scale
    for (int i = threadIdx.x; i < C::OFF_Q / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(ktiles)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        mbar_init(kfull, 1);
        mbar_init(kready, 4);
        mbar_init(kempty, PF_ISSUERS);
        for (int i = 0; i < PF_QSLOTS; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qready[i], 4);
            mbar_init(&qempty[i], PF_ISSUERS + C::EPI_WARPS);
        }
        for (int i = 0; i < PF_NACC; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], C::EPI_WARPS);
        }
        mbar_init(drain, PF_ISSUERS);
        sh->abort = 0;
        fence_mbar_init();
    }
    griddep_wait();
    griddep_launch_dependents();
    // the largest visible length of each query group, and of all of them
    int mall = 0;
    for (int g = threadIdx.x; g < p.ngroups; g += blockDim.x) {
        int m = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int n = p.n_vis[4 * g + i];
            if (n > p.max_vis) {
                raise_error(DEVERR_ARG);
                n = p.max_vis;
            }
            m = max(m, n);
        }
        gmax[g] = m;
        mall = max(mall, m);
    }
    if (threadIdx.x == 0) sh->count = 0;
    __syncthreads();
    mall = __reduce_max_sync(0xFFFFFFFFu, mall);
    if (lane == 0) atomicMax(reinterpret_cast<int*>(&sh->count), mall);
    fence_proxy_async_smem();  // the zeroed tiles before the bulk copies that refill them
    if (warp == C::MMA_WARP) tmem_alloc(&sh->tmem_base, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    const uint8_t* kbase = p.k_rec + (p.k_off ? p.k_off[0] : 0) * (int64_t)C::REC;
    // records holding a visible key: the copies read no further
    const int64_t cache_recs = (sh->count + 7) / 8;
    WaitTrace tr;
    PfWalk wk;
    wk.nchunks = nchunks;
    wk.ntiles = ntiles;
    wk.gmax = gmax;
    wk.ngroups = p.ngroups;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int qs = 0;  // query groups loaded (slot qs % PF_QSLOTS)
        int k_loaded = 0;
        int64_t last_q = -1;
        bool ok = true;
        for (int c = 0; ok && wk.set_chunk(c); ++c) {
            // the previous chunk's MMAs are done before its tiles are overwritten
            if (c > 0 && !(ok = wait_traced(kempty, (uint32_t)((c - 1) & 1), sh, tr, TR_PROD_EMPTY))) break;
            if (lane == 0) {
                const int64_t r0 = (int64_t)wk.t_lo * 16;
                const int64_t nrec = max((int64_t)0, min((int64_t)(wk.t_hi - wk.t_lo) * 16, cache_recs - r0));
                mbar_arrive_expect_tx(kfull, (uint32_t)(nrec * C::REC));
                for (int64_t r = 0; r < nrec; r += 16) {
                    const int64_t n = min((int64_t)16, nrec - r);
                    bulk_g2s(ktiles + r * C::REC, kbase + (r0 + r) * C::REC, (uint32_t)(n * C::REC), kfull);
                }
            }
            ++k_loaded;
            while (wk.next_group()) {
                const int slot = qs % PF_QSLOTS;
                if (!(ok = wait_traced(&qempty[slot], ((qs / PF_QSLOTS) & 1) ^ 1, sh, tr, TR_PROD_QEMPTY))) break;
                if (lane == 0) {
                    uint8_t* d = qslots + slot * C::SLOT_BYTES;
                    const int b0 = 4 * wk.g;
                    mbar_arrive_expect_tx(&qfull[slot], (uint32_t)(C::Q_BYTES + 512 + (FMT == FMT_NVFP4 ? 32 : 0)));
                    bulk_g2s(d, p.q_rec + (int64_t)b0 * 4 * C::REC, C::Q_BYTES, &qfull[slot]);
                    bulk_g2s(d + C::SLOT_W, p.w + (int64_t)b0 * 32, 512, &qfull[slot]);
                    if (FMT == FMT_NVFP4) {
                        bulk_g2s(d + C::SLOT_GQ, p.g_q + b0, 16, &qfull[slot]);
                        bulk_g2s(d + C::SLOT_GK, p.g_k + b0, 16, &qfull[slot]);
                    }
                }
                last_q = qs;
                ++qs;
            }
        }
        // drain: every copy issued has landed before the CTA exits
        if (lane == 0) {
            if (k_loaded > 0) wait_drain(kfull, (uint32_t)((k_loaded - 1) & 1));
            for (int64_t v = last_q - PF_QSLOTS + 1 > 0 ? last_q - PF_QSLOTS + 1 : 0; v <= last_q; ++v)
                wait_drain(&qfull[v % PF_QSLOTS], (uint32_t)((v / PF_QSLOTS) & 1));
        }
    } else if (warp < C::FIRST_SF_WARP) {
        // ----------------------------------------------------------------- MMA
        const int issuer = warp - C::MMA_WARP;
        if (lane == 0) {
            constexpr uint32_t idesc = FMT == FMT_MXFP4 ? idesc_mxf4(128, C::N) : idesc_nvf4(128, C::N);
            int qs = 0;
            int u = 0;  // units (tiles) of this CTA, in order
            bool ok = true;
            for (int c = 0; ok && wk.set_chunk(c); ++c) {
                if (!(ok = wait_one(kready, (uint32_t)(c & 1), sh, tr, TR_MMA_SFREADY))) break;
                while (ok && wk.next_group()) {
                    const int slot = qs % PF_QSLOTS;
                    if (!(ok = wait_one(&qready[slot], (uint32_t)((qs / PF_QSLOTS) & 1), sh, tr, TR_MMA_QREADY))) break;
                    const uint32_t b0 = smem_u32(qslots + slot * C::SLOT_BYTES);
                    const uint32_t sfb = tmem + C::COL_SFB + slot * 8;
                    for (int kt = 0; kt < wk.nt; ++kt, ++u) {
                        if ((int)(u % PF_ISSUERS) != issuer) continue;
                        const int ai = (int)(u % PF_NACC);
                        if (!(ok = wait_one(&acc_empty[ai], (uint32_t)(((u / PF_NACC) & 1) ^ 1), sh, tr,
                                            TR_MMA_ACCEMPTY)))
                            break;
                        tc_fence_after();
                        HSI_TSTART(t_issue);
                        const uint32_t d = tmem + C::COL_ACC + ai * C::N;
                        const uint32_t sfa = tmem + C::COL_SFA + kt * 8;
                        const uint32_t a0 = smem_u32(ktiles + kt * C::TILE_BYTES);
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint64_t ad = smem_desc(a0 + kk * 256, 128, C::REC);
                            const uint64_t bd = smem_desc(b0 + kk * 256, 128, C::REC);
                            if constexpr (FMT == FMT_MXFP4) mma_mxf4(d, ad, bd, idesc, sfa + kk * 4, sfb + kk * 4, kk);
                            else mma_nvf4(d, ad, bd, idesc, sfa + kk * 4, sfb + kk * 4, kk);
                        }
                        tc_commit(&acc_full[ai]);
                        HSI_TEND(t_issue, TR_MMA_ISSUE);
                    }
                    // the slot is free once this thread's MMAs on it finish
                    tc_commit(&qempty[slot]);
                    ++qs;
                }
                if (!ok) break;
                tc_commit(kempty);  // the chunk's tiles are free once this thread's MMAs finish
            }
            tc_commit(drain);
            wait_drain(drain, 0);
        }
        __syncwarp();
    } else if (warp < C::FIRST_EPI_WARP) {
        // ---------------------------------------------------- scale warpgroup
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        int qs = 0;
        bool ok = true;
        for (int c = 0; ok && wk.set_chunk(c); ++c) {
            if (!(ok = wait_traced(kfull, (uint32_t)(c & 1), sh, tr, TR_SF_FULL))) break;
            const int64_t cache_rows = (cache_recs - (int64_t)wk.t_lo * 16) * 8;  // rows of the chunk inside the cache
            for (int kt = 0; kt < wk.t_hi - wk.t_lo; ++kt) {
                uint32_t v[8];
                sf_quarter<FMT>(ktiles + kt * C::TILE_BYTES, (int)min((int64_t)TILE_KEYS, cache_rows - kt * TILE_KEYS),
                                lane, v);
                tmem_st8_wait(tmem + lane_base + C::COL_SFA + kt * 8, v);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(kready);
            while (wk.next_group()) {
                const int slot = qs % PF_QSLOTS;
                if (!(ok = wait_traced(&qfull[slot], (uint32_t)((qs / PF_QSLOTS) & 1), sh, tr, TR_SF_QFULL))) break;
                uint32_t v[8];
                sf_quarter<FMT>(qslots + slot * C::SLOT_BYTES, C::N, lane, v);
                tmem_st8_wait(tmem + lane_base + C::COL_SFB + slot * 8, v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&qready[slot]);
                ++qs;
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Software-pipelined over tiles: the previous tile's score, block
        // maximum (three dependent shuffles) and stores are issued while this
        // tile's TMEM load is in flight, since with four epilogue warps per
        // scheduler the latency of a tile's dependent chain is not hidden by
        // the other warps alone.
        const int grp = (warp - C::FIRST_EPI_WARP) >> 2;  // this warp scores queries PF_QPW grp .. + PF_QPW - 1
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + C::COL_ACC + grp * PF_QPW * 32;
        uint64_t w2[PF_QPW][16];
        int qs = 0;
        int u = 0;
        bool ok = true;
        // the previous tile's scores (of this group's queries), emitted one tile late
        float pend_s[PF_QPW];
        int pend_key = -1;
        int nv[PF_QPW];
        float* srow[PF_QPW];
        float* brow[PF_QPW];
        auto emit_pending = [&]() {
            if (pend_key < 0) return;
#pragma unroll
            for (int qi = 0; qi < PF_QPW; ++qi) {
                const bool vis = pend_key < nv[qi];
                if (vis) srow[qi][pend_key] = pend_s[qi];
                if (brow[qi]) {
                    float m = vis ? pend_s[qi] : __uint_as_float(0xFF800000u);
                    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
                    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
                    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
                    if ((lane & 7) == 0 && vis) brow[qi][pend_key / 8] = m;
                }
            }
            pend_key = -1;
        };
        for (int c = 0; ok && wk.set_chunk(c); ++c) {
            while (ok && wk.next_group()) {
                const int slot = qs % PF_QSLOTS;
                if (!(ok = wait_traced(&qfull[slot], (uint32_t)((qs / PF_QSLOTS) & 1), sh, tr, TR_EPI_ACCFULL))) break;
                const uint8_t* sl = qslots + slot * C::SLOT_BYTES;
#pragma unroll
                for (int qi = 0; qi < PF_QPW; ++qi) {
                    const int qg = grp * PF_QPW + qi;  // query within the group
                    const int b = 4 * wk.g + qg;
                    // the 2^-7 of the two unnormalised rotations; NVFP4 also its tensor scales
                    const float sc = (FMT == FMT_MXFP4 ? 1.0f
                                                       : reinterpret_cast<const float*>(sl + C::SLOT_GQ)[qg] *
                                                             reinterpret_cast<const float*>(sl + C::SLOT_GK)[qg]) *
                                     0.0078125f;
                    const float4* wv = reinterpret_cast<const float4*>(sl + C::SLOT_W) + qg * 8;
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 v = wv[j4];
                        w2[qi][2 * j4] = f2_pack(v.x * sc, v.y * sc);
                        w2[qi][2 * j4 + 1] = f2_pack(v.z * sc, v.w * sc);
                    }
                    const int n = p.n_vis[b];
                    nv[qi] = n > p.max_vis ? p.max_vis : n;
                    srow[qi] = p.scores + (int64_t)b * p.ld;
                    brow[qi] = p.bmax ? p.bmax + (int64_t)b * p.ldb : nullptr;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&qempty[slot]);  // this warp is done with the slot's weights
                for (int kt = 0; kt < wk.nt; ++kt, ++u) {
                    const int ai = (int)(u % PF_NACC);
                    if (!(ok = wait_traced(&acc_full[ai], (uint32_t)((u / PF_NACC) & 1), sh, tr, TR_EPI_ACCFULL)))
                        break;
                    HSI_TSTART(t_epi);
                    tc_fence_after();
                    const int key = (wk.t_lo + kt) * TILE_KEYS + row;
#pragma unroll
                    for (int qi = 0; qi < PF_QPW; ++qi) {
                        // the query's 32 columns in two loads of 16, the first overlapping
                        // the previous tile's stores
                        uint64_t a = f2_pack(0.f, 0.f), bb = a;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t r[16];
                            tmem_ld16_issue(tbase + ai * C::N + qi * 32 + h * 16, r);
                            if (qi == 0 && h == 0) emit_pending();
                            tmem_ld_wait(r);
                            if (qi == PF_QPW - 1 && h == 1) {  // the tile's columns of this warp are in registers
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0) mbar_arrive(&acc_empty[ai]);
                            }
                            head_sum_half(r, w2[qi], h, a, bb);
                        }
                        pend_s[qi] = head_sum_final(a, bb);
                    }
                    pend_key = key;
                    HSI_TEND(t_epi, TR_EPI_WORK);
                }
                emit_pending();  // the group's last tile, before its rows are replaced
                ++qs;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::MMA_WARP) tmem_dealloc(tmem, C::TMEM_COLS);
    (void)tr;
}

}  // namespace hsi
