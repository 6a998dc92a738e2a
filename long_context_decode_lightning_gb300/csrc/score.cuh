// K2 / K5: lightning-indexer scoring on the tensor cores.
//
//   I = (g_q g_k / 128) * sum_j w_j * ReLU(q_j . k)
//
// One tile = 128 keys (16 NVFP4 block records of 8 keys) x one query group
// (NQ queries x 32 heads). The contraction D[key][head] = K_tile . Q^T is
// tcgen05.mma kind::mxf4nvf4 with per-16-element E4M3 scales (M = 128,
// N = 32 NQ, K = 128 as two K = 64 steps), accumulated in fp32 in Tensor
// Memory. The epilogue reads D from TMEM (one key per thread), applies ReLU
// and the head weights and writes one fp32 score per key, so per-head logits
// never leave the SM.
//
// Warp roles in a persistent CTA (one per SM):
//   warp 0      producer: bulk copies (TMA engine) of K records into a ring of
//               shared-memory stages and of the group's q records into one of
//               two q slots. Full scan: one copy of up to 16 consecutive
//               records per tile. Pool gather: one 576-byte copy per pooled
//               block (a whole 8-key block: codes and scales).
//   warp 1      MMA issuer: rearranges each tile's scales into the 32x16-byte
//               layout tcgen05.cp takes, copies them to TMEM and issues the
//               MMAs; owns the TMEM allocation.
//   warps 2..5  epilogue (each owns one 32-lane quarter of TMEM).
// The block records are used in place as the MMA operands: a record is eight
// rows of four 8x16-byte core matrices (K-major, no swizzle, core matrices 128 B
// apart along K, records 576 B apart along M/N).
//
// Work: tiles of all queries are numbered in order (query group, then key
// tile) and each CTA takes one contiguous range, so it reloads q only when the
// group changes. Every wait is bounded; on a timeout the CTA records the error,
// drains its copies and MMAs, frees TMEM and returns.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace hsi {

constexpr int REC = 576;
constexpr int TILE_RECS = 16;
constexpr int TILE_KEYS = 128;

struct ScoreParams {
    const uint8_t* q_rec;
    const float* g_q;
    const float* w;
    const uint8_t* k_rec;
    const float* g_k;
    const int64_t* k_off;
    const int32_t* n_vis;
    int32_t B;
    int32_t ngroups;
    // full scan
    float* scores;
    int64_t ld;
    float* bmax;
    int64_t ldb;
    // pool gather
    const int32_t* block_ids;
    const int32_t* n_kept;
    int32_t n_keep;
    float* pool_scores;
    int64_t ld_pool;
};

template <int NQ, bool GATHER, int STAGES>
struct ScoreCfg {
    static constexpr int N = 32 * NQ;
    static constexpr int Q_BYTES = NQ * 4 * REC;
    static constexpr int STAGE_BYTES = TILE_RECS * REC + 2 * 512;  // records + two SFA atoms
    static constexpr int QSLOT_BYTES = ((Q_BYTES + 127) / 128) * 128 + 2 * 512;
    static constexpr int EPI_WARPS = 4;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    // TMEM columns: two accumulators, two SFA buffers (2 chunks x 4), two SFB slots
    static constexpr int COL_ACC = 0;
    static constexpr int COL_SFA = 2 * N;
    static constexpr int COL_SFB = 2 * N + 16;
    static constexpr int COLS_USED = 2 * N + 32;
    static constexpr int TMEM_COLS = COLS_USED <= 32 ? 32 : COLS_USED <= 64 ? 64 : COLS_USED <= 128 ? 128
                                     : COLS_USED <= 256 ? 256 : 512;
    static constexpr int OFF_STAGES = 0;
    static constexpr int OFF_QSLOTS = STAGES * STAGE_BYTES;
    static constexpr int OFF_BARS = OFF_QSLOTS + 2 * QSLOT_BYTES;
    static constexpr int NBARS = 2 * STAGES + 8 + 1;
    static constexpr int SMEM_BYTES = OFF_BARS + NBARS * 8 + 64 + 1024;  // + alignment slack
    static_assert(NQ <= 4, "one 128-row scale atom per K chunk for B");
    static_assert(COLS_USED <= 512, "TMEM");
};

struct ScoreShared {  // small control block after the barriers
    uint32_t tmem_base;
    int abort;
    int g0;
    int t0;
    long long count;
};

// Whole block: this CTA's first unit (g0, t0) and unit count.
template <class TilesFn>
__device__ void schedule_range(int ngroups, TilesFn tiles, ScoreShared* sh, long long* part_smem) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (ngroups + nt - 1) / nt;
    const int ga = min(ngroups, tid * per), gb = min(ngroups, ga + per);
    long long mine = 0;
    for (int g = ga; g < gb; ++g) mine += tiles(g);
    part_smem[tid] = mine;
    __syncthreads();
    if (tid == 0) {
        long long run = 0;
        for (int i = 0; i < nt; ++i) {
            const long long v = part_smem[i];
            part_smem[i] = run;
            run += v;
        }
        part_smem[nt] = run;
        sh->count = 0;
        sh->g0 = ngroups;
        sh->t0 = 0;
    }
    __syncthreads();
    const long long total = part_smem[nt];
    const long long lo = total * blockIdx.x / gridDim.x;
    const long long hi = total * (blockIdx.x + 1) / gridDim.x;
    const long long base = part_smem[tid];
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

// Bounded wait that ignores the abort flag (teardown: drain what is in flight).
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > HSI_WAIT_TIMEOUT_NS) {
            raise_error(DEVERR_TIMEOUT);
            return;
        }
    }
}

template <int NQ, bool GATHER>
__device__ __forceinline__ int group_tiles(const ScoreParams& p, int g) {
    if (GATHER) {
        const int nk = p.n_kept[g];
        return nk <= 0 ? 0 : (min(nk, p.n_keep) + TILE_RECS - 1) / TILE_RECS;
    } else {
        int m = 0;
#pragma unroll
        for (int i = 0; i < NQ; ++i) m = max(m, p.n_vis[g * NQ + i]);
        return (m + TILE_KEYS - 1) / TILE_KEYS;
    }
}

// Scale factors of 128 rows (16 records at stride 576) -> two 32x16-byte atoms:
// atom kk, byte (m%32)*16 + (m/32)*4 + i holds the scale of row m, values
// 64kk + 16i .. +16. Whole warp.
__device__ __forceinline__ void permute_sf(const uint8_t* recs, int nrows, uint8_t* atoms) {
    const int lane = threadIdx.x & 31;
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int m = lane + 32 * c;
        if (m < nrows) {
            const uint2 v = *reinterpret_cast<const uint2*>(recs + (m >> 3) * REC + 512 + (m & 7) * 8);
            lo[c] = v.x;
            hi[c] = v.y;
        } else {
            lo[c] = 0u;
            hi[c] = 0u;
        }
    }
    *reinterpret_cast<uint4*>(atoms + lane * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4*>(atoms + 512 + lane * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
}

template <int NQ, bool GATHER, int STAGES>
__global__ void __launch_bounds__(ScoreCfg<NQ, GATHER, STAGES>::THREADS, 1) score_kernel(ScoreParams p) {
    using C = ScoreCfg<NQ, GATHER, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem + C::OFF_STAGES;
    uint8_t* qslots = smem + C::OFF_QSLOTS;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* acc_full = bars + 2 * STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* q_full = acc_full + 4;
    uint64_t* q_empty = acc_full + 6;
    uint64_t* drain = acc_full + 8;
    ScoreShared* sh = reinterpret_cast<ScoreShared*>(bars + C::NBARS);
    __shared__ long long part[C::THREADS + 1];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], C::EPI_WARPS);
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
        }
        mbar_init(drain, 1);
        sh->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&sh->tmem_base, C::TMEM_COLS);
    schedule_range(p.ngroups, [&](int g) { return group_tiles<NQ, GATHER>(p, g); }, sh, part);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    const long long count = sh->count;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int g = sh->g0, t = sh->t0, ntiles = count > 0 ? group_tiles<NQ, GATHER>(p, g) : 0;
        int cur_g = -1, gc = -1;
        // what was issued, for the drain at teardown
        long long issued_units = 0;
        int last_q_gc[2] = {-1, -1};
        for (long long u = 0; u < count; ++u) {
            if (g != cur_g) {
                cur_g = g;
                ++gc;
                const int slot = gc & 1;
                if (!wait_role(&q_empty[slot], ((gc >> 1) & 1) ^ 1, sh)) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&q_full[slot], C::Q_BYTES);
                    bulk_g2s(qslots + slot * C::QSLOT_BYTES, p.q_rec + (int64_t)g * NQ * 4 * REC, C::Q_BYTES,
                             &q_full[slot]);
                }
                last_q_gc[slot] = gc;
            }
            const int s = (int)(u % STAGES);
            const uint32_t ph = (uint32_t)((u / STAGES) & 1);
            if (!wait_role(&empty[s], ph ^ 1, sh)) break;
            uint8_t* dst = stages + s * C::STAGE_BYTES;
            if (!GATHER) {
                const int b0 = g * NQ;
                int maxv = 0;
#pragma unroll
                for (int i = 0; i < NQ; ++i) maxv = max(maxv, p.n_vis[b0 + i]);
                const int64_t nrec_all = (maxv + 7) / 8;
                const int nrec = (int)min((int64_t)TILE_RECS, nrec_all - (int64_t)t * TILE_RECS);
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[s], (uint32_t)(nrec * REC));
                    bulk_g2s(dst, p.k_rec + (p.k_off[b0] + (int64_t)t * TILE_RECS) * REC, (uint32_t)(nrec * REC),
                             &full[s]);
                }
            } else {
                const int b = g;
                const int nk = min(p.n_kept[b], p.n_keep);
                const int j = t * TILE_RECS + lane;
                const int64_t nrec_vis = ((int64_t)p.n_vis[b] + 7) / 8;
                bool ok = false;
                int64_t id = 0;
                if (lane < TILE_RECS && j < nk) {
                    id = p.block_ids[(int64_t)b * p.n_keep + j];
                    ok = id >= 0 && id < nrec_vis;
                    if (!ok) raise_error(DEVERR_ARG);
                }
                const uint32_t m = __ballot_sync(0xFFFFFFFFu, ok);
                if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(__popc(m) * REC));
                __syncwarp();
                if (ok) bulk_g2s(dst + lane * REC, p.k_rec + (p.k_off[b] + id) * REC, REC, &full[s]);
            }
            issued_units = u + 1;
            if (++t == ntiles) {
                t = 0;
                do {
                    ++g;
                } while (g < p.ngroups && (ntiles = group_tiles<NQ, GATHER>(p, g)) == 0);
            }
        }
        // drain: every copy issued must have landed before the CTA exits
        if (lane == 0) {
            for (int s = 0; s < STAGES && s < issued_units; ++s) {
                const long long last = s + ((issued_units - 1 - s) / STAGES) * STAGES;  // last unit on stage s
                wait_drain(&full[s], (uint32_t)((last / STAGES) & 1));
            }
            for (int slot = 0; slot < 2; ++slot)
                if (last_q_gc[slot] >= 0) wait_drain(&q_full[slot], (uint32_t)((last_q_gc[slot] >> 1) & 1));
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        int g = sh->g0, t = sh->t0, ntiles = count > 0 ? group_tiles<NQ, GATHER>(p, g) : 0;
        int cur_g = -1, gc = -1;
        constexpr uint32_t idesc = idesc_nvf4(128, C::N);
        for (long long u = 0; u < count; ++u) {
            if (g != cur_g) {
                if (cur_g >= 0 && lane == 0) tc_commit(&q_empty[gc & 1]);  // old slot free once its MMAs finish
                cur_g = g;
                ++gc;
                const int slot = gc & 1;
                if (!wait_role(&q_full[slot], (gc >> 1) & 1, sh)) break;
                uint8_t* qs = qslots + slot * C::QSLOT_BYTES;
                uint8_t* atoms = qs + C::QSLOT_BYTES - 1024;
                permute_sf(qs, C::N, atoms);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t sfb = tmem + C::COL_SFB + slot * 8;
                    tc_cp_32x128b_x4(sfb, smem_desc(smem_u32(atoms), 128, 128));
                    tc_cp_32x128b_x4(sfb + 4, smem_desc(smem_u32(atoms + 512), 128, 128));
                }
                __syncwarp();
            }
            const int s = (int)(u % STAGES);
            const uint32_t ph = (uint32_t)((u / STAGES) & 1);
            const int acc = (int)(u & 1);
            const uint32_t aph = (uint32_t)((u >> 1) & 1);
            if (!wait_role(&full[s], ph, sh)) break;
            uint8_t* st = stages + s * C::STAGE_BYTES;
            uint8_t* sfa_atoms = st + TILE_RECS * REC;
            permute_sf(st, TILE_KEYS, sfa_atoms);
            fence_proxy_async_smem();
            __syncwarp();
            if (!wait_role(&acc_empty[acc], aph ^ 1, sh)) break;
            if (lane == 0) {
                tc_fence_after();
                const uint32_t sfa = tmem + C::COL_SFA + acc * 8;
                const uint32_t sfb = tmem + C::COL_SFB + (gc & 1) * 8;
                tc_cp_32x128b_x4(sfa, smem_desc(smem_u32(sfa_atoms), 128, 128));
                tc_cp_32x128b_x4(sfa + 4, smem_desc(smem_u32(sfa_atoms + 512), 128, 128));
                const uint32_t a0 = smem_u32(st);
                const uint32_t b0 = smem_u32(qslots + (gc & 1) * C::QSLOT_BYTES);
                const uint32_t d = tmem + C::COL_ACC + acc * C::N;
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    mma_nvf4(d, smem_desc(a0 + kk * 256, 128, REC), smem_desc(b0 + kk * 256, 128, REC), idesc,
                             sfa + kk * 4, sfb + kk * 4, kk);
                }
                tc_commit(&empty[s]);
                tc_commit(&acc_full[acc]);
            }
            __syncwarp();
            if (++t == ntiles) {
                t = 0;
                do {
                    ++g;
                } while (g < p.ngroups && (ntiles = group_tiles<NQ, GATHER>(p, g)) == 0);
            }
        }
        // drain: every MMA / copy into TMEM done before the allocation is freed
        if (lane == 0) {
            tc_commit(drain);
            wait_drain(drain, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // key within the tile
        int g = sh->g0, t = sh->t0, ntiles = count > 0 ? group_tiles<NQ, GATHER>(p, g) : 0;
        int cur_g = -1;
        float wq[NQ][32];
        for (long long u = 0; u < count; ++u) {
            if (g != cur_g) {
                cur_g = g;
#pragma unroll
                for (int qi = 0; qi < NQ; ++qi) {
                    const int b = g * NQ + qi;
                    const float sc = p.g_q[b] * p.g_k[b] * 0.0078125f;
                    const float4* wv = reinterpret_cast<const float4*>(p.w + (int64_t)b * 32);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 v = __ldg(wv + j4);
                        wq[qi][4 * j4 + 0] = v.x * sc;
                        wq[qi][4 * j4 + 1] = v.y * sc;
                        wq[qi][4 * j4 + 2] = v.z * sc;
                        wq[qi][4 * j4 + 3] = v.w * sc;
                    }
                }
            }
            const int acc = (int)(u & 1);
            const uint32_t aph = (uint32_t)((u >> 1) & 1);
            if (!wait_role(&acc_full[acc], aph, sh)) break;
            tc_fence_after();
            const uint32_t dbase = tmem + ((uint32_t)(quarter * 32) << 16) + C::COL_ACC + acc * C::N;
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                float a[32];
                tmem_ld32(dbase + qi * 32, a);
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    s0 = fmaf(wq[qi][j], fmaxf(a[j], 0.f), s0);
                    s1 = fmaf(wq[qi][j + 1], fmaxf(a[j + 1], 0.f), s1);
                }
                const float sc = s0 + s1;
                const int b = g * NQ + qi;
                if (!GATHER) {
                    const int nv = p.n_vis[b];
                    const int key = t * TILE_KEYS + row;
                    const bool vis = key < nv;
                    if (vis) p.scores[(int64_t)b * p.ld + key] = sc;
                    if (p.bmax) {
                        float m = vis ? sc : __uint_as_float(0xFF800000u);
                        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
                        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
                        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
                        if ((lane & 7) == 0 && vis) p.bmax[(int64_t)b * p.ldb + key / 8] = m;
                    }
                } else {
                    const int slot = t * TILE_KEYS + row;
                    const int j = slot >> 3;
                    const int nk = min(p.n_kept[b], p.n_keep);
                    if (j < nk) {
                        const int64_t pos = (int64_t)p.block_ids[(int64_t)b * p.n_keep + j] * 8 + (slot & 7);
                        const float v = pos < p.n_vis[b] ? sc : __uint_as_float(0xFF800000u);
                        p.pool_scores[(int64_t)b * p.ld_pool + slot] = v;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
            if (++t == ntiles) {
                t = 0;
                do {
                    ++g;
                } while (g < p.ngroups && (ntiles = group_tiles<NQ, GATHER>(p, g)) == 0);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace hsi
