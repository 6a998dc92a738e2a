// K7: compaction of a query's candidate pool. The Reindex layers of one decode
// step all score the same indexer K (the Full layer's) over the same pool, with
// different queries; copying the pooled block records (576 bytes NVFP4, 544
// MXFP4) of each query
// into one contiguous run once per step lets every Reindex layer stream them
// with the full-scan kernel (one bulk copy per unit) instead of gathering
// 2048 scattered records per query per layer.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace hsi {

constexpr int GATHER_THREADS = 256;
constexpr int GATHER_PER_THREAD = 4;  // chunks in flight per thread

// pool_rec[b][i] = k_rec[k_off[b] + block_ids[b][i]] for i < min(n_kept[b], n_keep),
// records of rec_chunks 16-byte chunks (36 or 34). grid = (ceil(n_keep *
// rec_chunks / (256 * 4)), B). Ids outside the query's visible records are
// reported through the device error word and skipped.
__global__ void __launch_bounds__(GATHER_THREADS) pool_gather_kernel(const uint4* __restrict__ k_rec,
                                                                     const int64_t* __restrict__ k_off,
                                                                     const int32_t* __restrict__ n_visible,
                                                                     const int32_t* __restrict__ block_ids,
                                                                     const int32_t* __restrict__ n_kept,
                                                                     int32_t n_keep, int rec_chunks,
                                                                     uint4* __restrict__ pool_rec) {
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.y;
    const int nk = min(n_kept[b], n_keep);
    const int64_t nrec = ((int64_t)n_visible[b] + 7) / 8;
    const int64_t base = k_off[b];
    const int64_t total = (int64_t)nk * rec_chunks;
    const int64_t c0 = (int64_t)blockIdx.x * GATHER_THREADS * GATHER_PER_THREAD + threadIdx.x;
    const int32_t* ids = block_ids + (int64_t)b * n_keep;
    uint4* out = pool_rec + (int64_t)b * n_keep * rec_chunks;
    uint4 v[GATHER_PER_THREAD];
    bool ok[GATHER_PER_THREAD];
    // all loads first, then all stores: GATHER_PER_THREAD reads in flight per thread
#pragma unroll
    for (int i = 0; i < GATHER_PER_THREAD; ++i) {
        const int64_t c = c0 + (int64_t)i * GATHER_THREADS;
        ok[i] = false;
        if (c < total) {
            const int r = (int)(c / rec_chunks), part = (int)(c % rec_chunks);
            const int64_t id = ids[r];
            ok[i] = id >= 0 && id < nrec;
            if (ok[i]) v[i] = __ldcs(k_rec + (base + id) * rec_chunks + part);
            else if (part == 0) raise_error(DEVERR_ARG);
        }
    }
#pragma unroll
    for (int i = 0; i < GATHER_PER_THREAD; ++i)
        if (ok[i]) out[c0 + (int64_t)i * GATHER_THREADS] = v[i];
}

}  // namespace hsi
