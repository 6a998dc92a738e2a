// K9: one decode token into every query's caches.
//
// A decode step appends the new position's indexer K row and main-KV entry to
// the query's caches before the indexer scores them. The K row is quantised
// with the cache's fixed tensor scale (NVFP4: the g_k the cache was built with;
// MXFP4: no tensor scale), as the quantiser's mode 1 would quantise the whole
// cache, so a cache built token by token equals the cache quantised at once.
// The visible length lives on the device and is advanced here, so a CUDA graph
// of a whole serving step replays over a growing cache.
//
// One CTA of 64 threads per query: warp 0 rotates and encodes the K row into
// row n = n_visible[b] of the cache's block records (only that row's bytes of
// record n/8 are written), warp 1 encodes the main-KV entry into entry n; then
// n_visible[b] = n + 1.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "mainkv.cuh"
#include "quantize.cuh"

namespace hsi {

struct AppendParams {
    QuantParams q;           // x: the new K rows [B][128] (bf16); neg_mask: the rotation's signs
    const float* g_k;        // [B] the K caches' tensor scales (NVFP4)
    uint8_t* k_rec;
    const int64_t* k_off;    // first record of query b's K cache
    const uint16_t* kv_x;    // the new main-KV entries [B][512] (bf16), or null
    uint8_t* kv;
    const int64_t* kv_off;   // first entry of query b's main-KV cache
    int32_t* n_vis;          // [B] in: the position to write; out: + 1
    const int32_t* capacity; // [B] rows (entries) each cache holds
    int mx;                  // MXFP4 K records
};

__global__ void __launch_bounds__(64) append_token_kernel(AppendParams p) {
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const int32_t n = p.n_vis[b];
    if (n < 0 || n >= __ldg(p.capacity + b)) {  // block-uniform: nothing is written
        if (threadIdx.x == 0) raise_error(DEVERR_ARG);
        return;
    }
    if (warp == 0) {
        float v[4];
        rotate_row_warp(p.q, b, v);
        if (p.mx) {
            encode_row_mx_warp(p.k_rec + __ldg(p.k_off + b) * 544, n, v, true);
        } else {
            QuantParams q = p.q;
            q.rec = p.k_rec + __ldg(p.k_off + b) * 576;  // tensor 0 of this cache
            q.rpt = (int64_t)n + 1;                       // row n is a real row
            encode_row_warp(q, 0, n, v, __ldg(p.g_k + b));
        }
    } else if (p.kv_x) {
        mainkv_encode_warp(p.kv_x + (int64_t)b * KV_DIM, p.kv + (__ldg(p.kv_off + b) + n) * KV_BYTES);
    }
    __syncthreads();  // every read of n_vis[b] precedes its update
    if (threadIdx.x == 0) p.n_vis[b] = n + 1;
}

}  // namespace hsi
