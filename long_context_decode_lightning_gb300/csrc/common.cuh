// Shared device-side definitions: the sticky error word and small helpers.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace hsi {

// Device error codes (bit flags, OR-ed into the sticky word).
enum : uint32_t {
    DEVERR_TIMEOUT = 1u,  // a bounded wait ran out
    DEVERR_ARG = 2u,      // a device-side argument was malformed
};

// The sticky error word of this module on the current device (the library is
// one translation unit, so this is its only definition).
__device__ uint32_t g_hsi_error = 0;

__device__ __forceinline__ void raise_error(uint32_t code) { atomicOr(&g_hsi_error, code); }

// Diagnostics (set from the host through hsi_debug_set): the wall-clock limit
// of every bounded wait, and a test switch that makes the scoring kernels'
// producer skip its first copy so that a consumer's wait runs out.
__device__ unsigned long long g_hsi_wait_limit_ns = HSI_WAIT_TIMEOUT_NS;
__device__ int g_hsi_skip_first_copy = 0;

// Optional wait tracing (build with -DHSI_TRACE): cycles each warp role spent
// blocked in each kind of wait, and its total loop cycles, summed over CTAs.
#ifdef HSI_TRACE
constexpr int TRACE_SLOTS = 32;
__device__ unsigned long long g_hsi_trace[TRACE_SLOTS];
// per-CTA wall-clock marks (ns): entry, work start, work end, exit
__device__ unsigned long long g_hsi_marks[1024][4];
#endif

struct WaitTrace {
#ifdef HSI_TRACE
    unsigned long long c[TRACE_SLOTS] = {};
    __device__ void add(int i, unsigned long long v) { c[i] += v; }
    __device__ void flush() {
        for (int i = 0; i < TRACE_SLOTS; ++i)
            if (c[i]) atomicAdd(&g_hsi_trace[i], c[i]);
    }
#else
    __device__ void add(int, unsigned long long) {}
    __device__ void flush() {}
#endif
};

// Wait for the phase of `bar` with the given parity to complete, bounded in
// wall-clock time. Returns false (after setting *abort and the device error
// word on a timeout) when the wait gave up, either by running out or because
// another warp of the block has already aborted.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const uint64_t limit = *(volatile unsigned long long*)&g_hsi_wait_limit_ns;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit) {
            raise_error(DEVERR_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag (teardown: drain what is in flight).
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    const uint64_t limit = *(volatile unsigned long long*)&g_hsi_wait_limit_ns;
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit) {
            raise_error(DEVERR_TIMEOUT);
            return;
        }
    }
}

// Order-preserving map of an fp32 score to a uint32 key (larger score ->
// larger key); -0 maps like +0. Scores must not be NaN.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
    const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

// Four pooled-block flags (bits 0..3 of nib) as the 32 position bits of their
// blocks of eight positions: bit q of the nibble fills byte q of the word.
__device__ __forceinline__ uint32_t expand_nibble(uint32_t nib) { return ((nib * 0x00204081u) & 0x01010101u) * 0xFFu; }

// The position bit table of one row (words 0 .. ceil(n_vis / 32) - 1) from the
// bitmap of its pooled blocks of eight positions (bit j of bm[j / 32] for
// block j): word w covers blocks 4w .. 4w + 3; bits of positions at or past
// n_vis are 0. Threads tid of nthreads share the words; when the row is
// 16-byte aligned the fully visible words go four to a store.
__device__ __forceinline__ void write_pos_bits8(uint32_t* bits, const uint32_t* bm, int64_t n_vis, int tid,
                                                int nthreads) {
    const int64_t pw = (n_vis + 31) / 32;
    int64_t w0 = 0;
    if ((reinterpret_cast<uintptr_t>(bits) & 15) == 0) {
        const int64_t quads = n_vis / 128;  // groups of four fully visible words: 16 blocks, half a bitmap word
        for (int64_t g = tid; g < quads; g += nthreads) {
            const uint32_t half = bm[g >> 1] >> (16 * (int)(g & 1));
            uint4 o;
            o.x = expand_nibble(half & 0xFu);
            o.y = expand_nibble((half >> 4) & 0xFu);
            o.z = expand_nibble((half >> 8) & 0xFu);
            o.w = expand_nibble((half >> 12) & 0xFu);
            reinterpret_cast<uint4*>(bits)[g] = o;
        }
        w0 = 4 * quads;
    }
    for (int64_t w = w0 + tid; w < pw; w += nthreads) {
        uint32_t v = expand_nibble((bm[w >> 3] >> (4 * (int)(w & 7))) & 0xFu);
        const int64_t left = n_vis - 32 * w;  // visible positions in this word
        if (left < 32) v &= (1u << left) - 1u;
        bits[w] = v;
    }
}

}  // namespace hsi
