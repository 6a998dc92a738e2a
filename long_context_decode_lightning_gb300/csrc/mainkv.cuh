// K8: the FP4 main KV that core attention reads, and gather(main_kv, topk).
//
// An entry is 512 values in 288 bytes: E2M1 codes (value i in byte i/2, low
// nibble for even i), then one E4M3 scale per 16 values (byte 256 + i/16); no
// global scale. Quantisation: scale = E4M3_RN(amax/6), code = E2M1_RN(x/scale).
// The gather decodes the selected entries of each query into bf16 rows for the
// attention kernel; every decoded value (an E2M1 value times an E4M3 scale, at
// most 6 significant bits, magnitude in [2^-10, 2688]) is exact in bf16.
//
// The quantiser gives each lane one 16-value group of an entry, so a group's
// amax and scale need no exchange between lanes; the gather gives each lane 8
// values of two groups, so that the warp's stores of a row are contiguous.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "quantize.cuh"

namespace hsi {

constexpr int KV_DIM = 512;
constexpr int KV_BYTES = 288;

// Eight codes (four bytes; value 2i in the low nibble of byte i) times one
// E4M3 scale, as four bf16 pairs. The hardware conversions give the E2M1
// values and the scale exactly in f16, and their product (at most 6
// significant bits, magnitude in [2^-10, 2688]) is exact in f16, so in fp32
// and in bf16: the same bits as decoding in fp32.
__device__ __forceinline__ void decode8_bf16(uint32_t codes, uint32_t scale_byte, uint32_t (&o)[4]) {
    uint32_t sc2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(sc2) : "h"((unsigned short)(scale_byte * 0x101u)));
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t v;
        asm("{ .reg .b8 t; cvt.u8.u16 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }"
            : "=r"(v)
            : "h"((unsigned short)((codes >> (8 * q)) & 0xFFu)));
        const __half2 prod = __hmul2(*reinterpret_cast<const __half2*>(&v), *reinterpret_cast<const __half2*>(&sc2));
        const float2 f = __half22float2(prod);
        const __nv_bfloat162 h = __floats2bfloat162_rn(f.x, f.y);
        o[q] = *reinterpret_cast<const uint32_t*>(&h);
    }
}

// One warp: the bf16 entry at x_row (512 values, 16-byte aligned) into the
// 288 bytes at dst. A non-finite value is reported through the error word.
__device__ __forceinline__ void mainkv_encode_warp(const uint16_t* __restrict__ x_row, uint8_t* __restrict__ dst) {
    const int lane = threadIdx.x & 31;
    const uint4* src = reinterpret_cast<const uint4*>(x_row + lane * 16);
    const uint4 a = __ldcs(src), b = __ldcs(src + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float v[16];
    float amax = 0.f;
    bool finite = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        finite = finite && isfinite(v[i]);
        amax = fmaxf(amax, fabsf(v[i]));
    }
    if (!finite) raise_error(DEVERR_ARG);
    const uint32_t sb = f32_to_e4m3_rn_sat(__fdiv_rn(amax, 6.0f));
    const float sc = e4m3_to_f32(sb);
    uint32_t c0 = 0u, c1 = 0u;
    if (sc != 0.0f) {
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = __fdiv_rn(v[i], sc);
        c0 = f32x4_to_e2m1x4(y[0], y[1], y[2], y[3]) | (f32x4_to_e2m1x4(y[4], y[5], y[6], y[7]) << 16);
        c1 = f32x4_to_e2m1x4(y[8], y[9], y[10], y[11]) | (f32x4_to_e2m1x4(y[12], y[13], y[14], y[15]) << 16);
    }
    *reinterpret_cast<uint2*>(dst + lane * 8) = make_uint2(c0, c1);
    dst[256 + lane] = (uint8_t)sb;
}

// x: bf16 [n][512] (16-byte aligned); kv: [n][288] (16-byte aligned). grid =
// ceil(n / 8) CTAs of 256 threads, one warp per entry.
__global__ void __launch_bounds__(256) mainkv_quant_kernel(const uint16_t* __restrict__ x, int64_t n,
                                                           uint8_t* __restrict__ kv) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t e = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (e >= n) return;
    mainkv_encode_warp(x + e * KV_DIM, kv + e * KV_BYTES);
}

// out[b][t][:] = entry kv_off[b] + idx[b][t] decoded (bf16 [B][k][512]),
// zeros where idx[b][t] < 0; an index at or past n_visible[b] is reported
// through the device error word and its row is zeroed. A warp takes
// GATHER_EPW consecutive (b, t) of the flattened list: lane j < GATHER_EPW
// resolves entry j's index, then every lane issues the loads of all its
// entries before decoding any, so one launch is about one wave of warps with
// two dependent memory round trips each. grid = ceil(B k / (8 GATHER_EPW))
// CTAs of 256 threads.
#ifndef HSI_GATHER_EPW
#define HSI_GATHER_EPW 4
#endif
constexpr int GATHER_EPW = HSI_GATHER_EPW;

// L lists of B x k indices (list l at idx + l idx_stride, its rows written
// at out + l out_stride) are one flattened list of L B k items, so a step's
// gathers for several layers run as one launch, one ramp instead of L.
__global__ void __launch_bounds__(256) mainkv_gather_kernel(const uint8_t* __restrict__ kv,
                                                            const int64_t* __restrict__ kv_off,
                                                            const int32_t* __restrict__ n_vis,
                                                            const int32_t* __restrict__ idx, int64_t ld_idx,
                                                            int64_t idx_stride, int32_t L, int32_t k, int32_t B,
                                                            uint16_t* __restrict__ out, int64_t out_stride) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t per = (int64_t)B * k;
    const int64_t total = per * L;
    const int64_t base = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * GATHER_EPW;
    if (base >= total) return;
    const int lane = threadIdx.x & 31;
    // lane j < GATHER_EPW: the entry (in entries of kv) of list item base + j, or -1
    long long src = -1;
    if (lane < GATHER_EPW && base + lane < total) {
        const int64_t f = base + lane;
        const int64_t l = f / per, r = f % per;
        const int b = (int)(r / k), t = (int)(r % k);
        const int32_t i = __ldg(idx + l * idx_stride + (int64_t)b * ld_idx + t);
        const int32_t nv = __ldg(n_vis + b);
        const int64_t o = __ldg(kv_off + b);
        if (i >= 0) {
            if (i < nv) src = o + i;
            else raise_error(DEVERR_ARG);
        }
    }
    // lane: values [8 lane, 8 lane + 8) and [256 + 8 lane, 256 + 8 lane + 8) of
    // each entry, so that each of the warp's two 16-byte stores per entry
    // covers 512 contiguous bytes of the row
    long long e[GATHER_EPW];
    uint32_t c0[GATHER_EPW], c1[GATHER_EPW], s0[GATHER_EPW], s1[GATHER_EPW];
#pragma unroll
    for (int j = 0; j < GATHER_EPW; ++j) {
        e[j] = __shfl_sync(0xFFFFFFFFu, src, j);
        c0[j] = c1[j] = s0[j] = s1[j] = 0u;
        if (e[j] >= 0) {
            const uint8_t* p = kv + e[j] * KV_BYTES;
            c0[j] = __ldcs(reinterpret_cast<const uint32_t*>(p) + lane);
            c1[j] = __ldcs(reinterpret_cast<const uint32_t*>(p + 128) + lane);
            s0[j] = __ldcs(p + 256 + (lane >> 1));
            s1[j] = __ldcs(p + 272 + (lane >> 1));
        }
    }
#pragma unroll
    for (int j = 0; j < GATHER_EPW; ++j) {
        if (base + j >= total) break;
        uint32_t o0[4] = {0u, 0u, 0u, 0u}, o1[4] = {0u, 0u, 0u, 0u};
        if (e[j] >= 0) {
            decode8_bf16(c0[j], s0[j], o0);
            decode8_bf16(c1[j], s1[j], o1);
        }
        const int64_t f = base + j;
        uint16_t* row = out + (f / per) * out_stride + (f % per) * KV_DIM;
        __stcs(reinterpret_cast<uint4*>(row + lane * 8), make_uint4(o0[0], o0[1], o0[2], o0[3]));
        __stcs(reinterpret_cast<uint4*>(row + 256 + lane * 8), make_uint4(o1[0], o1[1], o1[2], o1[3]));
    }
}

}  // namespace hsi
