// K1: random-sign Hadamard rotation + NVFP4 quantisation into block records.
//
// One warp per row of 128 values; lane l holds values 4l .. 4l+3. The
// unnormalised Sylvester transform runs stage by stage (h = 1, 2, ..., 64):
// the first two stages inside a lane, the last five across lanes with shuffles.
// Every output of a stage is the same single IEEE add or subtract of the same
// two operands regardless of which lane computes it, so the result is
// bit-identical to any other stage-ordered evaluation in fp32.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "common.cuh"

namespace hsi {

struct QuantParams {
    const uint16_t* x;      // bf16 bits [n_tensors * rpt][128]
    int64_t n_tensors;
    int64_t rpt;            // rows per tensor
    int64_t rec_per_tensor; // ceil(rpt / 8)
    uint32_t neg_mask[4];   // bit d set: sign d is -1
    float* g;               // [n_tensors]
    uint32_t* amax_bits;    // [n_tensors] (mode 0)
    uint8_t* rec;
};

// y = H (s .* x) for this warp's row; v holds values 4*lane .. 4*lane+3.
__device__ __forceinline__ void rotate_row_warp(const QuantParams& p, int64_t row, float (&v)[4]) {
    const int lane = threadIdx.x & 31;
    const uint2 raw = *reinterpret_cast<const uint2*>(p.x + row * 128 + lane * 4);
    const int wsel = lane >> 3;  // select without dynamic indexing of the parameter array
    const uint32_t word =
        wsel == 0 ? p.neg_mask[0] : wsel == 1 ? p.neg_mask[1] : wsel == 2 ? p.neg_mask[2] : p.neg_mask[3];
    const uint32_t bits = word >> ((lane & 7) * 4);
    uint32_t h[4] = {raw.x & 0xFFFFu, raw.x >> 16, raw.y & 0xFFFFu, raw.y >> 16};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float f = __uint_as_float(h[i] << 16);
        v[i] = ((bits >> i) & 1u) ? -f : f;
    }
    // h = 1 and h = 2: inside the lane.
    {
        float a0 = v[0], a1 = v[1], a2 = v[2], a3 = v[3];
        v[0] = __fadd_rn(a0, a1);
        v[1] = __fsub_rn(a0, a1);
        v[2] = __fadd_rn(a2, a3);
        v[3] = __fsub_rn(a2, a3);
        a0 = v[0], a1 = v[1], a2 = v[2], a3 = v[3];
        v[0] = __fadd_rn(a0, a2);
        v[2] = __fsub_rn(a0, a2);
        v[1] = __fadd_rn(a1, a3);
        v[3] = __fsub_rn(a1, a3);
    }
    // h = 4 .. 64: partner lane differs in bit log2(h) - 2.
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float other = __shfl_xor_sync(0xFFFFFFFFu, v[i], m);
            // lower element a, upper element b: lower <- a + b, upper <- a - b
            v[i] = upper ? __fsub_rn(other, v[i]) : __fadd_rn(v[i], other);
        }
    }
}

__global__ void __launch_bounds__(256) quant_amax_kernel(QuantParams p) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t warp = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t total = p.n_tensors * p.rpt;
    if (warp >= total) return;
    float v[4];
    rotate_row_warp(p, warp, v);
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) atomicMax(&p.amax_bits[warp / p.rpt], __float_as_uint(m));
}

__global__ void quant_scale_kernel(QuantParams p) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= p.n_tensors) return;
    const float amax = __uint_as_float(p.amax_bits[t]);
    p.g[t] = amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
}

// E4M3 bits -> fp32, exact (OCP FP8 E4M3: bias 7, subnormals m/8 * 2^-6).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    const float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
    return (b & 0x80u) ? -mag : mag;
}

__device__ __forceinline__ uint32_t f32_to_e4m3_rn_sat(float x) {
    uint32_t out;
    asm("{\n\t.reg .b16 t;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u16 %0, t;\n\t}"
        : "=r"(out)
        : "f"(0.0f), "f"(x));
    return out & 0xFFu;
}

// Four values -> four E2M1 codes, value 0 in the lowest nibble.
__device__ __forceinline__ uint32_t f32x4_to_e2m1x4(float a, float b, float c, float d) {
    unsigned short out;
    asm("{\n\t.reg .b8 lo, hi;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 hi, %4, %3;\n\t"
        "mov.b16 %0, {lo, hi};\n\t}"
        : "=h"(out)
        : "f"(a), "f"(b), "f"(c), "f"(d));
    return out;
}

// Encode one rotated row (this warp's v, tensor scale g) into row r of tensor
// t's records; rows at or past rpt are written as zeros.
__device__ __forceinline__ void encode_row_warp(const QuantParams& p, int64_t t, int64_t r, const float (&v)[4],
                                                float g) {
    const int lane = threadIdx.x & 31;
    uint8_t* rec = p.rec + (t * p.rec_per_tensor + r / 8) * 576;
    const int rr = (int)(r & 7);
    uint16_t codes = 0;
    uint8_t scale = 0;
    if (r < p.rpt) {
        float ab = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
        ab = fmaxf(ab, __shfl_xor_sync(0xFFFFFFFFu, ab, 1));
        ab = fmaxf(ab, __shfl_xor_sync(0xFFFFFFFFu, ab, 2));  // max over values 16j .. 16j+15
        const uint32_t sb = f32_to_e4m3_rn_sat(__fdiv_rn(ab, __fmul_rn(6.0f, g)));
        const float sc = __fmul_rn(e4m3_to_f32(sb), g);
        if (sc != 0.0f) {
            codes = (uint16_t)f32x4_to_e2m1x4(__fdiv_rn(v[0], sc), __fdiv_rn(v[1], sc), __fdiv_rn(v[2], sc),
                                              __fdiv_rn(v[3], sc));
        }
        scale = (uint8_t)sb;
    }
    // values 4*lane .. 4*lane+3 -> two bytes at (e/32)*128 + rr*16 + (e%32)/2
    *reinterpret_cast<uint16_t*>(rec + (lane >> 3) * 128 + rr * 16 + (lane & 7) * 2) = codes;
    if ((lane & 3) == 0) rec[512 + rr * 8 + (lane >> 2)] = scale;
}

__global__ void __launch_bounds__(256) quant_encode_kernel(QuantParams p) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t prow = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);  // padded row index
    const int64_t padded_rows = p.rec_per_tensor * 8;
    if (prow >= p.n_tensors * padded_rows) return;
    const int64_t t = prow / padded_rows;
    const int64_t r = prow % padded_rows;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < p.rpt) rotate_row_warp(p, t * p.rpt + r, v);
    encode_row_warp(p, t, r, v, r < p.rpt ? p.g[t] : 1.0f);
}

// ---- MXFP4 (32-element groups, E8M0 scales, no tensor scale) ----------------

// The exponent e of a group's scale 2^e: the smallest e in [-127, 127] with
// 6 * 2^e >= amax. With amax = m 2^E (m in [1, 2)), 6 * 2^(E-2) = 1.5 * 2^E, so
// e = E - 2 when m <= 1.5 and E - 1 otherwise; zero and subnormal amax (below
// 2^-126 < 6 * 2^-127) take e = -127, as does E - 2 = -128.
__device__ __forceinline__ int mx_scale_exp(float amax) {
    const uint32_t u = __float_as_uint(amax);
    const int E = (int)((u >> 23) & 0xFFu);
    if (E == 0) return -127;
    const int e = (E - 127) - ((u & 0x7FFFFFu) <= 0x400000u ? 2 : 1);
    return e < -127 ? -127 : e;
}

// Encode one rotated row (this warp's v, valid = a real row) as row r of the
// 544-byte MXFP4 records at `recs`: per group (lanes 8j .. 8j+7 hold values
// 32j .. 32j+31) the scale exponent and the codes E2M1_RN(v 2^-e). The product
// by 2^-e (a normal fp32 for every e) is exact unless it falls below the
// normal range, where every value rounds to a zero code of its sign either
// way. A padding row (valid false) is zero: codes 0, scale byte 0.
__device__ __forceinline__ void encode_row_mx_warp(uint8_t* recs, int64_t r, const float (&v)[4], bool valid) {
    const int lane = threadIdx.x & 31;
    uint8_t* rec = recs + (r / 8) * 544;
    const int rr = (int)(r & 7);
    uint16_t codes = 0;
    uint8_t sbyte = 0;
    if (valid) {
        const bool finite = isfinite(v[0]) && isfinite(v[1]) && isfinite(v[2]) && isfinite(v[3]);
        if (!__all_sync(0xFFFFFFFFu, finite) && lane == 0) raise_error(DEVERR_ARG);
        float a = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));  // max over values 32j .. 32j+31
        const int e = mx_scale_exp(a);
        const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
        codes = (uint16_t)f32x4_to_e2m1x4(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv), __fmul_rn(v[2], inv),
                                          __fmul_rn(v[3], inv));
        sbyte = (uint8_t)(e + 127);
    }
    // values 4*lane .. 4*lane+3 -> two bytes at (e/32)*128 + rr*16 + (e%32)/2
    *reinterpret_cast<uint16_t*>(rec + (lane >> 3) * 128 + rr * 16 + (lane & 7) * 2) = codes;
    if ((lane & 7) == 0) rec[512 + rr * 4 + (lane >> 3)] = sbyte;
}

// One warp per padded row of tensor t (grid over n_tensors * rec_per_tensor * 8
// rows, 8 per CTA) into 544-byte records: rotation as above, then the MXFP4
// encoding. A non-finite rotated value is reported through the error word.
__global__ void __launch_bounds__(256) quant_mx_kernel(QuantParams p) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t prow = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t padded_rows = p.rec_per_tensor * 8;
    if (prow >= p.n_tensors * padded_rows) return;
    const int64_t t = prow / padded_rows;
    const int64_t r = prow % padded_rows;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < p.rpt) rotate_row_warp(p, t * p.rpt + r, v);
    encode_row_mx_warp(p.rec + t * p.rec_per_tensor * 544, r, v, r < p.rpt);
}

// Small tensors (at most QUANT_SMALL_ROWS rows, e.g. the 32 heads of a query):
// one CTA per tensor rotates every row once, finds the tensor scale (mode 0)
// and encodes, in a single launch.
constexpr int QUANT_SMALL_ROWS = 64;

constexpr int QUANT_SMALL_WARPS = 32;  // one row per warp for a query's 32 heads

__global__ void __launch_bounds__(32 * QUANT_SMALL_WARPS) quant_small_kernel(QuantParams p, int mode) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ float wmax[QUANT_SMALL_WARPS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = blockIdx.x;
    constexpr int RPW = QUANT_SMALL_ROWS / QUANT_SMALL_WARPS;  // rows per warp
    float v[RPW][4];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int64_t r = warp + QUANT_SMALL_WARPS * i;
        v[i][0] = v[i][1] = v[i][2] = v[i][3] = 0.f;
        if (r < p.rpt) {
            rotate_row_warp(p, t * p.rpt + r, v[i]);
            m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i][0]), fabsf(v[i][1])), fmaxf(fabsf(v[i][2]), fabsf(v[i][3]))));
        }
    }
    float g;
    if (mode == 0) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) wmax[warp] = m;
        __syncthreads();
        float amax = wmax[lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        g = amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
        if (threadIdx.x == 0) p.g[t] = g;
    } else {
        g = p.g[t];
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int64_t r = warp + QUANT_SMALL_WARPS * i;
        if (r < p.rec_per_tensor * 8) encode_row_warp(p, t, r, v[i], g);
    }
}

}  // namespace hsi
