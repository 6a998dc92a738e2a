// K6: calibration kernels that measure the two rooflines the path is judged
// against on the running GPU: read-only HBM bandwidth (plain 16-byte loads, or
// the bulk-copy ring the scoring kernel uses) and the block-scaled FP4 tensor
// rate of tcgen05.mma kind::mxf4nvf4 at a given N.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace hsi {

// Grid-stride 16-byte loads over the buffer; one xor per CTA keeps them live.
__global__ void __launch_bounds__(512) calib_read_ldg_kernel(const uint4* __restrict__ buf, size_t n16,
                                                             unsigned long long* sink) {
    griddep_wait();  // the buffer may have just been written by the previous kernel
    uint32_t x = 0;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = __ldcs(buf + i), b = __ldcs(buf + i + stride), c = __ldcs(buf + i + 2 * stride),
                    d = __ldcs(buf + i + 3 * stride);
        x ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; i < n16; i += stride) {
        const uint4 a = __ldcs(buf + i);
        x ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    if (x == 0x9E3779B9u) atomicAdd(sink, 1ull);  // practically never; keeps the loads
}

// Each CTA streams one contiguous slice through a ring of `stages` shared-
// memory buffers of `chunk` bytes with bulk copies; one thread issues, one
// warp consumes (waits and releases). Mirrors the scoring kernel's producer.
__global__ void __launch_bounds__(64, 1) calib_read_bulk_kernel(const uint8_t* __restrict__ buf, size_t bytes,
                                                               int chunk, int stages, unsigned long long* sink) {
    griddep_wait();  // the buffer may have just been written by the previous kernel
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)stages * chunk);
    uint64_t* empty = full + stages;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t per = (bytes / gridDim.x) / chunk * chunk;
    const uint8_t* base = buf + per * blockIdx.x;
    const long long n = (long long)(per / chunk);
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        long long issued = 0;
        for (long long u = 0; u < n; ++u) {
            const int s = (int)(u % stages);
            if (!wait_bounded(&empty[s], (uint32_t)(((u / stages) & 1) ^ 1), &abort_flag)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[s], (uint32_t)chunk);
                bulk_g2s(smem + (size_t)s * chunk, base + (size_t)u * chunk, (uint32_t)chunk, &full[s]);
            }
            __syncwarp();
            issued = u + 1;
        }
        if (lane == 0)  // drain
            for (int s = 0; s < stages && s < issued; ++s) {
                const long long last = s + ((issued - 1 - s) / stages) * stages;
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&full[s], (uint32_t)((last / stages) & 1)))
                    if (globaltimer_ns() - t0 > HSI_WAIT_TIMEOUT_NS) {
                        raise_error(DEVERR_TIMEOUT);
                        break;
                    }
            }
    } else {
        uint32_t x = 0;
        for (long long u = 0; u < n; ++u) {
            const int s = (int)(u % stages);
            if (!wait_bounded(&full[s], (uint32_t)((u / stages) & 1), &abort_flag)) break;
            x ^= reinterpret_cast<const uint32_t*>(smem + (size_t)s * chunk)[lane];
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (x == 0x9E3779B9u) atomicAdd(sink, 1ull);
    }
    __syncthreads();
}

// Back-to-back tcgen05.mma kind::mxf4nvf4 (M = 128, N = n, K = 64) on
// shared-memory operands of zeros, one issuing thread per CTA.
template <int N>
__global__ void __launch_bounds__(128, 1) calib_mma_kernel(int iters, unsigned long long* sink) {
    constexpr int A_BYTES = 128 * 32, B_BYTES = N * 32;
    constexpr int COLS = N <= 32 ? 64 : N <= 64 ? 128 : N <= 128 ? 256 : 512;
    __shared__ __align__(1024) uint8_t ops[A_BYTES + B_BYTES + 1024];
    __shared__ uint64_t done;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < (A_BYTES + B_BYTES + 1024) / 4; i += blockDim.x)
        reinterpret_cast<uint32_t*>(ops)[i] = 0;
    if (threadIdx.x == 0) {
        mbar_init(&done, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    fence_proxy_async_smem();
    if (warp == 0) tmem_alloc(&tmem_base, COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    if (threadIdx.x == 0) {
        const uint32_t a = smem_u32(ops), b = a + A_BYTES, sf = b + B_BYTES;
        const uint32_t sfa = tmem + N, sfb = tmem + N + 4;
        tc_cp_32x128b_x4(sfa, smem_desc(sf, 128, 128));
        tc_cp_32x128b_x4(sfb, smem_desc(sf + 512, 128, 128));
        constexpr uint32_t idesc = idesc_nvf4(128, N);
        // K-major, no swizzle: 8-row core matrices, 2 of them along K (LBO 128), groups 256 B apart (SBO)
        const uint64_t ad = smem_desc(a, 128, 256), bd = smem_desc(b, 128, 256);
        for (int i = 0; i < iters; ++i) mma_nvf4(tmem, ad, bd, idesc, sfa, sfb, i > 0);
        tc_commit(&done);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&done, 0))
            if (globaltimer_ns() - t0 > HSI_WAIT_TIMEOUT_NS) {
                raise_error(DEVERR_TIMEOUT);
                break;
            }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, COLS);
    if (threadIdx.x == 0 && abort_flag) atomicAdd(sink, 1ull);
}

}  // namespace hsi
