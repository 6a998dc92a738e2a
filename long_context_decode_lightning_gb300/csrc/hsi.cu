// libhsi: the C-ABI entry points. Host-side validation, workspace carving and
// kernel launches; all arithmetic of the path runs in the kernels included here.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/hsi.h"
#include "append.cuh"
#include "calib.cuh"
#include "common.cuh"
#include "gather.cuh"
#include "mainkv.cuh"
#include "prefill.cuh"
#include "quantize.cuh"
#include "rowsel.cuh"
#include "score.cuh"
#include "select.cuh"

using namespace hsi;

namespace {

// Stage ring depth and 128-key tiles per stage of each scoring variant
// (the decode pair can be overridden at build time for tuning sweeps).
#ifndef HSI_DECODE_STAGES
#define HSI_DECODE_STAGES 4
#endif
#ifndef HSI_DECODE_UT
#define HSI_DECODE_UT 4
#endif
constexpr int kDecodeStages = HSI_DECODE_STAGES, kDecodeUT = HSI_DECODE_UT;
// scans of a compacted pool: 2048 records per query, a few units per CTA
#ifndef HSI_POOLED_STAGES
#define HSI_POOLED_STAGES 4
#endif
#ifndef HSI_POOLED_UT
#define HSI_POOLED_UT 4
#endif
constexpr int kPooledStages = HSI_POOLED_STAGES, kPooledUT = HSI_POOLED_UT;
#ifndef HSI_GATHER_STAGES
#define HSI_GATHER_STAGES 8
#endif
#ifndef HSI_GATHER_UT
#define HSI_GATHER_UT 2
#endif
constexpr int kGatherStages = HSI_GATHER_STAGES, kGatherUT = HSI_GATHER_UT;
constexpr int kPrefillStages = 8, kPrefillUT = 1;
constexpr int kCandCap = 65536;  // survivors of the histogram pass kept per query

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

hsi_status cuda_ok(cudaError_t e) { return e == cudaSuccess ? HSI_OK : HSI_ERR_CUDA; }

std::atomic<uint64_t> g_launches{0};

// Every kernel launch of the library is followed by this check.
hsi_status launch_ok() {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_ok(cudaGetLastError());
}

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous kernel on the stream finishes; it overlaps only its
// input-independent prologue and waits (griddep_wait) before touching memory
// the previous kernels write.
template <typename... KArgs, typename... Args>
hsi_status launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return e == cudaSuccess ? HSI_OK : HSI_ERR_CUDA;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kMaxDevices = 64;

// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device: the attribute is a property of the kernel on one
// device, so a process that drives several GPUs sets it on each. `done` is
// the caller's per-kernel table of devices already set; a race between host
// threads only sets the same value twice.
template <typename Kernel>
hsi_status smem_attr_once(Kernel kernel, int bytes, std::atomic<bool> (&done)[kMaxDevices]) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HSI_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return HSI_ERR_UNSUPPORTED;
    if (done[dev].load(std::memory_order_acquire)) return HSI_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return HSI_ERR_CUDA;
    done[dev].store(true, std::memory_order_release);
    return HSI_OK;
}

// Workspace of the selection passes for B queries of at most max_items items.
// A histogram region: [B][HIST_BINS] counts, then [B] counters of the
// histogram CTAs done (zeroed together).
size_t hist_region_bytes(int32_t B) { return align_up((size_t)B * HIST_BINS * 4 + (size_t)B * 4, 256); }

struct SelWs {
    uint32_t* hist;
    uint32_t* done;
    uint32_t* cnt;  // [B] survivor counts, then [B] threshold bins
    uint32_t* ckey;
    uint32_t* cidx;
    float* bmax;
};

size_t sel_ws_bytes(int32_t B, int64_t max_items, bool need_bmax, int64_t max_blocks, int cap = kCandCap) {
    size_t s = 0;
    if (max_items > SEL_CAP) {
        s += hist_region_bytes(B);
        s += align_up((size_t)B * 8, 256);
        s += 2 * align_up((size_t)B * cap * 4, 256);
    }
    if (need_bmax) s += align_up((size_t)B * (size_t)max_blocks * 4, 256);
    return s;
}

SelWs carve_sel(void* ws, int32_t B, int64_t max_items, bool need_bmax, int64_t max_blocks, int cap = kCandCap) {
    SelWs w{};
    uint8_t* p = static_cast<uint8_t*>(ws);
    if (max_items > SEL_CAP) {
        w.hist = reinterpret_cast<uint32_t*>(p);
        w.done = w.hist + (size_t)B * HIST_BINS;
        p += hist_region_bytes(B);
        w.cnt = reinterpret_cast<uint32_t*>(p);
        p += align_up((size_t)B * 8, 256);
        w.ckey = reinterpret_cast<uint32_t*>(p);
        p += align_up((size_t)B * cap * 4, 256);
        w.cidx = reinterpret_cast<uint32_t*>(p);
        p += align_up((size_t)B * cap * 4, 256);
    }
    if (need_bmax) w.bmax = reinterpret_cast<float*>(p);
    return w;
}

// The selection passes. With hist_ready, sp.hist already holds the key
// histogram (fused into the scoring kernel) and the histogram pass is skipped.
// Zero `bytes` of device memory in stream order: a kernel taking part in the
// programmatic launch chain when the range is 16-byte granular, else a memset.
hsi_status zero_async(void* ptr, size_t bytes, cudaStream_t s) {
    if (bytes == 0) return HSI_OK;
    if ((reinterpret_cast<uintptr_t>(ptr) & 15) == 0 && bytes % 16 == 0) {
        const int64_t n16 = (int64_t)(bytes / 16);
        const int64_t blocks = (n16 + 1023) / 1024;
        return launch(zero_kernel, dim3((unsigned)(blocks < 1024 ? blocks : 1024)), dim3(256), 0, s,
                      reinterpret_cast<uint4*>(ptr), n16);
    }
    return cudaMemsetAsync(ptr, 0, bytes, s) == cudaSuccess ? HSI_OK : HSI_ERR_CUDA;
}

hsi_status run_select(SelParams sp, int64_t max_items, cudaStream_t s, bool hist_ready = false) {
    if (max_items > SEL_CAP) {
        const dim3 grid((unsigned)((max_items + SCAN_CHUNK - 1) / SCAN_CHUNK), (unsigned)sp.B);
        if (!hist_ready) {
            // the histogram pass; its last CTA per query also finds the threshold bin
            sp.done = sp.hist + (size_t)sp.B * HIST_BINS;
            if (zero_async(sp.hist, (size_t)sp.B * (HIST_BINS + 1) * 4, s) != HSI_OK) return HSI_ERR_CUDA;
            if (launch(sel_hist_kernel, dim3(grid), dim3(SCAN_THREADS), 0, s, sp) != HSI_OK)
                return HSI_ERR_CUDA;
        } else {
            sp.done = nullptr;
            if (launch(sel_thresh_kernel, dim3(sp.B), dim3(SCAN_THREADS), 0, s, sp) != HSI_OK)
                return HSI_ERR_CUDA;
        }
        if (sp.blk_max) {  // block-guided: reads the block maxima and the few blocks that reach the bin
            const int64_t nblk = (max_items + 7) / 8;
            const dim3 bgrid((unsigned)((nblk + SCAN_CHUNK - 1) / SCAN_CHUNK), (unsigned)sp.B);
            if (launch(sel_collect_blocks_kernel, bgrid, dim3(SCAN_THREADS), 0, s, sp) != HSI_OK)
                return HSI_ERR_CUDA;
        } else if (launch(sel_collect_kernel, dim3(grid), dim3(SCAN_THREADS), 0, s, sp) != HSI_OK) {
            return HSI_ERR_CUDA;
        }
    }
    if (sp.mode == SEL_POOL && max_items > SEL_CAP) {
        static std::atomic<bool> pool_attr_set[kMaxDevices];
        if (smem_attr_once(pool_final_kernel, (int)sizeof(SelSmem), pool_attr_set) != HSI_OK) return HSI_ERR_CUDA;
        return launch(pool_final_kernel, dim3(sp.B), dim3(SEL_THREADS), sizeof(SelSmem), s, sp);
    }
    if (sp.hist_small && sp.mode == SEL_TOPK && max_items <= SEL_CAP) {
        static std::atomic<bool> small_attr_set[kMaxDevices];
        if (smem_attr_once(sel_small_kernel, (int)sizeof(SelSmem), small_attr_set) != HSI_OK) return HSI_ERR_CUDA;
        return launch(sel_small_kernel, dim3(sp.B), dim3(SEL_THREADS), sizeof(SelSmem), s, sp);
    }
    static std::atomic<bool> attr_set[kMaxDevices];
    if (smem_attr_once(sel_final_kernel, (int)sizeof(SelSmem), attr_set) != HSI_OK) return HSI_ERR_CUDA;
    return launch(sel_final_kernel, dim3(sp.B), dim3(SEL_THREADS), sizeof(SelSmem), s, sp);
}

SelParams topk_params(const float* scores, int64_t ld, const int32_t* n_valid, int64_t max_valid, int32_t B,
                      int32_t k, const int32_t* block_ids, int64_t ld_blocks, int32_t block_size, int32_t* out_idx,
                      float* out_val, const SelWs& wsp) {
    SelParams sp{};
    sp.src = scores;
    sp.ld = ld;
    sp.n_src = n_valid;
    sp.max_src = max_valid;
    sp.div = 1;
    sp.B = B;
    sp.k = k;
    sp.mode = SEL_TOPK;
    sp.hist = wsp.hist;
    sp.cand_cnt = wsp.cnt;
    sp.cand_key = wsp.ckey;
    sp.cand_idx = wsp.cidx;
    sp.thr = wsp.cnt ? wsp.cnt + B : nullptr;
    sp.cap = kCandCap;
    sp.block_ids = block_ids;
    sp.ld_blocks = ld_blocks;
    sp.block_size = block_size;
    sp.out_idx = out_idx;
    sp.out_val = out_val;
    return sp;
}

template <int NQ, bool GATHER, int STAGES, int UT, int FMT>
hsi_status launch_score_fmt(const ScoreParams& p, cudaStream_t s) {
    using C = ScoreCfg<NQ, GATHER, STAGES, UT, FMT>;
    static std::atomic<bool> attr_set[kMaxDevices];
    if (smem_attr_once(score_kernel<NQ, GATHER, STAGES, UT, FMT>, C::SMEM_BYTES, attr_set) != HSI_OK)
        return HSI_ERR_CUDA;
    const int sms = sm_count();
    if (sms <= 0) return HSI_ERR_CUDA;
    return launch(score_kernel<NQ, GATHER, STAGES, UT, FMT>, dim3(sms), dim3(C::THREADS), C::SMEM_BYTES, s, p);
}

// The chunked-prefill scorer (all queries on one cache), cache chunks spread
// over every SM, at most PF_KT_MAX tiles each.
template <int FMT>
hsi_status launch_prefill_fmt(const PrefillParams& p, int64_t max_visible, cudaStream_t s) {
    using C = PfCfg<FMT>;
    const int sms = sm_count();
    if (sms <= 0) return HSI_ERR_CUDA;
    const size_t smem = C::smem_bytes(p.ngroups);
    static std::atomic<bool> attr_set[kMaxDevices];
    if (smem_attr_once(prefill_kernel<FMT>, (int)smem, attr_set) != HSI_OK) return HSI_ERR_CUDA;
    const int64_t ntiles = (max_visible + TILE_KEYS - 1) / TILE_KEYS;
    const int64_t rounds = (ntiles + (int64_t)sms * PF_KT_MAX - 1) / ((int64_t)sms * PF_KT_MAX);
    const int64_t nchunks = (int64_t)sms * (rounds > 0 ? rounds : 1);
    return launch(prefill_kernel<FMT>, dim3(sms), dim3(C::THREADS), smem, s, p, (int)ntiles, (int)nchunks);
}

// The scoring kernel for the records' format (checked by the caller).
template <int NQ, bool GATHER, int STAGES, int UT>
hsi_status launch_score(const ScoreParams& p, hsi_format fmt, cudaStream_t s) {
    if (fmt == HSI_FMT_MXFP4) return launch_score_fmt<NQ, GATHER, STAGES, UT, FMT_MXFP4>(p, s);
    return launch_score_fmt<NQ, GATHER, STAGES, UT, FMT_NVFP4>(p, s);
}

bool format_ok(hsi_format fmt) { return fmt == HSI_FMT_NVFP4 || fmt == HSI_FMT_MXFP4; }
int64_t format_rec_bytes(hsi_format fmt) { return fmt == HSI_FMT_MXFP4 ? 544 : 576; }

// ---- fixed scratch of hsi_topk_noalloc ----------------------------------------
// A caller that cannot allocate device memory still needs somewhere for the
// long-row selection passes to keep their histogram and survivors. This array
// is that place: it lives in the library image, so every GPU that loads the
// library holds it (8 MiB) until the process exits, and every call of
// hsi_topk_noalloc on a device shares it.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
// Survivors of the histogram pass kept per query. It equals the final kernel's
// shared-memory capacity, so a noalloc call never takes the final kernel's
// middle branch (survivors selected in global memory): a query with more
// survivors than this (heavy ties near the k-th key) re-reads its row instead.
constexpr int kNoAllocCandCap = 16384;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// The device address of the scratch on the current device. Host code may not
// pass g_noalloc_scratch itself to a kernel (on the host that name is only a
// stand-in for the symbol); the address is looked up once per device, with the
// device current, and cached.
hsi_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HSI_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return HSI_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return HSI_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return HSI_OK;
}

// Scratch of the Full layer's top-k taken from its pool (scores == NULL): the
// pooled scores [B][8 kPooledTopkMaxKeep] and the key histogram the gathering
// scan fills (the Reindex layer's workspace for 8 kPooledTopkMaxKeep items).
constexpr int32_t kPooledTopkMaxKeep = SEL_CAP / 8;
size_t pooled_topk_ws_bytes(int32_t B) {
    return align_up((size_t)B * SEL_CAP * 4, 256) + sel_ws_bytes(B, SEL_CAP, false, 0) +
           align_up((size_t)B * HIST_BINS * 4, 256);
}

}  // namespace

extern "C" {

const char* hsi_status_string(hsi_status st) {
    switch (st) {
        case HSI_OK: return "ok";
        case HSI_ERR_INVALID_ARG: return "invalid argument";
        case HSI_ERR_UNSUPPORTED: return "unsupported device or shape";
        case HSI_ERR_CUDA: return "CUDA runtime error";
        case HSI_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait ran out";
        case HSI_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case HSI_ERR_DEVICE_ARG: return "a kernel found a malformed device-side argument";
        case HSI_ERR_TOO_LARGE: return "request needs more than the fixed scratch of hsi_topk_noalloc";
    }
    return "unknown status";
}

uint64_t hsi_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

#ifdef HSI_TRACE
// Trace builds only: copy out and clear the wait-cycle counters.
int hsi_trace_read(unsigned long long* out, int n) {
    if (n > TRACE_SLOTS) n = TRACE_SLOTS;
    if (cudaDeviceSynchronize() != cudaSuccess) return HSI_ERR_CUDA;
    if (cudaMemcpyFromSymbol(out, g_hsi_trace, n * sizeof(unsigned long long)) != cudaSuccess) return HSI_ERR_CUDA;
    static const unsigned long long zeros[TRACE_SLOTS] = {};
    if (cudaMemcpyToSymbol(g_hsi_trace, zeros, sizeof(zeros)) != cudaSuccess) return HSI_ERR_CUDA;
    return HSI_OK;
}

int hsi_trace_marks(unsigned long long* out /* [1024][4] */) {
    if (cudaDeviceSynchronize() != cudaSuccess) return HSI_ERR_CUDA;
    if (cudaMemcpyFromSymbol(out, g_hsi_marks, sizeof(g_hsi_marks)) != cudaSuccess) return HSI_ERR_CUDA;
    return HSI_OK;
}
#endif

hsi_status hsi_debug_set(int what, long long value) {
    if (what == HSI_DEBUG_WAIT_LIMIT_NS) {
        if (value <= 0) return HSI_ERR_INVALID_ARG;
        const unsigned long long v = (unsigned long long)value;
        return cuda_ok(cudaMemcpyToSymbol(g_hsi_wait_limit_ns, &v, sizeof(v)));
    }
    if (what == HSI_DEBUG_SKIP_FIRST_COPY) {
        const int v = value != 0;
        return cuda_ok(cudaMemcpyToSymbol(g_hsi_skip_first_copy, &v, sizeof(v)));
    }
    return HSI_ERR_INVALID_ARG;
}

hsi_status hsi_device_check(void) {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HSI_ERR_CUDA;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return HSI_ERR_CUDA;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return HSI_ERR_CUDA;
    return (major == 10 && minor == 3) ? HSI_OK : HSI_ERR_UNSUPPORTED;
}

hsi_status hsi_device_error(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return HSI_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpyFromSymbol(&word, g_hsi_error, sizeof(word)) != cudaSuccess) return HSI_ERR_CUDA;
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_hsi_error, &zero, sizeof(zero)) != cudaSuccess) return HSI_ERR_CUDA;
    if (word & DEVERR_TIMEOUT) return HSI_ERR_DEVICE_TIMEOUT;
    if (word & DEVERR_ARG) return HSI_ERR_DEVICE_ARG;
    return HSI_OK;
}

size_t hsi_workspace_size(hsi_ws_kind kind, int32_t B, int64_t max_n, int32_t k) {
    if (B <= 0 || max_n < 0) return 0;
    switch (kind) {
        case HSI_WS_QUANTIZE: return align_up((size_t)B * 4, 256);
        case HSI_WS_SCORE: return 0;
        case HSI_WS_TOPK: return sel_ws_bytes(B, max_n, false, 0);
        case HSI_WS_FULL_LAYER: {  // the top-k's and the pool's selection buffers, the block maxima (rows padded
                                   // to 16 bytes), and for the top-k from the pool its scores and key histogram
            const int64_t nb = (max_n + 7) / 8;
            return sel_ws_bytes(B, max_n, false, 0) + sel_ws_bytes(B, nb, false, 0) +
                   align_up((size_t)B * align_up((size_t)nb, 4) * 4, 256) + pooled_topk_ws_bytes(B);
        }
        case HSI_WS_PREFILL_LAYER:  // the block maxima, rows padded to 16 bytes
            return align_up((size_t)B * align_up((size_t)((max_n + 7) / 8), 4) * 4, 256);
        case HSI_WS_REINDEX_LAYER:  // + the key histogram the pooled scan accumulates
            return sel_ws_bytes(B, max_n, false, 0) + align_up((size_t)B * HIST_BINS * 4, 256);
        case HSI_WS_POOL: {
            // k is the block size here; block maxima are computed into the
            // workspace when they are not given
            const int64_t bs = k < 1 ? 1 : k;
            const int64_t nb = (max_n + bs - 1) / bs;
            return sel_ws_bytes(B, nb, true, nb);
        }
    }
    return 0;
}

hsi_status hsi_quantize_nvfp4(const uint16_t* x, int64_t n_tensors, int64_t rows_per_tensor, const int8_t* signs,
                              int mode, float* g, uint8_t* rec, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (!x || !signs || !g || !rec || n_tensors <= 0 || rows_per_tensor <= 0) return HSI_ERR_INVALID_ARG;
    if (mode != 0 && mode != 1) return HSI_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(rec, 16) || !aligned(g, 4)) return HSI_ERR_INVALID_ARG;
    QuantParams p{};
    p.x = x;
    p.n_tensors = n_tensors;
    p.rpt = rows_per_tensor;
    p.rec_per_tensor = (rows_per_tensor + 7) / 8;
    for (int d = 0; d < 128; ++d) {
        if (signs[d] != 1 && signs[d] != -1) return HSI_ERR_INVALID_ARG;
        if (signs[d] < 0) p.neg_mask[d >> 5] |= 1u << (d & 31);
    }
    p.g = g;
    p.rec = rec;
    if (mode == 0 && (!ws || ws_bytes < (size_t)n_tensors * 4 || !aligned(ws, 256))) return HSI_ERR_WORKSPACE;
    if (rows_per_tensor <= QUANT_SMALL_ROWS && n_tensors <= INT32_MAX) {
        return launch(quant_small_kernel, dim3((unsigned)n_tensors), dim3(32 * QUANT_SMALL_WARPS), 0, stream, p, mode);
    }
    if (mode == 0) {
        p.amax_bits = static_cast<uint32_t*>(ws);
        if (cudaMemsetAsync(ws, 0, (size_t)n_tensors * 4, stream) != cudaSuccess) return HSI_ERR_CUDA;
        const int64_t rows = n_tensors * rows_per_tensor;
        if (launch(quant_amax_kernel, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, stream, p) != HSI_OK)
            return HSI_ERR_CUDA;
        if (launch(quant_scale_kernel, dim3((unsigned)((n_tensors + 255) / 256)), dim3(256), 0, stream, p) !=
            HSI_OK)
            return HSI_ERR_CUDA;
    }
    const int64_t prows = n_tensors * p.rec_per_tensor * 8;
    return launch(quant_encode_kernel, dim3((unsigned)((prows + 7) / 8)), dim3(256), 0, stream, p);
}

hsi_status hsi_quantize_mxfp4(const uint16_t* x, int64_t n_tensors, int64_t rows_per_tensor, const int8_t* signs,
                              uint8_t* rec, cudaStream_t stream) {
    if (!x || !signs || !rec || n_tensors <= 0 || rows_per_tensor <= 0) return HSI_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(rec, 16)) return HSI_ERR_INVALID_ARG;
    QuantParams p{};
    p.x = x;
    p.n_tensors = n_tensors;
    p.rpt = rows_per_tensor;
    p.rec_per_tensor = (rows_per_tensor + 7) / 8;
    for (int d = 0; d < 128; ++d) {
        if (signs[d] != 1 && signs[d] != -1) return HSI_ERR_INVALID_ARG;
        if (signs[d] < 0) p.neg_mask[d >> 5] |= 1u << (d & 31);
    }
    p.rec = rec;
    const int64_t prows = n_tensors * p.rec_per_tensor * 8;
    if ((prows + 7) / 8 > INT32_MAX) return HSI_ERR_INVALID_ARG;
    return launch(quant_mx_kernel, dim3((unsigned)((prows + 7) / 8)), dim3(256), 0, stream, p);
}

// Pointers every scoring call needs; the tensor scales only for NVFP4.
static hsi_status check_score_common(hsi_format fmt, const uint8_t* q_rec, const float* g_q, const float* w,
                                     const uint8_t* k_rec, const float* g_k, const int64_t* k_rec_off,
                                     const int32_t* n_visible, int32_t B) {
    if (!format_ok(fmt)) return HSI_ERR_INVALID_ARG;
    if (fmt == HSI_FMT_NVFP4 && (!g_q || !g_k)) return HSI_ERR_INVALID_ARG;
    if (!q_rec || !w || !k_rec || !k_rec_off || !n_visible || B <= 0) return HSI_ERR_INVALID_ARG;
    if (!aligned(q_rec, 16) || !aligned(k_rec, 16) || !aligned(w, 16)) return HSI_ERR_INVALID_ARG;
    return HSI_OK;
}

hsi_status hsi_score_full(const uint8_t* q_rec, const float* g_q, const float* w, const uint8_t* k_rec,
                          const float* g_k, const int64_t* k_rec_off, const int32_t* n_visible, int32_t B,
                          int64_t max_visible, int32_t group, float* scores, int64_t ld, float* block_max,
                          int64_t ldb, hsi_format format, void* ws, size_t ws_bytes, cudaStream_t stream) {
    (void)ws;
    (void)ws_bytes;
    hsi_status st = check_score_common(format, q_rec, g_q, w, k_rec, g_k, k_rec_off, n_visible, B);
    if (st != HSI_OK) return st;
    if ((!scores && !block_max) || max_visible < 0 || max_visible > (int64_t)INT32_MAX - 128 ||
        (scores && ld < max_visible))
        return HSI_ERR_INVALID_ARG;
    if (block_max && ldb < (max_visible + 7) / 8) return HSI_ERR_INVALID_ARG;
    if (group != 1 && group != 4) return HSI_ERR_UNSUPPORTED;
    if (B % group) return HSI_ERR_INVALID_ARG;
    ScoreParams p{};
    p.q_rec = q_rec;
    p.g_q = g_q;
    p.w = w;
    p.k_rec = k_rec;
    p.g_k = g_k;
    p.k_off = k_rec_off;
    p.n_vis = n_visible;
    p.max_vis = (int32_t)max_visible;
    p.B = B;
    p.ngroups = B / group;
    p.scores = scores;
    p.ld = ld;
    p.bmax = block_max;
    p.ldb = ldb;
    if (group == 1) return launch_score<1, false, kDecodeStages, kDecodeUT>(p, format, stream);
    return launch_score<4, false, kPrefillStages, kPrefillUT>(p, format, stream);
}

hsi_status hsi_score_pool(const uint8_t* q_rec, const float* g_q, const float* w, const uint8_t* k_rec,
                          const float* g_k, const int64_t* k_rec_off, const int32_t* n_visible,
                          const int32_t* block_ids, const int32_t* n_kept, int32_t n_keep, int32_t B,
                          float* pool_scores, int64_t ld, hsi_format format, void* ws, size_t ws_bytes,
                          cudaStream_t stream) {
    (void)ws;
    (void)ws_bytes;
    hsi_status st = check_score_common(format, q_rec, g_q, w, k_rec, g_k, k_rec_off, n_visible, B);
    if (st != HSI_OK) return st;
    if (!block_ids || !n_kept || !pool_scores || n_keep <= 0 || n_keep > (1 << 20) || n_keep % (16 * kGatherUT) ||
        ld < (int64_t)n_keep * 8 || !aligned(block_ids, 16))
        return HSI_ERR_INVALID_ARG;
    ScoreParams p{};
    p.q_rec = q_rec;
    p.g_q = g_q;
    p.w = w;
    p.k_rec = k_rec;
    p.g_k = g_k;
    p.k_off = k_rec_off;
    p.n_vis = n_visible;
    p.max_vis = INT32_MAX;  // gathered ids are checked against ceil(n_vis / 8) records
    p.B = B;
    p.ngroups = B;
    p.block_ids = block_ids;
    p.n_kept = n_kept;
    p.n_keep = n_keep;
    p.pool_scores = pool_scores;
    p.ld_pool = ld;
    return launch_score<1, true, kGatherStages, kGatherUT>(p, format, stream);
}

hsi_status hsi_topk(const float* scores, int64_t ld, const int32_t* n_valid, int32_t B, int64_t max_valid, int32_t k,
                    const int32_t* block_ids, int64_t ld_blocks, int32_t block_size, int32_t* out_idx,
                    float* out_val, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (!scores || !n_valid || !out_idx || !out_val || B <= 0 || max_valid < 0 || ld < max_valid)
        return HSI_ERR_INVALID_ARG;
    if (max_valid > (int64_t)INT32_MAX) return HSI_ERR_INVALID_ARG;
    if (k < 1 || k > 2048) return HSI_ERR_INVALID_ARG;
    if (block_ids && (block_size < 1 || ld_blocks < (max_valid + block_size - 1) / block_size))
        return HSI_ERR_INVALID_ARG;
    const size_t need = sel_ws_bytes(B, max_valid, false, 0);
    if (need && (!ws || ws_bytes < need || !aligned(ws, 256))) return HSI_ERR_WORKSPACE;
    SelWs wsp = carve_sel(ws, B, max_valid, false, 0);
    const SelParams sp =
        topk_params(scores, ld, n_valid, max_valid, B, k, block_ids, ld_blocks, block_size, out_idx, out_val, wsp);
    return run_select(sp, max_valid, stream);
}

hsi_status hsi_topk_noalloc(const float* scores, int64_t ld, const int32_t* n_valid, int32_t B, int64_t max_valid,
                            int32_t k, const int32_t* block_ids, int64_t ld_blocks, int32_t block_size,
                            int32_t* out_idx, float* out_val, cudaStream_t stream) {
    if (!scores || !n_valid || !out_idx || !out_val || B <= 0 || max_valid < 0 || ld < max_valid)
        return HSI_ERR_INVALID_ARG;
    if (max_valid > (int64_t)INT32_MAX) return HSI_ERR_INVALID_ARG;
    if (k < 1 || k > 2048) return HSI_ERR_INVALID_ARG;
    if (block_ids && (block_size < 1 || ld_blocks < (max_valid + block_size - 1) / block_size))
        return HSI_ERR_INVALID_ARG;
    const size_t need = sel_ws_bytes(B, max_valid, false, 0, kNoAllocCandCap);
    if (need > kNoAllocScratchBytes) return HSI_ERR_TOO_LARGE;
    void* ws = nullptr;
    if (need) {
        const hsi_status st = noalloc_scratch(&ws);
        if (st != HSI_OK) return st;
    }
    SelWs wsp = carve_sel(ws, B, max_valid, false, 0, kNoAllocCandCap);
    SelParams sp{};
    sp.src = scores;
    sp.ld = ld;
    sp.n_src = n_valid;
    sp.max_src = max_valid;
    sp.div = 1;
    sp.B = B;
    sp.k = k;
    sp.mode = SEL_TOPK;
    sp.hist = wsp.hist;
    sp.cand_cnt = wsp.cnt;
    sp.cand_key = wsp.ckey;
    sp.cand_idx = wsp.cidx;
    sp.thr = wsp.cnt ? wsp.cnt + B : nullptr;
    sp.cap = kNoAllocCandCap;
    sp.block_ids = block_ids;
    sp.ld_blocks = ld_blocks;
    sp.block_size = block_size;
    sp.out_idx = out_idx;
    sp.out_val = out_val;
    return run_select(sp, max_valid, stream);  // clears the histogram and counters first
}

hsi_status hsi_candidate_pool(const float* scores, int64_t ld, const float* block_max, int64_t ldb,
                              const int32_t* n_visible, int32_t B, int64_t max_visible, int32_t block_size,
                              int32_t n_keep, int32_t* block_ids, int32_t* n_kept, int32_t* n_pool,
                              uint32_t* pool_bits, int64_t ld_bits, void* ws, size_t ws_bytes,
                              cudaStream_t stream) {
    if (!n_visible || !block_ids || !n_kept || !n_pool || B <= 0 || max_visible < 0) return HSI_ERR_INVALID_ARG;
    if (max_visible > (int64_t)INT32_MAX) return HSI_ERR_INVALID_ARG;
    if (block_size < 1 || block_size > 64 || n_keep < 1 || n_keep > SEL_MAXK) return HSI_ERR_INVALID_ARG;
    const int64_t max_blocks = (max_visible + block_size - 1) / block_size;
    if (block_max) {
        if (block_size != 8 || ldb < max_blocks) return HSI_ERR_INVALID_ARG;
    } else {
        if (!scores || ld < max_visible) return HSI_ERR_INVALID_ARG;
    }
    if (pool_bits && ld_bits < (max_visible + 31) / 32) return HSI_ERR_INVALID_ARG;
    const bool need_bmax = block_max == nullptr;
    const size_t need = sel_ws_bytes(B, max_blocks, need_bmax, max_blocks);
    if (need && (!ws || ws_bytes < need || !aligned(ws, 256))) return HSI_ERR_WORKSPACE;
    SelWs wsp = carve_sel(ws, B, max_blocks, need_bmax, max_blocks);
    const float* bm = block_max;
    int64_t bld = ldb;
    if (need_bmax) {
        const dim3 grid((unsigned)((max_blocks + 255) / 256 > 0 ? (max_blocks + 255) / 256 : 1), (unsigned)B);
        if (launch(block_max_kernel, dim3(grid), dim3(256), 0, stream, scores, ld, n_visible, max_visible, block_size,
                   wsp.bmax, max_blocks) != HSI_OK)
            return HSI_ERR_CUDA;
        bm = wsp.bmax;
        bld = max_blocks;
    }
    SelParams sp{};
    sp.src = bm;
    sp.ld = bld;
    sp.n_src = n_visible;
    sp.max_src = max_visible;
    sp.div = block_size;
    sp.B = B;
    sp.k = n_keep;
    sp.mode = SEL_POOL;
    sp.hist = wsp.hist;
    sp.cand_cnt = wsp.cnt;
    sp.cand_key = wsp.ckey;
    sp.cand_idx = wsp.cidx;
    sp.thr = wsp.cnt ? wsp.cnt + B : nullptr;
    sp.cap = kCandCap;
    sp.blk_out = block_ids;
    sp.n_kept = n_kept;
    sp.n_pool = n_pool;
    sp.bits = pool_bits;
    sp.ld_bits = ld_bits;
    return run_select(sp, max_blocks, stream);
}

hsi_status hsi_mask_scores(float* scores, int64_t ld, const int32_t* n_visible, const uint32_t* bits, int64_t ld_bits,
                           int32_t B, int64_t max_visible, cudaStream_t stream) {
    if (!scores || !n_visible || !bits || B <= 0 || B > 65535 || max_visible < 0 || ld < max_visible ||
        ld_bits < (max_visible + 31) / 32)
        return HSI_ERR_INVALID_ARG;
    if (max_visible == 0) return HSI_OK;
    const dim3 grid((unsigned)((max_visible + 255) / 256), (unsigned)B);
    return launch(mask_scores_kernel, grid, dim3(256), 0, stream, scores, ld, n_visible, max_visible, bits, ld_bits);
}

hsi_status hsi_calib_read(const void* buf, size_t bytes, int method, int chunk, int stages,
                          unsigned long long* sink, cudaStream_t stream) {
    if (!buf || !sink || bytes < 16 || !aligned(buf, 16)) return HSI_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms <= 0) return HSI_ERR_CUDA;
    if (method == 0) {
        return launch(calib_read_ldg_kernel, dim3(sms * 4), dim3(512), 0, stream, static_cast<const uint4*>(buf),
                      bytes / 16, sink);
    }
    if (method != 1 || chunk < 16 || chunk % 16 || stages < 1) return HSI_ERR_INVALID_ARG;
    const size_t smem = (size_t)stages * chunk + 2 * (size_t)stages * 8 + 1024;
    if (smem > 227 * 1024 || (size_t)chunk * sms > bytes) return HSI_ERR_INVALID_ARG;
    if (cudaFuncSetAttribute(calib_read_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return HSI_ERR_CUDA;
    return launch(calib_read_bulk_kernel, dim3(sms), dim3(64), smem, stream, static_cast<const uint8_t*>(buf), bytes,
                  chunk, stages, sink);
}

hsi_status hsi_calib_mma(int n, int iters, unsigned long long* sink, cudaStream_t stream) {
    if (!sink || iters < 1) return HSI_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms <= 0) return HSI_ERR_CUDA;
    switch (n) {
        case 32: calib_mma_kernel<32><<<sms, 128, 0, stream>>>(iters, sink); break;
        case 64: calib_mma_kernel<64><<<sms, 128, 0, stream>>>(iters, sink); break;
        case 128: calib_mma_kernel<128><<<sms, 128, 0, stream>>>(iters, sink); break;
        case 256: calib_mma_kernel<256><<<sms, 128, 0, stream>>>(iters, sink); break;
        default: return HSI_ERR_UNSUPPORTED;
    }
    return launch_ok();
}

hsi_status hsi_full_layer(const uint8_t* q_rec, const float* g_q, const float* w, const uint8_t* k_rec,
                          const float* g_k, const int64_t* k_rec_off, const int32_t* n_visible, int32_t B,
                          int64_t max_visible, float* scores, int64_t ld, int32_t k, int32_t* top_idx,
                          float* top_val, int32_t n_keep, int32_t* block_ids, int32_t* n_kept, int32_t* n_pool,
                          uint32_t* pool_bits, int64_t ld_bits, int32_t phases, hsi_format format, void* ws,
                          size_t ws_bytes, cudaStream_t stream) {
    if (phases != HSI_PHASE_SCORE && phases != HSI_PHASE_SELECT && phases != HSI_PHASE_ALL &&
        phases != HSI_PHASE_TOPK && phases != HSI_PHASE_POOL)
        return HSI_ERR_INVALID_ARG;
    hsi_status st = check_score_common(format, q_rec, g_q, w, k_rec, g_k, k_rec_off, n_visible, B);
    if (st != HSI_OK) return st;
    if (!top_idx || !top_val || max_visible < 0 || max_visible > (int64_t)INT32_MAX - 256 ||
        (scores && ld < max_visible) || k < 1 || k > 2048)
        return HSI_ERR_INVALID_ARG;
    const bool pool = block_ids != nullptr;
    if (pool && (!n_kept || !n_pool || n_keep < 1 || n_keep > SEL_MAXK)) return HSI_ERR_INVALID_ARG;
    // without scores the top-k comes from the pool: its n_keep - 1 unpinned
    // blocks hold the first k blocks by maximum, so the top-k lies in the pool
    const bool pooled_topk = scores == nullptr;
    if (pooled_topk && (!pool || n_keep - 1 < k)) return HSI_ERR_INVALID_ARG;
    if (pooled_topk && (n_keep > kPooledTopkMaxKeep || n_keep % (16 * kGatherUT))) return HSI_ERR_UNSUPPORTED;
    if (phases == HSI_PHASE_POOL && !pool) return HSI_ERR_INVALID_ARG;
    if (pool_bits && ld_bits < (max_visible + 31) / 32) return HSI_ERR_INVALID_ARG;
    const int64_t nb = (max_visible + 7) / 8;
    const int64_t ldb = (nb + 3) & ~(int64_t)3;  // rows of block maxima start on 16-byte boundaries
    const size_t need = hsi_workspace_size(HSI_WS_FULL_LAYER, B, max_visible, k);
    if (!ws || ws_bytes < need || !aligned(ws, 256)) return HSI_ERR_WORKSPACE;
    // workspace: the top-k's selection buffers, the pool's (separate, so that the
    // two selections may run at the same time on two streams), the block maxima
    SelWs wsp = carve_sel(ws, B, max_visible, false, 0);
    uint8_t* wpool = static_cast<uint8_t*>(ws) + sel_ws_bytes(B, max_visible, false, 0);
    SelWs wpp = carve_sel(wpool, B, nb, false, 0);
    float* bmax = reinterpret_cast<float*>(wpool + sel_ws_bytes(B, nb, false, 0));
    const bool big_topk = max_visible > SEL_CAP && !pooled_topk;  // the top-k's selection over the scores
    if (phases & 1) {
    // the pool's threshold comes from a histogram of the block maxima the scan
    // fills, like the top-k's from the scores' (rows past SEL_CAP blocks)
    const bool bmax_hist = pool && nb > SEL_CAP;
    if (big_topk && zero_async(wsp.hist, (size_t)B * HIST_BINS * 4, stream) != HSI_OK) return HSI_ERR_CUDA;
    if (bmax_hist && zero_async(wpp.hist, (size_t)B * HIST_BINS * 4, stream) != HSI_OK) return HSI_ERR_CUDA;
    ScoreParams p{};
    p.q_rec = q_rec;
    p.g_q = g_q;
    p.w = w;
    p.k_rec = k_rec;
    p.g_k = g_k;
    p.k_off = k_rec_off;
    p.n_vis = n_visible;
    p.max_vis = (int32_t)max_visible;
    p.B = B;
    p.ngroups = B;
    p.scores = scores;
    p.ld = ld;
    // block maxima: for the pool, and for the top-k's collect pass (it reads the
    // scores of the blocks whose maximum reaches the threshold bin only)
    p.bmax = pool || big_topk ? bmax : nullptr;  // scores == NULL: block maxima only
    p.ldb = ldb;
    p.key_hist = big_topk ? wsp.hist : nullptr;
    p.bmax_hist = bmax_hist ? wpp.hist : nullptr;
    st = launch_score<1, false, kDecodeStages, kDecodeUT>(p, format, stream);
    if (st != HSI_OK) return st;
    }
    const bool do_topk = phases == HSI_PHASE_ALL || phases == HSI_PHASE_SELECT || phases == HSI_PHASE_TOPK;
    const bool do_pool = pool && (phases == HSI_PHASE_ALL || phases == HSI_PHASE_SELECT || phases == HSI_PHASE_POOL);
    if (do_topk && pooled_topk) {
        // the pool's records re-scored with this layer's query (the same fp32
        // scores as the full scan's), its top-k mapped back to positions
        uint8_t* wt = reinterpret_cast<uint8_t*>(bmax) + align_up((size_t)B * ldb * 4, 256);
        float* pscores = reinterpret_cast<float*>(wt);
        uint8_t* rws = wt + align_up((size_t)B * SEL_CAP * 4, 256);
        const size_t rws_bytes = pooled_topk_ws_bytes(B) - align_up((size_t)B * SEL_CAP * 4, 256);
        if (phases == HSI_PHASE_ALL || phases == HSI_PHASE_SELECT) {  // the pool first
            st = hsi_full_layer(q_rec, g_q, w, k_rec, g_k, k_rec_off, n_visible, B, max_visible, scores, ld, k,
                                top_idx, top_val, n_keep, block_ids, n_kept, n_pool, pool_bits, ld_bits,
                                HSI_PHASE_POOL, format, ws, ws_bytes, stream);
            if (st != HSI_OK) return st;
        }
        return hsi_reindex_layer(q_rec, g_q, w, k_rec, g_k, k_rec_off, nullptr, 0, n_visible, block_ids, n_kept,
                                 n_pool, n_keep, B, pscores, (int64_t)n_keep * 8, k, top_idx, top_val, format, rws,
                                 rws_bytes, stream);
    }
    if (do_topk) {
    SelParams sp{};
    sp.src = scores;
    sp.ld = ld;
    sp.n_src = n_visible;
    sp.max_src = max_visible;
    sp.div = 1;
    sp.B = B;
    sp.k = k;
    sp.mode = SEL_TOPK;
    sp.hist = wsp.hist;
    sp.cand_cnt = wsp.cnt;
    sp.cand_key = wsp.ckey;
    sp.cand_idx = wsp.cidx;
    sp.thr = wsp.cnt ? wsp.cnt + B : nullptr;
    sp.cap = kCandCap;
    sp.out_idx = top_idx;
    sp.out_val = top_val;
    if (big_topk) {
        sp.blk_max = bmax;
        sp.ld_bmax = ldb;
    }
    st = run_select(sp, max_visible, stream, true);
    if (st != HSI_OK) return st;
    }
    if (!do_pool) return HSI_OK;
    SelParams pp{};
    pp.src = bmax;
    pp.ld = ldb;
    pp.n_src = n_visible;
    pp.max_src = max_visible;
    pp.div = 8;
    pp.B = B;
    pp.k = n_keep;
    pp.mode = SEL_POOL;
    pp.hist = wpp.hist;
    pp.cand_cnt = wpp.cnt;
    pp.cand_key = wpp.ckey;
    pp.cand_idx = wpp.cidx;
    pp.thr = wpp.cnt ? wpp.cnt + B : nullptr;
    pp.cap = kCandCap;
    pp.blk_out = block_ids;
    pp.n_kept = n_kept;
    pp.n_pool = n_pool;
    pp.bits = pool_bits;
    pp.ld_bits = ld_bits;
    // rows past SEL_CAP blocks: the histogram of the block maxima comes from the
    // scoring phase (its pinned block counted at its own maximum, one bin too
    // low at most: the threshold bin can only drop, the candidates still hold
    // the pool); shorter rows are selected in shared memory whole
    return run_select(pp, nb, stream, nb > SEL_CAP);
}

hsi_status hsi_prefill_layer(const uint8_t* q_rec, const float* g_q, const float* w, const uint8_t* k_rec,
                             const float* g_k, const int64_t* k_rec_off, const int32_t* n_visible, int32_t B,
                             int64_t max_visible, int32_t group, float* scores, int64_t ld, int32_t k,
                             int32_t* top_idx, float* top_val, int32_t n_keep, int32_t* block_ids, int32_t* n_kept,
                             int32_t* n_pool, uint32_t* pool_bits, int64_t ld_bits, int32_t phases,
                             hsi_format format, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (phases != HSI_PHASE_SCORE && phases != HSI_PHASE_SELECT && phases != HSI_PHASE_ALL)
        return HSI_ERR_INVALID_ARG;
    hsi_status st = check_score_common(format, q_rec, g_q, w, k_rec, g_k, k_rec_off, n_visible, B);
    if (st != HSI_OK) return st;
    if (!scores || !top_idx || !top_val || max_visible < 0 || ld < max_visible || k < 1 || k > RS_MAXK)
        return HSI_ERR_INVALID_ARG;
    if (max_visible > (int64_t)RS_MAX_BLOCKS * 8) return HSI_ERR_UNSUPPORTED;
    if (group != 1 && group != 4) return HSI_ERR_UNSUPPORTED;
    if (B % group) return HSI_ERR_INVALID_ARG;
    if (group == 4) {  // the queries' tensor scales are copied 16 bytes at a time with their records
        if (B / 4 > PF_MAX_GROUPS) return HSI_ERR_UNSUPPORTED;
        if (format == HSI_FMT_NVFP4 && (!aligned(g_q, 16) || !aligned(g_k, 16))) return HSI_ERR_INVALID_ARG;
    }
    const bool pool = block_ids != nullptr;
    if (pool && (!n_kept || !n_pool || n_keep < 1 || n_keep > SEL_MAXK)) return HSI_ERR_INVALID_ARG;
    if (pool_bits && ld_bits < (max_visible + 31) / 32) return HSI_ERR_INVALID_ARG;
    const int64_t nb = (int64_t)align_up((size_t)((max_visible + 7) / 8), 4);  // rows of block maxima, 16-byte aligned
    const size_t need = hsi_workspace_size(HSI_WS_PREFILL_LAYER, B, max_visible, k);
    if (!ws || ws_bytes < need || !aligned(ws, 256)) return HSI_ERR_WORKSPACE;
    float* bmax = static_cast<float*>(ws);
    if (phases & HSI_PHASE_SCORE) {
        ScoreParams p{};
        p.q_rec = q_rec;
        p.g_q = g_q;
        p.w = w;
        p.k_rec = k_rec;
        p.g_k = g_k;
        p.k_off = k_rec_off;
        p.n_vis = n_visible;
        p.max_vis = (int32_t)max_visible;
        p.B = B;
        p.ngroups = B / group;
        p.scores = scores;
        p.ld = ld;
        p.bmax = bmax;
        p.ldb = nb;
        if (group == 1) {
            st = launch_score<1, false, kDecodeStages, kDecodeUT>(p, format, stream);
        } else {
            PrefillParams pp{};
            pp.q_rec = q_rec;
            pp.g_q = g_q;
            pp.w = w;
            pp.k_rec = k_rec;
            pp.g_k = g_k;
            pp.k_off = k_rec_off;
            pp.n_vis = n_visible;
            pp.max_vis = (int32_t)max_visible;
            pp.B = B;
            pp.ngroups = B / 4;
            pp.scores = scores;
            pp.ld = ld;
            pp.bmax = bmax;
            pp.ldb = nb;
            st = format == HSI_FMT_MXFP4 ? launch_prefill_fmt<FMT_MXFP4>(pp, max_visible, stream)
                                         : launch_prefill_fmt<FMT_NVFP4>(pp, max_visible, stream);
        }
        if (st != HSI_OK) return st;
    }
    if (!(phases & HSI_PHASE_SELECT)) return HSI_OK;
    RowSelParams rp{};
    rp.bmax = bmax;
    rp.ldb = nb;
    rp.scores = scores;
    rp.ld = ld;
    rp.n_vis = n_visible;
    rp.max_vis = max_visible;
    rp.B = B;
    rp.k = k;
    rp.out_idx = top_idx;
    rp.out_val = top_val;
    rp.n_keep = pool ? n_keep : 0;
    rp.blk_out = block_ids;
    rp.n_kept = n_kept;
    rp.n_pool = n_pool;
    rp.bits = pool_bits;
    rp.ld_bits = ld_bits;
    static std::atomic<bool> attr_set[kMaxDevices];
    if (smem_attr_once(rowsel_kernel, (int)sizeof(RowSelSmem), attr_set) != HSI_OK) return HSI_ERR_CUDA;
    return launch(rowsel_kernel, dim3((unsigned)B), dim3(RS_THREADS), sizeof(RowSelSmem), stream, rp);
}

hsi_status hsi_quantize_mainkv(const uint16_t* x, int64_t n, uint8_t* kv, cudaStream_t stream) {
    if (!x || !kv || n <= 0 || !aligned(x, 16) || !aligned(kv, 16)) return HSI_ERR_INVALID_ARG;
    if ((n + 7) / 8 > INT32_MAX) return HSI_ERR_INVALID_ARG;
    return launch(mainkv_quant_kernel, dim3((unsigned)((n + 7) / 8)), dim3(256), 0, stream, x, n, kv);
}

hsi_status hsi_gather_mainkv_layers(const uint8_t* kv, const int64_t* kv_off, const int32_t* n_visible,
                                    const int32_t* idx, int64_t ld_idx, int64_t idx_stride, int32_t L, int32_t k,
                                    int32_t B, uint16_t* out, int64_t out_stride, cudaStream_t stream) {
    if (!kv || !kv_off || !n_visible || !idx || !out || B <= 0 || L <= 0 || k < 1 || k > 4096 || ld_idx < k)
        return HSI_ERR_INVALID_ARG;
    if (L > 1 && (idx_stride < (int64_t)B * ld_idx || out_stride < (int64_t)B * k * HSI_KV_DIM || out_stride % 8))
        return HSI_ERR_INVALID_ARG;
    if (!aligned(kv, 16) || !aligned(out, 16)) return HSI_ERR_INVALID_ARG;
    const int64_t warps = ((int64_t)L * B * k + GATHER_EPW - 1) / GATHER_EPW;
    if ((warps + 7) / 8 > INT32_MAX) return HSI_ERR_INVALID_ARG;
    return launch(mainkv_gather_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, stream, kv, kv_off,
                  n_visible, idx, ld_idx, idx_stride, L, k, B, out, out_stride);
}

hsi_status hsi_gather_mainkv(const uint8_t* kv, const int64_t* kv_off, const int32_t* n_visible, const int32_t* idx,
                             int64_t ld_idx, int32_t k, int32_t B, uint16_t* out, cudaStream_t stream) {
    return hsi_gather_mainkv_layers(kv, kv_off, n_visible, idx, ld_idx, 0, 1, k, B, out, 0, stream);
}

hsi_status hsi_append_token(const uint16_t* k_x, const int8_t* signs, const float* g_k, uint8_t* k_rec,
                            const int64_t* k_rec_off, const uint16_t* kv_x, uint8_t* kv, const int64_t* kv_off,
                            int32_t* n_visible, const int32_t* capacity, int32_t B, hsi_format format,
                            cudaStream_t stream) {
    if (!k_x || !signs || !k_rec || !k_rec_off || !n_visible || !capacity || B <= 0 || !format_ok(format))
        return HSI_ERR_INVALID_ARG;
    if (format == HSI_FMT_NVFP4 && !g_k) return HSI_ERR_INVALID_ARG;
    if (kv_x && (!kv || !kv_off)) return HSI_ERR_INVALID_ARG;
    if (!aligned(k_x, 16) || !aligned(k_rec, 16) || (kv_x && (!aligned(kv_x, 16) || !aligned(kv, 16))))
        return HSI_ERR_INVALID_ARG;
    AppendParams p{};
    p.q.x = k_x;
    p.q.n_tensors = B;
    p.q.rpt = 1;
    p.q.rec_per_tensor = 1;
    for (int d = 0; d < 128; ++d) {
        if (signs[d] != 1 && signs[d] != -1) return HSI_ERR_INVALID_ARG;
        if (signs[d] < 0) p.q.neg_mask[d >> 5] |= 1u << (d & 31);
    }
    p.g_k = g_k;
    p.k_rec = k_rec;
    p.k_off = k_rec_off;
    p.kv_x = kv_x;
    p.kv = kv;
    p.kv_off = kv_off;
    p.n_vis = n_visible;
    p.capacity = capacity;
    p.mx = format == HSI_FMT_MXFP4;
    return launch(append_token_kernel, dim3((unsigned)B), dim3(64), 0, stream, p);
}

hsi_status hsi_pool_gather(const uint8_t* k_rec, const int64_t* k_rec_off, const int32_t* n_visible,
                           const int32_t* block_ids, const int32_t* n_kept, int32_t n_keep, int32_t B,
                           uint8_t* pool_rec, hsi_format format, cudaStream_t stream) {
    if (!k_rec || !k_rec_off || !n_visible || !block_ids || !n_kept || !pool_rec || B <= 0 || B > 65535 ||
        n_keep <= 0 || n_keep > (1 << 20) || pool_rec == k_rec || !format_ok(format))
        return HSI_ERR_INVALID_ARG;
    if (!aligned(k_rec, 16) || !aligned(pool_rec, 16)) return HSI_ERR_INVALID_ARG;
    const int rec_chunks = (int)(format_rec_bytes(format) / 16);
    const int64_t chunks = (int64_t)n_keep * rec_chunks;
    const dim3 grid((unsigned)((chunks + GATHER_THREADS * GATHER_PER_THREAD - 1) / (GATHER_THREADS * GATHER_PER_THREAD)),
                    (unsigned)B);
    return launch(pool_gather_kernel, grid, dim3(GATHER_THREADS), 0, stream, reinterpret_cast<const uint4*>(k_rec),
                  k_rec_off, n_visible, block_ids, n_kept, n_keep, rec_chunks, reinterpret_cast<uint4*>(pool_rec));
}

hsi_status hsi_reindex_layer(const uint8_t* q_rec, const float* g_q, const float* w, const uint8_t* k_rec,
                             const float* g_k, const int64_t* k_rec_off, uint8_t* pool_rec, int32_t pool_rec_ready,
                             const int32_t* n_visible, const int32_t* block_ids, const int32_t* n_kept,
                             const int32_t* n_pool, int32_t n_keep, int32_t B, float* pool_scores, int64_t ld,
                             int32_t k, int32_t* top_idx, float* top_val, hsi_format format, void* ws,
                             size_t ws_bytes, cudaStream_t stream) {
    if (!n_pool || !format_ok(format)) return HSI_ERR_INVALID_ARG;
    hsi_status st;
    if (!pool_rec || !pool_rec_ready) {
        // gather from k_rec (and, with pool_rec, leave the compacted pool there)
        st = check_score_common(format, q_rec, g_q, w, k_rec, g_k, k_rec_off, n_visible, B);
        if (st != HSI_OK) return st;
        if (!block_ids || !n_kept || !pool_scores || n_keep <= 0 || n_keep > (1 << 20) ||
            n_keep % (16 * kGatherUT) || ld < (int64_t)n_keep * 8 || !aligned(block_ids, 16))
            return HSI_ERR_INVALID_ARG;
        if (pool_rec && (!aligned(pool_rec, 16) || pool_rec == k_rec)) return HSI_ERR_INVALID_ARG;
        if (!top_idx || !top_val || k < 1 || k > 2048) return HSI_ERR_INVALID_ARG;
        const int64_t max_valid = (int64_t)n_keep * 8;
        const size_t need = hsi_workspace_size(HSI_WS_REINDEX_LAYER, B, max_valid, k);
        if (!ws || ws_bytes < need || !aligned(ws, 256)) return HSI_ERR_WORKSPACE;
        SelWs wsp = carve_sel(ws, B, max_valid, false, 0);
        uint32_t* hist = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + sel_ws_bytes(B, max_valid, false, 0));
        if (zero_async(hist, (size_t)B * HIST_BINS * 4, stream) != HSI_OK) return HSI_ERR_CUDA;
        ScoreParams p{};
        p.q_rec = q_rec;
        p.g_q = g_q;
        p.w = w;
        p.k_rec = k_rec;
        p.g_k = g_k;
        p.k_off = k_rec_off;
        p.n_vis = n_visible;
        p.max_vis = INT32_MAX;  // gathered ids are checked against ceil(n_vis / 8) records
        p.B = B;
        p.ngroups = B;
        p.block_ids = block_ids;
        p.n_kept = n_kept;
        p.n_keep = n_keep;
        p.pool_scores = pool_scores;
        p.ld_pool = ld;
        p.key_hist = hist;
        p.pool_out = pool_rec;
        st = launch_score<1, true, kGatherStages, kGatherUT>(p, format, stream);
        if (st != HSI_OK) return st;
        SelParams sp =
            topk_params(pool_scores, ld, n_pool, max_valid, B, k, block_ids, n_keep, 8, top_idx, top_val, wsp);
        sp.hist = hist;
        sp.hist_small = 1;
        return run_select(sp, max_valid, stream, true);
    } else {
        // the compacted pool is a contiguous scan: query b's keys are its pool
        // slots (n_pool[b] of them visible, the newest block last), its records
        // n_keep apart; slots up to 8 n_kept[b] past the visible ones get -inf
        if (!q_rec || !w || !block_ids || !n_kept || B <= 0 || n_keep <= 0 || n_keep > (1 << 20) ||
            !pool_scores || ld < (int64_t)n_keep * 8)
            return HSI_ERR_INVALID_ARG;
        if (format == HSI_FMT_NVFP4 && (!g_q || !g_k)) return HSI_ERR_INVALID_ARG;
        if (!aligned(q_rec, 16) || !aligned(pool_rec, 16) || !aligned(w, 16)) return HSI_ERR_INVALID_ARG;
        if (!top_idx || !top_val || k < 1 || k > 2048) return HSI_ERR_INVALID_ARG;
        const int64_t max_valid = (int64_t)n_keep * 8;
        const size_t need = hsi_workspace_size(HSI_WS_REINDEX_LAYER, B, max_valid, k);
        if (!ws || ws_bytes < need || !aligned(ws, 256)) return HSI_ERR_WORKSPACE;
        // the scan accumulates the key histogram that the selection starts from
        SelWs wsp = carve_sel(ws, B, max_valid, false, 0);
        uint32_t* hist = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + sel_ws_bytes(B, max_valid, false, 0));
        if (zero_async(hist, (size_t)B * HIST_BINS * 4, stream) != HSI_OK) return HSI_ERR_CUDA;
        ScoreParams p{};
        p.q_rec = q_rec;
        p.g_q = g_q;
        p.w = w;
        p.k_rec = pool_rec;
        p.g_k = g_k;
        p.k_off = nullptr;
        p.k_stride = n_keep;
        p.n_vis = n_pool;
        p.max_vis = (int32_t)max_valid;  // slots of the compacted pool
        p.B = B;
        p.ngroups = B;
        p.scores = pool_scores;
        p.ld = ld;
        p.pad_blocks = n_kept;
        p.n_keep = n_keep;
        p.key_hist = hist;
        st = launch_score<1, false, kPooledStages, kPooledUT>(p, format, stream);
        if (st != HSI_OK) return st;
        SelParams sp =
            topk_params(pool_scores, ld, n_pool, max_valid, B, k, block_ids, n_keep, 8, top_idx, top_val, wsp);
        sp.hist = hist;
        sp.hist_small = 1;
        return run_select(sp, max_valid, stream, true);
    }
}

}  // extern "C"
