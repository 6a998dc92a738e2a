/*
 * libhsi -- the decode-time hot path of DeepSeek-V4.1's Hierarchical Sparse
 * Indexer on one GB300 (sm_103a).
 *
 * The method (sources are the pages' titles and sections):
 *  - Lightning-indexer score, "DeepSeek-V4.1 模型结构（3）：序列维度（下），
 *    Hierarchical Sparse Indexer 与 FP4 KV cache", section "Reindex 层每个 token
 *    要给 100 万条打分", equation I_{t,s} = sum_{j=1..32} w_{t,j} ReLU(q_{t,j} . k_s),
 *    32 heads x 128 dims, FP4 q and k.
 *  - Per-layer top-512 and the two-level candidate pool (blocks of 8, block
 *    score = max, keep 2048 blocks), same page, section "用浅层的打分结果限制深层
 *    的打分范围"; pinning of the newest block and the per-query boolean table,
 *    section "候选池的三个细节在代码里".
 *  - Reindex layers score only inside the pool; a deployed kernel reads only
 *    the pooled indexer K (same section, last paragraph).
 *  - Random Hadamard rotation before FP4 quantisation, "DeepSeek-V4 模型结构（2）：
 *    序列维度（中），Lightning Indexer 与稀疏选择", Q&A on quantisation.
 *
 * Conventions for every call:
 *  - Pointers marked (dev) are device pointers, (host) host pointers. The
 *    caller owns every buffer; no call allocates or frees memory.
 *  - Every call is enqueued on `stream` and returns without synchronising.
 *    Host-side argument errors are returned at once and launch nothing.
 *  - A kernel that detects a problem on the device (a bounded wait that ran
 *    out, a malformed argument only visible on the device) records it in a
 *    sticky device error word; hsi_device_error() reports and clears it.
 *  - Scratch memory is passed in as (ws, ws_bytes); hsi_workspace_size() says
 *    how much a call needs. ws must be 256-byte aligned.
 *  - The library runs only on compute capability 10.3 devices.
 */
#ifndef HSI_H_
#define HSI_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    HSI_OK = 0,
    HSI_ERR_INVALID_ARG = -1,    /* a null pointer, a bad size or a misaligned buffer */
    HSI_ERR_UNSUPPORTED = -2,    /* a valid request the library does not serve (device, shape) */
    HSI_ERR_CUDA = -3,           /* a CUDA runtime call failed (launch, attribute, sync) */
    HSI_ERR_DEVICE_TIMEOUT = -4, /* a kernel's bounded wait ran out (reported by hsi_device_error) */
    HSI_ERR_WORKSPACE = -5,      /* ws is NULL, too small or not 256-byte aligned */
    HSI_ERR_DEVICE_ARG = -6,     /* a kernel found a bad device-side argument (reported by hsi_device_error) */
    HSI_ERR_TOO_LARGE = -7       /* more than the fixed scratch of hsi_topk_noalloc holds */
} hsi_status;

#define HSI_HEADS 32      /* indexer heads H */
#define HSI_DIM 128       /* head dimension d */
#define HSI_REC_ROWS 8    /* rows per NVFP4 block record */
#define HSI_REC_BYTES 576 /* bytes per NVFP4 block record: 8 rows x (64 B codes + 8 B scales) */
#define HSI_MX_REC_BYTES 544 /* bytes per MXFP4 block record: 8 rows x (64 B codes + 4 B scales) */

/* Record format of the indexer q and K (every scoring call takes one). */
typedef enum {
    HSI_FMT_NVFP4 = 0, /* 576-byte records, per-16 E4M3 scales, fp32 tensor scale g */
    HSI_FMT_MXFP4 = 1  /* 544-byte records, per-32 E8M0 scales, no tensor scale */
} hsi_format;

/*
 * NVFP4 block-record storage, used for indexer queries and indexer K.
 *
 * A tensor of R rows of 128 values is stored as ceil(R/8) records of 576 bytes
 * plus one fp32 tensor scale g. Record i holds rows 8i .. 8i+7 (missing rows
 * of the last record are zero):
 *   bytes [0, 512):   E2M1 codes. Value e (0..127) of row r sits in byte
 *                     (e/32)*128 + r*16 + (e%32)/2, low nibble for even e,
 *                     high nibble for odd e (bit 3 of a code is its sign).
 *   bytes [512, 576): E4M3 block scales. The scale of row r, values
 *                     16j .. 16j+15, is byte 512 + r*8 + j.
 * The decoded value is E2M1(code) * E4M3(scale) * g. A query (32 heads) is
 * 4 records; a K cache of n keys is ceil(n/8) records, and its block of
 * positions 8b .. 8b+7 is exactly record b: 8 keys x 72 B = 576 B.
 *
 * MXFP4 block records (HSI_FMT_MXFP4), the indexer format the pages describe
 * ("DeepSeek-V4.1 模型结构（3）", table in section "scale 的格式决定了精度":
 * groups of 32, E8M0 scales, 4.25 bits per value; 68 B per indexer key in
 * section "890 字节的分项"): 544 bytes per 8 rows, no tensor scale.
 *   bytes [0, 512):   E2M1 codes, placed exactly as in NVFP4 records.
 *   bytes [512, 544): E8M0 scales. The scale of row r, values 32j .. 32j+31,
 *                     is byte 512 + r*4 + j; its value is 2^(byte - 127).
 * The decoded value is E2M1(code) * 2^(scale - 127): 8 keys x 68 B = 544 B.
 */

/* ------------------------------------------------------------------------- */

/*
 * Rotate and quantise bf16 rows to NVFP4 block records.
 * Page: "DeepSeek-V4 模型结构（2）", Q&A on quantisation (random Hadamard
 * rotation before FP4); "DeepSeek-V4.1 模型结构（3）", section "E2M1 只能表示
 * 15 个值" (q = round_E2M1(x/s), s = max|x|/6) and section "去掉全局 scale 之后
 * 范围仍然够用" (448 x 6 = 2688).
 *
 * Per row: y = H (signs .* x), H the unnormalised 128-point Sylvester Hadamard
 * transform evaluated in fp32 stage by stage (h = 1, 2, ..., 64). Per tensor:
 * g = amax|y| / 2688 (g = 1 for an all-zero tensor). Per 16 values:
 * sb = E4M3_RN(amax_b / (6 g)), code = E2M1_RN(y / (E4M3(sb) g)) (0 when that
 * scale is 0). Rounding is to nearest, ties to even, saturating at 448 / 6.
 *
 *  x         (dev)  bf16 bit patterns [n_tensors * rows_per_tensor][128].
 *  signs     (host) 128 values, each +1 or -1 (the rotation's random signs;
 *                   queries and keys scored together must share them).
 *  mode      0: compute g per tensor and write it to g; 1: read g (> 0) from g.
 *  g         (dev)  fp32 [n_tensors].
 *  rec       (dev)  out: n_tensors * ceil(rows_per_tensor/8) records; tensor t
 *                   starts at record t * ceil(rows_per_tensor/8).
 *  ws        (dev)  mode 0: 4 * n_tensors bytes. Mode 1: may be NULL.
 * Errors: INVALID_ARG for null pointers, non-positive sizes, signs not +-1,
 * unaligned rec (16 B) or x (16 B); WORKSPACE when ws is short in mode 0.
 */
hsi_status hsi_quantize_nvfp4(const uint16_t* x, int64_t n_tensors, int64_t rows_per_tensor,
                              const int8_t* signs, int mode, float* g, uint8_t* rec, void* ws,
                              size_t ws_bytes, cudaStream_t stream);

/*
 * Rotate and quantise bf16 rows to MXFP4 block records (no tensor scale).
 * Page: "DeepSeek-V4.1 模型结构（3）", section "scale 的格式决定了精度" (groups of
 * 32 with an E8M0 scale, which can only be a power of two: the ideal scale
 * max|x|/6 rounded up to one); section "E2M1 只能表示 15 个值" (the codes).
 *
 * Per row the same rotation as hsi_quantize_nvfp4; per 32 values the scale
 * 2^e with e the smallest integer in [-127, 127] such that 6 * 2^e >= amax of
 * the group (e = -127 for an all-zero group), then code = E2M1_RN(y / 2^e),
 * ties to even, saturating at 6. Inputs must be finite; a non-finite rotated
 * value is reported as HSI_ERR_DEVICE_ARG by hsi_device_error.
 *
 *  x, signs  as for hsi_quantize_nvfp4.
 *  rec       (dev) out: n_tensors * ceil(rows_per_tensor/8) 544-byte records;
 *                  tensor t starts at record t * ceil(rows_per_tensor/8).
 * Errors: INVALID_ARG for null pointers, non-positive sizes, signs not +-1,
 * unaligned rec (16 B) or x (16 B).
 */
hsi_status hsi_quantize_mxfp4(const uint16_t* x, int64_t n_tensors, int64_t rows_per_tensor,
                              const int8_t* signs, uint8_t* rec, cudaStream_t stream);

/*
 * Lightning-indexer scores of every visible key (a Full layer).
 * Page: "DeepSeek-V4.1 模型结构（3）", section "Reindex 层每个 token 要给 100 万条打分"
 * (the equation); section "用浅层的打分结果限制深层的打分范围" (the Full layer
 * scores all visible positions).
 *
 *   scores[b][s] = (g_q[b] g_k[b] / 128) * sum_j w[b][j] * max(a_j, 0),
 *   a_j = sum_d qhat[b][j][d] * khat_s[d]      (0 <= s < n_visible[b])
 * with qhat, khat the decoded values without tensor scales; the factor 1/128
 * undoes the unnormalised rotation of both operands. The contraction runs on
 * the tensor cores (FP4 x FP4, fp32 accumulation); ReLU and the weighted head
 * sum are fused, so per-head logits never reach memory.
 *
 *  q_rec   (dev) B*4 records (query b = records 4b .. 4b+3); g_q (dev) [B].
 *  w       (dev) fp32 [B][32].
 *  k_rec   (dev) base of the K records; query b reads the cache starting at
 *                record k_rec_off[b] (dev, int64 [B]); g_k (dev) [B] is that
 *                cache's tensor scale.
 *  n_visible (dev) int32 [B], 0 <= n_visible[b] <= max_visible (host bound).
 *  group   1, or 4: queries 4i .. 4i+3 share one cache (equal k_rec_off and
 *          g_k) and are scored in one tensor-core tile (chunked prefill);
 *          B must then be a multiple of 4.
 *  scores  (dev) fp32 [B][ld]; entries s < n_visible[b] are written, the
 *          rest are left untouched. ld >= max_visible. May be NULL when
 *          block_max is given (the block maxima only).
 *  block_max (dev, may be NULL) fp32 [B][ldb]: the max of each run of 8
 *          consecutive visible scores (block b8 = positions 8*b8 .. 8*b8+7,
 *          invisible positions count as -inf), for the blocks that hold a
 *          visible position. ldb >= ceil(max_visible/8).
 *  format  HSI_FMT_NVFP4 (576-byte records, g_q and g_k required) or
 *          HSI_FMT_MXFP4 (544-byte records; g_q and g_k are not read and may
 *          be NULL: the formula above with g_q = g_k = 1). q and K share it.
 *  ws      may be NULL (0 bytes needed).
 */
hsi_status hsi_score_full(const uint8_t* q_rec, const float* g_q, const float* w, const uint8_t* k_rec,
                          const float* g_k, const int64_t* k_rec_off, const int32_t* n_visible,
                          int32_t B, int64_t max_visible, int32_t group, float* scores, int64_t ld,
                          float* block_max, int64_t ldb, hsi_format format, void* ws, size_t ws_bytes,
                          cudaStream_t stream);

/*
 * Exact per-query top-k of fp32 scores.
 * Page: "DeepSeek-V4.1 模型结构（3）", section "用浅层的打分结果限制深层的打分范围"
 * (each Full and Reindex layer keeps its own top-512).
 *
 * For query b the eligible entries are i < n_valid[b] of row scores[b][.]
 * (ld floats per row). Order: value descending (-0 and +0 compare equal),
 * ties by index ascending. Writes min(k, n_valid[b]) entries to out_idx[b][.]
 * and out_val[b][.] in that order and pads the rest with -1 / -inf.
 * Scores must not be NaN.
 *
 *  block_ids (dev, may be NULL) int32 [B][ld_blocks]: when given, an eligible
 *          local index i is reported as the position block_ids[b][i/block_size]
 *          * block_size + i % block_size (pool-local -> global; the block ids
 *          must be ascending so that the tie order carries over).
 *  max_valid (host) upper bound of n_valid; k in [1, 2048].
 *  ws      (dev) hsi_workspace_size(HSI_WS_TOPK, B, max_valid, k) bytes.
 */
hsi_status hsi_topk(const float* scores, int64_t ld, const int32_t* n_valid, int32_t B, int64_t max_valid,
                    int32_t k, const int32_t* block_ids, int64_t ld_blocks, int32_t block_size,
                    int32_t* out_idx, float* out_val, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * hsi_topk without a workspace: for callers that cannot allocate device
 * memory and have none to lend -- code running inside a host framework that
 * owns every byte of device memory through its own pool, or a latency-critical
 * loop where cudaMalloc's implicit device synchronisation is not acceptable.
 * The pages have no counterpart; this is a convenience of the library.
 *
 * Results are exactly those of hsi_topk with the same arguments. Instead of
 * `ws`, the long-row passes (rows longer than 16384 items) use one fixed 8 MiB
 * array compiled into the library, which every GPU that loads the library
 * keeps until the process exits. That bounds the request: with
 * max_valid > 16384, B may be at most 56 (HSI_ERR_TOO_LARGE beyond that);
 * shorter rows use no scratch and have no limit on B.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - Every call on a device shares the array and clears what must start at
 *    zero itself; calls whose work overlaps on the GPU (other streams, other
 *    host threads) race on the array and must be ordered by the caller.
 *  - No call allocates or frees memory.
 *  - The fixed scratch keeps at most 16384 survivors of the histogram pass
 *    per query (hsi_topk keeps 65536). A row with more (heavy ties near the
 *    k-th score) is selected by re-reading it from `scores`: the same result,
 *    more slowly than hsi_topk.
 */
hsi_status hsi_topk_noalloc(const float* scores, int64_t ld, const int32_t* n_valid, int32_t B, int64_t max_valid,
                            int32_t k, const int32_t* block_ids, int64_t ld_blocks, int32_t block_size,
                            int32_t* out_idx, float* out_val, cudaStream_t stream);

/*
 * The candidate pool of each query.
 * Page: "DeepSeek-V4.1 模型结构（3）", sections "用浅层的打分结果限制深层的打分范围"
 * (blocks of 8, block score = max, top 2048 blocks, at most 16384 positions)
 * and "候选池的三个细节在代码里" (the newest block pinned, -inf padding, blocks
 * whose value is -inf dropped, a per-query boolean table).
 *
 * Query b sees positions [0, n_visible[b]). Blocks are runs of block_size
 * positions; a block's value is the max of its visible scores; the block of
 * position n_visible[b]-1 gets +inf. The pool keeps the first
 * min(n_keep, nblk) blocks by (value desc, block index asc) whose value is
 * > -inf, intersected with the visible positions.
 *
 *  scores  (dev) fp32 [B][ld] (read for s < n_visible[b]); may be NULL when
 *          block_max is given.
 *  block_max (dev, may be NULL) fp32 [B][ldb]: precomputed block maxima for
 *          block_size 8, as hsi_score_full writes them.
 *  block_ids (dev) out int32 [B][n_keep]: kept block indices ascending, -1 padded.
 *  n_kept  (dev) out int32 [B]: number of kept blocks.
 *  n_pool  (dev) out int32 [B]: number of visible positions in the pool (the
 *          kept blocks' positions in block-list order, less the invisible tail
 *          of the newest block, which is always last).
 *  pool_bits (dev, may be NULL) out uint32 [B][ld_bits]: the boolean table,
 *          bit s%32 of word s/32 set iff position s is in the pool; words up to
 *          ceil(n_visible[b]/32) are written. ld_bits >= ceil(max_visible/32).
 *  block_size in [1, 64]; n_keep in [1, 4096].
 *  ws      (dev) hsi_workspace_size(HSI_WS_POOL, B, max_visible, n_keep) bytes.
 */
hsi_status hsi_candidate_pool(const float* scores, int64_t ld, const float* block_max, int64_t ldb,
                              const int32_t* n_visible, int32_t B, int64_t max_visible, int32_t block_size,
                              int32_t n_keep, int32_t* block_ids, int32_t* n_kept, int32_t* n_pool,
                              uint32_t* pool_bits, int64_t ld_bits, void* ws, size_t ws_bytes,
                              cudaStream_t stream);

/*
 * The pages' masked form of a Reindex layer, kept for comparison with the
 * pooled layers: after hsi_score_full has scored every visible position with
 * the Reindex layer's query, every score of query b at a visible position s
 * (< n_visible[b]) whose pool bit is clear (bit s%32 of bits[b][s/32], as
 * written by hsi_candidate_pool or hsi_full_layer) becomes -inf; hsi_topk of
 * the result is the layer's top-k. Page: "DeepSeek-V4.1 模型结构（3）", section
 * "候选池的三个细节在代码里" (the Reindex code masks the full score row with the
 * pool's boolean table and then takes its top-k) and the last paragraph of
 * "用浅层的打分结果限制深层的打分范围" (16384 of 1M positions: 1/64 of the work).
 *  scores  (dev) fp32 [B][ld], ld >= max_visible (host bound on n_visible).
 *  bits    (dev) uint32 [B][ld_bits], ld_bits >= ceil(max_visible / 32).
 */
hsi_status hsi_mask_scores(float* scores, int64_t ld, const int32_t* n_visible, const uint32_t* bits, int64_t ld_bits,
                           int32_t B, int64_t max_visible, cudaStream_t stream);

/*
 * Reindex-layer scores restricted to the pool, reading only pooled K.
 * Page: "DeepSeek-V4.1 模型结构（3）", section "用浅层的打分结果限制深层的打分范围"
 * (Reindex layers score only pooled positions, 16384 x 4096 MACs per token)
 * and the last paragraph of "候选池的三个细节在代码里" (a deployed kernel fetches
 * only the pooled indexer K).
 *
 * Slot i = 8j + r of query b holds the score of position block_ids[b][j]*8 + r
 * (same formula as hsi_score_full), -inf if that position is not visible.
 * Slots i < 8 * n_kept[b] are written; the rest are left untouched. Each
 * pooled block is one K record (576 or 544 bytes), fetched whole.
 *
 *  block_ids, n_kept: as written by hsi_candidate_pool with block_size 8;
 *          block_ids 16-byte aligned, n_keep a multiple of 32.
 *  pool_scores (dev) fp32 [B][ld], ld >= 8 * n_keep.
 *  format  as for hsi_score_full.
 *  ws      may be NULL.
 */
hsi_status hsi_score_pool(const uint8_t* q_rec, const float* g_q, const float* w, const uint8_t* k_rec,
                          const float* g_k, const int64_t* k_rec_off, const int32_t* n_visible,
                          const int32_t* block_ids, const int32_t* n_kept, int32_t n_keep, int32_t B,
                          float* pool_scores, int64_t ld, hsi_format format, void* ws, size_t ws_bytes,
                          cudaStream_t stream);

/*
 * Compaction of each query's candidate pool, once per decode step: the pooled
 * K records of query b (576 or 544 bytes), in block-list order, into one
 * contiguous run,
 *   pool_rec[b][i] = the record k_rec_off[b] + block_ids[b][i],  i < min(n_kept[b], n_keep).
 * Records of slots at or past n_kept[b] are left untouched.
 * Page: "DeepSeek-V4.1 模型结构（3）", section "用浅层的打分结果限制深层的打分范围"
 * (the Reindex layers score the same indexer K as the Full layer, each with
 * its own query, inside the same per-query pool): the layers of a step can
 * then stream the pool instead of each gathering it (hsi_reindex_layer with
 * pool_rec). The method itself fixes only which records are scored; this
 * layout is this library's.
 *
 *  k_rec, k_rec_off, n_visible: as for hsi_score_full.
 *  block_ids, n_kept: as written by hsi_candidate_pool (block_size 8).
 *  pool_rec (dev) [B][n_keep][record bytes], 16-byte aligned; distinct from k_rec.
 *  format  the records' format (it fixes their size).
 * A block id outside [0, ceil(n_visible[b] / 8)) is skipped and reported as
 * HSI_ERR_DEVICE_ARG by hsi_device_error.
 */
hsi_status hsi_pool_gather(const uint8_t* k_rec, const int64_t* k_rec_off, const int32_t* n_visible,
                           const int32_t* block_ids, const int32_t* n_kept, int32_t n_keep, int32_t B,
                           uint8_t* pool_rec, hsi_format format, cudaStream_t stream);

/*
 * FP4 main KV for core attention, and gather(main_kv, topk).
 * Page: "DeepSeek-V4.1 模型结构（3）", section "scale 的格式决定了精度" (the main KV
 * uses groups of 16 with an E4M3 scale, NVFP4's layout without its global
 * scale: a 512-dim entry is 256 B of codes plus 32 B of scales, 288 B) and
 * section "官方的参考实现里" (dequantised before attention); the CSA2 layer
 * pseudocode of "DeepSeek V4.1 Flash KV cache" (selected = gather(main_kv,
 * topk), then core attention).
 *
 * Entry layout (288 bytes, 512 values): the E2M1 code of value i in byte i/2
 * (low nibble for even i), then the E4M3 scale of values 16g .. 16g+15 in
 * byte 256 + g. Value = E2M1(code) * E4M3(scale); every such product is exact
 * in bf16. Quantisation: scale = E4M3_RN(amax/6) (amax of the 16 values, the
 * division in fp32), code = E2M1_RN(x / scale), 0 where the scale decodes to
 * 0; no rotation. Scale bytes 0x7F and 0xFF (NaN) never occur in valid entries.
 */
#define HSI_KV_DIM 512
#define HSI_KV_ENTRY_BYTES 288

/*
 *  x   (dev) bf16 bit patterns [n][512], 16-byte aligned; finite (a non-finite
 *      value is reported as HSI_ERR_DEVICE_ARG by hsi_device_error).
 *  kv  (dev) out: [n][288] bytes, 16-byte aligned.
 */
hsi_status hsi_quantize_mainkv(const uint16_t* x, int64_t n, uint8_t* kv, cudaStream_t stream);

/*
 * out[b][t] = entry kv_off[b] + idx[b][t] of kv, decoded to bf16, for t < k;
 * a zero row where idx[b][t] < 0 (the -1 padding of a short top-k list).
 *  kv      (dev) entries, 16-byte aligned; query b's cache starts at entry
 *          kv_off[b] (dev, int64 [B]) and holds n_visible[b] (dev, int32 [B])
 *          entries. An index at or past n_visible[b] is reported as
 *          HSI_ERR_DEVICE_ARG by hsi_device_error and its row is zeroed.
 *  idx     (dev) int32 [B][ld_idx], ld_idx >= k (e.g. the top_idx of a layer).
 *  k       1 .. 4096.
 *  out     (dev) bf16 bit patterns [B][k][512], 16-byte aligned.
 */
hsi_status hsi_gather_mainkv(const uint8_t* kv, const int64_t* kv_off, const int32_t* n_visible,
                             const int32_t* idx, int64_t ld_idx, int32_t k, int32_t B, uint16_t* out,
                             cudaStream_t stream);

/*
 * hsi_gather_mainkv for the top-k lists of L layers of one decode step in
 * one launch (the pages' step gathers the selected entries of every layer;
 * one launch has one ramp where L launches have L): list l is read at
 * idx + l * idx_stride ([B][ld_idx]) and its rows are written at
 * out + l * out_stride (bf16 elements, [B][k][512]), against the same caches.
 * Results equal L calls of hsi_gather_mainkv.
 *  idx_stride >= B * ld_idx and out_stride >= B * k * 512 (a multiple of 8)
 *  when L > 1; other arguments as for hsi_gather_mainkv.
 */
hsi_status hsi_gather_mainkv_layers(const uint8_t* kv, const int64_t* kv_off, const int32_t* n_visible,
                                    const int32_t* idx, int64_t ld_idx, int64_t idx_stride, int32_t L, int32_t k,
                                    int32_t B, uint16_t* out, int64_t out_stride, cudaStream_t stream);

/*
 * Append one decode token to every query's caches: the new position's
 * indexer K row (rotated and quantised as hsi_quantize_nvfp4 does in mode 1,
 * with the cache's fixed tensor scale g_k[b]; or as hsi_quantize_mxfp4 does)
 * into row n_visible[b] of query b's K records, and (kv_x given) the new
 * main-KV entry (as hsi_quantize_mainkv does) into entry n_visible[b] of its
 * main-KV cache; then n_visible[b] += 1. A cache built token by token is
 * byte for byte the cache quantised at once with the same tensor scale.
 * Page: "DeepSeek-V4.1 模型结构（3）", section "去掉全局 scale 之后范围仍然够用"
 * (a fixed scale is enough for the range of later entries) and section
 * "用浅层的打分结果限制深层的打分范围" (every decode step scores the visible
 * positions, including the newest, whose block the pool pins).
 *
 * The lengths live on the device, so a CUDA graph that holds this call and
 * the step's scoring calls (their max_visible set to the caches' capacity)
 * replays over a growing cache.
 *  k_x     (dev) bf16 bit patterns [B][128], 16-byte aligned: row b is query b's new K row.
 *  signs   (host) the rotation's 128 signs (+1 / -1), as for the quantisers.
 *  g_k     (dev) [B] the K caches' tensor scales (NVFP4; may be NULL for MXFP4).
 *  k_rec, k_rec_off: the K records and each query's first record, as for
 *          hsi_score_full; the record of row n_visible[b] must be allocated.
 *  kv_x    (dev, may be NULL) bf16 [B][512]; kv, kv_off: the main-KV entries
 *          and each query's first entry, as for hsi_gather_mainkv.
 *  n_visible (dev) int32 [B], read and advanced.
 *  capacity  (dev) int32 [B]: rows (entries) each query's caches hold. A query
 *          whose n_visible is not below its capacity is left unchanged and
 *          reported as HSI_ERR_DEVICE_ARG by hsi_device_error.
 * One query per cache: two queries that share a cache would append twice.
 */
hsi_status hsi_append_token(const uint16_t* k_x, const int8_t* signs, const float* g_k, uint8_t* k_rec,
                            const int64_t* k_rec_off, const uint16_t* kv_x, uint8_t* kv, const int64_t* kv_off,
                            int32_t* n_visible, const int32_t* capacity, int32_t B, hsi_format format,
                            cudaStream_t stream);

/*
 * A decoder Full layer in one call: hsi_score_full, then the top-k of the
 * scores, then (block_ids != NULL) the candidate pool with blocks of 8, with
 * the selections' key histograms accumulated inside the scoring kernel
 * instead of in separate passes. Results equal those of the three separate
 * calls (same scores, same top-k, same pool).
 * Page: "DeepSeek-V4.1 模型结构（3）", section "用浅层的打分结果限制深层的打分范围"
 * (the Full layer scores every visible position, keeps its top-512 and builds
 * the pool from the same scores).
 *
 *  Arguments as in hsi_score_full (group 1, format), hsi_topk (n_valid =
 *  n_visible) and hsi_candidate_pool (block_size 8). scores [B][ld] is written.
 *  block_ids NULL: no pool (n_kept, n_pool, pool_bits ignored).
 *  scores NULL (with a pool, n_keep - 1 >= k, n_keep <= 2048 and a multiple
 *          of 32): no score row is written, and the top-k is taken from the
 *          pool. The pool's n_keep - 1 unpinned blocks are the first by
 *          (maximum desc, index asc), and every top-k position lies in the
 *          first k blocks of that order (a position outside them is outranked
 *          by each of those blocks' maxima), so the pool holds the top-k. The
 *          pooled blocks are scored again from k_rec with the layer's query
 *          (the same fp32 scores as the full scan) and their top-k taken as in
 *          hsi_reindex_layer: the same top_idx and top_val as with scores.
 *          HSI_PHASE_TOPK then needs the pool first (HSI_PHASE_POOL, or
 *          HSI_PHASE_SELECT / HSI_PHASE_ALL, which run it first).
 *  phases  HSI_PHASE_ALL, or the parts as separate calls with the same
 *          arguments and workspace, scoring first (the workspace carries the
 *          histograms and block maxima from one to the other):
 *          HSI_PHASE_SCORE, then HSI_PHASE_SELECT (the top-k, then the pool),
 *          or HSI_PHASE_TOPK and HSI_PHASE_POOL, which use separate parts of
 *          the workspace and may run at the same time on two streams (both
 *          after the scoring call).
 *  ws      (dev) hsi_workspace_size(HSI_WS_FULL_LAYER, B, max_visible, k).
 */
#define HSI_PHASE_SCORE 1
#define HSI_PHASE_SELECT 2
#define HSI_PHASE_ALL 3
#define HSI_PHASE_TOPK 4
#define HSI_PHASE_POOL 8
hsi_status hsi_full_layer(const uint8_t* q_rec, const float* g_q, const float* w, const uint8_t* k_rec,
                          const float* g_k, const int64_t* k_rec_off, const int32_t* n_visible, int32_t B,
                          int64_t max_visible, float* scores, int64_t ld, int32_t k, int32_t* top_idx,
                          float* top_val, int32_t n_keep, int32_t* block_ids, int32_t* n_kept, int32_t* n_pool,
                          uint32_t* pool_bits, int64_t ld_bits, int32_t phases, hsi_format format, void* ws,
                          size_t ws_bytes, cudaStream_t stream);

/*
 * A chunked-prefill layer in one call: the scores of every visible key with
 * groups of `group` consecutive queries sharing one cache and one tensor-core
 * tile (as hsi_score_full), then per query its top-k and (block_ids != NULL)
 * its candidate pool, equal to what hsi_topk and hsi_candidate_pool give on
 * the same scores. The selection reads the block maxima the scoring kernel
 * writes, not the score rows: a top-k position lies in one of the first k
 * blocks by (block max desc, block asc), since the maximum of every block
 * ranked ahead of its own outranks it, so only the scores of the first k + 1
 * blocks of the pool's order (the newest block pinned first) are read.
 * Page: "DeepSeek-V4.1 模型结构（3）", sections "Reindex 层每个 token 要给 100 万条
 * 打分" (the score), "用浅层的打分结果限制深层的打分范围" (top-512 and the pool of
 * every query) and "候选池的三个细节在代码里" (pinning, -inf blocks dropped).
 *
 *  Arguments as in hsi_score_full (group 1 or 4; max_visible <= 524288) and
 *  hsi_full_layer (k <= 2048; block_ids NULL: no pool; block size 8).
 *  phases  HSI_PHASE_ALL, or HSI_PHASE_SCORE then HSI_PHASE_SELECT with the
 *          same arguments and workspace.
 *  ws      (dev) hsi_workspace_size(HSI_WS_PREFILL_LAYER, B, max_visible, k).
 */
hsi_status hsi_prefill_layer(const uint8_t* q_rec, const float* g_q, const float* w, const uint8_t* k_rec,
                             const float* g_k, const int64_t* k_rec_off, const int32_t* n_visible, int32_t B,
                             int64_t max_visible, int32_t group, float* scores, int64_t ld, int32_t k,
                             int32_t* top_idx, float* top_val, int32_t n_keep, int32_t* block_ids, int32_t* n_kept,
                             int32_t* n_pool, uint32_t* pool_bits, int64_t ld_bits, int32_t phases,
                             hsi_format format, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * A decoder Reindex layer in one call: the pooled scores (hsi_score_pool),
 * then the top-k inside the pool reported as global positions (hsi_topk with
 * the block map).
 * Page: "DeepSeek-V4.1 模型结构（3）", section "用浅层的打分结果限制深层的打分范围"
 * (Reindex layers score only pooled positions and keep their own top-512).
 *
 *  pool_rec, pool_rec_ready: pool_rec NULL: the pooled records are gathered
 *          from k_rec (as by hsi_score_pool). pool_rec (dev, [B][n_keep][record
 *          bytes], 16-byte aligned) with pool_rec_ready 0: gathered from k_rec, and
 *          also left in pool_rec in the layout hsi_pool_gather writes, so that
 *          the step's later Reindex layers can stream them. pool_rec_ready 1:
 *          pool_rec already holds them (an earlier layer of this pool, or
 *          hsi_pool_gather); they are streamed and k_rec is not read. All
 *          forms give the same pool_scores, top_idx and top_val.
 *  n_pool (dev) int32 [B] as written by hsi_candidate_pool / hsi_full_layer.
 *  pool_scores [B][ld], ld >= 8 * n_keep, is written (as by hsi_score_pool).
 *  format  as for hsi_score_full; the pooled records and q share it.
 *  ws      (dev) hsi_workspace_size(HSI_WS_REINDEX_LAYER, B, 8 * n_keep, k).
 */
hsi_status hsi_reindex_layer(const uint8_t* q_rec, const float* g_q, const float* w, const uint8_t* k_rec,
                             const float* g_k, const int64_t* k_rec_off, uint8_t* pool_rec, int32_t pool_rec_ready,
                             const int32_t* n_visible, const int32_t* block_ids, const int32_t* n_kept,
                             const int32_t* n_pool, int32_t n_keep, int32_t B, float* pool_scores, int64_t ld,
                             int32_t k, int32_t* top_idx, float* top_val, hsi_format format, void* ws,
                             size_t ws_bytes, cudaStream_t stream);

typedef enum {
    HSI_WS_QUANTIZE = 0,
    HSI_WS_SCORE = 1,
    HSI_WS_TOPK = 2,
    HSI_WS_POOL = 3,
    HSI_WS_FULL_LAYER = 4,
    HSI_WS_REINDEX_LAYER = 5,
    HSI_WS_PREFILL_LAYER = 6
} hsi_ws_kind;

/* Scratch bytes a call needs for B queries of at most max_n entries.
 * QUANTIZE: B = number of tensors (max_n, k unused). SCORE: 0. TOPK: max_n =
 * max_valid (k unused). POOL: max_n = max_visible and k = block_size.
 * FULL_LAYER, PREFILL_LAYER: max_n = max_visible. REINDEX_LAYER: max_n = 8 * n_keep. */
size_t hsi_workspace_size(hsi_ws_kind kind, int32_t B, int64_t max_n, int32_t k);

/* Synchronise `stream`, then report and clear the sticky device error word of
 * the current device: HSI_OK, HSI_ERR_DEVICE_TIMEOUT or HSI_ERR_DEVICE_ARG
 * (or HSI_ERR_CUDA if the synchronisation itself failed). */
hsi_status hsi_device_error(cudaStream_t stream);

/*
 * Diagnostics for the failure path (no counterpart on the pages), current
 * device, synchronous:
 *  HSI_DEBUG_WAIT_LIMIT_NS: the wall-clock limit of every bounded wait in the
 *    kernels (default 1 s). When a wait runs out the kernel records
 *    HSI_ERR_DEVICE_TIMEOUT, drains what it has in flight, frees its TMEM and
 *    returns; the context stays usable.
 *  HSI_DEBUG_SKIP_FIRST_COPY: nonzero makes the scoring kernels' producer skip
 *    the copy of its first unit, so that the consumer's wait runs out (a test
 *    of the path above). Zero restores normal operation.
 */
#define HSI_DEBUG_WAIT_LIMIT_NS 1
#define HSI_DEBUG_SKIP_FIRST_COPY 2
hsi_status hsi_debug_set(int what, long long value);

/* HSI_OK if the current device is compute capability 10.3, else UNSUPPORTED. */
hsi_status hsi_device_check(void);

/* A static English description of a status code. */
const char* hsi_status_string(hsi_status status);

/* Number of kernels this library has launched in this process (all devices,
 * all streams), for tracing and launch accounting. */
uint64_t hsi_kernel_launches(void);

/*
 * Calibration: the rooflines of the running GPU, measured with the same
 * instructions the path uses (no counterpart on the pages; the report states
 * these beside every roofline fraction).
 *
 * hsi_calib_read streams `bytes` of `buf` (dev, 16-byte aligned) once.
 * method 0: 16-byte loads from every SM; method 1: one contiguous slice per SM
 * through a ring of `stages` shared-memory buffers of `chunk` bytes filled by
 * bulk copies (chunk a multiple of 16). Time it with events on `stream`.
 * `sink` (dev) is a scratch counter that keeps the loads live.
 *
 * hsi_calib_mma issues `iters` back-to-back tcgen05.mma kind::mxf4nvf4 of
 * M = 128, N = n (32, 64, 128 or 256), K = 64 per SM on shared-memory operands:
 * 2 * 128 * n * 64 * iters FP4 flops per SM.
 */
hsi_status hsi_calib_read(const void* buf, size_t bytes, int method, int chunk, int stages,
                          unsigned long long* sink, cudaStream_t stream);
hsi_status hsi_calib_mma(int n, int iters, unsigned long long* sink, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* HSI_H_ */
