/*
 * ORACLE -- test infrastructure, not the product.
 *
 * A plain, slow, single-threaded CPU restatement of the decode-time path of
 * DeepSeek-V4.1's Hierarchical Sparse Indexer, written from the pages'
 * statement of the method. Only the tests, the smoke check and the bench's
 * CPU-baseline leg load it. It shares no code with the CUDA path.
 *
 * Sources (page titles and sections):
 *  [J] "DeepSeek-V4.1 模型结构（3）：序列维度（下），Hierarchical Sparse Indexer 与
 *      FP4 KV cache" (blog.javazero.top): the indexer score equation I_{t,s} in
 *      "Reindex 层每个 token 要给 100 万条打分"; the two-level pool in
 *      "用浅层的打分结果限制深层的打分范围"; the select_candidate_blocks code and the
 *      masked Reindex code in "候选池的三个细节在代码里"; the E2M1 value set in
 *      "E2M1 只能表示 15 个值"; group quantisation s = max|x|/6 in the same section;
 *      448*6 = 2688 in "去掉全局 scale 之后范围仍然够用".
 *  [X] "DeepSeek-V4 模型结构（2）：序列维度（中），Lightning Indexer 与稀疏选择"
 *      (xhh.club): FP4 q/k after a random Hadamard rotation (Q&A on quantisation).
 *
 * Readings where the pages are silent (each is a stated choice):
 *  - NVFP4 storage: 16-element groups with an E4M3 scale and one fp32 tensor
 *    scale g; g = amax_T / 2688 (2688 = 448 * 6), g = 1 for an all-zero tensor;
 *    block scale sb = E4M3_RN(amax_b / (6 g)); code = E2M1_RN(y / (sb g)),
 *    code 0 when sb g == 0. Rounding is to nearest, ties to the even code,
 *    saturating at +-6 (E2M1) and 448 (E4M3); the sign of the input is kept.
 *  - Rotation: y = H (s .* x) with the unnormalised 128-point Sylvester
 *    Hadamard transform evaluated in fp32 stage by stage (h = 1, 2, ..., 64,
 *    pairs (i, i+h) with bit h of i clear -> (a+b, a-b)). The 1/sqrt(128)
 *    normalisation of q and k is folded into the score as an exact 2^-7.
 *  - Score: a_j = sum_d qhat_jd khat_d accumulated in double over exactly
 *    decoded values (each product is exact), then
 *    I = (g_q g_k / 128) * sum_j w_j * max(a_j, 0) in double, rounded to fp32 once.
 *  - Top-k: order by value descending (numeric compare, so -0 == +0), ties by
 *    index ascending; fewer than k eligible entries -> pad with -1 / -inf.
 *  - Pool: blocks of positions [b*bs, b*bs+bs); block value = max over its
 *    visible positions; the block of position n_vis-1 is set to +inf; keep the
 *    first min(n_keep, nblk) blocks in (value desc, block asc) order whose value
 *    is > -inf; the pool is the kept blocks intersected with [0, n_vis).
 *
 *  - MXFP4 (the indexer format the pages describe, [J] table in "scale 的格式
 *    决定了精度"): 32-element groups, one E8M0 scale each (a power of two, no
 *    tensor scale). The pages give the ideal scale max|x|/6 and say an E8M0
 *    scale can only take it rounded up to a power of two; so the group scale is
 *    the smallest 2^e (e in [-127, 127]) with 6 * 2^e >= amax_group (2^-127
 *    for an all-zero group), and code = E2M1_RN(y / 2^e), saturating at +-6.
 *    The score is the same sum with g_q = g_k = 1.
 *
 *  - Main KV for core attention ([J] "scale 的格式决定了精度": groups of 16 with
 *    an E4M3 scale, the NVFP4 layout without its second, global scale; 512
 *    values = 256 B of codes + 32 B of scales = 288 B; [J] "官方的参考实现里"
 *    and [P] section 5.1: dequantised before attention; the gather of the
 *    selected positions is the pseudocode's gather(main_kv, topk)). Per 16
 *    values: s = E4M3_RN(amax/6) (division in fp32), code = E2M1_RN(x / s)
 *    (0 when s decodes to 0), no rotation (the Hadamard rotation belongs to
 *    the indexer). An entry is stored whole: code of value i in byte i/2 (low
 *    nibble for even i), the scale of values 16g .. 16g+15 in byte 256 + g.
 *    Decoded values E2M1 * E4M3 are exact in bf16, which the gather returns.
 *
 * Storage formats decoded here (the product's "block records"): rows are
 * grouped 8 to a record. In record R (rows 8R .. 8R+7), element e of row r has
 * its 4-bit code in byte (e/32)*128 + r*16 + (e%32)/2, low nibble for even e.
 * NVFP4 records are 576 bytes: the E4M3 scale of row r, group e/16, is byte
 * 512 + r*8 + e/16. MXFP4 records are 544 bytes: the E8M0 scale of row r,
 * group e/32, is byte 512 + r*4 + e/32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define REC_BYTES 576
#define MX_REC_BYTES 544
#define FMT_NVFP4 0
#define FMT_MXFP4 1
#define ROWS_PER_REC 8
#define DIM 128
#define HEADS 32

/* ---------------------------------------------------------------- codecs -- */

/* E2M1: 1 sign bit, 2 exponent bits, 1 mantissa bit. Magnitudes as listed on
 * the page: 0, 0.5, 1, 1.5, 2, 3, 4, 6 for codes 0..7; bit 3 is the sign. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double hsio_e2m1_value(uint8_t code) {
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* E4M3 as in the OCP 8-bit floating point specification (the "fn" variant):
 * bias 7, exponent field 0 is subnormal (m/8 * 2^-6), 0x7F and 0xFF are NaN,
 * no infinities; largest finite magnitude 448. */
double hsio_e4m3_value(uint8_t code) {
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round |x| to the nearest of n ascending magnitudes tab[0..n-1] (codes 0..n-1),
 * ties to the even code, saturating at the largest. */
static int nearest_code(double ax, const double* tab, int n) {
    if (ax >= tab[n - 1]) return n - 1;
    int hi = 1;
    while (tab[hi] < ax) ++hi; /* tab[hi-1] < ax <= tab[hi] */
    int lo = hi - 1;
    if (ax == tab[hi]) return hi;
    double dl = ax - tab[lo], dh = tab[hi] - ax;
    if (dl < dh) return lo;
    if (dh < dl) return hi;
    return (lo & 1) ? hi : lo;
}

static double E4M3_MAG[127]; /* codes 0x00 .. 0x7E */
static int e4m3_ready = 0;

static void e4m3_init(void) {
    if (e4m3_ready) return;
    for (int c = 0; c < 127; ++c) E4M3_MAG[c] = hsio_e4m3_value((uint8_t)c);
    e4m3_ready = 1;
}

uint8_t hsio_e4m3_encode(float x) {
    e4m3_init();
    double ax = fabs((double)x);
    int c = nearest_code(ax, E4M3_MAG, 127);
    return (uint8_t)(c | (signbit(x) ? 0x80 : 0));
}

static uint8_t e2m1_encode_d(double x) {
    int c = nearest_code(fabs(x), E2M1_MAG, 8);
    return (uint8_t)(c | (signbit(x) ? 8 : 0));
}

uint8_t hsio_e2m1_encode(float x) { return e2m1_encode_d((double)x); }

/* E8M0 (OCP MX scale): an unsigned biased exponent, value 2^(b - 127); 0xFF is NaN. */
double hsio_e8m0_value(uint8_t b) { return b == 0xFF ? NAN : ldexp(1.0, (int)b - 127); }

/* The MXFP4 group scale exponent: the smallest e in [-127, 127] with
 * 6 * 2^e >= amax (the ideal scale amax / 6 rounded up to a power of two). */
int hsio_mx_scale_exp(float amax) {
    int e = -127;
    while (e < 127 && ldexp(6.0, e) < (double)amax) ++e;
    return e;
}

static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ------------------------------------------------------------- rotation -- */

/* Unnormalised 128-point Walsh-Hadamard transform in Sylvester order, fp32. */
void hsio_fwht128(float* v) {
    for (int h = 1; h < DIM; h <<= 1)
        for (int i = 0; i < DIM; ++i)
            if (!(i & h)) {
                float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
}

static void rotate_row(const uint16_t* x, const int8_t* signs, float* y) {
    for (int d = 0; d < DIM; ++d) y[d] = (float)signs[d] * bf16_to_f32(x[d]);
    hsio_fwht128(y);
}

/* --------------------------------------------------------- record format -- */

static inline uint8_t rec_code(const uint8_t* rec, int r, int e) {
    uint8_t byte = rec[(e >> 5) * 128 + r * 16 + ((e & 31) >> 1)];
    return (e & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
}

static inline void rec_put_code(uint8_t* rec, int r, int e, uint8_t code) {
    uint8_t* p = &rec[(e >> 5) * 128 + r * 16 + ((e & 31) >> 1)];
    if (e & 1)
        *p = (uint8_t)((*p & 0x0F) | (code << 4));
    else
        *p = (uint8_t)((*p & 0xF0) | (code & 15));
}

static inline uint8_t rec_scale(const uint8_t* rec, int r, int g) { return rec[512 + r * 8 + g]; }

static inline uint8_t mx_rec_scale(const uint8_t* rec, int r, int g) { return rec[512 + r * 4 + g]; }

/* Decoded row `row` of a record array: code value * block scale * tensor scale g,
 * in double (exact). */
void hsio_decode_row(const uint8_t* records, int64_t row, float g, double* out) {
    const uint8_t* rec = records + (row / ROWS_PER_REC) * REC_BYTES;
    int r = (int)(row % ROWS_PER_REC);
    for (int e = 0; e < DIM; ++e)
        out[e] = hsio_e2m1_value(rec_code(rec, r, e)) * hsio_e4m3_value(rec_scale(rec, r, e >> 4)) *
                 (double)g;
}

/* Decoded row `row` of an MXFP4 record array: code value * 2^(scale - 127). */
void hsio_decode_row_mx(const uint8_t* records, int64_t row, double* out) {
    const uint8_t* rec = records + (row / ROWS_PER_REC) * MX_REC_BYTES;
    int r = (int)(row % ROWS_PER_REC);
    for (int e = 0; e < DIM; ++e)
        out[e] = hsio_e2m1_value(rec_code(rec, r, e)) * hsio_e8m0_value(mx_rec_scale(rec, r, e >> 5));
}

/* Same without the tensor scale (code value * block scale), either format. */
static void decode_row_unscaled(int fmt, const uint8_t* records, int64_t row, double* out) {
    if (fmt == FMT_MXFP4) {
        hsio_decode_row_mx(records, row, out);
        return;
    }
    const uint8_t* rec = records + (row / ROWS_PER_REC) * REC_BYTES;
    int r = (int)(row % ROWS_PER_REC);
    for (int e = 0; e < DIM; ++e)
        out[e] = hsio_e2m1_value(rec_code(rec, r, e)) * hsio_e4m3_value(rec_scale(rec, r, e >> 4));
}

/* ------------------------------------------------------------- quantise -- */

/* Quantise one tensor of `rows` bf16 rows of 128 into NVFP4 block records.
 * mode 0: g is computed from the tensor's amax and written to *g_io.
 * mode 1: *g_io is used as given.
 * records must hold ceil(rows/8) * 576 bytes; padding rows are zero.
 * Returns 0, or -1 on a non-finite input or a non-positive given scale. */
int hsio_quantize(const uint16_t* x, int64_t rows, const int8_t* signs, int mode, float* g_io,
                  uint8_t* records) {
    float y[DIM];
    float g;
    if (mode == 0) {
        float amax = 0.0f;
        for (int64_t i = 0; i < rows; ++i) {
            rotate_row(x + i * DIM, signs, y);
            for (int d = 0; d < DIM; ++d) {
                if (!isfinite(y[d])) return -1;
                float a = fabsf(y[d]);
                if (a > amax) amax = a;
            }
        }
        g = amax > 0.0f ? amax / 2688.0f : 1.0f;
        *g_io = g;
    } else {
        g = *g_io;
        if (!(g > 0.0f) || !isfinite(g)) return -1;
    }
    int64_t nrec = (rows + ROWS_PER_REC - 1) / ROWS_PER_REC;
    memset(records, 0, (size_t)nrec * REC_BYTES);
    for (int64_t i = 0; i < rows; ++i) {
        uint8_t* rec = records + (i / ROWS_PER_REC) * REC_BYTES;
        int r = (int)(i % ROWS_PER_REC);
        rotate_row(x + i * DIM, signs, y);
        for (int grp = 0; grp < DIM / 16; ++grp) {
            float amax_b = 0.0f;
            for (int t = 0; t < 16; ++t) {
                if (!isfinite(y[grp * 16 + t])) return -1;
                float a = fabsf(y[grp * 16 + t]);
                if (a > amax_b) amax_b = a;
            }
            float six_g = 6.0f * g;
            uint8_t sb = hsio_e4m3_encode(amax_b / six_g);
            float sc = (float)hsio_e4m3_value(sb) * g;
            rec[512 + r * 8 + grp] = sb;
            for (int t = 0; t < 16; ++t) {
                int e = grp * 16 + t;
                uint8_t code = (sc == 0.0f) ? 0 : hsio_e2m1_encode(y[e] / sc);
                rec_put_code(rec, r, e, code);
            }
        }
    }
    return 0;
}

/* Quantise `rows` bf16 rows of 128 into MXFP4 block records (no tensor
 * scale): per row the same rotation, then per 32-element group the scale
 * exponent e of hsio_mx_scale_exp and codes E2M1_RN(y / 2^e) (y / 2^e is exact
 * in double). records must hold ceil(rows/8) * 544 bytes; padding rows are
 * zero (codes 0, scale byte 0). Returns 0, or -1 on a non-finite input. */
int hsio_quantize_mx(const uint16_t* x, int64_t rows, const int8_t* signs, uint8_t* records) {
    float y[DIM];
    int64_t nrec = (rows + ROWS_PER_REC - 1) / ROWS_PER_REC;
    memset(records, 0, (size_t)nrec * MX_REC_BYTES);
    for (int64_t i = 0; i < rows; ++i) {
        uint8_t* rec = records + (i / ROWS_PER_REC) * MX_REC_BYTES;
        int r = (int)(i % ROWS_PER_REC);
        rotate_row(x + i * DIM, signs, y);
        for (int grp = 0; grp < DIM / 32; ++grp) {
            float amax = 0.0f;
            for (int t = 0; t < 32; ++t) {
                if (!isfinite(y[grp * 32 + t])) return -1;
                float a = fabsf(y[grp * 32 + t]);
                if (a > amax) amax = a;
            }
            int e = hsio_mx_scale_exp(amax);
            rec[512 + r * 4 + grp] = (uint8_t)(e + 127);
            for (int t = 0; t < 32; ++t) {
                int el = grp * 32 + t;
                rec_put_code(rec, r, el, e2m1_encode_d(ldexp((double)y[el], -e)));
            }
        }
    }
    return 0;
}

/* -------------------------------------------------------------- main KV -- */

#define KV_DIM 512
#define KV_BYTES 288

/* Quantise n bf16 main-KV entries of 512 values into 288-byte entries.
 * Returns 0, or -1 on a non-finite input. */
int hsio_mainkv_quantize(const uint16_t* x, int64_t n, uint8_t* kv) {
    for (int64_t i = 0; i < n; ++i) {
        uint8_t* e = kv + i * KV_BYTES;
        memset(e, 0, KV_BYTES);
        for (int g = 0; g < KV_DIM / 16; ++g) {
            float v[16], amax = 0.0f;
            for (int t = 0; t < 16; ++t) {
                v[t] = bf16_to_f32(x[i * KV_DIM + g * 16 + t]);
                if (!isfinite(v[t])) return -1;
                if (fabsf(v[t]) > amax) amax = fabsf(v[t]);
            }
            uint8_t sb = hsio_e4m3_encode(amax / 6.0f);
            float sc = (float)hsio_e4m3_value(sb);
            e[256 + g] = sb;
            for (int t = 0; t < 16; ++t) {
                int c = g * 16 + t;
                uint8_t code = (sc == 0.0f) ? 0 : hsio_e2m1_encode(v[t] / sc);
                e[c / 2] |= (uint8_t)((c & 1) ? code << 4 : code);
            }
        }
    }
    return 0;
}

/* The 512 decoded values of main-KV entry i: E2M1(code) * E4M3(scale). */
void hsio_mainkv_decode(const uint8_t* kv, int64_t i, double* out) {
    const uint8_t* e = kv + i * KV_BYTES;
    for (int c = 0; c < KV_DIM; ++c) {
        uint8_t code = (c & 1) ? (uint8_t)(e[c / 2] >> 4) : (uint8_t)(e[c / 2] & 15);
        out[c] = hsio_e2m1_value(code) * hsio_e4m3_value(e[256 + c / 16]);
    }
}

/* gather(main_kv, topk) for one query: row t of out (bf16 bits [k][512]) is
 * entry idx[t] of the cache decoded, zeros where idx[t] < 0 (padding).
 * Returns 0, -1 if an index is at or past n_vis, -2 if a decoded value is
 * not exact in bf16 (impossible for these formats; checked anyway). */
int hsio_mainkv_gather(const uint8_t* kv, int64_t n_vis, const int32_t* idx, int k, uint16_t* out) {
    double d[KV_DIM];
    for (int t = 0; t < k; ++t) {
        uint16_t* row = out + (int64_t)t * KV_DIM;
        if (idx[t] < 0) {
            memset(row, 0, KV_DIM * sizeof(uint16_t));
            continue;
        }
        if (idx[t] >= n_vis) return -1;
        hsio_mainkv_decode(kv, idx[t], d);
        for (int c = 0; c < KV_DIM; ++c) {
            float f = (float)d[c];
            uint32_t u;
            memcpy(&u, &f, 4);
            if ((double)f != d[c] || (u & 0xFFFFu)) return -2;
            row[c] = (uint16_t)(u >> 16);
        }
    }
    return 0;
}

/* ---------------------------------------------------------------- score -- */

typedef struct {
    double qv[HEADS][DIM]; /* decoded q without the tensor scale */
    double w[HEADS];
    double scale;          /* g_q * g_k / 128 */
    int fmt;               /* FMT_NVFP4 or FMT_MXFP4, for q and K alike */
} query_ctx;

static void query_setup(query_ctx* c, int fmt, const uint8_t* q_rec, float g_q, const float* w, float g_k) {
    c->fmt = fmt;
    for (int j = 0; j < HEADS; ++j) {
        decode_row_unscaled(fmt, q_rec, j, c->qv[j]);
        c->w[j] = (double)w[j];
    }
    c->scale = (double)g_q * (double)g_k / 128.0;
}

/* I = (g_q g_k / 128) * sum_j w_j * ReLU(qhat_j . khat), qhat/khat without
 * tensor scales. Adds the multiply-adds done to *macs. */
static float score_one(const query_ctx* c, const uint8_t* k_rec, int64_t row, int64_t* macs) {
    double kv[DIM];
    decode_row_unscaled(c->fmt, k_rec, row, kv);
    double acc = 0.0;
    int64_t m = 0;
    for (int j = 0; j < HEADS; ++j) {
        double a = 0.0;
        for (int d = 0; d < DIM; ++d) {
            a += c->qv[j][d] * kv[d];
            ++m;
        }
        acc += c->w[j] * (a > 0.0 ? a : 0.0);
    }
    *macs += m;
    return (float)(c->scale * acc);
}

/* Scores of keys [0, n_vis) of one K cache for one query, records of format
 * fmt (MXFP4: pass g_q = g_k = 1). Returns MACs done. */
int64_t hsio_score_full_fmt(int fmt, const uint8_t* q_rec, float g_q, const float* w, const uint8_t* k_rec,
                            float g_k, int64_t n_vis, float* scores) {
    query_ctx* c = (query_ctx*)malloc(sizeof(query_ctx));
    query_setup(c, fmt, q_rec, g_q, w, g_k);
    int64_t macs = 0;
    for (int64_t s = 0; s < n_vis; ++s) scores[s] = score_one(c, k_rec, s, &macs);
    free(c);
    return macs;
}

int64_t hsio_score_full(const uint8_t* q_rec, float g_q, const float* w, const uint8_t* k_rec, float g_k,
                        int64_t n_vis, float* scores) {
    return hsio_score_full_fmt(FMT_NVFP4, q_rec, g_q, w, k_rec, g_k, n_vis, scores);
}

/* Scores of the listed keys, and for each the parity tolerance
 * 1e-4 * sum_j |w_j| * sum_d |qhat_jd khat_d| (tensor scales and the 2^-7 fold
 * applied, as in the score). */
int64_t hsio_score_rows_fmt(int fmt, const uint8_t* q_rec, float g_q, const float* w, const uint8_t* k_rec,
                            float g_k, const int64_t* rows, int64_t n, float* out, double* tol) {
    query_ctx* c = (query_ctx*)malloc(sizeof(query_ctx));
    query_setup(c, fmt, q_rec, g_q, w, g_k);
    int64_t macs = 0;
    for (int64_t i = 0; i < n; ++i) {
        out[i] = score_one(c, k_rec, rows[i], &macs);
        if (tol) {
            double kv[DIM];
            decode_row_unscaled(c->fmt, k_rec, rows[i], kv);
            double t = 0.0;
            for (int j = 0; j < HEADS; ++j) {
                double sabs = 0.0;
                for (int d = 0; d < DIM; ++d) sabs += fabs(c->qv[j][d] * kv[d]);
                t += fabs(c->w[j]) * sabs;
            }
            tol[i] = 1e-4 * c->scale * t;
        }
    }
    free(c);
    return macs;
}

int64_t hsio_score_rows(const uint8_t* q_rec, float g_q, const float* w, const uint8_t* k_rec, float g_k,
                        const int64_t* rows, int64_t n, float* out, double* tol) {
    return hsio_score_rows_fmt(FMT_NVFP4, q_rec, g_q, w, k_rec, g_k, rows, n, out, tol);
}

/* ---------------------------------------------------------------- top-k -- */

typedef struct {
    float v;
    int64_t i;
} entry;

static int cmp_desc(const void* pa, const void* pb) {
    const entry* a = (const entry*)pa;
    const entry* b = (const entry*)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->i < b->i) ? -1 : (a->i > b->i);
}

/* The k best of scores[0 .. n_valid), by value desc then index asc (full sort).
 * Writes min(k, n_valid) entries, pads the rest with -1 / -inf. Returns the
 * count written, or -1 if a score is NaN. */
int64_t hsio_topk(const float* scores, int64_t n_valid, int k, int32_t* idx, float* val) {
    entry* e = (entry*)malloc(sizeof(entry) * (size_t)(n_valid > 0 ? n_valid : 1));
    for (int64_t i = 0; i < n_valid; ++i) {
        if (isnan(scores[i])) {
            free(e);
            return -1;
        }
        e[i].v = scores[i];
        e[i].i = i;
    }
    qsort(e, (size_t)n_valid, sizeof(entry), cmp_desc);
    int64_t m = n_valid < k ? n_valid : k;
    for (int64_t t = 0; t < k; ++t) {
        idx[t] = t < m ? (int32_t)e[t].i : -1;
        val[t] = t < m ? e[t].v : -INFINITY;
    }
    free(e);
    return m;
}

/* ----------------------------------------------------------------- pool -- */

/* The candidate pool of one query, following the page's select_candidate_blocks:
 * block max with -inf padding, the newest block pinned to +inf, the top
 * min(n_keep, nblk) blocks, only those with value > -inf kept.
 * Outputs: block_ids[0 .. n_kept) ascending (rest -1), *n_kept, *n_pool = number
 * of visible positions in the pool, mask[0 .. n_vis) as 0/1 when mask != NULL.
 * Returns 0, or -1 on a NaN score. */
int hsio_pool(const float* scores, int64_t n_vis, int bs, int n_keep, int32_t* block_ids,
              int32_t* n_kept_out, int64_t* n_pool_out, uint8_t* mask) {
    int64_t nblk = (n_vis + bs - 1) / bs;
    entry* blk = (entry*)malloc(sizeof(entry) * (size_t)(nblk > 0 ? nblk : 1));
    for (int64_t b = 0; b < nblk; ++b) {
        float m = -INFINITY;
        for (int t = 0; t < bs; ++t) {
            int64_t s = b * bs + t;
            float v = s < n_vis ? scores[s] : -INFINITY;
            if (isnan(v)) {
                free(blk);
                return -1;
            }
            if (v > m) m = v;
        }
        blk[b].v = m;
        blk[b].i = b;
    }
    if (n_vis > 0) blk[(n_vis - 1) / bs].v = INFINITY;
    qsort(blk, (size_t)nblk, sizeof(entry), cmp_desc);
    int64_t take = nblk < n_keep ? nblk : n_keep;
    uint8_t* keep = (uint8_t*)calloc((size_t)(nblk > 0 ? nblk : 1), 1);
    for (int64_t t = 0; t < take; ++t)
        if (blk[t].v > -INFINITY) keep[blk[t].i] = 1;
    int32_t nk = 0;
    int64_t npool = 0;
    for (int64_t b = 0; b < nblk; ++b) {
        if (keep[b]) {
            block_ids[nk++] = (int32_t)b;
            for (int t = 0; t < bs; ++t)
                if (b * bs + t < n_vis) ++npool;
        }
    }
    for (int32_t t = nk; t < n_keep; ++t) block_ids[t] = -1;
    if (mask)
        for (int64_t s = 0; s < n_vis; ++s) mask[s] = keep[s / bs];
    *n_kept_out = nk;
    *n_pool_out = npool;
    free(keep);
    free(blk);
    return 0;
}

/* Reindex scoring restricted to the pool: slot j*bs + r holds the score of
 * position block_ids[j]*bs + r, -inf where that position is not visible and for
 * every slot at or past n_kept*bs, up to n_keep*bs. Returns MACs done. */
int64_t hsio_score_pool_fmt(int fmt, const uint8_t* q_rec, float g_q, const float* w, const uint8_t* k_rec,
                            float g_k, int64_t n_vis, const int32_t* block_ids, int32_t n_kept,
                            int32_t n_keep, int bs, float* pool_scores) {
    query_ctx* c = (query_ctx*)malloc(sizeof(query_ctx));
    query_setup(c, fmt, q_rec, g_q, w, g_k);
    int64_t macs = 0;
    for (int64_t slot = 0; slot < (int64_t)n_keep * bs; ++slot) {
        int64_t j = slot / bs, r = slot % bs;
        float v = -INFINITY;
        if (j < n_kept) {
            int64_t pos = (int64_t)block_ids[j] * bs + r;
            if (pos < n_vis) v = score_one(c, k_rec, pos, &macs);
        }
        pool_scores[slot] = v;
    }
    free(c);
    return macs;
}

int64_t hsio_score_pool(const uint8_t* q_rec, float g_q, const float* w, const uint8_t* k_rec, float g_k,
                        int64_t n_vis, const int32_t* block_ids, int32_t n_kept, int32_t n_keep, int bs,
                        float* pool_scores) {
    return hsio_score_pool_fmt(FMT_NVFP4, q_rec, g_q, w, k_rec, g_k, n_vis, block_ids, n_kept, n_keep, bs,
                               pool_scores);
}

/* Top-k inside the pool, reported as global positions: the pool-local top-k of
 * pool_scores[0 .. n_pool), slot i mapped to block_ids[i/bs]*bs + i%bs. */
int64_t hsio_topk_pool(const float* pool_scores, int64_t n_pool, const int32_t* block_ids, int bs,
                       int k, int32_t* idx, float* val) {
    int64_t m = hsio_topk(pool_scores, n_pool, k, idx, val);
    for (int64_t t = 0; t < m; ++t) idx[t] = block_ids[idx[t] / bs] * bs + idx[t] % bs;
    return m;
}

/* The page's masked form, literally: score every visible position, set the
 * positions outside the pool mask to -inf, take the top-k of what is left
 * (eligible = pool positions). Used to cross-check the pooled path. */
int64_t hsio_topk_masked(const float* scores_all, int64_t n_vis, const uint8_t* mask, int k,
                         int32_t* idx, float* val) {
    float* masked = (float*)malloc(sizeof(float) * (size_t)(n_vis > 0 ? n_vis : 1));
    int64_t n_in = 0;
    for (int64_t s = 0; s < n_vis; ++s) {
        masked[s] = mask[s] ? scores_all[s] : -INFINITY;
        n_in += mask[s] ? 1 : 0;
    }
    entry* e = (entry*)malloc(sizeof(entry) * (size_t)(n_vis > 0 ? n_vis : 1));
    for (int64_t s = 0; s < n_vis; ++s) {
        e[s].v = masked[s];
        e[s].i = s;
    }
    qsort(e, (size_t)n_vis, sizeof(entry), cmp_desc);
    int64_t m = n_in < k ? n_in : k;
    for (int64_t t = 0; t < k; ++t) {
        idx[t] = t < m ? (int32_t)e[t].i : -1;
        val[t] = t < m ? e[t].v : -INFINITY;
    }
    free(e);
    free(masked);
    return m;
}
