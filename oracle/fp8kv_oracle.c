/*
 * fp8kv_oracle.c -- plain, slow, single-threaded CPU oracle for the FP8 paged
 * KV-cache hot path.  TEST INFRASTRUCTURE ONLY: the product library never links,
 * loads or calls this file; only the tests, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it computes (sources are the four "b70-optimization-lab" pages):
 *  - E4M3FN codec: the OCP 8-bit float with 4 exponent bits (bias 7), 3 mantissa
 *    bits, no infinities, S.1111.111 = NaN, largest finite 448.  The KV cache is
 *    "explicit E4M3 FP8" ("Laguna S 2.1 INT4 -- calibrated FP8 KV on Intel B70",
 *    section "Contract"); the FN flavour is the one the campaign ledger names
 *    ("Laguna S 2.1 B70 campaign transfer ledger", table "Result progression").
 *  - Cache insert: "quantize, store FP8" ("Laguna S 2.1 KV-cache precision
 *    decision", section "BF16 versus FP8 in concrete terms", property table,
 *    row "Cache write/read work") with one static symmetric per-tensor scalar
 *    scale per K and per V (same page, section "What the official checkpoint
 *    requests": kv_cache_scheme with strategy "tensor", symmetric, dynamic false).
 *    Reading: stored code = E4M3(fp32(x) / scale), round to nearest even,
 *    saturating to +-448.
 *  - Per-head scales (an extension the pages do not use: the checkpoint asks for
 *    strategy "tensor"): one scale per KV head for K and one for V, each the
 *    same kind of static symmetric scalar; every element of head h is encoded
 *    and decoded with that head's scale, nothing else changes.
 *  - Q/K RMSNorm + RoPE ahead of the insert ("calibrated FP8 KV on Intel B70",
 *    section "Initial optimization order", item 3; ledger table "Result
 *    progression", row "Exact fusion stack").  The pages give no epsilon, no
 *    rotary style and no precision; the op order below is the reading chosen so
 *    that the FP8 bytes are reproducible bit for bit.
 *  - Exact paged attention over the dequantized cache ("calibrated FP8 KV on
 *    Intel B70", "Initial optimization order", item 2: exact q1/M12 paged
 *    attention), in float64, with GQA, a causal mask among the M new rows and an
 *    optional sliding window ("KV-cache precision decision", section "BF16
 *    versus FP8 in concrete terms": 36 sliding-window layers of 512 and 12
 *    global layers).
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (no fast-math): every
 * fp32 operation below must round exactly as written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1

/* ------------------------------------------------------------------ bits */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bfloat16 is the top half of an fp32 bit pattern. */
static float bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* fp32 -> bfloat16, round to nearest, ties to even (NaN kept quiet). */
static uint16_t f32_to_bf16(float f)
{
    uint32_t u = f32_bits(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* --------------------------------------------------------------- E4M3FN */

/* Decode one E4M3FN code: sign bit 7, exponent bits 6..3 (bias 7), mantissa
 * bits 2..0.  Exponent field 0 is subnormal (m * 2^-9); S.1111.111 is NaN. */
double oracle_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m, -9);
    else mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Encode an fp32 value to E4M3FN: NaN -> 0x7F with the input's sign bit;
 * |x| >= 448 (infinities included) saturates to +-448 (0x7E / 0xFE);
 * otherwise round |x| to the nearest point of the E4M3 grid, ties to the even
 * code.  The grid spacing is 2^(e-3) in binade [2^e, 2^(e+1)) for e >= -6 and
 * 2^-9 below 2^-6 (subnormals).  Integer arithmetic on the fp32 bits keeps the
 * rounding exact (no double rounding). */
uint8_t oracle_e4m3_encode(float x)
{
    uint32_t u = f32_bits(x);
    uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return (uint8_t)(sign | 0x7f);           /* NaN */
    if (a >= 0x43e00000u) return (uint8_t)(sign | 0x7e);          /* >= 448 */
    if (a == 0) return sign;                                      /* +-0 */
    int be = (int)(a >> 23);                                      /* biased exp */
    uint32_t mant;
    int e;                                                        /* |x| = mant * 2^(e-23) */
    if (be == 0) { mant = a & 0x7fffffu; e = -126; }              /* fp32 subnormal */
    else { mant = (a & 0x7fffffu) | 0x800000u; e = be - 127; }
    int eq = (e < -6 ? -6 : e);                                   /* grid binade */
    int qe = eq - 3;                                              /* grid step 2^qe */
    int shift = 23 + qe - e;                                      /* >= 20 */
    uint32_t q;
    if (shift >= 25) {
        q = 0;                                                    /* below half a step */
    } else {
        uint32_t rem = mant & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        q = mant >> shift;
        if (rem > half || (rem == half && (q & 1u))) q += 1u;
    }
    /* value = q * 2^qe; code = 8 * (eq + 6) + q carries into the exponent field
     * when q reaches 16, and gives the subnormal codes for eq == -6, q < 8. */
    uint32_t code = 8u * (uint32_t)(eq + 6) + q;
    return (uint8_t)(sign | code);
}

void oracle_e4m3_encode_array(const float* x, size_t n, uint8_t* out)
{
    for (size_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t* c, size_t n, double* out)
{
    for (size_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
}

/* ---------------------------------------------------------------- insert */

/* Cache layout: [num_pages][Hkv][page_size][D]; slot s lives in page
 * s / page_size at offset s % page_size.  Negative slots are skipped. */
static size_t cache_index(int64_t slot, int h, int d, int Hkv, int page_size, int D)
{
    int64_t page = slot / page_size, off = slot % page_size;
    return (((size_t)page * Hkv + h) * page_size + (size_t)off) * D + d;
}

/* cache_dtype 0 = E4M3 bytes, 1 = bfloat16 (stored unchanged, scales unused). */
int oracle_cache_insert(const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
                        int T, int Hkv, int D, float k_scale, float v_scale,
                        void* k_cache, void* v_cache, int num_pages, int page_size,
                        int cache_dtype)
{
    if (T < 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages < 0) return ORACLE_BAD_ARG;
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_pages * page_size) return ORACLE_BAD_ARG;
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < D; ++d) {
                size_t src = ((size_t)t * Hkv + h) * D + d;
                size_t dst = cache_index(slot, h, d, Hkv, page_size, D);
                if (cache_dtype == 0) {
                    float xk = bf16_to_f32(k[src]) / k_scale;
                    float xv = bf16_to_f32(v[src]) / v_scale;
                    ((uint8_t*)k_cache)[dst] = oracle_e4m3_encode(xk);
                    ((uint8_t*)v_cache)[dst] = oracle_e4m3_encode(xv);
                } else {
                    ((uint16_t*)k_cache)[dst] = k[src];
                    ((uint16_t*)v_cache)[dst] = v[src];
                }
            }
        }
    }
    return ORACLE_OK;
}

/* Per-head scales: head h of K (V) is encoded with k_scale[h] (v_scale[h]);
 * E4M3 cache only. */
int oracle_cache_insert_per_head(const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
                                 int T, int Hkv, int D, const float* k_scale, const float* v_scale,
                                 uint8_t* k_cache, uint8_t* v_cache, int num_pages, int page_size)
{
    if (T < 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages < 0) return ORACLE_BAD_ARG;
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_pages * page_size) return ORACLE_BAD_ARG;
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < D; ++d) {
                size_t src = ((size_t)t * Hkv + h) * D + d;
                size_t dst = cache_index(slot, h, d, Hkv, page_size, D);
                k_cache[dst] = oracle_e4m3_encode(bf16_to_f32(k[src]) / k_scale[h]);
                v_cache[dst] = oracle_e4m3_encode(bf16_to_f32(v[src]) / v_scale[h]);
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------ RMSNorm and RoPE */

/* Rotary table, one row per position: cos of the D/2 frequencies, then their
 * sines; frequency k is theta^(-2k/D), evaluated in double, rounded to fp32. */
void oracle_rope_table(double theta, int max_pos, int D, float* cos_sin)
{
    int half = D / 2;
    for (int p = 0; p < max_pos; ++p) {
        for (int k = 0; k < half; ++k) {
            double inv_freq = pow(theta, -2.0 * k / (double)D);
            double ang = (double)p * inv_freq;
            cos_sin[(size_t)p * D + k] = (float)cos(ang);
            cos_sin[(size_t)p * D + half + k] = (float)sin(ang);
        }
    }
}

/* One head row: RMSNorm then rotate-half RoPE, all in fp32 with a fixed order.
 *   sum of squares: 32 partial sums, part l covers x[l*E .. l*E+E-1] (E = D/32)
 *     accumulated as fma(x_i, x_i, acc) from acc = x_0*x_0; the 32 parts are
 *     then added pairwise (l with l+16, then +8, +4, +2, +1).
 *   r = 1 / sqrt(ss / D + eps)                (IEEE sqrt and divide)
 *   n = bf16(x * r); y = bf16(n * w)
 *   o_k   = bf16(fma(y_k,   c_k, -(y_k+h * s_k)))
 *   o_k+h = bf16(fma(y_k+h, c_k,  (y_k   * s_k)))      h = D/2
 * Output is bf16 bits. */
int oracle_norm_rope_row(const uint16_t* x, const uint16_t* w, float eps,
                         const float* cs_row, int D, uint16_t* out)
{
    if (D <= 0 || D % 64 != 0 || D > 1024) return ORACLE_BAD_ARG;
    int E = D / 32, half = D / 2;
    float part[32];
    for (int l = 0; l < 32; ++l) {
        float x0 = bf16_to_f32(x[l * E]);
        float acc = x0 * x0;
        for (int i = 1; i < E; ++i) {
            float xi = bf16_to_f32(x[l * E + i]);
            acc = fmaf(xi, xi, acc);
        }
        part[l] = acc;
    }
    for (int width = 16; width >= 1; width /= 2)
        for (int l = 0; l < width; ++l) part[l] = part[l] + part[l + width];
    float ss = part[0];
    float r = 1.0f / sqrtf(ss / (float)D + eps);
    float y[1024];
    for (int i = 0; i < D; ++i) {
        float n = bf16_to_f32(f32_to_bf16(bf16_to_f32(x[i]) * r));
        y[i] = bf16_to_f32(f32_to_bf16(n * bf16_to_f32(w[i])));
    }
    for (int k = 0; k < half; ++k) {
        float c = cs_row[k], s = cs_row[half + k];
        float t1 = y[k + half] * s;
        float t2 = y[k] * s;
        out[k] = f32_to_bf16(fmaf(y[k], c, -t1));
        out[k + half] = f32_to_bf16(fmaf(y[k + half], c, t2));
    }
    return ORACLE_OK;
}

/* Fused boundary: Q and K heads get RMSNorm + RoPE at their token's position;
 * V gets neither; the rotated K and the raw V are then inserted as E4M3. */
int oracle_qk_norm_rope_insert(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const int64_t* positions, const uint16_t* q_norm_w,
                               const uint16_t* k_norm_w, float eps, const float* cos_sin,
                               int max_pos, uint16_t* q_out, const int64_t* slot_mapping,
                               int T, int Hq, int Hkv, int D, float k_scale, float v_scale,
                               uint8_t* k_cache, uint8_t* v_cache, int num_pages, int page_size)
{
    if (T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || D % 64 != 0 || D > 1024) return ORACLE_BAD_ARG;
    uint16_t row[1024];
    for (int t = 0; t < T; ++t) {
        int64_t pos = positions[t];
        if (pos < 0 || pos >= max_pos) return ORACLE_BAD_ARG;
        const float* cs = cos_sin + (size_t)pos * D;
        for (int h = 0; h < Hq; ++h) {
            size_t base = ((size_t)t * Hq + h) * D;
            int rc = oracle_norm_rope_row(q + base, q_norm_w, eps, cs, D, q_out + base);
            if (rc) return rc;
        }
        int64_t slot = slot_mapping[t];
        if (slot >= (int64_t)num_pages * page_size) return ORACLE_BAD_ARG;
        for (int h = 0; h < Hkv; ++h) {
            size_t base = ((size_t)t * Hkv + h) * D;
            int rc = oracle_norm_rope_row(k + base, k_norm_w, eps, cs, D, row);
            if (rc) return rc;
            if (slot < 0) continue;
            for (int d = 0; d < D; ++d) {
                size_t dst = cache_index(slot, h, d, Hkv, page_size, D);
                k_cache[dst] = oracle_e4m3_encode(bf16_to_f32(row[d]) / k_scale);
                v_cache[dst] = oracle_e4m3_encode(bf16_to_f32(v[base + d]) / v_scale);
            }
        }
    }
    return ORACLE_OK;
}

/* -------------------------------------------------------------- attention */

typedef struct {
    const uint16_t* q;            /* bf16 [B][M][Hq][D] */
    const void* k_cache;          /* [num_pages][Hkv][ps][D], E4M3 bytes or bf16 */
    const void* v_cache;
    int cache_dtype;              /* 0 = E4M3, 1 = bf16 */
    const int32_t* block_table;   /* [B][max_pages_per_seq] */
    int max_pages_per_seq;
    const int32_t* seq_lens;      /* [B], context length including the M new rows */
    int B, M, Hq, Hkv, D, page_size, num_pages;
    double k_scale, v_scale, sm_scale;
    int window_left;              /* -1: global; else keys j >= p - window_left */
    const double* k_scale_h;      /* per-head scales [Hkv] (E4M3), or NULL: k_scale, v_scale */
    const double* v_scale_h;
} attn_args;

/* Dequantized element d of key/value j (logical position) for kv head hk. */
static double cache_value(const attn_args* a, const void* cache, double scale,
                          int b, int hk, int j, int d, int* bad)
{
    int32_t page = a->block_table[(size_t)b * a->max_pages_per_seq + j / a->page_size];
    if (page < 0 || page >= a->num_pages) { *bad = 1; return 0.0; }
    size_t idx = (((size_t)page * a->Hkv + hk) * a->page_size + (size_t)(j % a->page_size)) * a->D + d;
    if (a->cache_dtype == 0) return oracle_e4m3_decode(((const uint8_t*)cache)[idx]) * scale;
    return (double)bf16_to_f32(((const uint16_t*)cache)[idx]);
}

/* Visible keys of query row m in sequence b: [lo, p] with p = L - M + m. */
static void visible_range(const attn_args* a, int b, int m, int* lo, int* hi)
{
    int L = a->seq_lens[b];
    int p = L - a->M + m;
    int l = 0;
    if (a->window_left >= 0 && p - a->window_left > 0) l = p - a->window_left;
    *lo = l;
    *hi = p;
}

/* Partial softmax over keys [j0, j1] of one row: returns the max logit mx, the
 * sum of exp(s - mx) in *l and the unnormalised sum of exp(s - mx) * Vd in acc.
 * An empty range gives mx = -inf, l = 0, acc = 0. */
static int row_partial(const attn_args* a, int b, int m, int h, int j0, int j1,
                       double* mx_out, double* l_out, double* acc, double* scratch_s)
{
    int G = a->Hq / a->Hkv, hk = h / G, D = a->D, bad = 0;
    const uint16_t* q = a->q + (((size_t)b * a->M + m) * a->Hq + h) * D;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    if (j1 < j0) { *mx_out = -INFINITY; *l_out = 0.0; return 0; }
    double k_scale = a->cache_dtype == 0 ? (a->k_scale_h ? a->k_scale_h[hk] : a->k_scale) : 1.0;
    double v_scale = a->cache_dtype == 0 ? (a->v_scale_h ? a->v_scale_h[hk] : a->v_scale) : 1.0;
    double mx = -INFINITY;
    for (int j = j0; j <= j1; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += (double)bf16_to_f32(q[d]) * cache_value(a, a->k_cache, k_scale, b, hk, j, d, &bad);
        double s = dot * a->sm_scale;
        scratch_s[j - j0] = s;
        if (s > mx) mx = s;
    }
    double l = 0.0;
    for (int j = j0; j <= j1; ++j) {
        double w = exp(scratch_s[j - j0] - mx);
        l += w;
        for (int d = 0; d < D; ++d)
            acc[d] += w * cache_value(a, a->v_cache, v_scale, b, hk, j, d, &bad);
    }
    *mx_out = mx;
    *l_out = l;
    return bad;
}

static int check_args(const attn_args* a)
{
    if (a->B < 0 || a->M < 1 || a->Hq <= 0 || a->Hkv <= 0 || a->Hq % a->Hkv) return ORACLE_BAD_ARG;
    if (a->D <= 0 || a->page_size <= 0 || a->max_pages_per_seq <= 0) return ORACLE_BAD_ARG;
    for (int b = 0; b < a->B; ++b) {
        int L = a->seq_lens[b];
        if (L < a->M || (L + a->page_size - 1) / a->page_size > a->max_pages_per_seq) return ORACLE_BAD_ARG;
    }
    return ORACLE_OK;
}

/* Attention for selected rows; rows[3*i..3*i+2] = (b, m, h); out [n_rows][D]. */
static int attention_rows_impl(const attn_args* a, const int32_t* rows, int n_rows,
                               int split_tokens, double* out)
{
    int rc = check_args(a);
    if (rc) return rc;
    int maxL = 0;
    for (int b = 0; b < a->B; ++b) if (a->seq_lens[b] > maxL) maxL = a->seq_lens[b];
    double* s = (double*)malloc(sizeof(double) * (size_t)(maxL + 1));
    double* acc = (double*)malloc(sizeof(double) * (size_t)a->D);
    double* tot = (double*)malloc(sizeof(double) * (size_t)a->D);
    if (!s || !acc || !tot) { free(s); free(acc); free(tot); return ORACLE_BAD_ARG; }
    for (int i = 0; i < n_rows && rc == 0; ++i) {
        int b = rows[3 * i], m = rows[3 * i + 1], h = rows[3 * i + 2];
        if (b < 0 || b >= a->B || m < 0 || m >= a->M || h < 0 || h >= a->Hq) { rc = ORACLE_BAD_ARG; break; }
        int lo, hi;
        visible_range(a, b, m, &lo, &hi);
        double* o = out + (size_t)i * a->D;
        if (split_tokens <= 0) {
            /* plain definition: one softmax over all visible keys */
            double mx, l;
            if (row_partial(a, b, m, h, lo, hi, &mx, &l, acc, s)) { rc = ORACLE_BAD_ARG; break; }
            for (int d = 0; d < a->D; ++d) o[d] = acc[d] / l;
        } else {
            /* partitions [p*S, (p+1)*S) of the key axis, combined through
             * their log-sum-exp: O = sum_p e^(m_p - m*) acc_p / sum_p e^(m_p - m*) l_p */
            int np = hi / split_tokens + 1;
            double* pm = (double*)malloc(sizeof(double) * (size_t)np);
            double* pl = (double*)malloc(sizeof(double) * (size_t)np);
            double* pacc = (double*)malloc(sizeof(double) * (size_t)np * a->D);
            if (!pm || !pl || !pacc) { free(pm); free(pl); free(pacc); rc = ORACLE_BAD_ARG; break; }
            double mstar = -INFINITY;
            for (int p = 0; p < np; ++p) {
                int j0 = p * split_tokens, j1 = (p + 1) * split_tokens - 1;
                if (j0 < lo) j0 = lo;
                if (j1 > hi) j1 = hi;
                if (row_partial(a, b, m, h, j0, j1, &pm[p], &pl[p], pacc + (size_t)p * a->D, s)) rc = ORACLE_BAD_ARG;
                if (pm[p] > mstar) mstar = pm[p];
            }
            double den = 0.0;
            for (int d = 0; d < a->D; ++d) tot[d] = 0.0;
            for (int p = 0; p < np; ++p) {
                if (pl[p] == 0.0) continue;
                double f = exp(pm[p] - mstar);
                den += f * pl[p];
                for (int d = 0; d < a->D; ++d) tot[d] += f * pacc[(size_t)p * a->D + d];
            }
            for (int d = 0; d < a->D; ++d) o[d] = tot[d] / den;
            free(pm); free(pl); free(pacc);
        }
    }
    free(s); free(acc); free(tot);
    return rc;
}

#define ATTN_PARAMS                                                                     \
    const uint16_t *q, const void *k_cache, const void *v_cache, int cache_dtype,        \
        const int32_t *block_table, int max_pages_per_seq, const int32_t *seq_lens,      \
        int B, int M, int Hq, int Hkv, int D, int page_size, int num_pages,              \
        double k_scale, double v_scale, double sm_scale, int window_left

#define ATTN_INIT                                                                       \
    attn_args a = {q, k_cache, v_cache, cache_dtype, block_table, max_pages_per_seq,     \
                   seq_lens, B, M, Hq, Hkv, D, page_size, num_pages, k_scale, v_scale,  \
                   sm_scale, window_left, NULL, NULL}

int oracle_paged_attention_rows(ATTN_PARAMS, const int32_t* rows, int n_rows, double* out)
{
    ATTN_INIT;
    return attention_rows_impl(&a, rows, n_rows, 0, out);
}

int oracle_paged_attention_split_rows(ATTN_PARAMS, int split_tokens, const int32_t* rows,
                                      int n_rows, double* out)
{
    ATTN_INIT;
    if (split_tokens <= 0) return ORACLE_BAD_ARG;
    return attention_rows_impl(&a, rows, n_rows, split_tokens, out);
}

/* All rows; out is [B][M][Hq][D]. */
int oracle_paged_attention(ATTN_PARAMS, double* out)
{
    ATTN_INIT;
    size_t n = (size_t)B * M * Hq;
    int32_t* rows = (int32_t*)malloc(sizeof(int32_t) * 3 * (n ? n : 1));
    if (!rows) return ORACLE_BAD_ARG;
    size_t i = 0;
    for (int b = 0; b < B; ++b)
        for (int m = 0; m < M; ++m)
            for (int h = 0; h < Hq; ++h) {
                rows[3 * i] = b; rows[3 * i + 1] = m; rows[3 * i + 2] = h;
                ++i;
            }
    int rc = attention_rows_impl(&a, rows, (int)n, 0, out);
    free(rows);
    return rc;
}

/* All rows over an E4M3 cache with per-head scales k_scale[Hkv], v_scale[Hkv];
 * out is [B][M][Hq][D]. */
int oracle_paged_attention_per_head(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                    const int32_t* block_table, int max_pages_per_seq,
                                    const int32_t* seq_lens, int B, int M, int Hq, int Hkv, int D,
                                    int page_size, int num_pages, const double* k_scale,
                                    const double* v_scale, double sm_scale, int window_left, double* out)
{
    attn_args a = {q, k_cache, v_cache, 0, block_table, max_pages_per_seq, seq_lens, B, M, Hq, Hkv, D,
                   page_size, num_pages, 0.0, 0.0, sm_scale, window_left, k_scale, v_scale};
    size_t n = (size_t)B * M * Hq;
    int32_t* rows = (int32_t*)malloc(sizeof(int32_t) * 3 * (n ? n : 1));
    if (!rows) return ORACLE_BAD_ARG;
    size_t i = 0;
    for (int b = 0; b < B; ++b)
        for (int m = 0; m < M; ++m)
            for (int h = 0; h < Hq; ++h) {
                rows[3 * i] = b; rows[3 * i + 1] = m; rows[3 * i + 2] = h;
                ++i;
            }
    int rc = attention_rows_impl(&a, rows, (int)n, 0, out);
    free(rows);
    return rc;
}

/* Encode the fp32 bit patterns first .. first+n-1 (exhaustive encoder checks). */
void oracle_e4m3_encode_bits_range(uint32_t first, size_t n, uint8_t* out)
{
    for (size_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(bits_f32(first + (uint32_t)i));
}
