/*
 * pa_oracle.c -- plain, slow, CPU reference for paged-KV decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This library exists to check the CUDA path; it is
 * never part of it.  Only the test suite, the smoke check in __graft_entry__ and
 * the CPU-baseline / reference legs of bench.py may load it.  It shares no code,
 * header, table or constant with the CUDA library, and it includes nothing from
 * the package.
 *
 * Every function computes the plain definition of its step, in double precision
 * unless the step itself fixes another precision (the FP8 writer is defined in
 * fp32 arithmetic, see oracle_reshape_and_cache_fp8).  No blocking, fusion,
 * online softmax or reordering beyond what the definition states.
 *
 * Sources (web pages this method is described on):
 *   [P1] "appendonly" (rajatmohan.com), sections "Paging, because contiguous
 *        allocation is a disaster" and "Prefix sharing is where the real win lives".
 *   [P3] "KV Cache Engineering for LLM Serving" (dailydoseofds), sections
 *        1 "GQA and MQA cache fewer heads", 8 "Quantization", 10 "Paging".
 *   [P4] "Taming the Token Torrent" (architects-blueprint), sections
 *        "The Block Table Logic" and "Custom PagedAttention Kernels".
 *   OCP 8-bit Floating Point Specification (OFP8), E4M3 format.
 *
 * Layouts (all row-major):
 *   q            [B, Hq, D]                 bf16 bit patterns (uint16)
 *   k/v pool     [nblocks, bs, Hkv, D]      bf16 bit patterns, or E4M3 codes (uint8)
 *   k/v scale    [nblocks, Hkv]             fp32 (FP8 pools only)
 *   block_tables [B, max_blocks]            int32
 *   seq_lens     [B]                        int32 (tokens in the cache, incl. this step's)
 *   slot_mapping [T]                        int64 (slot = block * bs + offset; < 0 = skip)
 *   out          [B, Hq, D]                 double
 *
 * Parity status of each function is listed in the header comment of
 * oracle/__init__.py together with the tests that pin it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Scalar formats                                                             */
/* ------------------------------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32. */
static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

double oracle_bf16_to_double(uint16_t h) { return (double)bf16_bits_to_float(h); }

/*
 * OFP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 *   exponent field 0      : subnormal, |x| = 2^-6 * (m / 8)
 *   exponent field 1..15  : normal,    |x| = 2^(e-7) * (1 + m / 8)
 *   S.1111.111            : NaN (the only non-finite encoding; no infinities)
 * Largest finite magnitude: S.1111.110 = 448.
 */
double oracle_e4m3_to_double(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/*
 * Round a float to E4M3, to nearest with ties to the even code, saturating
 * finite values of magnitude >= 448 to +-448 ("satfinite").  NaN maps to the
 * NaN code.  The sign of the input is kept, so values that round to zero give
 * +0 (0x00) or -0 (0x80).
 *
 * Written as the definition: scan the 127 non-negative finite codes (their
 * magnitudes increase with the code), take the two that bracket |x| and pick the
 * nearer one, comparing against their exact midpoint.
 */
uint8_t oracle_e4m3_from_float(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a, lo_v, hi_v, mid;
    int hi;
    if (isnan(x))
        return 0x7F;
    a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    hi = 0;
    while (oracle_e4m3_to_double((uint8_t)hi) < a)
        hi++;                                   /* stops at <= 0x7E since a < 448 */
    hi_v = oracle_e4m3_to_double((uint8_t)hi);
    if (hi_v == a || hi == 0)
        return (uint8_t)(sign | hi);
    lo_v = oracle_e4m3_to_double((uint8_t)(hi - 1));
    mid = 0.5 * (lo_v + hi_v);                  /* exact: both have few significant bits */
    if (a < mid)
        return (uint8_t)(sign | (hi - 1));
    if (a > mid)
        return (uint8_t)(sign | hi);
    return (uint8_t)(sign | (((hi & 1) == 0) ? hi : hi - 1));   /* tie: even code */
}

/* Array forms of the two E4M3 conversions (same definitions, element by element). */
void oracle_e4m3_to_double_array(const uint8_t *c, long long n, double *out)
{
    long long i;
    for (i = 0; i < n; i++)
        out[i] = oracle_e4m3_to_double(c[i]);
}

void oracle_e4m3_from_float_array(const float *x, long long n, uint8_t *out)
{
    long long i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; i++)
        out[i] = oracle_e4m3_from_float(x[i]);
}

/* ------------------------------------------------------------------------- */
/* Small definitions pinned by the pages' printed examples                   */
/* ------------------------------------------------------------------------- */

/* [P3] section 1: query head h reads KV head h / (Hq / Hkv); a group of Hq/Hkv
 * consecutive query heads shares one KV head. */
int oracle_kv_head(int h, int Hq, int Hkv) { return h / (Hq / Hkv); }

/* [P3] "The cache formula" / section 1: scalars cached = 2 (K and V) x KV heads
 * x tokens x head size, per layer. */
long long oracle_cached_scalars(int layers, int Hkv, long long tokens, int D)
{
    return 2LL * layers * Hkv * tokens * D;
}

/*
 * [P3] section 3: a sliding-window layer keeps only the most recent `window`
 * positions.  After a sequence of `len` tokens it retains positions
 * [max(0, len - window), len); window <= 0 means no window (all positions).
 * Writes the retained positions to out and returns how many there are.
 */
int oracle_window_positions(int len, int window, int *out)
{
    int first = (window > 0 && len > window) ? len - window : 0;
    int t, n = 0;
    for (t = first; t < len; t++)
        out[n++] = t;
    return n;
}

/*
 * [P3] section 7 (Quest): a page's summary is the per-channel minimum and maximum
 * of its n keys; a query scores the page by sum_d max(q_d * min_d, q_d * max_d), an
 * upper bound of q . k over the page's keys.  Pages are chosen by score.
 */
void oracle_page_summary(const double *keys, int n, int D, double *mn, double *mx)
{
    int i, d;
    for (d = 0; d < D; d++) {
        mn[d] = keys[d];
        mx[d] = keys[d];
    }
    for (i = 1; i < n; i++)
        for (d = 0; d < D; d++) {
            if (keys[(size_t)i * D + d] < mn[d]) mn[d] = keys[(size_t)i * D + d];
            if (keys[(size_t)i * D + d] > mx[d]) mx[d] = keys[(size_t)i * D + d];
        }
}

/*
 * Directed rounding of a finite double to the bf16 grid: 8 significant bits with
 * fp32's exponent range, subnormal spacing 2^-133.  down: the largest bf16 value
 * <= x; up: the smallest bf16 value >= x.  Used for Quest summaries of quantised
 * pools, whose restored keys (code * scale) are not bf16 values: the minimum is
 * rounded down and the maximum up, so the page score stays an upper bound of q . k.
 */
static double bf16_ulp(double x)
{
    int e;
    (void)frexp(x, &e);                 /* |x| in [2^(e-1), 2^e) */
    if (e < -125) e = -125;             /* below 2^-126: subnormal spacing */
    return ldexp(1.0, e - 8);
}

double oracle_bf16_round_down(double x)
{
    double u;
    if (x == 0.0) return 0.0;
    u = bf16_ulp(x);
    return floor(x / u) * u;
}

double oracle_bf16_round_up(double x)
{
    double u;
    if (x == 0.0) return 0.0;
    u = bf16_ulp(x);
    return ceil(x / u) * u;
}

double oracle_page_score(const double *q, const double *mn, const double *mx, int D)
{
    double s = 0.0;
    int d;
    for (d = 0; d < D; d++) {
        double a = q[d] * mn[d], b = q[d] * mx[d];
        s += (a > b) ? a : b;
    }
    return s;
}

/* The k highest-scoring of n pages (all of them when n <= k), ties to the lower
 * page index, returned in increasing page order.  Returns how many were chosen. */
int oracle_select_pages(const double *scores, int n, int k, int *out)
{
    int i, j, m = (n < k) ? n : k;
    char *taken = (char *)calloc((size_t)(n > 0 ? n : 1), 1);
    for (j = 0; j < m; j++) {
        int best = -1;
        for (i = 0; i < n; i++)
            if (!taken[i] && (best < 0 || scores[i] > scores[best]))
                best = i;
        taken[best] = 1;
    }
    for (i = 0, j = 0; i < n; i++)
        if (taken[i])
            out[j++] = i;
    free(taken);
    return m;
}

/*
 * [P3] section 8: absmax quantiser onto signed integer codes.
 *   scale = max|x| / largest_code, largest_code = 2^(bits-1) - 1
 *   code  = clip(rint(x / scale), -largest_code, largest_code)   (rint: ties to even)
 *   restored = code * scale
 * Double precision, as in the page's example.  A zero absmax gives scale 0 and
 * all-zero codes.
 */
void oracle_quantize_absmax_int(const double *x, int n, int bits, int *codes,
                                double *restored, double *scale_out)
{
    int i, largest = (1 << (bits - 1)) - 1;
    double amax = 0.0, scale;
    for (i = 0; i < n; i++)
        if (fabs(x[i]) > amax)
            amax = fabs(x[i]);
    scale = amax / (double)largest;
    for (i = 0; i < n; i++) {
        double c = (scale == 0.0) ? 0.0 : nearbyint(x[i] / scale);
        if (c > largest) c = largest;
        if (c < -largest) c = -largest;
        codes[i] = (int)c;
        restored[i] = c * scale;
    }
    *scale_out = scale;
}

/* ------------------------------------------------------------------------- */
/* Cache write (reshape_and_cache)                                            */
/* ------------------------------------------------------------------------- */

/*
 * [P4] "How Paging Works": a new token goes into a physical block taken from
 * the pool; [P4] "The Block Table Logic": logical index -> (block, offset).
 * Slot s addresses row (s / bs, s % bs) of the pool.  For each token t with
 * slot_mapping[t] >= 0 the K/V vectors of all KV heads are copied bit for bit:
 *   pool[s / bs][s % bs][h][:] = new[t][h][:]
 * Negative slots are padding and write nothing.
 */
void oracle_reshape_and_cache_bf16(int T, int Hkv, int D, int bs,
                                   const uint16_t *k_new, const uint16_t *v_new,
                                   uint16_t *k_pool, uint16_t *v_pool,
                                   const int64_t *slot_mapping)
{
    int t, h, d;
    for (t = 0; t < T; t++) {
        int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        for (h = 0; h < Hkv; h++)
            for (d = 0; d < D; d++) {
                size_t dst = (((size_t)(s / bs) * bs + (size_t)(s % bs)) * Hkv + h) * D + d;
                size_t src = ((size_t)t * Hkv + h) * D + d;
                k_pool[dst] = k_new[src];
                v_pool[dst] = v_new[src];
            }
    }
}

/*
 * One (block, kv head) of an FP8 pool receives the token vector x[0..D) at
 * offset off.  Reading of [P3] section 8 for a paged cache with one fp32 scale
 * per (block, kv head):
 *   - the scale is absmax / 448 over every value ever written into this
 *     (block, head) since its offset 0 was written (448 = largest E4M3 code),
 *     computed as an fp32 IEEE division.  Writing offset 0 starts afresh.
 *   - code = E4M3(x / scale), fp32 IEEE division, ties-to-even, saturating.
 *   - when a write raises the scale, the codes already stored at offsets
 *     0..off-1 are re-encoded from their restored values:
 *       restored = float(E4M3 value) * old_scale   (one fp32 product)
 *       code'    = E4M3(restored / new_scale)
 *   - a zero scale stores +0 codes.
 * Because fp32 division is monotone, keeping max(old, absmax_new / 448) equals
 * absmax_over_all / 448.
 */
static void fp8_write_row(uint8_t *pool, float *scale, int Hkv, int D, int bs,
                          int64_t blk, int off, int h, const uint16_t *x)
{
    float amax = 0.0f, cand, old, s_new;
    int d, r;
    float *sp = &scale[blk * Hkv + h];
    for (d = 0; d < D; d++) {
        float v = fabsf(bf16_bits_to_float(x[d]));
        if (v > amax)
            amax = v;
    }
    cand = amax / 448.0f;
    old = *sp;
    s_new = (off == 0 || cand > old) ? cand : old;
    if (off > 0 && s_new > old) {
        for (r = 0; r < off; r++)
            for (d = 0; d < D; d++) {
                uint8_t *c = &pool[(((size_t)blk * bs + r) * Hkv + h) * D + d];
                float restored = (float)oracle_e4m3_to_double(*c) * old;
                *c = (s_new == 0.0f) ? 0x00 : oracle_e4m3_from_float(restored / s_new);
            }
    }
    for (d = 0; d < D; d++) {
        float v = bf16_bits_to_float(x[d]);
        pool[(((size_t)blk * bs + off) * Hkv + h) * D + d] =
            (s_new == 0.0f) ? 0x00 : oracle_e4m3_from_float(v / s_new);
    }
    *sp = s_new;
}

/* FP8 variant of the cache write: the slot mapping of oracle_reshape_and_cache_bf16
 * and the per-(block, head) quantiser of fp8_write_row.  Tokens are applied in
 * index order. */
void oracle_reshape_and_cache_fp8(int T, int Hkv, int D, int bs,
                                  const uint16_t *k_new, const uint16_t *v_new,
                                  uint8_t *k_pool, uint8_t *v_pool,
                                  float *k_scale, float *v_scale,
                                  const int64_t *slot_mapping)
{
    int t, h;
    for (t = 0; t < T; t++) {
        int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        for (h = 0; h < Hkv; h++) {
            fp8_write_row(k_pool, k_scale, Hkv, D, bs, s / bs, (int)(s % bs), h,
                          &k_new[((size_t)t * Hkv + h) * D]);
            fp8_write_row(v_pool, v_scale, Hkv, D, bs, s / bs, (int)(s % bs), h,
                          &v_new[((size_t)t * Hkv + h) * D]);
        }
    }
}

/*
 * 4-bit variant of the cache write ([P3] section 8 with bits = 4, largest code
 * 7), per (block, kv head) and separately for K and V, with the same reading as
 * the FP8 writer:
 *   scale = absmax of all values written since offset 0 / 7 (fp32 division);
 *   code  = clip(rint(x / scale), -7, 7) (fp32 division, ties to even);
 *   a write that raises the scale re-encodes rows 0..off-1 from
 *   restored = code * old_scale (fp32 product); a zero scale stores code 0.
 * Storage: a code is kept as the nibble code + 8 (offset binary, 1..15); the
 * byte at column j of a row holds elements 2j (low nibble) and 2j + 1 (high).
 */
static int int4_get(const uint8_t *row, int d)
{
    int nib = (d & 1) ? (row[d >> 1] >> 4) : (row[d >> 1] & 0xF);
    return nib - 8;
}

static void int4_put(uint8_t *row, int d, int code)
{
    uint8_t nib = (uint8_t)(code + 8);
    if (d & 1)
        row[d >> 1] = (uint8_t)((row[d >> 1] & 0x0F) | (nib << 4));
    else
        row[d >> 1] = (uint8_t)((row[d >> 1] & 0xF0) | nib);
}

static int int4_code(float x, float scale)
{
    float c;
    if (scale == 0.0f)
        return 0;
    c = nearbyintf(x / scale);
    if (c > 7.0f) c = 7.0f;
    if (c < -7.0f) c = -7.0f;
    return (int)c;
}

static void int4_write_row(uint8_t *pool, float *scale, int Hkv, int D, int bs,
                           int64_t blk, int off, int h, const uint16_t *x)
{
    float amax = 0.0f, cand, old, s_new;
    int d, r;
    float *sp = &scale[blk * Hkv + h];
    size_t rowb = (size_t)D / 2;
    for (d = 0; d < D; d++) {
        float v = fabsf(bf16_bits_to_float(x[d]));
        if (v > amax)
            amax = v;
    }
    cand = amax / 7.0f;
    old = *sp;
    s_new = (off == 0 || cand > old) ? cand : old;
    if (off > 0 && s_new > old) {
        for (r = 0; r < off; r++) {
            uint8_t *row = &pool[(((size_t)blk * bs + r) * Hkv + h) * rowb];
            for (d = 0; d < D; d++) {
                float restored = (float)int4_get(row, d) * old;
                int4_put(row, d, int4_code(restored, s_new));
            }
        }
    }
    {
        uint8_t *row = &pool[(((size_t)blk * bs + off) * Hkv + h) * rowb];
        for (d = 0; d < D; d++)
            int4_put(row, d, int4_code(bf16_bits_to_float(x[d]), s_new));
    }
    *sp = s_new;
}

void oracle_reshape_and_cache_int4(int T, int Hkv, int D, int bs,
                                   const uint16_t *k_new, const uint16_t *v_new,
                                   uint8_t *k_pool, uint8_t *v_pool,
                                   float *k_scale, float *v_scale,
                                   const int64_t *slot_mapping)
{
    int t, h;
    for (t = 0; t < T; t++) {
        int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        for (h = 0; h < Hkv; h++) {
            int4_write_row(k_pool, k_scale, Hkv, D, bs, s / bs, (int)(s % bs), h,
                           &k_new[((size_t)t * Hkv + h) * D]);
            int4_write_row(v_pool, v_scale, Hkv, D, bs, s / bs, (int)(s % bs), h,
                           &v_new[((size_t)t * Hkv + h) * D]);
        }
    }
}

/* Restored values of one 4-bit row: (nibble - 8) * scale, exactly in double. */
void oracle_int4_restore(const uint8_t *row, int D, float scale, double *out)
{
    int d;
    for (d = 0; d < D; d++)
        out[d] = (double)int4_get(row, d) * (double)scale;
}

/* ------------------------------------------------------------------------- */
/* Decode attention                                                           */
/* ------------------------------------------------------------------------- */

typedef struct {
    int Hq, Hkv, D, bs, max_blocks, kv_kind;
    const void *k_pool, *v_pool;
    const float *k_scale, *v_scale;
    const int32_t *block_tables;
} paged_kv;

/* Gather: the key (or value) row of logical token t of sequence b, KV head kvh
 * ([P4] "The Block Table Logic"; [P1] "Paging"):
 *   block = block_tables[b][t / bs], row = pool[block][t % bs][kvh][:]
 * written into dst[0..D) as doubles.  FP8 and 4-bit pools are restored as
 * code value * scale[block][kvh], exactly in double (kv_kind: 0 bf16, 1 E4M3,
 * 2 4-bit). */
/* Row (blk, off, kvh) of one pool, restored into dst[0..D) as doubles. */
static void pool_row(int Hkv, int D, int bs, int kv_kind, const void *pool, const float *sc,
                     long long blk, int off, int kvh, double *dst)
{
    size_t idx = (((size_t)blk * bs + (size_t)off) * Hkv + kvh) * D;
    int d;
    if (kv_kind == 0) {
        for (d = 0; d < D; d++)
            dst[d] = oracle_bf16_to_double(((const uint16_t *)pool)[idx + d]);
    } else if (kv_kind == 2) {
        oracle_int4_restore(&((const uint8_t *)pool)[idx / 2], D, sc[(size_t)blk * Hkv + kvh],
                            dst);
    } else {
        double scale = (double)sc[(size_t)blk * Hkv + kvh];
        for (d = 0; d < D; d++)
            dst[d] = oracle_e4m3_to_double(((const uint8_t *)pool)[idx + d]) * scale;
    }
}

static void kv_row(const paged_kv *p, int is_v, int b, int t, int kvh, double *dst)
{
    int32_t blk = p->block_tables[(size_t)b * p->max_blocks + t / p->bs];
    pool_row(p->Hkv, p->D, p->bs, p->kv_kind, is_v ? p->v_pool : p->k_pool,
             is_v ? p->v_scale : p->k_scale, blk, t % p->bs, kvh, dst);
}

/*
 * Quest's stored summary ([P3] section 7) of pool page `page` (pool rows
 * 16 page .. 16 page + rows - 1, i.e. slots of one block) for KV head kvh: the
 * per-channel minimum and maximum of the restored keys (oracle_page_summary),
 * the minimum rounded down and the maximum up to bf16.
 */
void oracle_quest_page_summary(int Hkv, int D, int bs, int kv_kind, const void *k_pool,
                               const float *k_scale, long long page, int rows, int kvh,
                               double *mn, double *mx)
{
    double *keys = (double *)malloc(sizeof(double) * 16 * (size_t)D);
    int t, d;
    for (t = 0; t < rows; t++) {
        long long r = 16 * page + t;
        pool_row(Hkv, D, bs, kv_kind, k_pool, k_scale, r / bs, (int)(r % bs), kvh,
                 &keys[(size_t)t * D]);
    }
    oracle_page_summary(keys, rows, D, mn, mx);
    for (d = 0; d < D; d++) {
        mn[d] = oracle_bf16_round_down(mn[d]);
        mx[d] = oracle_bf16_round_up(mx[d]);
    }
    free(keys);
}

/*
 * Textbook attention of one query head over tokens [t0, t1) of sequence b:
 *   s_t = sm_scale * <q, K_t>,   w_t = exp(s_t - max_t s_t)
 *   o   = sum_t w_t V_t / sum_t w_t,   lse = max_t s_t + ln(sum_t w_t)
 * An empty range gives o = 0 and lse = -inf.
 */
static void attend_range(const paged_kv *p, const uint16_t *q_row, int b, int h,
                         int t0, int t1, double sm_scale, double *o, double *lse)
{
    int kvh = oracle_kv_head(h, p->Hq, p->Hkv);
    int n = t1 - t0, t, d;
    double mx = -INFINITY, sum = 0.0;
    double *s, *row, *q;
    for (d = 0; d < p->D; d++)
        o[d] = 0.0;
    if (n <= 0) {
        *lse = -INFINITY;
        return;
    }
    s = (double *)malloc(sizeof(double) * (size_t)n);
    row = (double *)malloc(sizeof(double) * (size_t)p->D);
    q = (double *)malloc(sizeof(double) * (size_t)p->D);
    for (d = 0; d < p->D; d++)
        q[d] = oracle_bf16_to_double(q_row[d]);
    for (t = 0; t < n; t++) {
        double acc = 0.0;
        kv_row(p, 0, b, t0 + t, kvh, row);
        for (d = 0; d < p->D; d++)
            acc += q[d] * row[d];
        s[t] = sm_scale * acc;
        if (s[t] > mx)
            mx = s[t];
    }
    for (t = 0; t < n; t++) {
        s[t] = exp(s[t] - mx);
        sum += s[t];
    }
    for (t = 0; t < n; t++) {
        kv_row(p, 1, b, t0 + t, kvh, row);
        for (d = 0; d < p->D; d++)
            o[d] += s[t] * row[d];
    }
    for (d = 0; d < p->D; d++)
        o[d] /= sum;
    *lse = mx + log(sum);
    free(s);
    free(row);
    free(q);
}

/*
 * Decode attention for a batch: out[b][h] = softmax(sm_scale * q[b,h] K_b^T) V_b
 * over the L_b = seq_lens[b] tokens of sequence b, gathered through its block
 * table ([P4] "Custom PagedAttention Kernels": grid over (sequence, head),
 * walk the block table, load K and V, scaled dot-product attention).  With
 * window > 0 only the positions oracle_window_positions retains are attended
 * ([P3] section 3).
 * With rows == NULL every (b, h) is computed into out[B][Hq][D]; otherwise only
 * the nrows pairs (rows_b[i], rows_h[i]) into out[nrows][D].
 * Parallel over rows with OpenMP when nthreads > 1 (each row is independent).
 */
void oracle_paged_decode(int B, int Hq, int Hkv, int D, int bs, int max_blocks, int kv_kind,
                         const uint16_t *q, const void *k_pool, const void *v_pool,
                         const float *k_scale, const float *v_scale,
                         const int32_t *block_tables, const int32_t *seq_lens,
                         double sm_scale, int window, int nrows, const int32_t *rows_b,
                         const int32_t *rows_h, double *out, int nthreads)
{
    paged_kv p;
    long long i, n;
    p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.bs = bs; p.max_blocks = max_blocks; p.kv_kind = kv_kind;
    p.k_pool = k_pool; p.v_pool = v_pool; p.k_scale = k_scale; p.v_scale = v_scale;
    p.block_tables = block_tables;
    n = rows_b ? (long long)nrows : (long long)B * Hq;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (i = 0; i < n; i++) {
        int b = rows_b ? rows_b[i] : (int)(i / Hq);
        int h = rows_b ? rows_h[i] : (int)(i % Hq);
        double lse;
        int L = seq_lens[b];
        int first = (window > 0 && L > window) ? L - window : 0;
        attend_range(&p, &q[((size_t)b * Hq + h) * D], b, h, first, L, sm_scale,
                     &out[(size_t)i * D], &lse);
    }
}

/*
 * Query-aware sparse decode ([P3] section 7), pages of 16 tokens, over bf16, E4M3 or
 * 4-bit pools (kv_kind as in kv_row; keys and values restored exactly):
 * for every (b, kv head) the pages of sequence b are summarised from their valid
 * keys (oracle_page_summary), the summary stored as bf16 with the minimum rounded
 * down and the maximum up (a no-op on bf16 keys), each page is scored with every
 * query head of the group and keeps the largest score (the group shares one
 * selection), the topk best pages are chosen (oracle_select_pages) and every query
 * head of the group attends over the tokens of the chosen pages only (textbook
 * softmax).  The chosen pages go to sel[b][kvh][0..topk) (-1 where fewer exist).
 */
void oracle_quest_decode(int B, int Hq, int Hkv, int D, int bs, int max_blocks, int kv_kind,
                         const uint16_t *q, const void *k_pool, const void *v_pool,
                         const float *k_scale, const float *v_scale,
                         const int32_t *block_tables, const int32_t *seq_lens, double sm_scale,
                         int topk, double *out, int32_t *sel, int nthreads)
{
    paged_kv p;
    long long i;
    int G = Hq / Hkv;
    p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.bs = bs; p.max_blocks = max_blocks; p.kv_kind = kv_kind;
    p.k_pool = k_pool; p.v_pool = v_pool; p.k_scale = k_scale; p.v_scale = v_scale;
    p.block_tables = block_tables;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (i = 0; i < (long long)B * Hkv; i++) {
        int b = (int)(i / Hkv), kvh = (int)(i % Hkv);
        int L = seq_lens[b], np = (L + 15) / 16, j, t, g, d, m, c;
        double *keys = (double *)malloc(sizeof(double) * 16 * (size_t)D);
        double *mn = (double *)malloc(sizeof(double) * (size_t)D);
        double *mx = (double *)malloc(sizeof(double) * (size_t)D);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        double *row = (double *)malloc(sizeof(double) * (size_t)D);
        double *scores = (double *)malloc(sizeof(double) * (size_t)(np > 0 ? np : 1));
        int *chosen = (int *)malloc(sizeof(int) * (size_t)(np > 0 ? np : 1));
        for (j = 0; j < np; j++) {
            int n = (L - 16 * j < 16) ? L - 16 * j : 16;
            /* logical page j: 16 rows of one block, at pool page blk * bs / 16 + ... */
            long long blk = block_tables[(size_t)b * max_blocks + 16 * j / bs];
            oracle_quest_page_summary(Hkv, D, bs, kv_kind, k_pool, k_scale,
                                      blk * (bs / 16) + (16 * j % bs) / 16, n, kvh, mn, mx);
            scores[j] = -INFINITY;
            for (g = 0; g < G; g++) {
                double sc;
                for (d = 0; d < D; d++)
                    qd[d] = oracle_bf16_to_double(q[((size_t)b * Hq + kvh * G + g) * D + d]);
                sc = oracle_page_score(qd, mn, mx, D);
                if (sc > scores[j]) scores[j] = sc;
            }
        }
        m = oracle_select_pages(scores, np, topk, chosen);
        for (c = 0; c < topk; c++)
            sel[(size_t)i * topk + c] = (c < m) ? chosen[c] : -1;
        for (g = 0; g < G; g++) {
            int h = kvh * G + g, nt = 0;
            double mxs = -INFINITY, sum = 0.0;
            double *o = &out[((size_t)b * Hq + h) * D];
            double *sv = (double *)malloc(sizeof(double) * 16 * (size_t)(m > 0 ? m : 1));
            for (d = 0; d < D; d++) {
                qd[d] = oracle_bf16_to_double(q[((size_t)b * Hq + h) * D + d]);
                o[d] = 0.0;
            }
            for (c = 0; c < m; c++) {
                int pg = chosen[c], n = (L - 16 * pg < 16) ? L - 16 * pg : 16;
                for (t = 0; t < n; t++) {
                    double acc = 0.0;
                    kv_row(&p, 0, b, 16 * pg + t, kvh, row);
                    for (d = 0; d < D; d++)
                        acc += qd[d] * row[d];
                    sv[nt] = sm_scale * acc;
                    if (sv[nt] > mxs) mxs = sv[nt];
                    nt++;
                }
            }
            nt = 0;
            for (c = 0; c < m; c++) {
                int pg = chosen[c], n = (L - 16 * pg < 16) ? L - 16 * pg : 16;
                for (t = 0; t < n; t++) {
                    double w = exp(sv[nt++] - mxs);
                    sum += w;
                    kv_row(&p, 1, b, 16 * pg + t, kvh, row);
                    for (d = 0; d < D; d++)
                        o[d] += w * row[d];
                }
            }
            for (d = 0; d < D; d++)
                o[d] = (sum > 0.0) ? o[d] / sum : 0.0;
            free(sv);
        }
        free(keys); free(mn); free(mx); free(qd); free(row); free(scores); free(chosen);
    }
}

/*
 * Split-KV partials of one (b, h): split i covers logical blocks
 * [blk_begin[i], blk_begin[i+1]) of the sequence, clipped to its length.
 * Each split is attended on its own (attend_range), giving o_i (normalised) and
 * lse_i (natural log).  Empty splits give o_i = 0, lse_i = -inf.
 */
void oracle_split_partials(int Hq, int Hkv, int D, int bs, int max_blocks, int kv_kind,
                           const uint16_t *q, const void *k_pool, const void *v_pool,
                           const float *k_scale, const float *v_scale,
                           const int32_t *block_tables, const int32_t *seq_lens,
                           double sm_scale, int b, int h, int nsplit,
                           const int32_t *blk_begin, double *o_parts, double *lse)
{
    paged_kv p;
    int i, L = seq_lens[b];
    p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.bs = bs; p.max_blocks = max_blocks; p.kv_kind = kv_kind;
    p.k_pool = k_pool; p.v_pool = v_pool; p.k_scale = k_scale; p.v_scale = v_scale;
    p.block_tables = block_tables;
    for (i = 0; i < nsplit; i++) {
        int t0 = blk_begin[i] * bs, t1 = blk_begin[i + 1] * bs;
        if (t1 > L) t1 = L;
        if (t0 > L) t0 = L;
        attend_range(&p, &q[((size_t)b * Hq + h) * D], b, h, t0, t1, sm_scale,
                     &o_parts[(size_t)i * D], &lse[i]);
    }
}

/*
 * Split-KV partials of one (b, h) over token ranges: piece i covers tokens
 * [tok_begin[i], tok_begin[i+1]) of the sequence, clipped to its length, attended on
 * its own (attend_range): o_i normalised, lse_i natural log; an empty piece gives
 * o_i = 0 and lse_i = -inf.  (oracle_split_partials is the block-aligned case.)
 */
void oracle_token_partials(int Hq, int Hkv, int D, int bs, int max_blocks, int kv_kind,
                           const uint16_t *q, const void *k_pool, const void *v_pool,
                           const float *k_scale, const float *v_scale,
                           const int32_t *block_tables, const int32_t *seq_lens,
                           double sm_scale, int b, int h, int npiece,
                           const int32_t *tok_begin, double *o_parts, double *lse)
{
    paged_kv p;
    int i, L = seq_lens[b];
    p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.bs = bs; p.max_blocks = max_blocks; p.kv_kind = kv_kind;
    p.k_pool = k_pool; p.v_pool = v_pool; p.k_scale = k_scale; p.v_scale = v_scale;
    p.block_tables = block_tables;
    for (i = 0; i < npiece; i++) {
        int t0 = tok_begin[i], t1 = tok_begin[i + 1];
        if (t1 > L) t1 = L;
        if (t0 > L) t0 = L;
        attend_range(&p, &q[((size_t)b * Hq + h) * D], b, h, t0, t1, sm_scale,
                     &o_parts[(size_t)i * D], &lse[i]);
    }
}

/*
 * Decode over chosen pages ([P3] section 7, the read that follows the selection):
 * query head h of sequence b attends over the tokens of the 16-token pages
 * sel[b][h / G][0 .. topk) only -- page j holds tokens [16 j, min(16 j + 16, L)) --
 * with textbook softmax (max-subtracted, in double).  Entries that name no page of
 * the sequence (-1, or j * 16 >= L) are skipped; a head with no token gets zeros.
 * Pages are visited in the order given.
 */
void oracle_paged_decode_pages(int B, int Hq, int Hkv, int D, int bs, int max_blocks,
                               int kv_kind, const uint16_t *q, const void *k_pool,
                               const void *v_pool, const float *k_scale, const float *v_scale,
                               const int32_t *block_tables, const int32_t *seq_lens,
                               double sm_scale, int topk, const int32_t *sel, double *out,
                               int nthreads)
{
    paged_kv p;
    long long i;
    p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.bs = bs; p.max_blocks = max_blocks; p.kv_kind = kv_kind;
    p.k_pool = k_pool; p.v_pool = v_pool; p.k_scale = k_scale; p.v_scale = v_scale;
    p.block_tables = block_tables;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (i = 0; i < (long long)B * Hq; i++) {
        int b = (int)(i / Hq), h = (int)(i % Hq), kvh = oracle_kv_head(h, Hq, Hkv);
        int L = seq_lens[b], c, t, d, n = 0;
        const int32_t *pages = &sel[((size_t)b * Hkv + kvh) * topk];
        double mx = -INFINITY, sum = 0.0;
        double *o = &out[(size_t)i * D];
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        double *row = (double *)malloc(sizeof(double) * (size_t)D);
        double *sv = (double *)malloc(sizeof(double) * 16 * (size_t)(topk > 0 ? topk : 1));
        for (d = 0; d < D; d++) {
            qd[d] = oracle_bf16_to_double(q[(size_t)i * D + d]);
            o[d] = 0.0;
        }
        for (c = 0; c < topk; c++) {            /* scores of the chosen tokens */
            int pg = pages[c], t0 = 16 * pg, t1 = 16 * pg + 16;
            if (pg < 0 || t0 >= L) continue;
            if (t1 > L) t1 = L;
            for (t = t0; t < t1; t++) {
                double acc = 0.0;
                kv_row(&p, 0, b, t, kvh, row);
                for (d = 0; d < D; d++)
                    acc += qd[d] * row[d];
                sv[n] = sm_scale * acc;
                if (sv[n] > mx) mx = sv[n];
                n++;
            }
        }
        n = 0;
        for (c = 0; c < topk; c++) {            /* weights and values, same order */
            int pg = pages[c], t0 = 16 * pg, t1 = 16 * pg + 16;
            if (pg < 0 || t0 >= L) continue;
            if (t1 > L) t1 = L;
            for (t = t0; t < t1; t++) {
                double w = exp(sv[n++] - mx);
                sum += w;
                kv_row(&p, 1, b, t, kvh, row);
                for (d = 0; d < D; d++)
                    o[d] += w * row[d];
            }
        }
        for (d = 0; d < D; d++)
            o[d] = (sum > 0.0) ? o[d] / sum : 0.0;
        free(qd); free(row); free(sv);
    }
}

/*
 * Log-sum-exp merge of split partials of one head:
 *   M = max_i lse_i,  w_i = exp(lse_i - M),  out = sum_i w_i o_i / sum_i w_i
 * Splits with lse_i = -inf carry no weight; if all are -inf the output is 0.
 */
void oracle_merge_lse(int nsplit, int D, const double *o_parts, const double *lse, double *out)
{
    int i, d;
    double M = -INFINITY, wsum = 0.0;
    for (d = 0; d < D; d++)
        out[d] = 0.0;
    for (i = 0; i < nsplit; i++)
        if (lse[i] > M)
            M = lse[i];
    if (M == -INFINITY)
        return;
    for (i = 0; i < nsplit; i++) {
        double w;
        if (lse[i] == -INFINITY)
            continue;
        w = exp(lse[i] - M);
        wsum += w;
        for (d = 0; d < D; d++)
            out[d] += w * o_parts[(size_t)i * D + d];
    }
    for (d = 0; d < D; d++)
        out[d] /= wsum;
}
