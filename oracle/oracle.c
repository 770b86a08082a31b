/*
 * CPU oracle for the paged FP8-KV grouped-query decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into a separate host
 * library that the tests, the smoke check and the CPU-baseline leg of the
 * benchmark load.  The CUDA library never links, includes or calls it, and it
 * shares no header, table or helper with the CUDA sources.
 *
 * It is deliberately plain: scalar loops, fp64 arithmetic, no blocking, no
 * fusion.  Each function restates the definition it follows:
 *
 *   - E4M3 (FN variant) format: 1 sign bit, 4 exponent bits (bias 7), 3
 *     mantissa bits; largest finite value 448, smallest non-zero 2^-9.
 *     "FP8量化与长上下文实测：Llama 3 70B部署优化指南", §1.1.
 *   - Quantisation is a division by a scale followed by the cast to E4M3
 *     ("FP8量化与长上下文实测", §3.1 weight code; §3.2 applies the same scale
 *     idea to the KV cache).  Rounding is round-to-nearest-even straight from
 *     fp32 and out-of-range values saturate to +-448.
 *   - The KV cache is cut into fixed pages of P tokens addressed through a
 *     per-sequence block table (0539edu.com Llama 3 notes, §2.2 and §5.2;
 *     default P = 16 in §3.3).
 *   - GQA: several query heads share one KV head; query head i reads KV head
 *     i / G ("FP8量化与长上下文实测", §1.2: 64 query heads over 8 KV heads).
 *   - Decode attention: for the one new query of every sequence,
 *     o = softmax(q . K^T / sqrt(D)) . V over every cached token.
 *   - Chunked prefill (0539edu.com Llama 3 notes, §2.2: a 128K prompt is
 *     prefilled as 8 chunks of 16K, each chunk's KV joined to the cache): the
 *     chunk's K/V are appended to the pages first, then the query at position
 *     p attends to every cached token t <= p (causal, the earlier chunks
 *     included).
 *   - KV-scale calibration: every attention layer keeps a running maximum of
 *     |K| and |V| over the prefill batches it has seen, per kv head, and the
 *     scale is that maximum / 448, floored at 1e-12 ("FP8量化与长上下文实测",
 *     §3.2 running max per layer, §3.1 absmax / 448 and the 1e-12 clamp).
 *
 * Readings where the pages are silent (all listed in the design notes):
 *   NaN input -> a NaN code (0x7F); |y| > 448 (and +-Inf) -> +-448; the sign of
 *   zero is kept; q widens exactly from bf16; sm_scale = 1/sqrt(D); tokens at
 *   t >= seq_len are never read; seq_len = 0 gives an all-zero output; NaN
 *   inputs do not enter the running maximum.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* E4M3 codec, written from the format definition.                         */
/* ---------------------------------------------------------------------- */

/* Value of one E4M3 code.  Normal: (-1)^s 2^(e-7) (1 + m/8) for e in 1..15
 * (except e=15, m=7, which is NaN).  Subnormal (e = 0): (-1)^s 2^-6 (m/8). */
double oracle_e4m3_value(uint8_t code)
{
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* fp32 -> E4M3 code, round to nearest with ties to even, saturating.
 * The exponent of |y| is found with frexp; below 2^-6 the quantum stays at
 * the subnormal spacing 2^-9.  |y| / quantum is exact (power-of-two scale)
 * and rint() rounds it to the nearest integer, ties to even. */
uint8_t oracle_e4m3_encode(float y)
{
    uint8_t sign;
    double a, n;
    int ex, E;

    if (isnan(y))
        return 0x7F;
    sign = signbit(y) ? 0x80 : 0x00;
    a = fabs((double)y);
    if (a > 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a == 0.0)
        return sign;

    frexp(a, &ex);            /* a = f * 2^ex, f in [0.5, 1) */
    E = ex - 1;               /* floor(log2(a)) */
    if (E < -6)
        E = -6;
    n = rint(ldexp(a, -(E - 3)));   /* a / 2^(E-3), rounded */

    if (n < 8.0)              /* only possible when E == -6: subnormal */
        return (uint8_t)(sign | (uint8_t)n);
    if (n >= 16.0) {          /* rounding carried into the next binade */
        n = 8.0;
        E += 1;
    }
    /* a <= 448 keeps E + 7 <= 15 and the mantissa <= 6 here. */
    return (uint8_t)(sign | ((E + 7) << 3) | ((int)n - 8));
}

void oracle_e4m3_encode_array(const float *y, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(y[i]);
}

void oracle_e4m3_value_array(const uint8_t *c, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_value(c[i]);
}

/* Multi-threaded encode for the exhaustive fp32 sweep (same scalar routine,
 * split into contiguous ranges). */
struct enc_job { const float *y; uint8_t *out; int64_t n; };

static void *enc_worker(void *arg)
{
    struct enc_job *j = (struct enc_job *)arg;
    oracle_e4m3_encode_array(j->y, j->out, j->n);
    return NULL;
}

int oracle_e4m3_encode_array_mt(const float *y, uint8_t *out, int64_t n, int threads)
{
    pthread_t tid[256];
    struct enc_job job[256];
    int k, created[256];
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    for (k = 0; k < threads; ++k) {
        int64_t lo = n * k / threads, hi = n * (k + 1) / threads;
        job[k].y = y + lo;
        job[k].out = out + lo;
        job[k].n = hi - lo;
        created[k] = (threads > 1) && pthread_create(&tid[k], NULL, enc_worker, &job[k]) == 0;
        if (!created[k])
            enc_worker(&job[k]);
    }
    for (k = 0; k < threads; ++k)
        if (created[k])
            pthread_join(tid[k], NULL);
    return threads;
}

/* ---------------------------------------------------------------------- */
/* kv_append: quantise new tokens and write them into their pages.         */
/* ---------------------------------------------------------------------- */

/* bf16 widens to fp32 exactly: its 16 bits are the top half of the fp32. */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* x:       new K or V rows, [T][Hkv][D], fp32 (in_bf16 = 0) or bf16 bits.
 * slots:   [T]; token t goes to cache slot slots[t] (< 0: not written).
 * scale:   [Hkv] fp32.
 * cache:   [num_pages][Hkv][P][D] bytes.
 * byte = E4M3(x / scale[h]) with the division done in IEEE fp32, written to
 * page slot / P, row slot % P.  Returns the number of tokens whose slot was
 * outside the pool (those are skipped). */
int64_t oracle_kv_append(const void *x, int in_bf16, int64_t T, int Hkv, int D,
                         const int64_t *slots, const float *scale,
                         uint8_t *cache, int64_t num_pages, int P)
{
    int64_t bad = 0;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slots[t];
        if (slot < 0)
            continue;
        if (slot >= num_pages * (int64_t)P) {
            ++bad;
            continue;
        }
        int64_t page = slot / P, off = slot % P;
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < D; ++d) {
                int64_t src = (t * Hkv + h) * (int64_t)D + d;
                float v = in_bf16 ? bf16_bits_to_float(((const uint16_t *)x)[src])
                                  : ((const float *)x)[src];
                float q = v / scale[h];   /* one IEEE fp32 division */
                cache[((page * Hkv + h) * P + off) * (int64_t)D + d] =
                    oracle_e4m3_encode(q);
            }
        }
    }
    return bad;
}

/* ---------------------------------------------------------------------- */
/* Paged GQA decode attention in fp64.                                     */
/* ---------------------------------------------------------------------- */

struct decode_args {
    const uint16_t *q;                 /* [B][Hq][D] bf16 bits */
    const uint8_t *kc, *vc;            /* [num_pages][Hkv][P][D] */
    const float *ks, *vs;              /* [Hkv] */
    const int32_t *bt;                 /* [B][max_pages] */
    int max_pages;
    const int32_t *lens;               /* [B] */
    const int32_t *page_sizes;         /* [B] tokens per page of each sequence, or NULL (all P) */
    int B, Hq, Hkv, D, P;
    int64_t num_pages;
    double sm_scale;
    const int32_t *sel;                /* [n_sel][2] = (b, q_head) */
    int64_t n_sel;
    double *out;                       /* [n_sel][D] */
    double *weights;                   /* [n_sel][w_stride] or NULL */
    int64_t w_stride;
    int status;                        /* 0 ok, 1 bad block-table entry */
};

/* Where token t of sequence b lives.  A page of P_b tokens (P_b = P unless
 * per-sequence page sizes are given: 0539edu.com Llama 3 notes, §3.2, 16-token
 * pages for short sequences and 64-token pages for long ones) is a run of
 * P_b / P consecutive pool pages whose first page is the table entry
 * block_table[b][t / P_b]; offset o = t % P_b of the logical page lies in pool
 * page entry + o / P at row o % P.  Returns the pool page, or -1 if the table
 * runs out or the page lies outside the pool. */
static int64_t token_pool_page(const struct decode_args *a, int b, int t)
{
    int Pb = a->page_sizes ? a->page_sizes[b] : a->P;
    int32_t entry;
    int64_t page;
    if (Pb <= 0 || t / Pb >= a->max_pages)
        return -1;
    entry = a->bt[(int64_t)b * a->max_pages + t / Pb];
    page = (int64_t)entry + (t % Pb) / a->P;
    if (entry < 0 || page >= a->num_pages)
        return -1;
    return page;
}

/* One (sequence b, query head i) output row.
 *   K^_td = value(k byte) * k_scale[h], V^_td likewise, h = i / G;
 *   s_t   = (sum_d q_id K^_td) * sm_scale,  t < L_b, token t found at
 *           pool page token_pool_page(b, t), row t % P;
 *   w_t   = exp(s_t - max s) / sum_u exp(s_u - max s);
 *   o_id  = sum_t w_t V^_td.                                               */
static int decode_one(const struct decode_args *a, int64_t k)
{
    int b = a->sel[2 * k], i = a->sel[2 * k + 1];
    int G = a->Hq / a->Hkv;
    int h = i / G;
    int L = a->lens[b];
    int D = a->D, P = a->P;
    double *o = a->out + k * D;
    double *s, smax, denom;
    double q[1024];

    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (L <= 0)
        return 0;
    for (int d = 0; d < D; ++d)
        q[d] = (double)bf16_bits_to_float(a->q[((int64_t)b * a->Hq + i) * D + d]);

    s = (double *)malloc(sizeof(double) * (size_t)L);
    if (!s)
        return 2;
    for (int t = 0; t < L; ++t) {
        int64_t phys = token_pool_page(a, b, t);
        if (phys < 0) {
            free(s);
            return 1;
        }
        const uint8_t *krow = a->kc + ((phys * a->Hkv + h) * P + t % P) * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += q[d] * (oracle_e4m3_value(krow[d]) * (double)a->ks[h]);
        s[t] = acc * a->sm_scale;
    }
    smax = s[0];
    for (int t = 1; t < L; ++t)
        if (s[t] > smax)
            smax = s[t];
    denom = 0.0;
    for (int t = 0; t < L; ++t) {
        s[t] = exp(s[t] - smax);
        denom += s[t];
    }
    for (int t = 0; t < L; ++t) {
        double w = s[t] / denom;
        int64_t phys = token_pool_page(a, b, t);
        const uint8_t *vrow = a->vc + ((phys * a->Hkv + h) * P + t % P) * D;
        for (int d = 0; d < D; ++d)
            o[d] += w * (oracle_e4m3_value(vrow[d]) * (double)a->vs[h]);
        if (a->weights && t < a->w_stride)
            a->weights[k * a->w_stride + t] = w;
    }
    free(s);
    return 0;
}

struct decode_job { const struct decode_args *a; int64_t lo, hi; int status; };

static void *decode_worker(void *arg)
{
    struct decode_job *j = (struct decode_job *)arg;
    j->status = 0;
    for (int64_t k = j->lo; k < j->hi; ++k) {
        int st = decode_one(j->a, k);
        if (st && !j->status)
            j->status = st;
    }
    return NULL;
}

/* Computes the selected (b, q_head) rows; `threads` workers split the list.
 * Returns 0, or 1 if a needed block-table entry is outside the pool, or 2 on
 * allocation failure. */
int oracle_paged_decode(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                        const float *k_scale, const float *v_scale,
                        const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                        const int32_t *page_sizes,
                        int B, int Hq, int Hkv, int D, int P, int64_t num_pages,
                        double sm_scale, const int32_t *sel, int64_t n_sel,
                        double *out, double *weights, int64_t w_stride, int threads)
{
    struct decode_args a;
    pthread_t tid[256];
    struct decode_job job[256];
    int k, status = 0, created[256];

    if (D > 1024 || Hkv <= 0 || Hq % Hkv != 0)
        return 3;
    a.q = q; a.kc = k_cache; a.vc = v_cache; a.ks = k_scale; a.vs = v_scale;
    a.bt = block_table; a.max_pages = max_pages; a.lens = seq_lens; a.page_sizes = page_sizes;
    a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.P = P; a.num_pages = num_pages;
    a.sm_scale = sm_scale; a.sel = sel; a.n_sel = n_sel; a.out = out;
    a.weights = weights; a.w_stride = w_stride; a.status = 0;

    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    for (k = 0; k < threads; ++k) {
        job[k].a = &a;
        job[k].lo = n_sel * k / threads;
        job[k].hi = n_sel * (k + 1) / threads;
        created[k] = (threads > 1) && pthread_create(&tid[k], NULL, decode_worker, &job[k]) == 0;
        if (!created[k])
            decode_worker(&job[k]);
    }
    for (k = 0; k < threads; ++k) {
        if (created[k])
            pthread_join(tid[k], NULL);
        if (job[k].status && !status)
            status = job[k].status;
    }
    return status;
}

/* ---------------------------------------------------------------------- */
/* KV-scale calibration: running |x| maximum per kv head, scale = max/448.  */
/* ---------------------------------------------------------------------- */

/* running_max[h] = max(running_max[h], |x[t][h][d]| for all t, d); NaN is
 * skipped (a comparison with NaN is false). */
void oracle_kv_absmax_update(const void *x, int in_bf16, int64_t T, int Hkv, int D, float *running_max)
{
    for (int h = 0; h < Hkv; ++h) {
        float m = running_max[h];
        for (int64_t t = 0; t < T; ++t) {
            for (int d = 0; d < D; ++d) {
                int64_t i = (t * Hkv + h) * (int64_t)D + d;
                float v = in_bf16 ? bf16_bits_to_float(((const uint16_t *)x)[i]) : ((const float *)x)[i];
                float a = fabsf(v);
                if (a > m)
                    m = a;
            }
        }
        running_max[h] = m;
    }
}

/* scale[h] = max(running_max[h] / 448, 1e-12), the division in IEEE fp32. */
void oracle_kv_scale_from_max(const float *running_max, int Hkv, float *scale)
{
    for (int h = 0; h < Hkv; ++h) {
        float s = running_max[h] / 448.0f;
        scale[h] = s > 1e-12f ? s : 1e-12f;
    }
}

/* ---------------------------------------------------------------------- */
/* Chunked-prefill attention: a chunk of queries per sequence, causal.     */
/* ---------------------------------------------------------------------- */

/* q: [T][Hq][D] bf16 bits, the queries of all sequences back to back;
 * cu_q[B + 1]: sequence b owns query rows cu_q[b] .. cu_q[b+1] - 1.  seq_lens[b]
 * counts the chunk, so with n = cu_q[b+1] - cu_q[b] its queries sit at
 * positions L - n .. L - 1.  The query at position p attends to cached tokens
 * 0 .. p, exactly as oracle_paged_decode does for a sequence of length p + 1.
 * page_sizes: per-sequence page sizes as in oracle_paged_decode, or NULL.
 * out: [T][Hq][D] fp64.  A sequence with L < n is an error (status 3); its
 * rows are left untouched.  `threads` workers split each row's heads.
 * Returns 0 or the first non-zero status. */
int oracle_paged_prefill(const uint16_t *q, const int32_t *cu_q, const uint8_t *k_cache, const uint8_t *v_cache,
                         const float *k_scale, const float *v_scale,
                         const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                         const int32_t *page_sizes,
                         int B, int Hq, int Hkv, int D, int P, int64_t num_pages,
                         double sm_scale, double *out, int threads)
{
    int status = 0;
    int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * 2 * (size_t)(Hq > 0 ? Hq : 1));
    if (!sel)
        return 2;
    for (int i = 0; i < Hq; ++i) {                       /* every query head of the row */
        sel[2 * i] = 0;
        sel[2 * i + 1] = i;
    }
    for (int b = 0; b < B; ++b) {
        int32_t n = cu_q[b + 1] - cu_q[b];
        if (n < 0 || seq_lens[b] < n) {
            if (!status)
                status = 3;
            continue;
        }
        for (int32_t c = 0; c < n; ++c) {
            int32_t len = seq_lens[b] - n + c + 1;       /* keys 0 .. position */
            int64_t row = (int64_t)cu_q[b] + c;
            int st = oracle_paged_decode(q + row * Hq * D, k_cache, v_cache, k_scale, v_scale,
                                         block_table + (int64_t)b * max_pages, max_pages, &len,
                                         page_sizes ? page_sizes + b : NULL, 1, Hq, Hkv, D, P,
                                         num_pages, sm_scale, sel, Hq, out + row * Hq * D, NULL, 0, threads);
            if (st && !status)
                status = st;
        }
    }
    free(sel);
    return status;
}
