/*
 * sdpa_oracle.c -- plain, slow, fp64 CPU oracle for the fused SDPA forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library; its inputs come from the seeded generators in attn_inputs.py.
 *
 * Sources (page titles as cited throughout this repository):
 *   [ALG]  "gfx942 unified attention, from the math up" (ALGORITHM.md of the
 *          gfx942 unified-attention example)
 *   [RDM]  "gfx942 unified attention - parity + benchmark harness" (README.md
 *          of the same example)
 *   [MM]   "MoonMath.ai abre un nucleo de atencion HIP para AMD MI300X que
 *          supera a AITER v3 en todas las formas y modos de redondeo"
 *          (7minutos.es news article)
 *
 * What is computed (all arithmetic in IEEE binary64), by oracle_sdpa_run:
 *   variant 0, the definition -- [ALG] sec. 1 (softmax of tau*q.K^T times V,
 *       one query row at a time), with the stability shift of [ALG] sec. 2,
 *       the bottom-right causal mask of [ALG] sec. 4 and [RDM]
 *       "Troubleshooting", the paged KV layout, block table and GQA head
 *       grouping of [ALG] sec. 5, and the gather -> repeat_interleave ->
 *       mask -> softmax -> .V recipe of the correctness gate, [ALG] sec. 10.
 *   variant 1, the online-softmax recurrence of [ALG] sec. 3 (running max m,
 *       denominator l, rescale alpha = e^(m_old - m_new), un-normalised o,
 *       final o / l) over key tiles of a given width.  Self-test only: it
 *       must equal the definition.
 *   variant 2, a split of the key range into P contiguous parts, each reduced
 *       to (o_p / l_p, lse_p) and combined by the log-sum-exp rule (the
 *       split-KV decode of [ALG] sec. 8).  Self-test only.
 * and by the two helpers:
 *   oracle_round_f32         -- rounding of binary32 values to bf16 / fp16 in
 *                               the three modes named in [MM] "Punto de
 *                               referencia": nearest-even, nearest with ties
 *                               away from zero, toward zero.
 *   oracle_widen16           -- exact widening of bf16 / fp16 bit patterns to
 *                               binary64, from the formats' definitions.
 *   oracle_widen8            -- exact widening of fp8 E4M3 bit patterns (the
 *                               OCP 8-bit format with 4 exponent bits, bias 7,
 *                               3 fraction bits, no infinities, S.1111.111 NaN).
 *
 * Feature-flagged variants (variant 0 only).  [ALG] sec. 9 names sinks,
 * ALiBi, softcap, sliding window (and fp8) as flags the dispatcher keeps out
 * of graph replay, without defining them; the oracle takes their usual
 * definitions, with diag = i + (kv_len - query_len) the key aligned with
 * query row i:
 *   sliding window (left W_l, right W_r; -1 = unbounded): key j is visible
 *       only if diag - W_l <= j <= diag + W_r (on top of j < kv_len and, when
 *       causal, j <= diag);
 *   softcap c > 0: the scaled score s = tau q.k becomes c * tanh(s / c);
 *   ALiBi slope a_h: the score gains -a_h * |diag - j| (after the softcap);
 *   sink z_h: one more logit in the softmax denominator with no value row,
 *       O = sum_j e^(s_j) V_j / (sum_j e^(s_j) + e^(z_h)); the log-sum-exp
 *       includes it.
 *   fp8 K/V caches: the caches hold E4M3 bytes and the key and value used
 *       are the widened byte times a per-tensor factor, K = k_scale * e4m3(k),
 *       V = v_scale * e4m3(v) (the common "descale" convention); queries and
 *       outputs keep the 16-bit dtype.
 *
 * Readings where the pages are silent:
 *   - A query row with no visible key (causal with query_len > kv_len, or
 *     kv_len == 0) has output 0 and log-sum-exp -inf (z_h with a sink).
 *   - Non-causal attention (the [MM] kernel) sees every key j < kv_len.
 *   - kv head of q head h is h / (num_q_heads / num_kv_heads).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F16 = 0, OR_BF16 = 1 };
enum { OR_RTNE = 0, OR_RTNA = 1, OR_RTZ = 2 };

/* ------------------------------------------------------------------------ */
/* 16-bit formats -> binary64                                               */
/* ------------------------------------------------------------------------ */

/* E4M3: bit 7 sign, bits 6..3 exponent e (bias 7), bits 2..0 fraction f.
 * e = 0: subnormal, f/8 * 2^-6.  e >= 1: (1 + f/8) * 2^(e-7), except that
 * e = 15 with f = 7 is NaN (the format has no infinities; 448 is the largest
 * finite magnitude). */
double oracle_widen8(uint8_t b)
{
    const int s = (b >> 7) & 1;
    const int e = (b >> 3) & 15;
    const int f = b & 7;
    double mag;
    if (e == 15 && f == 7) return NAN;
    if (e == 0) mag = ldexp((double)f / 8.0, -6);
    else mag = ldexp(1.0 + (double)f / 8.0, e - 7);
    return s ? -mag : mag;
}

void oracle_widen8_array(double *out, const uint8_t *in, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_widen8(in[i]);
}

/* bf16 is the upper half of a binary32 pattern; fp16 is IEEE binary16
 * (1 sign, 5 exponent bits with bias 15, 10 fraction bits). */
double oracle_widen16(uint16_t h, int32_t dtype)
{
    int sign = (h >> 15) & 1;
    double v;
    if (dtype == OR_BF16) {
        int e = (h >> 7) & 0xFF;
        int f = h & 0x7F;
        if (e == 0xFF)
            v = f ? NAN : INFINITY;
        else if (e == 0)
            v = ldexp((double)f, -126 - 7);
        else
            v = ldexp((double)(128 + f), e - 127 - 7);
    } else {
        int e = (h >> 10) & 0x1F;
        int f = h & 0x3FF;
        if (e == 0x1F)
            v = f ? NAN : INFINITY;
        else if (e == 0)
            v = ldexp((double)f, -14 - 10);
        else
            v = ldexp((double)(1024 + f), e - 15 - 10);
    }
    return sign ? -v : v;
}

void oracle_widen16_array(double *out, const uint16_t *in, int64_t n, int32_t dtype)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_widen16(in[i], dtype);
}

/* ------------------------------------------------------------------------ */
/* binary32 -> 16-bit rounding in three modes                               */
/* ------------------------------------------------------------------------ */

/* Rounds the binary32 value x to the target format by exact integer
 * arithmetic on its significand: x = M * 2^E with an integer M; the target's
 * quantum at x's magnitude is 2^Q; the kept integer is M >> (Q - E) and the
 * discarded remainder decides the rounding.  Overflow follows IEEE 754: the
 * nearest modes go to infinity, toward-zero stops at the largest finite.
 * NaN becomes the format's quiet NaN with the sign kept. */
static uint16_t round_one(float xf, int32_t dtype, int32_t mode)
{
    uint32_t u;
    memcpy(&u, &xf, 4);
    uint16_t sign = (uint16_t)((u >> 31) << 15);
    int e32 = (int)((u >> 23) & 0xFF);
    uint32_t f32 = u & 0x7FFFFF;

    /* format parameters */
    int fbits, emin, emax, ebias;
    if (dtype == OR_BF16) { fbits = 7; ebias = 127; emin = -126; emax = 127; }
    else                  { fbits = 10; ebias = 15; emin = -14;  emax = 15;  }
    uint16_t inf = (uint16_t)(((1u << (15 - fbits)) - 1u) << fbits);
    uint16_t maxfin = (uint16_t)(inf - 1u);

    if (e32 == 0xFF) {
        if (f32) return (uint16_t)(sign | inf | (1u << (fbits - 1)));  /* quiet NaN */
        return (uint16_t)(sign | inf);
    }
    if (e32 == 0 && f32 == 0) return sign;

    /* |x| = M * 2^E, M < 2^24 */
    uint64_t M;
    int E;
    if (e32 == 0) { M = f32; E = -126 - 23; }
    else          { M = f32 | 0x800000u; E = e32 - 127 - 23; }

    /* exponent of x: floor(log2 |x|) */
    int top = 63 - __builtin_clzll(M);      /* index of the leading one */
    int ex = E + top;
    /* quantum exponent of the target at this magnitude */
    int qexp = (ex < emin ? emin : ex) - fbits;

    uint64_t kept;       /* |x| / 2^qexp rounded toward zero */
    int cmp_half;        /* sign of (remainder - half quantum) */
    int rem_nonzero;
    if (qexp <= E) {
        kept = M << (E - qexp);
        cmp_half = -1;
        rem_nonzero = 0;
    } else {
        int sh = qexp - E;
        if (sh >= 63) {
            kept = 0;
            /* remainder is |x| itself, well below half a quantum */
            cmp_half = -1;
            rem_nonzero = 1;
        } else {
            kept = M >> sh;
            uint64_t rem = M - (kept << sh);
            uint64_t half = 1ull << (sh - 1);
            cmp_half = rem > half ? 1 : (rem == half ? 0 : -1);
            rem_nonzero = rem != 0;
        }
    }
    (void)rem_nonzero;

    int up = 0;
    if (mode == OR_RTZ) up = 0;
    else if (mode == OR_RTNA) up = cmp_half >= 0;
    else /* RTNE */ up = cmp_half > 0 || (cmp_half == 0 && (kept & 1));
    uint64_t q = kept + (uint64_t)up;

    /* q * 2^qexp -> encoding.  For normal results q is in [2^fbits, 2^(fbits+1)]
     * (the upper end is a carry into the next binade). */
    int be;  /* biased exponent */
    uint64_t frac;
    if (q == 0) return sign;
    int qtop = 63 - __builtin_clzll(q);
    int vexp = qexp + qtop;                 /* exponent of the rounded value */
    if (vexp < emin) {                      /* subnormal: q < 2^fbits */
        be = 0;
        frac = q;
    } else {
        if (vexp > emax) {
            if (mode == OR_RTZ) return (uint16_t)(sign | maxfin);
            return (uint16_t)(sign | inf);
        }
        be = vexp + ebias;
        /* renormalise q to fbits fraction bits (exact: trailing bits are 0
         * when q carried into the next binade) */
        if (qtop > fbits) frac = (q >> (qtop - fbits)) & ((1u << fbits) - 1u);
        else frac = (q << (fbits - qtop)) & ((1u << fbits) - 1u);
    }
    return (uint16_t)(sign | ((uint32_t)be << fbits) | (uint32_t)frac);
}

void oracle_round_f32(uint16_t *out, const float *in, int64_t n, int32_t dtype, int32_t mode)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = round_one(in[i], dtype, mode);
}

/* ------------------------------------------------------------------------ */
/* problem description shared by the three SDPA routines                    */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q;           /* [total_q, Hq, d] */
    const void *k_cache;         /* [num_blocks, bs, Hkv, d], 16-bit or E4M3 */
    const void *v_cache;         /* [num_blocks, bs, Hkv, d], 16-bit or E4M3 */
    const int32_t *block_table;  /* [num_seqs, bt_stride] */
    int32_t bt_stride;
    const int32_t *query_start_loc;  /* [num_seqs + 1] */
    const int32_t *seq_lens;         /* [num_seqs] */
    int32_t num_seqs, Hq, Hkv, d, bs;
    double scale;
    int32_t causal, dtype;
    int32_t variant;             /* 0 direct, 1 streaming, 2 split */
    int32_t param;               /* tile width (streaming) or parts (split) */
    int32_t win_left, win_right; /* sliding window, -1 = unbounded */
    double softcap;              /* 0 = off */
    const double *alibi;         /* [Hq] slopes or NULL */
    const double *sinks;         /* [Hq] sink logits or NULL */
    int32_t kv_fp8;              /* 1: caches hold E4M3 bytes */
    double k_scale, v_scale;     /* factors applied to widened E4M3 K / V */
    const int64_t *rows;         /* optional list of row ids t*Hq + h */
    int64_t n_rows;
    double *out;                 /* [n_rows, d] */
    double *lse;                 /* [n_rows] or NULL */
    int64_t max_kv;
} problem_t;

typedef struct {
    const problem_t *p;
    int64_t begin, end;
} job_t;

/* element (key j of sequence b, kv head kvh, channel c) of a paged cache,
 * found through the block table as in [ALG] sec. 5 */
static double cache_at(const problem_t *p, const void *cache, double fp8_scale, int32_t b,
                       int64_t j, int32_t kvh, int32_t c)
{
    int32_t page = p->block_table[(int64_t)b * p->bt_stride + j / p->bs];
    int64_t slot = j % p->bs;
    int64_t idx = (((int64_t)page * p->bs + slot) * p->Hkv + kvh) * p->d + c;
    if (p->kv_fp8) return fp8_scale * oracle_widen8(((const uint8_t *)cache)[idx]);
    return oracle_widen16(((const uint16_t *)cache)[idx], p->dtype);
}

static int32_t seq_of_token(const problem_t *p, int64_t t)
{
    int32_t lo = 0, hi = p->num_seqs - 1;
    while (lo < hi) {            /* last b with query_start_loc[b] <= t */
        int32_t mid = (lo + hi + 1) / 2;
        if (p->query_start_loc[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

/* One output row (token t, query head h).  s and qv are scratch buffers of
 * max_kv and d doubles. */
static void one_row(const problem_t *p, int64_t t, int32_t h, double *o,
                    double *lse, double *s, double *qv)
{
    const int32_t d = p->d;
    int32_t b = seq_of_token(p, t);
    int64_t i = t - p->query_start_loc[b];
    int64_t Sq = p->query_start_loc[b + 1] - p->query_start_loc[b];
    int64_t Sk = p->seq_lens[b];
    int32_t kvh = h / (p->Hq / p->Hkv);

    /* visible keys: j < Sk, and for causal j <= i + (Sk - Sq) (bottom-right
     * alignment: the masked set is triu(diagonal = Sk - Sq + 1)); a sliding
     * window narrows the range to [diag - W_l, diag + W_r] */
    const int64_t diag = i + (Sk - Sq);
    int64_t lo = 0, limit = Sk;
    if (p->causal && diag + 1 < limit) limit = diag + 1;
    if (p->win_right >= 0 && diag + p->win_right + 1 < limit) limit = diag + p->win_right + 1;
    if (p->win_left >= 0 && diag - p->win_left > lo) lo = diag - p->win_left;
    const double sink = p->sinks ? p->sinks[h] : -INFINITY;
    for (int32_t c = 0; c < d; ++c) o[c] = 0.0;
    if (limit <= lo) {
        if (lse) *lse = sink;      /* -inf without a sink */
        return;
    }
    for (int32_t c = 0; c < d; ++c)
        qv[c] = oracle_widen16(p->q[(t * p->Hq + h) * (int64_t)d + c], p->dtype);

    /* scores s_j = tau * <q, K_j>, then the softcap and the ALiBi bias */
    for (int64_t j = lo; j < limit; ++j) {
        double acc = 0.0;
        for (int32_t c = 0; c < d; ++c)
            acc += qv[c] * cache_at(p, p->k_cache, p->k_scale, b, j, kvh, c);
        double x = p->scale * acc;
        if (p->softcap > 0.0) x = p->softcap * tanh(x / p->softcap);
        if (p->alibi) x -= p->alibi[h] * fabs((double)(diag - j));
        s[j] = x;
    }

    if (p->variant == 0) {
        /* [ALG] sec. 1-2: weights e^(s_j - max) / sum, output sum of w_j V_j;
         * a sink adds e^(z - max) to the sum only */
        double m = sink;
        for (int64_t j = lo; j < limit; ++j) if (s[j] > m) m = s[j];
        double den = p->sinks ? exp(sink - m) : 0.0;
        for (int64_t j = lo; j < limit; ++j) {
            double w = exp(s[j] - m);
            den += w;
            for (int32_t c = 0; c < d; ++c)
                o[c] += w * cache_at(p, p->v_cache, p->v_scale, b, j, kvh, c);
        }
        for (int32_t c = 0; c < d; ++c) o[c] /= den;
        if (lse) *lse = m + log(den);
    } else if (p->variant == 1) {
        /* [ALG] sec. 3: online recurrence over tiles of width T */
        int64_t T = p->param;
        double m = -INFINITY, l = 0.0;
        for (int64_t j0 = 0; j0 < limit; j0 += T) {
            int64_t j1 = j0 + T < limit ? j0 + T : limit;
            double tmax = -INFINITY;
            for (int64_t j = j0; j < j1; ++j) if (s[j] > tmax) tmax = s[j];
            double m_new = m > tmax ? m : tmax;
            double alpha = exp(m - m_new);      /* e^(-inf) = 0 on the first tile */
            double tsum = 0.0;
            for (int32_t c = 0; c < d; ++c) o[c] *= alpha;
            for (int64_t j = j0; j < j1; ++j) {
                double pj = exp(s[j] - m_new);
                tsum += pj;
                for (int32_t c = 0; c < d; ++c)
                    o[c] += pj * cache_at(p, p->v_cache, p->v_scale, b, j, kvh, c);
            }
            l = alpha * l + tsum;
            m = m_new;
        }
        for (int32_t c = 0; c < d; ++c) o[c] /= l;
        if (lse) *lse = m + log(l);
    } else {
        /* [ALG] sec. 8: P contiguous parts of ceil(ceil(limit / P) / 16) * 16
         * keys; each part gives its normalised output and its log-sum-exp;
         * combine: lse* = max lse_p, w_p = e^(lse_p - lse*),
         * O = sum w_p O_p / sum w_p.  Empty parts have lse_p = -inf. */
        int64_t P = p->param;
        int64_t per = (limit + P - 1) / P;
        per = (per + 15) / 16 * 16;
        double part_lse[256];
        double *part_o = (double *)calloc((size_t)P * (size_t)d, sizeof(double));
        for (int64_t q = 0; q < P; ++q) {
            int64_t j0 = q * per, j1 = (q + 1) * per < limit ? (q + 1) * per : limit;
            if (j0 >= j1) { part_lse[q] = -INFINITY; continue; }
            double m = -INFINITY;
            for (int64_t j = j0; j < j1; ++j) if (s[j] > m) m = s[j];
            double den = 0.0;
            double *po = part_o + q * d;
            for (int64_t j = j0; j < j1; ++j) {
                double w = exp(s[j] - m);
                den += w;
                for (int32_t c = 0; c < d; ++c)
                    po[c] += w * cache_at(p, p->v_cache, p->v_scale, b, j, kvh, c);
            }
            for (int32_t c = 0; c < d; ++c) po[c] /= den;
            part_lse[q] = m + log(den);
        }
        double L = -INFINITY;
        for (int64_t q = 0; q < P; ++q) if (part_lse[q] > L) L = part_lse[q];
        double wsum = 0.0;
        for (int64_t q = 0; q < P; ++q) {
            if (part_lse[q] == -INFINITY) continue;
            double w = exp(part_lse[q] - L);
            wsum += w;
            for (int32_t c = 0; c < d; ++c) o[c] += w * part_o[q * d + c];
        }
        for (int32_t c = 0; c < d; ++c) o[c] /= wsum;
        if (lse) *lse = L + log(wsum);
        free(part_o);
    }
}

static void *run_job(void *arg)
{
    job_t *job = (job_t *)arg;
    const problem_t *p = job->p;
    double *s = (double *)malloc((size_t)(p->max_kv > 0 ? p->max_kv : 1) * sizeof(double));
    double *qv = (double *)malloc((size_t)p->d * sizeof(double));
    for (int64_t r = job->begin; r < job->end; ++r) {
        int64_t id = p->rows ? p->rows[r] : r;
        int64_t t = id / p->Hq;
        int32_t h = (int32_t)(id % p->Hq);
        one_row(p, t, h, p->out + r * p->d, p->lse ? p->lse + r : NULL, s, qv);
    }
    free(s);
    free(qv);
    return NULL;
}

static int run_problem(problem_t *p, int32_t n_threads)
{
    if (p->Hkv <= 0 || p->Hq % p->Hkv != 0 || p->d <= 0 || p->bs <= 0) return 1;
    if (p->variant == 2 && (p->param < 1 || p->param > 256)) return 1;
    if (p->variant == 1 && p->param < 1) return 1;
    /* the self-test variants take the plain problem only */
    if (p->variant != 0 && (p->win_left >= 0 || p->win_right >= 0 || p->softcap != 0.0 ||
                            p->alibi || p->sinks))
        return 1;
    if (!(p->softcap >= 0.0) || p->win_left < -1 || p->win_right < -1) return 1;
    int64_t total_q = p->query_start_loc[p->num_seqs];
    if (!p->rows) p->n_rows = total_q * p->Hq;
    p->max_kv = 0;
    for (int32_t b = 0; b < p->num_seqs; ++b)
        if (p->seq_lens[b] > p->max_kv) p->max_kv = p->seq_lens[b];
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 512) n_threads = 512;
    if (p->n_rows < n_threads) n_threads = p->n_rows > 0 ? (int32_t)p->n_rows : 1;

    pthread_t th[512];
    int created[512];
    job_t jobs[512];
    int64_t per = (p->n_rows + n_threads - 1) / n_threads;
    for (int32_t k = 0; k < n_threads; ++k) {
        jobs[k].p = p;
        jobs[k].begin = k * per < p->n_rows ? k * per : p->n_rows;
        jobs[k].end = (k + 1) * per < p->n_rows ? (k + 1) * per : p->n_rows;
        created[k] = 0;
        if (k == 0) continue;
        if (pthread_create(&th[k], NULL, run_job, &jobs[k]) == 0)
            created[k] = 1;
        else
            run_job(&jobs[k]);   /* could not start a thread: do the share here */
    }
    run_job(&jobs[0]);
    for (int32_t k = 1; k < n_threads; ++k)
        if (created[k]) pthread_join(th[k], NULL);
    return 0;
}

/* Common entry.  out is [n_rows, d] (n_rows = total_q * Hq when rows is
 * NULL, in (token, head) order), lse is [n_rows] or NULL.  win_left /
 * win_right = -1, softcap = 0, alibi = sinks = NULL give the plain problem;
 * kv_fp8 = 1 reads the caches as E4M3 bytes scaled by k_scale / v_scale. */
int oracle_sdpa_run_ex(double *out, double *lse,
                       const uint16_t *q, const void *k_cache, const void *v_cache,
                       const int32_t *block_table, int32_t bt_stride,
                       const int32_t *query_start_loc, const int32_t *seq_lens,
                       int32_t num_seqs, int32_t Hq, int32_t Hkv, int32_t d, int32_t bs,
                       double scale, int32_t causal, int32_t dtype,
                       int32_t variant, int32_t param,
                       const int64_t *rows, int64_t n_rows, int32_t n_threads,
                       int32_t win_left, int32_t win_right, double softcap,
                       const double *alibi, const double *sinks,
                       int32_t kv_fp8, double k_scale, double v_scale)
{
    problem_t p;
    memset(&p, 0, sizeof(p));
    p.win_left = win_left; p.win_right = win_right; p.softcap = softcap;
    p.alibi = alibi; p.sinks = sinks;
    p.kv_fp8 = kv_fp8; p.k_scale = k_scale; p.v_scale = v_scale;
    p.q = q; p.k_cache = k_cache; p.v_cache = v_cache;
    p.block_table = block_table; p.bt_stride = bt_stride;
    p.query_start_loc = query_start_loc; p.seq_lens = seq_lens;
    p.num_seqs = num_seqs; p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.bs = bs;
    p.scale = scale; p.causal = causal; p.dtype = dtype;
    p.variant = variant; p.param = param;
    p.rows = rows; p.n_rows = n_rows;
    p.out = out; p.lse = lse;
    return run_problem(&p, n_threads);
}

int oracle_sdpa_run(double *out, double *lse,
                    const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                    const int32_t *block_table, int32_t bt_stride,
                    const int32_t *query_start_loc, const int32_t *seq_lens,
                    int32_t num_seqs, int32_t Hq, int32_t Hkv, int32_t d, int32_t bs,
                    double scale, int32_t causal, int32_t dtype,
                    int32_t variant, int32_t param,
                    const int64_t *rows, int64_t n_rows, int32_t n_threads)
{
    return oracle_sdpa_run_ex(out, lse, q, k_cache, v_cache, block_table, bt_stride,
                              query_start_loc, seq_lens, num_seqs, Hq, Hkv, d, bs, scale,
                              causal, dtype, variant, param, rows, n_rows, n_threads,
                              -1, -1, 0.0, NULL, NULL, 0, 1.0, 1.0);
}
