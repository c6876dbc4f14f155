/*
 * zyfa_oracle.c -- CPU oracle for causal FP8 / BF16 flash attention with
 * Lean P, exact P, per-64-key power-of-two block scaling and division by the
 * sum of the rounded probabilities.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; it is used by tests/, by __graft_entry__.smoke() and by the
 * cpu_baseline / reference leg of bench.py.  It shares no code, header, table
 * or constant generator with the CUDA library.
 *
 * Source: "ZYFA: Speed and Accuracy of FP8 FlashAttention on AMD CDNA4"
 * (arXiv 2611.07496).  Every step cites the section it follows:
 *   - causal attention, base-2 scores t = c*q.k*log2(e), running maximum and
 *     rescale of acc and l by 2^(m_old - m): Sec. II-B and its footnotes 3, 4;
 *   - e4m3 format (bias 7, 3 mantissa bits, max 448, normal >= 2^-6,
 *     subnormal spacing 2^-9, underflow below 2^-10) and one FP32 scale per
 *     tensor folded into c and the output: Sec. II-C and footnote 5;
 *   - Lean P, y = 8(x + sigma + 7) - beta rounded to an integer code,
 *     sigma = 6, beta = 0.35, clamp to [0, 255]: Sec. IV-B1, Eq. (2);
 *   - exact P, e4m3 rounding of 2^(x+sigma): Sec. IV-B1;
 *   - lazy rescaling with threshold tau: Sec. IV-A ("Lazy rescaling") and
 *     footnote 9;
 *   - per-64-key block exponent o = whole binades between block max and row
 *     max, probabilities multiplied by 2^o and the product by 2^-o:
 *     Sec. IV-B2 and Fig. 5;
 *   - row sum of the rounded probabilities as the denominator: Sec. IV-B3 and
 *     footnote 12; the unrounded-denominator variant is the baseline that
 *     Fig. 5 (panel 1) describes;
 *   - LSE of the rounded probabilities: Sec. IV-B3;
 *   - fp64 attention on the quantised inputs as the error reference:
 *     Sec. V-D and footnote 15; the P term emulated with the exact row maximum:
 *     Sec. V-E ("Error of each stage of one call").
 *
 * Everything is computed in fp64 (binary64); the build uses
 * -ffp-contract=off so that results do not depend on FMA contraction.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* e4m3 (the "fn" variant: no infinities, code 0x7F/0xFF is NaN)            */
/* Sec. II-C: 4 exponent bits with bias 7, 3 mantissa bits, max 448.         */
/* Footnote 5: normal values 1.f x 2^e down to 2^-6, subnormal 0.f x 2^-6    */
/* spaced 2^-9 apart.                                                        */
/* ------------------------------------------------------------------------ */
double zo_e4m3_decode(unsigned code)
{
    code &= 0xFFu;
    unsigned s = code >> 7, E = (code >> 3) & 15u, M = code & 7u;
    double v;
    if (E == 15u && M == 7u) return NAN;
    if (E == 0u)
        v = ldexp((double)M, -9);                 /* 0.M x 2^-6 = M x 2^-9 */
    else
        v = ldexp(1.0 + (double)M / 8.0, (int)E - 7);
    return s ? -v : v;
}

/* Round-to-nearest-even onto the e4m3 grid, saturating to +-448 (finite
 * values only ever saturate; NaN maps to the NaN code). */
unsigned zo_e4m3_encode(double x)
{
    if (isnan(x)) return 0x7Fu;
    unsigned sign = signbit(x) ? 0x80u : 0u;
    double a = fabs(x);
    unsigned code;
    if (isinf(a)) return sign | 0x7Eu;            /* saturates like any a > 448 */
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: value = n x 2^-9, code = n (n = 8 is 2^-6) */
        double n = nearbyint(a * 512.0);          /* ties to even */
        code = (unsigned)n;
    } else {
        int e;
        (void)frexp(a, &e);                       /* a = f 2^e, f in [0.5,1) */
        int E = e - 1;                            /* a in [2^E, 2^(E+1))     */
        if (E > 8) {
            code = 0x7Eu;                         /* beyond 448: saturate    */
        } else {
            double q = ldexp(a, 3 - E);           /* in [8,16): 8 steps/binade */
            double n = nearbyint(q);              /* ties to even            */
            long c = 8L * E + 48L + (long)n;      /* (E+7)*8 + (n-8)         */
            code = c > 0x7E ? 0x7Eu : (unsigned)c;
        }
    }
    return sign | code;
}

/* Element-wise zo_e4m3_encode over an array (the quantisation oracle). */
void zo_e4m3_encode_n(const double* x, unsigned char* out, long long n)
{
    for (long long i = 0; i < n; ++i) out[i] = (unsigned char)zo_e4m3_encode(x[i]);
}

/* ------------------------------------------------------------------------ */
/* bfloat16: 8 significant bits.  Round-to-nearest-even directly from fp64. */
/* ------------------------------------------------------------------------ */
unsigned zo_bf16_encode(double x)
{
    if (isnan(x)) return 0x7FC0u;
    unsigned sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);                           /* a = f 2^e, f in [0.5,1) */
    int ulp_exp = e - 8;                          /* 8 significant bits      */
    if (ulp_exp < -133) ulp_exp = -133;           /* subnormal spacing 2^-133 */
    double n = nearbyint(ldexp(a, -ulp_exp));     /* ties to even            */
    double r = ldexp(n, ulp_exp);
    if (r > 3.3895313892515355e38) return sign | 0x7F80u;   /* overflow -> inf */
    float f = (float)r;                           /* exact: r has <= 8 bits  */
    uint32_t u;
    memcpy(&u, &f, 4);
    return sign | (u >> 16);
}

double zo_bf16_decode(unsigned bits)
{
    uint32_t u = (bits & 0xFFFFu) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Probability codes.  u = x + o, where x = t - m (base-2 score relative to   */
/* the reference maximum) and o the block exponent.                          */
/* ------------------------------------------------------------------------ */

/* Eq. (2) before rounding: y = 8 (u + sigma + 7) - beta. */
double zo_lean_y(double u, double sigma, double beta)
{
    return 8.0 * (u + sigma + 7.0) - beta;
}

/* Eq. (2) rounded to the nearest integer (ties to even), clamped to
 * [0, 255]; a NaN score gives code 0 (Sec. IV-B "Non-finite inputs"). */
unsigned zo_lean_code(double u, double sigma, double beta)
{
    double y = zo_lean_y(u, sigma, beta);
    if (!(y > 0.0)) return 0u;                    /* also NaN and -inf       */
    double n = nearbyint(y);
    if (n > 255.0) n = 255.0;
    return (unsigned)n;
}

/* Exact P: the e4m3 value nearest to 2^(u + sigma) (Sec. IV-B1). */
unsigned zo_exact_code(double u, double sigma)
{
    return zo_e4m3_encode(exp2(u + sigma));
}

/* ------------------------------------------------------------------------ */
/* Forward pass                                                              */
/* ------------------------------------------------------------------------ */
typedef struct {
    int dtype;            /* 0: e4m3 codes (1 byte);  1: bf16 bits (2 bytes); */
                          /* 2: bf16 Q and K, e4m3 V, FP8 probabilities      */
    int B, Hq, Hkv, N, d_qk, d_v;
    int causal;           /* 1: key j visible to query i iff j <= i           */
    double descale_q, descale_k, descale_v;   /* per-tensor scales (Sec. II-C) */
    double softmax_scale; /* c                                                */
    int p_mode;           /* 0: exact P, 1: Lean P, 2: unrounded p            */
    int block_scale;      /* 1: per-64-key power-of-two scaling (Sec. IV-B2)  */
    int max_mode;         /* 0: exact row maximum; 1: running maximum updated */
                          /*    once per key block of kv_block keys, lazily   */
    double tau;           /* lazy-rescaling threshold in base-2 units         */
    int kv_block;         /* keys per running-maximum step (max_mode 1)       */
    int scale_block;      /* keys per block exponent (64)                     */
    int denom_mode;       /* 0: sum of rounded p; 1: sum of unrounded p       */
    double sigma;         /* probability shift (6 in FP8, 0 in BF16)          */
    double beta;          /* Lean P bias (0.35)                               */
    int o_max;            /* largest block exponent (UE8M0 range: 127)        */
    int key_begin;        /* keys [key_begin, key_end) only (split-key       */
    int key_end;          /* partial attention, Sec. IV-B3); key_end < 0: N   */
} zo_params;

static double e4m3_table[256];
static pthread_once_t table_once = PTHREAD_ONCE_INIT;
static void build_table(void)
{
    for (int i = 0; i < 256; ++i) e4m3_table[i] = zo_e4m3_decode((unsigned)i);
}

static inline double load_e4m3(const void* base, size_t idx)
{
    return e4m3_table[((const uint8_t*)base)[idx]];
}
static inline double load_bf16(const void* base, size_t idx)
{
    return zo_bf16_decode(((const uint16_t*)base)[idx]);
}
/* Q and K elements: e4m3 in dtype 0, bf16 otherwise. */
static inline double load_qk(const zo_params* p, const void* base, size_t idx)
{
    return p->dtype == 0 ? load_e4m3(base, idx) : load_bf16(base, idx);
}
/* V elements: bf16 in dtype 1, e4m3 otherwise. */
static inline double load_v(const zo_params* p, const void* base, size_t idx)
{
    return p->dtype == 1 ? load_bf16(base, idx) : load_e4m3(base, idx);
}

/* Probability of one key given u = x + o: returns the rounded value used in
 * the numerator (*pr) and the unrounded value (*pu), both including 2^sigma
 * and the factor 2^o. */
static inline void prob(const zo_params* p, double u, double* pr, double* pu)
{
    double exact = exp2(u + p->sigma);
    *pu = exact;
    if (p->p_mode == 2) { *pr = exact; return; }
    if (p->dtype == 1) { *pr = zo_bf16_decode(zo_bf16_encode(exact)); return; }
    if (p->p_mode == 1)
        *pr = e4m3_table[zo_lean_code(u, p->sigma, p->beta)];
    else
        *pr = e4m3_table[zo_e4m3_encode(exact)];
}

typedef struct {
    const zo_params* p;
    const void *q, *k, *v;
    const long long* rows;
    long long nrows;
    double* out;          /* nrows x d_v, fp64 result before BF16 rounding   */
    unsigned short* out_bf16;   /* nrows x d_v BF16 bits (optional)          */
    double* lse;          /* nrows, natural log (optional)                    */
    int reference;        /* 1: fp64 exact softmax attention                  */
    long long next;       /* shared work counter                              */
} zo_job;

/* First key of the range. */
static inline int key0(const zo_params* p) { return p->key_begin > 0 ? p->key_begin : 0; }

/* Scores of row r: fills t[j] = c * dq * dk * log2(e) * (q_i . k_(key0 + j))
 * for the visible keys of the key range and returns their count. */
static int row_scores(const zo_params* p, const void* q, const void* k,
                      long long r, double* qv, double* t)
{
    int N = p->N, Hq = p->Hq;
    long long b = r / ((long long)Hq * N);
    int h = (int)((r / N) % Hq);
    int i = (int)(r % N);
    int g = h / (Hq / p->Hkv);
    int kend = p->causal ? i + 1 : N;
    if (p->key_end >= 0 && p->key_end < kend) kend = p->key_end;
    int nk = kend - key0(p);
    if (nk < 0) nk = 0;
    size_t qoff = (((size_t)b * N + i) * Hq + h) * (size_t)p->d_qk;
    for (int d = 0; d < p->d_qk; ++d) qv[d] = load_qk(p, q, qoff + d);
    double cst = p->softmax_scale * p->descale_q * p->descale_k * M_LOG2E;
    for (int jj = 0; jj < nk; ++jj) {
        const int j = key0(p) + jj;
        size_t koff = (((size_t)b * N + j) * p->Hkv + g) * (size_t)p->d_qk;
        double s = 0.0;
        for (int d = 0; d < p->d_qk; ++d) s += qv[d] * load_qk(p, k, koff + d);
        t[jj] = cst * s;
    }
    return nk;
}

static inline void add_value(const zo_params* p, const void* v, long long b,
                             int g, int j, double w, double* acc)
{
    size_t voff = (((size_t)b * p->N + key0(p) + j) * p->Hkv + g) * (size_t)p->d_v;
    for (int d = 0; d < p->d_v; ++d) acc[d] += w * load_v(p, v, voff + d);
}

static inline double nanmax(double a, double b)
{
    return fmax(a, b);                            /* NaN operands are ignored */
}

/* One query row of the method.  Keys are visited in segments that share one
 * reference maximum: a single segment holding every visible key with the
 * exact row maximum (max_mode 0), or blocks of kv_block keys in ascending
 * order with the lazily updated running maximum (max_mode 1).  Within a
 * segment each scale_block-aligned block of keys gets its own exponent o. */
static void method_row(const zo_params* p, const void* v, long long r,
                       const double* t, int nk, double* acc, double* out,
                       double* lse_out)
{
    int N = p->N, Hq = p->Hq;
    long long b = r / ((long long)Hq * N);
    int h = (int)((r / N) % Hq);
    int g = h / (Hq / p->Hkv);
    for (int d = 0; d < p->d_v; ++d) acc[d] = 0.0;
    double l = 0.0;
    double m_ref = -INFINITY;
    if (nk == 0) {        /* no visible key in the range: nothing to merge */
        for (int d = 0; d < p->d_v; ++d) out[d] = 0.0;
        if (lse_out) *lse_out = -INFINITY;
        return;
    }

    int seg = p->max_mode == 0 ? nk : p->kv_block;
    if (p->max_mode == 0)
        for (int j = 0; j < nk; ++j) m_ref = nanmax(m_ref, t[j]);

    for (int s0 = 0; s0 < nk; s0 += seg) {
        int s1 = s0 + seg < nk ? s0 + seg : nk;
        if (p->max_mode == 1) {
            double bm = -INFINITY;
            for (int j = s0; j < s1; ++j) bm = nanmax(bm, t[j]);
            double m_new = m_ref;
            if (s0 == 0 || bm - m_ref > p->tau) m_new = bm;
            if (s0 > 0 && m_new != m_ref) {
                /* footnote 4: rescale acc and l by 2^(m_old - m_new) */
                double f = exp2(m_ref - m_new);
                for (int d = 0; d < p->d_v; ++d) acc[d] *= f;
                l *= f;
            }
            m_ref = m_new;
        }
        int sb = p->scale_block;
        for (int c0 = (s0 / sb) * sb; c0 < s1; c0 += sb) {
            int a0 = c0 > s0 ? c0 : s0;
            int a1 = c0 + sb < s1 ? c0 + sb : s1;
            double hm = -INFINITY;
            for (int j = a0; j < a1; ++j) hm = nanmax(hm, t[j]);
            int o = 0;
            if (p->block_scale && hm > -INFINITY) {
                double gap = floor(m_ref - hm);
                if (gap > (double)p->o_max) gap = (double)p->o_max;
                o = gap > 0.0 ? (int)gap : 0;
            }
            double inv = ldexp(1.0, -o);
            for (int j = a0; j < a1; ++j) {
                double pr, pu;
                prob(p, t[j] - m_ref + (double)o, &pr, &pu);
                double w = pr * inv;
                add_value(p, v, b, g, j, w, acc);
                l += p->denom_mode == 0 ? w : pu * inv;
            }
        }
    }
    for (int d = 0; d < p->d_v; ++d) out[d] = p->descale_v * acc[d] / l;
    if (lse_out)   /* ln sum_j exp(score_j), from the same weights: l 2^(m - sigma) */
        *lse_out = log(l) + (m_ref - p->sigma) * M_LN2;
}

/* fp64 softmax attention on the dequantised inputs (Sec. V-D). */
static void reference_row(const zo_params* p, const void* v, long long r,
                          const double* t, int nk, double* acc, double* out,
                          double* lse_out)
{
    int N = p->N, Hq = p->Hq;
    long long b = r / ((long long)Hq * N);
    int h = (int)((r / N) % Hq);
    int g = h / (Hq / p->Hkv);
    if (nk == 0) {
        for (int d = 0; d < p->d_v; ++d) out[d] = 0.0;
        if (lse_out) *lse_out = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int j = 0; j < nk; ++j) m = nanmax(m, t[j] * M_LN2);
    for (int d = 0; d < p->d_v; ++d) acc[d] = 0.0;
    double l = 0.0;
    for (int j = 0; j < nk; ++j) {
        double w = exp(t[j] * M_LN2 - m);
        add_value(p, v, b, g, j, w, acc);
        l += w;
    }
    for (int d = 0; d < p->d_v; ++d) out[d] = p->descale_v * acc[d] / l;
    if (lse_out) *lse_out = m + log(l);
}

static void* worker(void* arg)
{
    zo_job* job = (zo_job*)arg;
    const zo_params* p = job->p;
    double* t = (double*)malloc(sizeof(double) * (size_t)(p->N > 0 ? p->N : 1));
    double* qv = (double*)malloc(sizeof(double) * (size_t)p->d_qk);
    double* acc = (double*)malloc(sizeof(double) * (size_t)p->d_v);
    if (!t || !qv || !acc) { free(t); free(qv); free(acc); return (void*)1; }
    for (;;) {
        long long n = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
        if (n >= job->nrows) break;
        long long r = job->rows[n];
        int nk = row_scores(p, job->q, job->k, r, qv, t);
        double* o = job->out + (size_t)n * p->d_v;
        double* lse = job->lse ? job->lse + n : NULL;
        if (job->reference)
            reference_row(p, job->v, r, t, nk, acc, o, lse);
        else
            method_row(p, job->v, r, t, nk, acc, o, lse);
        if (job->out_bf16)
            for (int d = 0; d < p->d_v; ++d)
                job->out_bf16[(size_t)n * p->d_v + d] = (unsigned short)zo_bf16_encode(o[d]);
    }
    free(t); free(qv); free(acc);
    return NULL;
}

static int check(const zo_params* p, const long long* rows, long long nrows)
{
    if (!p || p->B < 0 || p->N < 0 || p->Hq <= 0 || p->Hkv <= 0 || p->Hq % p->Hkv)
        return -2;
    if (p->d_qk <= 0 || p->d_v <= 0 || p->kv_block <= 0 || p->scale_block <= 0)
        return -2;
    long long total = (long long)p->B * p->Hq * p->N;
    for (long long n = 0; n < nrows; ++n)
        if (rows[n] < 0 || rows[n] >= total) return -2;
    return 0;
}

static int run(const zo_params* p, const void* q, const void* k, const void* v,
               const long long* rows, long long nrows, double* out,
               unsigned short* out_bf16, double* lse, int nthreads, int reference)
{
    int rc = check(p, rows, nrows);
    if (rc) return rc;
    pthread_once(&table_once, build_table);
    if (nrows == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    zo_job job = { p, q, k, v, rows, nrows, out, out_bf16, lse, reference, 0 };
    pthread_t th[512];
    int started = 0;
    for (int i = 1; i < nthreads; ++i)
        if (pthread_create(&th[started], NULL, worker, &job) == 0) ++started;
    void* res0 = worker(&job);
    int failed = res0 != NULL;
    for (int i = 0; i < started; ++i) {
        void* res;
        pthread_join(th[i], &res);
        failed |= res != NULL;
    }
    return failed ? -5 : 0;
}

/* The method (Lean P / exact P / unrounded, with block scaling and the chosen
 * maximum and denominator), for the listed rows.  rows[n] is the flat index
 * (b*Hq + h)*N + i.  Returns 0, or -2 on bad parameters. */
int zo_fwd(const zo_params* p, const void* q, const void* k, const void* v,
           const long long* rows, long long nrows, double* out,
           unsigned short* out_bf16, double* lse, int nthreads)
{
    return run(p, q, k, v, rows, nrows, out, out_bf16, lse, nthreads, 0);
}

/* fp64 exact softmax attention on the same (dequantised) inputs. */
int zo_attn_fp64(const zo_params* p, const void* q, const void* k, const void* v,
                 const long long* rows, long long nrows, double* out,
                 double* lse, int nthreads)
{
    return run(p, q, k, v, rows, nrows, out, NULL, lse, nthreads, 1);
}
