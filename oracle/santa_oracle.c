/*
 * santa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * The plain, slow, fp64 CPU oracle for SANTA decode-step attention
 * ("Stochastic Sparse Attention for Memory-Bound Inference", abstract).  Only the
 * tests, the smoke check and the CPU-baseline leg of the benchmark may load it.  It
 * shares no code, header, table or constant generator with the CUDA library: the mode
 * numbers and the Philox layout below are written out again here on purpose.
 *
 * What it computes, per (batch b, query head h), with g = h / (H_q / H_kv) the KV head
 * and n = seq_lens[b] valid keys (all arithmetic in IEEE fp64):
 *
 *   s_j = sigma * sum_i q[b,h,i] * K[b,g,j,i]            (abstract: the score stage
 *                                                         reads all n_k keys)
 *   m = max_j s_j,   w_j = exp(s_j - m),   W_j = w_0 + ... + w_j,   Z = W_{n-1}
 *   p_j = w_j / Z                                        (post-softmax distribution)
 *   dense:    o = sum_j p_j v_j                          (exact attention, the value
 *                                                         the estimator targets)
 *   sampled:  S points t_0 <= ... <= t_{S-1} in [0,1), T_s = t_s * Z,
 *             i_s = min{ j : W_j > T_s } (clamped to n-1),
 *             o_hat = (1/S) * sum_s v_{i_s}              (abstract: sample S << n_k
 *                                                         indices from the post-softmax
 *                                                         distribution and aggregate only
 *                                                         those value rows; unbiased)
 *
 * Points (abstract: "stratified and systematic sampling"; the pages give no formula,
 * so the plainest unbiased readings are used):
 *   systematic:  one uniform u per (b,h);  t_s = (u + s) * r_S
 *   stratified:  one uniform u_s per stratum;  t_s = (s + u_s) * r_S
 *   iid:         S independent uniforms, sorted ascending
 * with r_S = 1/S rounded once to fp64: the pages leave the arithmetic open, and one
 * correctly rounded multiply is reproducible bit for bit by any IEEE implementation
 * (u + s is exact, since u has 32 fraction bits and s < 2^21).
 * Uniforms: the top 32 bits of a Philox4x64-10 word times 2^-32 (an exact fp64 in
 * [0, 1 - 2^-32]).  Philox4x64-10 is the counter-based generator of Salmon, Moraes,
 * Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11), written here
 * from that definition.  key = (seed, 0); counter = (block, b, h, domain) with domain
 * 1 = stratified, 2 = systematic, 3 = iid.  Systematic uses word 0 of block 0;
 * stratified and iid use word (s mod 4) of block floor(s/4).
 *
 * Inputs q, K, V arrive as bf16 bit patterns (uint16) and are widened exactly to fp64.
 * sigma is the fp64 value of the fp32 scale the caller passes.
 *
 * Bernoulli qK^T (abstract, last sentences: the score stage is sparsified by
 * "stochastic ternary queries" that reduce key-feature access; the pages give no
 * formula).  Reading taken, the plainest unbiased one: before scoring, each query head
 * q (d features) is replaced by one ternary draw q~ with q~_i in {-a, 0, +a},
 * a = max_i |q_i|, where q~_i = sign(q_i) * a with probability |q_i| / a and 0
 * otherwise, independently per feature; so E[q~_i] = q_i and E[q~ . k] = q . k for every
 * key.  The same q~ scores all keys of the head (it is one query), and a score then needs
 * only the features where q~_i != 0.  The uniform of feature i is the top 32 bits x_i of
 * word (i mod 4) of the Philox block (floor(i/4), b, h, 4) (domain 4, apart from the
 * sampling's domains), and the draw keeps the sign when x_i * 2^-32 < |q_i| / a, i.e.
 * when x_i * a < |q_i| * 2^32: both products are exact in fp64 (x_i has 32 bits, a and
 * q_i are bf16 values with 8), so the decision has no rounding.  q~ is a vector of bf16
 * values (a is one), and the rest of the step runs on it unchanged.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_DENSE 0
#define ORC_STRATIFIED 1
#define ORC_SYSTEMATIC 2
#define ORC_IID 3

/* ---------------- Philox4x64-10 (Salmon et al., SC'11) ---------------- */

static uint64_t mulhilo64(uint64_t a, uint64_t b, uint64_t *hi)
{
    unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
    *hi = (uint64_t)(p >> 64);
    return (uint64_t)p;
}

/* One Philox4x64 round: two 64x64->128 multiplies, then a xor with the key and the
 * other two counter words, with the words permuted. */
static void philox4x64_round(uint64_t x[4], const uint64_t k[2])
{
    uint64_t hi0, hi1;
    uint64_t lo0 = mulhilo64(0xD2E7470EE14C6C93ULL, x[0], &hi0);
    uint64_t lo1 = mulhilo64(0xCA5A826395121157ULL, x[2], &hi1);
    uint64_t y0 = hi1 ^ x[1] ^ k[0];
    uint64_t y2 = hi0 ^ x[3] ^ k[1];
    x[0] = y0;
    x[1] = lo1;
    x[2] = y2;
    x[3] = lo0;
}

void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4])
{
    uint64_t x[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint64_t k[2] = {key[0], key[1]};
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {               /* Weyl key schedule between rounds */
            k[0] += 0x9E3779B97F4A7C15ULL;
            k[1] += 0xBB67AE8584CAA73BULL;
        }
        philox4x64_round(x, k);
    }
    memcpy(out, x, sizeof x);
}

/* Uniform in [0,1): top 32 bits of a 64-bit word times 2^-32 (exact in fp64). */
static double word_to_uniform(uint64_t x)
{
    return (double)(x >> 32) * 0x1p-32;
}

static int cmp_double(const void *a, const void *b)
{
    double x = *(const double *)a, y = *(const double *)b;
    return (x > y) - (x < y);
}

/* The S sorted sample points of one (b, h).  Returns 0, or -1 on a bad mode/S. */
int oracle_points(int mode, int32_t S, uint64_t seed, int32_t b, int32_t h, double *t)
{
    if (S < 1) return -1;
    const uint64_t key[2] = {seed, 0};
    if (mode == ORC_SYSTEMATIC) {
        const uint64_t ctr[4] = {0, (uint64_t)b, (uint64_t)h, 2};
        uint64_t r[4];
        oracle_philox4x64_10(ctr, key, r);
        const double u = word_to_uniform(r[0]);
        const double rS = 1.0 / (double)S;
        for (int32_t s = 0; s < S; ++s) t[s] = (u + (double)s) * rS;
        return 0;
    }
    if (mode == ORC_STRATIFIED || mode == ORC_IID) {
        const uint64_t dom = (mode == ORC_STRATIFIED) ? 1 : 3;
        const double rS = 1.0 / (double)S;
        uint64_t r[4];
        for (int32_t s = 0; s < S; ++s) {
            if (s % 4 == 0) {
                const uint64_t ctr[4] = {(uint64_t)(s / 4), (uint64_t)b, (uint64_t)h, dom};
                oracle_philox4x64_10(ctr, key, r);
            }
            const double u = word_to_uniform(r[s % 4]);
            t[s] = (mode == ORC_STRATIFIED) ? ((double)s + u) * rS : u;
        }
        if (mode == ORC_IID) qsort(t, (size_t)S, sizeof(double), cmp_double);
        return 0;
    }
    return -1;
}

/* ---------------- exact attention pieces ---------------- */

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Scores s[0..n-1] and unnormalised CDF W[0..n-1] (inclusive prefix of
 * w_j = exp(s_j - m)) of one (b, h); returns m via *m_out. */
static void cdf_one(int32_t H_q, int32_t H_kv, int32_t d, int32_t n_max, double sigma,
                    const uint16_t *qh, const uint16_t *k, int32_t b, int32_t h, int32_t n,
                    double *s, double *W, double *m_out)
{
    const int32_t G = H_q / H_kv;
    const int32_t g = h / G;
    const uint16_t *kg = k + ((size_t)b * H_kv + g) * (size_t)n_max * d;
    double m = -INFINITY;
    for (int32_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int32_t i = 0; i < d; ++i)
            dot += bf16_to_double(qh[i]) * bf16_to_double(kg[(size_t)j * d + i]);
        s[j] = sigma * dot;
        if (s[j] > m) m = s[j];
    }
    double acc = 0.0;
    for (int32_t j = 0; j < n; ++j) {
        acc += exp(s[j] - m);
        W[j] = acc;
    }
    *m_out = m;
}

/* Bernoulli qK^T: the ternary draw q~ of one query head qh [d] (bf16 bits) as bf16 bits
 * qt [d].  Returns the number of non-zero features. */
int32_t oracle_ternary_query(int32_t d, const uint16_t *qh, uint64_t seed, int32_t b, int32_t h,
                             uint16_t *qt)
{
    double a = 0.0;
    uint16_t abits = 0;
    for (int32_t i = 0; i < d; ++i) {
        const double x = fabs(bf16_to_double(qh[i]));
        if (x > a) {
            a = x;
            abits = (uint16_t)(qh[i] & 0x7fffu);
        }
    }
    const uint64_t key[2] = {seed, 0};
    uint64_t r[4] = {0, 0, 0, 0};
    int32_t nnz = 0;
    for (int32_t i = 0; i < d; ++i) {
        if (i % 4 == 0) {
            const uint64_t ctr[4] = {(uint64_t)(i / 4), (uint64_t)b, (uint64_t)h, 4};
            oracle_philox4x64_10(ctr, key, r);
        }
        const double x = (double)(r[i % 4] >> 32);
        const double qi = fabs(bf16_to_double(qh[i]));
        /* keep with probability |q_i| / a: x 2^-32 < |q_i| / a  <=>  x a < |q_i| 2^32 */
        if (a > 0.0 && x * a < qi * 0x1p32) {
            qt[i] = (uint16_t)((qh[i] & 0x8000u) | abits);
            ++nnz;
        } else {
            qt[i] = 0;
        }
    }
    return nnz;
}

/* i = min{ j : W_j > T }, clamped to n-1 (plain binary search over a nondecreasing
 * array). */
static int32_t search_cdf(const double *W, int32_t n, double T)
{
    int32_t lo = 0, hi = n;            /* answer in [lo, hi] */
    while (lo < hi) {
        int32_t mid = lo + (hi - lo) / 2;
        if (W[mid] > T) hi = mid; else lo = mid + 1;
    }
    return lo < n ? lo : n - 1;
}

static int check_shape(int32_t B, int32_t H_q, int32_t H_kv, int32_t d, int32_t n_max)
{
    if (B < 0 || H_q <= 0 || H_kv <= 0 || d <= 0 || n_max < 0) return -1;
    if (H_q % H_kv != 0) return -1;
    return 0;
}

/*
 * Full decode step.  mode: 0 dense, 1 stratified, 2 systematic, 3 iid; ternary != 0
 * first replaces every query head by its Bernoulli qK^T draw (seeded by `seed`).
 * q [B,H_q,d], k/v [B,H_kv,n_max,d] as bf16 bits; seq_lens [B] (0 <= n_b <= n_max).
 * t_in: optional caller-chosen points [B,H_q,S] replacing the Philox points.
 * pairs: optional list of n_pairs (b,h) pairs to compute (NULL: all B*H_q pairs).
 * out [B,H_q,d] fp64; idx [B,H_q,S] int32 (optional); Z_out [B,H_q] (optional).
 * n_b = 0 yields out = 0, idx = -1, Z = 0.  Returns 0 or -1 on bad arguments.
 */
int oracle_decode(int32_t B, int32_t H_q, int32_t H_kv, int32_t d, int32_t n_max, float scale,
                  const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  const int32_t *seq_lens, int32_t S, int mode, uint64_t seed, int ternary,
                  const double *t_in, const int32_t *pairs, int32_t n_pairs,
                  double *out, int32_t *idx, double *Z_out)
{
    if (check_shape(B, H_q, H_kv, d, n_max)) return -1;
    if (mode < 0 || mode > 3) return -1;
    if (mode != ORC_DENSE && S < 1) return -1;
    for (int32_t b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > n_max) return -1;
    const int32_t G = H_q / H_kv;
    const double sigma = (double)scale;
    const int32_t total = pairs ? n_pairs : B * H_q;
    const int32_t Sa = S > 0 ? S : 1;
    int bad = 0;

#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(n_max > 0 ? n_max : 1));
        double *W = (double *)malloc(sizeof(double) * (size_t)(n_max > 0 ? n_max : 1));
        double *t = (double *)malloc(sizeof(double) * (size_t)Sa);
        double *acc = (double *)malloc(sizeof(double) * (size_t)d);
        uint16_t *qt = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)d);
        if (!s || !W || !t || !acc || !qt) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int32_t pi = 0; pi < total; ++pi) {
            if (bad) continue;
            const int32_t b = pairs ? pairs[2 * pi] : pi / H_q;
            const int32_t h = pairs ? pairs[2 * pi + 1] : pi % H_q;
            if (b < 0 || b >= B || h < 0 || h >= H_q) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const int32_t n = seq_lens[b];
            const int32_t g = h / G;
            double *o = out + ((size_t)b * H_q + h) * d;
            int32_t *ix = (idx && mode != ORC_DENSE) ? idx + ((size_t)b * H_q + h) * (size_t)S : NULL;
            if (n == 0) {
                for (int32_t i = 0; i < d; ++i) o[i] = 0.0;
                if (ix) for (int32_t si = 0; si < S; ++si) ix[si] = -1;
                if (Z_out) Z_out[(size_t)b * H_q + h] = 0.0;
                continue;
            }
            double m;
            const uint16_t *qh = q + ((size_t)b * H_q + h) * d;
            if (ternary) {  /* step 1 of Bernoulli qK^T: the ternary query */
                oracle_ternary_query(d, qh, seed, b, h, qt);
                qh = qt;
            }
            cdf_one(H_q, H_kv, d, n_max, sigma, qh, k, b, h, n, s, W, &m);
            const double Z = W[n - 1];
            if (Z_out) Z_out[(size_t)b * H_q + h] = Z;
            const uint16_t *vg = v + ((size_t)b * H_kv + g) * (size_t)n_max * d;
            for (int32_t i = 0; i < d; ++i) acc[i] = 0.0;
            if (mode == ORC_DENSE) {
                for (int32_t j = 0; j < n; ++j) {
                    const double p = exp(s[j] - m) / Z;
                    for (int32_t i = 0; i < d; ++i)
                        acc[i] += p * bf16_to_double(vg[(size_t)j * d + i]);
                }
                for (int32_t i = 0; i < d; ++i) o[i] = acc[i];
            } else {
                if (t_in) {
                    memcpy(t, t_in + ((size_t)b * H_q + h) * S, sizeof(double) * (size_t)S);
                } else if (oracle_points(mode, S, seed, b, h, t)) {
#pragma omp atomic write
                    bad = 1;
                    continue;
                }
                for (int32_t si = 0; si < S; ++si) {
                    const double T = t[si] * Z;
                    const int32_t j = search_cdf(W, n, T);
                    if (ix) ix[si] = j;
                    for (int32_t i = 0; i < d; ++i) acc[i] += bf16_to_double(vg[(size_t)j * d + i]);
                }
                for (int32_t i = 0; i < d; ++i) o[i] = acc[i] / (double)S;
            }
        }
        free(s); free(W); free(t); free(acc); free(qt);
    }
    return bad ? -1 : 0;
}

/* Unnormalised CDF W[0..n-1] and max score m of one (b, h), for boundary analysis. */
int oracle_cdf(int32_t B, int32_t H_q, int32_t H_kv, int32_t d, int32_t n_max, float scale,
               const uint16_t *q, const uint16_t *k, const int32_t *seq_lens,
               int32_t b, int32_t h, double *W, double *m_out)
{
    if (check_shape(B, H_q, H_kv, d, n_max)) return -1;
    if (b < 0 || b >= B || h < 0 || h >= H_q) return -1;
    const int32_t n = seq_lens[b];
    if (n < 0 || n > n_max) return -1;
    if (n == 0) { *m_out = -INFINITY; return 0; }
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    if (!s) return -1;
    cdf_one(H_q, H_kv, d, n_max, (double)scale, q + ((size_t)b * H_q + h) * d, k, b, h, n, s, W, m_out);
    free(s);
    return 0;
}

/* o_hat = (1/S) * sum_s v_{idx[b,h,s]} for given indices (any source), fp64.  An index
 * outside [0, seq_lens[b]) makes the call fail with -1. */
int oracle_gather(int32_t B, int32_t H_q, int32_t H_kv, int32_t d, int32_t n_max,
                  const uint16_t *v, const int32_t *seq_lens, const int32_t *idx, int32_t S,
                  double *out)
{
    if (check_shape(B, H_q, H_kv, d, n_max) || S < 1) return -1;
    const int32_t G = H_q / H_kv;
    int bad = 0;
#pragma omp parallel for schedule(static)
    for (int32_t pi = 0; pi < B * H_q; ++pi) {
        const int32_t b = pi / H_q, h = pi % H_q, g = h / G;
        const int32_t n = seq_lens[b];
        const uint16_t *vg = v + ((size_t)b * H_kv + g) * (size_t)n_max * d;
        double *o = out + (size_t)pi * d;
        for (int32_t i = 0; i < d; ++i) o[i] = 0.0;
        if (n == 0) continue;
        for (int32_t si = 0; si < S; ++si) {
            const int32_t j = idx[(size_t)pi * S + si];
            if (j < 0 || j >= n) {
#pragma omp atomic write
                bad = 1;
                break;
            }
            for (int32_t i = 0; i < d; ++i) o[i] += bf16_to_double(vg[(size_t)j * d + i]);
        }
        for (int32_t i = 0; i < d; ++i) o[i] /= (double)S;
    }
    return bad ? -1 : 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
