/*
 * eb_oracle.c -- plain CPU oracle of the Entropy-Bounded (EB) denoising sampler step
 * of DiffusionGemma's block-autoregressive text diffusion.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct statement of what
 * the GPU path computes.  Only the test suite, the smoke check and the benchmark's CPU
 * baseline call it.  It shares no code, header, table or constant generator with the
 * CUDA library; it carries its own Philox4x32-10.
 *
 * Precision: every floating-point quantity is computed in IEEE binary64 with the C
 * library's exp/log; logits are converted exactly from their binary32 / bfloat16 bits.
 * Parallelism: OpenMP over canvas rows only (rows are independent); every row and every
 * canvas selection is a plain sequential loop.
 *
 * Source passages (DiffusionGemma model card, "Best practices" section 1, "Diffusion
 * sampling settings"; the same list appears in the Korean model card's "Recommendations"
 * section 1 and in the aitrends.kr summary, "Good to know" / "Technical features"):
 *   - at most 48 denoising steps;
 *   - temperature schedule for logit shaping, linear from 0.8 down to 0.4;
 *   - each step selects the lowest-entropy tokens while their mutual-information bound
 *     stays under the entropy bound 0.1;
 *   - the tokens that were not selected are fully re-noised (re-masked);
 *   - adaptive stop only when the mean model entropy over the whole canvas is below
 *     0.005 AND the top-probability prediction is unchanged over two consecutive steps.
 * The pages give no selection formula.  The one used here: sort the still-masked
 * positions by entropy ascending (ties: lower position first) and accept sorted index i
 * iff the sum of the entropies before it is <= the bound (index 0 always accepted), i.e.
 * the longest prefix whose (sum - max) stays within the bound.
 *
 * Readings of points the pages leave open (each one also listed in the design notes):
 *   - entropy and sampling both use the shaped logits z = x / T;
 *   - T_s = t_start + (t_end - t_start) * s / (max_steps - 1);
 *   - the stop rule's mean runs over all L positions, committed ones included;
 *   - "unchanged over two consecutive steps" = argmax at step s equals argmax at s-1
 *     at every position, so the earliest stop is at s = 1;
 *   - on adaptive stop and at the step cap the positions still masked take the current
 *     step's argmax; committed tokens are never revised;
 *   - sampling is Gumbel-max: Y = argmax_v z_v - ln(-ln u_v), u_v a Philox uniform.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ----------------------------------------------------------------------------------
 * Philox4x32-10, written from its published definition: Salmon, Moraes, Dror, Shaw,
 * "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11, section 3 (the Philox S-P
 * network): per round two 32x32->64 products of counter words 0 and 2 with the
 * multipliers 0xD2511F53 and 0xCD9E8D57, the high halves xored with the other counter
 * words and the round key, the low halves passed through; the key is bumped by the Weyl
 * constants 0x9E3779B9 (golden ratio) and 0xBB67AE85 (sqrt(3)-1) between rounds.
 * -------------------------------------------------------------------------------- */
void eb_oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Random-number streams (field 3 of the counter, bits 24..31). */
#define EB_ORACLE_STREAM_GUMBEL 1u

/* The 32-bit Philox word that feeds the Gumbel noise of vocabulary entry v of canvas
 * row (b, p) at denoising step s.  Counter = (v / 4, p, s, stream << 24 | b), key =
 * (low, high) 32 bits of the seed; word v % 4 of the output belongs to entry v. */
uint32_t eb_oracle_gumbel_word(uint64_t seed, int b, int p, int s, int64_t v)
{
    uint32_t ctr[4] = {(uint32_t)(v >> 2), (uint32_t)p, (uint32_t)s,
                       (EB_ORACLE_STREAM_GUMBEL << 24) | (uint32_t)b};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    eb_oracle_philox4x32_10(ctr, key, out);
    return out[v & 3];
}

/* Uniform in (0,1) from a word: the low 23 bits j give u = (j + 1/2) / 2^23. */
double eb_oracle_uniform(uint32_t w)
{
    return ((double)(w & 0x7FFFFFu) + 0.5) / 8388608.0;
}

/* Standard Gumbel variate g = -ln(-ln u). */
double eb_oracle_gumbel(uint32_t w)
{
    double u = eb_oracle_uniform(w);
    return -log(-log(u));
}

/* Linear temperature schedule from t_start (step 0) to t_end (step max_steps-1). */
double eb_oracle_temperature(int step, int max_steps, double t_start, double t_end)
{
    if (max_steps <= 1) return t_start;
    return t_start + (t_end - t_start) * (double)step / (double)(max_steps - 1);
}

/* Value of one OCP FP8 e4m3 code: sign s, exponent field e (bias 7), mantissa m (3 bits);
 * e = 0 is subnormal, m / 8 * 2^-6; S.1111.111 is NaN; there are no infinities. */
static double e4m3_value(uint8_t code)
{
    const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(8.0 + (double)m, e - 10);
    return s ? -v : v;
}

/* Exact conversion of one logit to binary64. dtype: 0 = binary32, 1 = bfloat16 bits,
 * 2 = binary64, 3 = e4m3 codes. */
static double load_logit(const void *x, int dtype, int64_t i)
{
    if (dtype == 0) return (double)((const float *)x)[i];
    if (dtype == 1) {
        uint32_t bits = (uint32_t)((const uint16_t *)x)[i] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    if (dtype == 3) return e4m3_value(((const uint8_t *)x)[i]);
    return ((const double *)x)[i];
}

/* The e4m3 decoding above, exported for the tests. */
double eb_oracle_e4m3_value(int code) { return e4m3_value((uint8_t)code); }

/* One canvas row of V logits at temperature T.
 * Outputs: H = softmax entropy of z = x/T in nats; A = first index of the largest raw
 * logit; if masked, Y = first index of the largest z_v + g_v and gap = the distance
 * between the two largest perturbed scores divided by max(1, |largest|) (tie
 * accounting).  Unmasked rows get Y = -1 and gap = +inf. */
void eb_oracle_row(const void *x, int dtype, int64_t V, double T, int masked,
                   uint64_t seed, int b, int p, int s,
                   double *H, int32_t *A, int32_t *Y, double *gap)
{
    /* argmax of the raw logits (first index on equality) */
    int64_t a = 0;
    double amax = load_logit(x, dtype, 0);
    for (int64_t v = 1; v < V; ++v) {
        double xv = load_logit(x, dtype, v);
        if (xv > amax) { amax = xv; a = v; }
    }
    *A = (int32_t)a;

    /* softmax of z = x/T, then H = -sum p ln p */
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        double z = load_logit(x, dtype, v) / T;
        if (z > m) m = z;
    }
    double S = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double z = load_logit(x, dtype, v) / T;
        S += exp(z - m);
    }
    double logS = log(S);
    double h = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double z = load_logit(x, dtype, v) / T;
        double pv = exp(z - m) / S;
        if (pv > 0.0) {
            double logp = (z - m) - logS;
            h -= pv * logp;
        }
    }
    *H = h;

    /* Gumbel-max sample */
    if (masked) {
        double best = -INFINITY, second = -INFINITY;
        int64_t y = -1;
        for (int64_t v = 0; v < V; ++v) {
            double z = load_logit(x, dtype, v) / T;
            double score = z + eb_oracle_gumbel(eb_oracle_gumbel_word(seed, b, p, s, v));
            if (score > best) {
                second = best;
                best = score;
                y = v;
            } else if (score > second) {
                second = score;
            }
        }
        *Y = (int32_t)y;
        double scale = fabs(best) > 1.0 ? fabs(best) : 1.0;
        *gap = (V > 1) ? (best - second) / scale : INFINITY;
    } else {
        *Y = -1;
        *gap = INFINITY;
    }
}

/* Canvas status codes (stop reasons). */
#define EB_ORACLE_RUNNING 0
#define EB_ORACLE_ADAPTIVE 1
#define EB_ORACLE_COMPLETE 2
#define EB_ORACLE_CAP 3

typedef struct {
    double H;
    int32_t p;
} keyed_entropy;

static int cmp_keyed(const void *pa, const void *pb)
{
    const keyed_entropy *a = (const keyed_entropy *)pa, *b = (const keyed_entropy *)pb;
    if (a->H < b->H) return -1;
    if (a->H > b->H) return 1;
    return (a->p > b->p) - (a->p < b->p);
}

/* Entropy-bounded selection for one canvas.  Given the entropies H[0..L) and the mask,
 * writes accept[p] = 1 for the accepted masked positions and returns their count.
 * sum_margin = min over sorted indices i >= 1 of |sum_{j<i} H_(j) - bound| and
 * order_margin = H_(k) - H_(k-1) at the acceptance cut (k accepted, k < n), both +inf
 * when undefined; they let a comparison with a lower-precision implementation count
 * the cases a rounding difference could flip. */
int eb_oracle_select(int L, const double *H, const uint8_t *mask, double bound,
                     uint8_t *accept, double *sum_margin, double *order_margin)
{
    keyed_entropy *list = (keyed_entropy *)malloc(sizeof(keyed_entropy) * (size_t)(L > 0 ? L : 1));
    int n = 0;
    for (int p = 0; p < L; ++p) {
        accept[p] = 0;
        if (mask[p]) { list[n].H = H[p]; list[n].p = p; ++n; }
    }
    qsort(list, (size_t)n, sizeof(keyed_entropy), cmp_keyed);
    double prefix = 0.0;   /* sum of the entropies before sorted index i */
    double smargin = INFINITY;
    int k = 0;
    for (int i = 0; i < n; ++i) {
        if (i >= 1) {
            double d = fabs(prefix - bound);
            if (d < smargin) smargin = d;
        }
        if (i == 0 || prefix <= bound) {
            accept[list[i].p] = 1;
            ++k;
        }
        prefix += list[i].H;
    }
    double omargin = INFINITY;
    if (k >= 1 && k < n) omargin = list[k].H - list[k - 1].H;
    if (sum_margin) *sum_margin = smargin;
    if (order_margin) *order_margin = omargin;
    free(list);
    return k;
}

/* Reading variants (bits of `flags` in eb_oracle_step; the values match the library's
 * parameter flags, an interface convention only):
 *   STOP_MASKED_ONLY  the stop rule's mean entropy and its argmax-stability test run over
 *                     the positions still masked at the start of the step, instead of all L;
 *   FINALIZE_SAMPLED  on adaptive stop and at the step cap the positions still masked take
 *                     their sampled token Y instead of the argmax A;
 *   STOP_RAW_ENTROPY  the stop rule's mean entropy is that of the raw logits (T = 1) instead
 *                     of the shaped ones; selection keeps the shaped entropy. */
#define ORACLE_FLAG_STOP_MASKED_ONLY 2u
#define ORACLE_FLAG_FINALIZE_SAMPLED 4u
#define ORACLE_FLAG_STOP_RAW_ENTROPY 8u

/* One full EB sampler step over B canvases of L positions (logits [B, L, V]).
 *
 * State (in/out): mask [B*L] (1 = still masked), tokens [B*L] (-1 while masked),
 * prev_argmax [B*L], status [B] (0 running, 1 adaptive stop, 2 complete, 3 step cap),
 * steps_taken [B].  Canvases whose status is not 0 are left untouched.
 * Outputs per row: H, A, Y, gap (see eb_oracle_row) and selected (1 = committed now).
 * Outputs per canvas (may be NULL): committed count, mean entropy, sum_margin,
 * order_margin (see eb_oracle_select), stop_margin = |mean H - stop_entropy|.
 *
 * Order within a step: row statistics -> stop test (s >= 1) -> on stop, every masked
 * position takes its argmax; otherwise selection and commit of the sampled tokens, then
 * the complete / cap check (at the cap the rest take their argmax) -> prev_argmax = A.
 * temperature <= 0 selects the linear schedule; flags selects the reading variants above;
 * canvas_ids (NULL: b) gives each canvas's id in the Gumbel noise's Philox counter, which the
 * block driver sets to the block number. */
void eb_oracle_step(int B, int L, int64_t V, int dtype, const void *logits,
                    int step, double temperature,
                    int max_steps, double t_start, double t_end, double bound,
                    double stop_entropy, uint64_t seed, uint32_t flags, const int32_t *canvas_ids,
                    uint8_t *mask, int32_t *tokens, int32_t *prev_argmax,
                    int32_t *status, int32_t *steps_taken,
                    double *H, int32_t *A, int32_t *Y, double *gap, uint8_t *selected,
                    int32_t *committed, double *mean_entropy,
                    double *sum_margin, double *order_margin, double *stop_margin)
{
    double T = temperature > 0.0 ? temperature
                                 : eb_oracle_temperature(step, max_steps, t_start, t_end);
    size_t esize = dtype == 0 ? 4 : (dtype == 1 ? 2 : (dtype == 3 ? 1 : 8));
    int64_t rows = (int64_t)B * L;

    /* the raw-logit entropies of STOP_RAW_ENTROPY: the same row at T = 1, no sampling */
    double *Hraw = (flags & ORACLE_FLAG_STOP_RAW_ENTROPY) ? (double *)malloc((size_t)rows * sizeof(double)) : NULL;

    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        int b = (int)(r / L), p = (int)(r % L);
        selected[r] = 0;
        if (status[b] != EB_ORACLE_RUNNING) {
            H[r] = NAN; A[r] = -1; Y[r] = -1; gap[r] = INFINITY;
            continue;
        }
        const char *row = (const char *)logits + (size_t)r * (size_t)V * esize;
        eb_oracle_row(row, dtype, V, T, mask[r], seed, canvas_ids ? canvas_ids[b] : b, p, step,
                      &H[r], &A[r], &Y[r], &gap[r]);
        if (Hraw) {
            int32_t a2, y2;
            double g2;
            eb_oracle_row(row, dtype, V, 1.0, 0, seed, b, p, step, &Hraw[r], &a2, &y2, &g2);
        }
    }

    for (int b = 0; b < B; ++b) {
        if (committed) committed[b] = 0;
        if (mean_entropy) mean_entropy[b] = NAN;
        if (sum_margin) sum_margin[b] = INFINITY;
        if (order_margin) order_margin[b] = INFINITY;
        if (stop_margin) stop_margin[b] = INFINITY;
        if (status[b] != EB_ORACLE_RUNNING) continue;
        int64_t base = (int64_t)b * L;
        const int masked_only = (flags & ORACLE_FLAG_STOP_MASKED_ONLY) != 0;
        const int fin_sampled = (flags & ORACLE_FLAG_FINALIZE_SAMPLED) != 0;
        double sumH = 0.0;
        int nstat = 0;
        int stable = 1;
        for (int p = 0; p < L; ++p) {
            if (masked_only && !mask[base + p]) continue;
            sumH += Hraw ? Hraw[base + p] : H[base + p];
            ++nstat;
            if (A[base + p] != prev_argmax[base + p]) stable = 0;
        }
        double meanH = nstat > 0 ? sumH / (double)nstat : NAN;
        if (mean_entropy) mean_entropy[b] = meanH;
        if (stop_margin && step >= 1 && stable && nstat > 0) stop_margin[b] = fabs(meanH - stop_entropy);
        int count = 0;
        if (step >= 1 && stable && nstat > 0 && meanH < stop_entropy) {
            for (int p = 0; p < L; ++p) {
                if (mask[base + p]) {
                    tokens[base + p] = fin_sampled ? Y[base + p] : A[base + p];
                    mask[base + p] = 0;
                    selected[base + p] = 1;
                    ++count;
                }
            }
            status[b] = EB_ORACLE_ADAPTIVE;
            steps_taken[b] = step + 1;
        } else {
            uint8_t *accept = (uint8_t *)malloc((size_t)L);
            eb_oracle_select(L, &H[base], &mask[base], bound, accept,
                             sum_margin ? &sum_margin[b] : NULL,
                             order_margin ? &order_margin[b] : NULL);
            int remaining = 0;
            for (int p = 0; p < L; ++p) {
                if (accept[p]) {
                    tokens[base + p] = Y[base + p];
                    mask[base + p] = 0;
                    selected[base + p] = 1;
                    ++count;
                }
                if (mask[base + p]) ++remaining;
            }
            free(accept);
            if (remaining == 0) {
                status[b] = EB_ORACLE_COMPLETE;
                steps_taken[b] = step + 1;
            } else if (step >= max_steps - 1) {
                for (int p = 0; p < L; ++p) {
                    if (mask[base + p]) {
                        tokens[base + p] = fin_sampled ? Y[base + p] : A[base + p];
                        mask[base + p] = 0;
                        selected[base + p] = 1;
                        ++count;
                    }
                }
                status[b] = EB_ORACLE_CAP;
                steps_taken[b] = step + 1;
            }
        }
        for (int p = 0; p < L; ++p) prev_argmax[base + p] = A[base + p];
        if (committed) committed[b] = count;
    }
    free(Hraw);
}

/* Number of OpenMP threads the oracle's row loop uses. */
int eb_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void eb_oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
