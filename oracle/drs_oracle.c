/*
 * drs_oracle.c -- TEST INFRASTRUCTURE, not part of the product path.
 *
 * A plain, slow, single-threaded CPU restatement of what the DiffusionGemma
 * per-row sampler statistics compute, used only to check the CUDA library.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this code. It shares nothing with the CUDA sources: no header, no
 * helper, no table.
 *
 * Sources (page "vllm.model_executor.models.diffusion_gemma_sampler"):
 *   - module docstring: per canvas position, the argmax of the temperature-
 *     scaled logits, a Gumbel-max sample, the softmax entropy and the softmax
 *     in the model dtype;
 *   - sample_row_stats docstring: row i uses temps[i // canvas_len]; a zero
 *     temperature is greedy, and the entropy clamps T at 1e-10;
 *   - sample_row_stats_reference, read for its definitions (not transcribed):
 *     the scaled logit is the logit over the temperature clamped at 1e-10;
 *     the noise is a Gumbel variate -log(-log u) of a uniform u clamped
 *     below at 1e-20, added only where T > 0; the sample is the Gumbel-max
 *     argmax of scaled + noise; the entropy is that of the softmax of the
 *     scaled row, masked columns contributing nothing; the probabilities are
 *     the softmax in the model dtype; ties go to the lowest column;
 *   - stash_converged_logprobs docstring and _lp_topk_kernel docstring: the
 *     num_topk largest scaled logits of kept rows, ordered by value and then
 *     by lower index, and their logprobs; the stash layout (request rows
 *     src * canvas_len + p for p < valid, stash row (slots, p), the argmax,
 *     then token_ids or the num_topk largest, padding with id 0 at -inf).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - the noise: the reference draws it with an unseeded rand_like; the
 *     kernel takes a seed. Here u comes from Philox4x32-10 (Salmon, Moraes,
 *     Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11) with
 *     key (lo32(seed), hi32(seed)) and counter
 *     (lo32(col/4), hi32(col/4), lo32(row), hi32(row)), word col%4, mapped to
 *     u = (word >> 8) * 2^-24 and clamped below at 1e-20f;
 *   - ties: lowest index for argmax, sample and top-k;
 *   - -0.0 and +0.0 are the same value for the top-k order;
 *   - the top-k logprob clamps T at 1e-10 like the row statistics;
 *   - a row that is -inf everywhere: argmax = sample = 0, entropy = 0,
 *     probs = NaN, top-k logprobs = NaN (what the PyTorch definition gives);
 *   - the stash: temps[j] is clamped at 1e-10; a token id outside the
 *     vocabulary gets NaN; logits mode writes the scaled logit instead of
 *     the logprob; out_ranks holds, per stash row, 1 + the number of
 *     columns whose scaled logit exceeds column 0's (the pages do not say
 *     what the rank counts: parity unpinned beyond this reading).
 *
 * Floating point: the scaled logit is one IEEE fp32 division; everything
 * after it is in double. Build with -ffp-contract=off and without fast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- Philox */

/* Philox4x32 round constants from the SC'11 paper: the two multipliers and
 * the two Weyl-sequence key increments. */
#define ORACLE_PHILOX_M0 0xD2511F53u
#define ORACLE_PHILOX_M1 0xCD9E8D57u
#define ORACLE_PHILOX_W0 0x9E3779B9u
#define ORACLE_PHILOX_W1 0xBB67AE85u

/* Ten rounds of the Philox4x32 bijection. Each round multiplies words 0 and
 * 2 by the two constants, takes the high halves xor the other two words xor
 * the round key as the new words 0 and 2, and the low halves as the new
 * words 1 and 3 (crossed). The key advances by the Weyl increments between
 * rounds. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                          uint32_t out[4]) {
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t prod_a = (uint64_t)ORACLE_PHILOX_M0 * (uint64_t)x0;
        uint64_t prod_b = (uint64_t)ORACLE_PHILOX_M1 * (uint64_t)x2;
        uint32_t hi_a = (uint32_t)(prod_a >> 32), lo_a = (uint32_t)prod_a;
        uint32_t hi_b = (uint32_t)(prod_b >> 32), lo_b = (uint32_t)prod_b;
        uint32_t y0 = hi_b ^ x1 ^ k0;
        uint32_t y1 = lo_b;
        uint32_t y2 = hi_a ^ x3 ^ k1;
        uint32_t y3 = lo_a;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += ORACLE_PHILOX_W0;
        k1 += ORACLE_PHILOX_W1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* The 32 random bits that drive the noise of (row, col). */
uint32_t oracle_noise_bits(uint64_t seed, int64_t row, int64_t col) {
    uint64_t group = (uint64_t)col >> 2;
    uint32_t ctr[4] = {(uint32_t)group, (uint32_t)(group >> 32),
                       (uint32_t)(uint64_t)row, (uint32_t)((uint64_t)row >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return out[(uint64_t)col & 3u];
}

/* u in [0, 1 - 2^-24] on a 2^-24 grid, then clamp(min=1e-20) in fp32. */
float oracle_uniform(uint32_t bits) {
    float u = (float)(bits >> 8) * 0x1p-24f; /* exact: 24-bit integer */
    const float lo = 1e-20f;
    return u < lo ? lo : u;
}

/* The Gumbel noise -log(-log u), in double. */
double oracle_gumbel_of_bits(uint32_t bits) {
    double u = (double)oracle_uniform(bits);
    return -log(-log(u));
}

/* Fill bits[r, c] and gumbel[r, c] (either may be NULL) for rows
 * row0 .. row0 + rows - 1 and columns 0 .. vocab - 1, row-major. */
void oracle_philox_gumbel(uint64_t seed, int64_t row0, int64_t rows,
                          int64_t vocab, uint32_t *bits, double *gumbel) {
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < vocab; ++c) {
            uint32_t b = oracle_noise_bits(seed, row0 + r, c);
            if (bits) bits[r * vocab + c] = b;
            if (gumbel) gumbel[r * vocab + c] = oracle_gumbel_of_bits(b);
        }
    }
}

/* ------------------------------------------------- narrowing conversions */

/* fp32 -> bfloat16 bits, round to nearest even (the top 16 bits of the
 * fp32 encoding after adding half an ulp of bf16 plus the tie bit). */
uint16_t oracle_f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
    uint32_t tie = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + tie) >> 16);
}

/* fp32 -> IEEE binary16 bits, round to nearest even, through the compiler's
 * _Float16 conversion. */
uint16_t oracle_f32_to_f16_bits(float f) {
    _Float16 h = (_Float16)f;
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

/* ------------------------------------------------------------ row stats */

enum { ORACLE_PROBS_NONE = 0, ORACLE_PROBS_BF16 = 1, ORACLE_PROBS_FP16 = 2 };

/* The clamp(min=1e-10) of the temperature, in fp32 like the tensor it
 * applies to. */
static float oracle_clamped_temp(float t) {
    const float lo = 1e-10f;
    return t > lo ? t : lo;
}

/*
 * Row statistics of one row: x[0 .. vocab-1] is row `row` (its global index,
 * which keys the noise) and `temp` its slot's temperature. Outputs:
 *   *argmax, *sample      lowest index of the max of scaled / noisy;
 *   *entropy              log S - W / S (S, W over the finite columns);
 *   *entropy_check        -sum_{p>0} p log p, the PyTorch form;
 *   probs                 vocab 16-bit codes (probs_dtype NONE: not touched);
 *   *sample_gap           best minus second-best noisy score, or +inf when
 *                         the sample is not drawn by noise;
 *   *sample_best          the best noisy score, or the max scaled logit
 *                         when no noise is drawn.
 * `scaled` is caller scratch of vocab floats.
 */
static void oracle_one_row(const float *x, int64_t vocab, int64_t row, float temp,
                           uint64_t seed, float *scaled, int64_t *argmax,
                           int64_t *sample, double *entropy, double *entropy_check,
                           int probs_dtype, uint16_t *probs, double *sample_gap,
                           double *sample_best) {
    float te = oracle_clamped_temp(temp);

    /* scaled = logits / clamp(temp, 1e-10): one fp32 division each. */
    for (int64_t j = 0; j < vocab; ++j) scaled[j] = x[j] / te;

    /* argmax of scaled: first index attaining the maximum. */
    int64_t arg = 0;
    float mx = scaled[0];
    for (int64_t j = 1; j < vocab; ++j) {
        if (scaled[j] > mx) { mx = scaled[j]; arg = j; }
    }
    *argmax = arg;

    /* softmax statistics in double. */
    double m = (double)mx;
    double h = 0.0, h_check = 0.0;
    double s_sum = 0.0;
    if (m != -INFINITY) {
        double w_sum = 0.0;
        for (int64_t j = 0; j < vocab; ++j) {
            if (scaled[j] == -INFINITY) continue; /* 0 * -inf dropped */
            double d = (double)scaled[j] - m;
            double e = exp(d);
            s_sum += e;
            w_sum += e * d;
        }
        double log_s = log(s_sum);
        h = log_s - w_sum / s_sum;
        for (int64_t j = 0; j < vocab; ++j) {
            double d = (double)scaled[j] - m;
            double p = exp(d) / s_sum;
            if (p > 0.0) h_check -= p * (d - log_s);
        }
    } /* else: log_softmax is NaN everywhere; where(p > 0) drops it all. */
    *entropy = h;
    *entropy_check = h_check;

    /* probs = exp(log_softmax) -> fp32 -> model dtype. */
    if (probs_dtype != ORACLE_PROBS_NONE && probs) {
        for (int64_t j = 0; j < vocab; ++j) {
            float pf = (m == -INFINITY) ? NAN : (float)(exp((double)scaled[j] - m) / s_sum);
            probs[j] = probs_dtype == ORACLE_PROBS_BF16 ? oracle_f32_to_bf16_bits(pf)
                                                         : oracle_f32_to_f16_bits(pf);
        }
    }

    /* Gumbel-max sample: noise only where temp > 0. */
    if (temp > 0.0f) {
        double best = -INFINITY, second = -INFINITY;
        int64_t best_j = 0;
        int have = 0;
        for (int64_t j = 0; j < vocab; ++j) {
            double score = (double)scaled[j] +
                           oracle_gumbel_of_bits(oracle_noise_bits(seed, row, j));
            if (!have || score > best) {
                if (have) second = best > second ? best : second;
                best = score;
                best_j = j;
                have = 1;
            } else if (score > second) {
                second = score;
            }
        }
        *sample = best_j;
        *sample_gap = (best == -INFINITY) ? INFINITY : best - second;
        *sample_best = best;
    } else {
        *sample = arg;
        *sample_gap = INFINITY;
        *sample_best = m;
    }
}

/*
 * Row statistics for rows [row_begin, row_end) of a [rows, row_stride] fp32
 * buffer whose first `vocab` columns are the logits; row i uses
 * temps[i / canvas_len]. Outputs are indexed by the row (probs: row i at
 * probs + i * probs_row_stride); only that range is written. NULL is
 * allowed for entropy_check, sample_gap, sample_best and (with probs_dtype
 * NONE) probs. Returns 0, or -1 if scratch memory could not be allocated.
 */
int oracle_row_stats(const float *logits, int64_t rows, int64_t vocab,
                     int64_t row_stride, const float *temps, int64_t canvas_len,
                     uint64_t seed, int64_t row_begin, int64_t row_end,
                     int64_t *argmax, int64_t *sample, double *entropy,
                     double *entropy_check, int probs_dtype, uint16_t *probs,
                     int64_t probs_row_stride, double *sample_gap,
                     double *sample_best) {
    (void)rows;
    float *scaled = (float *)malloc((size_t)vocab * sizeof(float));
    if (!scaled) return -1;
    for (int64_t i = row_begin; i < row_end; ++i) {
        double hc, gap, best;
        oracle_one_row(logits + i * row_stride, vocab, i, temps[i / canvas_len], seed, scaled,
                       &argmax[i], &sample[i], &entropy[i], &hc, probs_dtype,
                       probs ? probs + i * probs_row_stride : NULL, &gap, &best);
        if (entropy_check) entropy_check[i] = hc;
        if (sample_gap) sample_gap[i] = gap;
        if (sample_best) sample_best[i] = best;
    }
    free(scaled);
    return 0;
}

/*
 * The same statistics for n rows given one by one: rows[t] points at
 * `vocab` logits of global row row_ids[t], whose temperature is temps[t].
 * Output t of each array (probs: probs + t * vocab) receives row t.
 */
int oracle_row_stats_rows(const float *const *row_ptrs, const int64_t *row_ids,
                          const float *temps, int64_t n, int64_t vocab, uint64_t seed,
                          int64_t *argmax, int64_t *sample, double *entropy,
                          double *entropy_check, int probs_dtype, uint16_t *probs,
                          double *sample_gap, double *sample_best) {
    float *scaled = (float *)malloc((size_t)vocab * sizeof(float));
    if (!scaled) return -1;
    for (int64_t t = 0; t < n; ++t) {
        oracle_one_row(row_ptrs[t], vocab, row_ids[t], temps[t], seed, scaled, &argmax[t],
                       &sample[t], &entropy[t], &entropy_check[t], probs_dtype,
                       probs ? probs + t * vocab : NULL, &sample_gap[t], &sample_best[t]);
    }
    free(scaled);
    return 0;
}

/* --------------------------------------------------------------- top-k */

typedef struct {
    float value;
    int64_t index;
} oracle_ranked;

/* Descending value, then ascending index: a total order, so the first k
 * after sorting are unique. */
static int oracle_rank_cmp(const void *pa, const void *pb) {
    const oracle_ranked *a = (const oracle_ranked *)pa;
    const oracle_ranked *b = (const oracle_ranked *)pb;
    if (a->value > b->value) return -1;
    if (a->value < b->value) return 1;
    if (a->index < b->index) return -1;
    if (a->index > b->index) return 1;
    return 0;
}

/* Top-k of one row x[0 .. vocab-1] scaled by clamp(temp, 1e-10): the k
 * columns of largest scaled value (ties by lower column, -0.0 == +0.0) and
 * their logprobs scaled - max - log(sum exp(scaled - max)). */
static void oracle_topk_one(const float *x, int64_t vocab, float temp, int32_t k,
                            oracle_ranked *items, int32_t *ids, double *lps) {
    float te = oracle_clamped_temp(temp);
    float mx = -INFINITY;
    for (int64_t j = 0; j < vocab; ++j) {
        float s = x[j] / te;
        s = s + 0.0f; /* -0.0 and +0.0 are one value */
        items[j].value = s;
        items[j].index = j;
        if (s > mx) mx = s;
    }
    double m = (double)mx;
    double log_s = NAN;
    if (m != -INFINITY) {
        double s_sum = 0.0;
        for (int64_t j = 0; j < vocab; ++j)
            if (items[j].value != -INFINITY) s_sum += exp((double)items[j].value - m);
        log_s = log(s_sum);
    }
    qsort(items, (size_t)vocab, sizeof(oracle_ranked), oracle_rank_cmp);
    for (int32_t r = 0; r < k; ++r) {
        ids[r] = (int32_t)items[r].index;
        lps[r] = (m == -INFINITY) ? NAN : (double)items[r].value - m - log_s;
    }
}

/*
 * Top-k logprobs of the rows of kept slots in [row_begin, row_end): row i is
 * kept when keep[i / canvas_len] != 0 and then fills out_ids[i * k + r] and
 * out_logprobs[i * k + r], r < k. Rows of slots that are not kept are not
 * touched. Returns 0, or -1 on allocation failure.
 */
int oracle_topk_logprobs(const float *logits, int64_t rows, int64_t vocab,
                         int64_t row_stride, const float *temps,
                         int64_t canvas_len, const uint8_t *keep, int32_t k,
                         int64_t row_begin, int64_t row_end, int32_t *out_ids,
                         double *out_logprobs) {
    (void)rows;
    if (k <= 0) return 0;
    oracle_ranked *items = (oracle_ranked *)malloc((size_t)vocab * sizeof(oracle_ranked));
    if (!items) return -1;
    for (int64_t i = row_begin; i < row_end; ++i) {
        int64_t slot = i / canvas_len;
        if (!keep[slot]) continue;
        oracle_topk_one(logits + i * row_stride, vocab, temps[slot], k, items,
                        out_ids + i * k, out_logprobs + i * k);
    }
    free(items);
    return 0;
}

/* Top-k of n rows given one by one (all kept): rows[t] has temperature
 * temps[t]; out_ids / out_logprobs + t * k receive row t. */
int oracle_topk_rows(const float *const *row_ptrs, const float *temps, int64_t n,
                     int64_t vocab, int32_t k, int32_t *out_ids, double *out_logprobs) {
    if (k <= 0) return 0;
    oracle_ranked *items = (oracle_ranked *)malloc((size_t)vocab * sizeof(oracle_ranked));
    if (!items) return -1;
    for (int64_t t = 0; t < n; ++t)
        oracle_topk_one(row_ptrs[t], vocab, temps[t], k, items, out_ids + t * k,
                        out_logprobs + t * k);
    free(items);
    return 0;
}

/*
 * The stash written by stash_converged_logprobs (page
 * "vllm.model_executor.models.diffusion_gemma_sampler", its docstring).
 * Request j < m owns logits rows src[j] * canvas_len + p for p < valid[j]
 * (at most canvas_len), scaled by clamp(temps[j], 1e-10). Where keep[j],
 * stash row (slots[j], p) -- row slots[j] * canvas_len + p of the outputs --
 * receives `width` columns of (id, value):
 *   column 0              the argmax (lowest column of the max);
 *   the next columns      token_ids[j * ids_stride + c] for c < n_j when
 *                         token_ids is given and n_j = min(num_token_ids[j],
 *                         ids_stride) > 0 (a request's list has ids_stride
 *                         entries),
 *                         else the num_topk largest (value descending, lower
 *                         column first);
 *   the rest              id 0 with value -inf.
 * value = scaled - max - log(sum exp(scaled - max)) (NaN when the row is
 * -inf everywhere, and for a token id outside [0, vocab)), or the scaled
 * logit itself when logits_mode. out_ranks[stash row] = 1 + #{k : scaled_k >
 * scaled of column 0's id}. -0.0 is taken as +0.0. Stash rows of requests
 * that are not kept, and positions p >= valid[j], are not touched; out_ids,
 * out_vals hold width entries per stash row. Returns 0, or -1 on
 * allocation failure.
 */
int oracle_stash(const float *logits, int64_t row_stride, int64_t vocab, int64_t canvas_len,
                 int64_t m, const int32_t *src, const int32_t *slots, const uint8_t *keep,
                 const int32_t *valid, const float *temps, int32_t num_topk,
                 const int32_t *num_token_ids, const int32_t *token_ids, int64_t ids_stride,
                 int32_t width, int logits_mode, int32_t *out_ids, double *out_vals,
                 int32_t *out_ranks) {
    float *scaled = (float *)malloc((size_t)vocab * sizeof(float));
    oracle_ranked *items = (oracle_ranked *)malloc((size_t)vocab * sizeof(oracle_ranked));
    if (!scaled || !items) {
        free(scaled);
        free(items);
        return -1;
    }
    for (int64_t j = 0; j < m; ++j) {
        if (!keep[j]) continue;
        float te = oracle_clamped_temp(temps[j]);
        int64_t npos = valid[j] < canvas_len ? valid[j] : canvas_len;
        for (int64_t p = 0; p < npos; ++p) {
            const float *x = logits + ((int64_t)src[j] * canvas_len + p) * row_stride;
            int64_t out_row = (int64_t)slots[j] * canvas_len + p;
            int32_t *ids = out_ids + out_row * width;
            double *vals = out_vals + out_row * width;

            /* scaled logits, their max, log of the sum of exponentials */
            float mx = -INFINITY;
            int64_t arg = 0;
            for (int64_t c = 0; c < vocab; ++c) {
                scaled[c] = x[c] / te + 0.0f;
                if (scaled[c] > mx) {
                    mx = scaled[c];
                    arg = c;
                }
            }
            double big_m = (double)mx, log_s = NAN;
            if (mx != -INFINITY) {
                double s_sum = 0.0;
                for (int64_t c = 0; c < vocab; ++c)
                    if (scaled[c] != -INFINITY) s_sum += exp((double)scaled[c] - big_m);
                log_s = log(s_sum);
            }
#define ORACLE_VALUE(col)                                                              \
    ((col) < 0 || (col) >= vocab ? NAN                                                 \
     : logits_mode              ? (double)scaled[(col)]                               \
     : mx == -INFINITY          ? NAN                                                 \
                                : (double)scaled[(col)] - big_m - log_s)

            int32_t w = 0;
            if (w < width) {
                ids[w] = (int32_t)arg;
                vals[w] = ORACLE_VALUE(arg);
                ++w;
            }
            int64_t n_ids = token_ids && num_token_ids ? num_token_ids[j] : 0;
            if (n_ids > ids_stride) n_ids = ids_stride;
            if (n_ids > 0) {
                for (int64_t c = 0; c < n_ids && w < width; ++c, ++w) {
                    int32_t id = token_ids[j * ids_stride + c];
                    ids[w] = id;
                    vals[w] = ORACLE_VALUE(id);
                }
            } else if (num_topk > 0) {
                for (int64_t c = 0; c < vocab; ++c) {
                    items[c].value = scaled[c];
                    items[c].index = c;
                }
                qsort(items, (size_t)vocab, sizeof(oracle_ranked), oracle_rank_cmp);
                for (int32_t r = 0; r < num_topk && r < vocab && w < width; ++r, ++w) {
                    ids[w] = (int32_t)items[r].index;
                    vals[w] = ORACLE_VALUE(items[r].index);
                }
            }
            for (; w < width; ++w) {
                ids[w] = 0;
                vals[w] = -INFINITY;
            }
#undef ORACLE_VALUE
            int32_t above = 0;
            for (int64_t c = 0; c < vocab; ++c) above += scaled[c] > scaled[arg];
            out_ranks[out_row] = 1 + above;
        }
    }
    free(scaled);
    free(items);
    return 0;
}
