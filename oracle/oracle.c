/*
 * Oracle for the EntropyCache per-step hot path: a plain, slow, float64 CPU
 * implementation written from the method's definitions.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library.  It shares no code, header
 * or table with the CUDA library, and the CUDA library never calls it.
 *
 * Sources (cited by page title and section):
 *   [EC-it]  "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion
 *            Language Models", Italian summary (gist.science/it/paper/2603.18489),
 *            section "2. Metodologia", subsection "Algoritmo di Funzionamento".
 *   [EC-ar]  the same paper, Arabic technical summary
 *            (gist.science/ar/paper/2603.18489), section "2. Methodology",
 *            subsection "Algorithm workflow" and its equation for E_{t+1}.
 *
 * Readings taken where the pages are silent (all listed in the design notes):
 *   - "log" in the entropy is the natural logarithm (nats);
 *   - decoding a row is greedy: token = argmax of the logits (lowest index on a
 *     tie), confidence = the softmax probability of that token;
 *   - unmasking takes, per sequence, the n rows of highest confidence (ties:
 *     lower position first);
 *   - the gate is the strict comparison E > tau, E the maximum entropy over the
 *     rows unmasked this step (E = -inf when none is);
 *   - "currently masked" means the masked positions of the active block, and the
 *     k most recently decoded positions are those with the largest decode step
 *     (ties: lower position first);
 *   - attention is bidirectional softmax(q K^T * scale) V over all L keys of the
 *     cache after the fresh K/V rows were written into it.
 *
 * Parallelism: the loops over independent items (logits rows, attention outputs,
 * projection rows) may run on several host threads (OpenMP, orc_set_threads);
 * each item is still computed by one thread with the loop body below, so the
 * result of every item is the same whatever the thread count.
 *
 * Element types: 0 = float32, 1 = bfloat16 (raw uint16 bits), 2 = float64.
 * Every value is widened exactly to double before any arithmetic.
 * Return codes: 0 = ok, -2 = bad shape/argument, -3 = bad dtype, -9 = out of memory.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_BAD_ARG (-2)
#define ORC_BAD_DTYPE (-3)
#define ORC_NOMEM (-9)

/* Host threads the item loops use (1 unless set). */
static int g_threads = 1;

void orc_set_threads(int n) { g_threads = n > 0 ? n : 1; }

int orc_get_threads(void)
{
#ifdef _OPENMP
    return g_threads;
#else
    return 1;
#endif
}

static int dtype_ok(int dtype) { return dtype == 0 || dtype == 1 || dtype == 2; }

static size_t dtype_size(int dtype) { return dtype == 0 ? 4 : (dtype == 1 ? 2 : 8); }

/* Exact widening of element i of a typed array to double. */
static double load(const void *base, int dtype, int64_t i)
{
    if (dtype == 0)
        return (double)((const float *)base)[i];
    if (dtype == 1) {
        uint32_t bits = ((uint32_t)((const uint16_t *)base)[i]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return ((const double *)base)[i];
}

/*
 * Per-row decode statistics.  [EC-it] step 1 ("decode new tokens and compute
 * the entropy of their distributions"); [EC-ar] phase 2, the inner sum of the
 * E_{t+1} equation: H_i = -sum_j p_ij log p_ij with p_i = softmax(x_i).
 *
 * For each of n_rows rows (row i starts at element i * row_stride):
 *   token[i]   = smallest j with x_ij = max_j x_ij
 *   conf[i]    = p_{i, token[i]}
 *   entropy[i] = -sum_j p_ij ln p_ij   (terms with p_ij = 0 contribute 0)
 */
static void row_stats_one(const void *logits, int dtype, int64_t row_stride, int32_t vocab,
                          int32_t i, double *x, double *p, double *entropy, double *conf,
                          int32_t *token)
{
    const int64_t base = (int64_t)i * row_stride;
    for (int32_t j = 0; j < vocab; ++j)
        x[j] = load(logits, dtype, base + j);

    /* greedy decode: the first index holding the maximum */
    double m = x[0];
    int32_t a = 0;
    for (int32_t j = 1; j < vocab; ++j)
        if (x[j] > m) {
            m = x[j];
            a = j;
        }

    /* softmax, shifted by the maximum for range */
    double z = 0.0;
    for (int32_t j = 0; j < vocab; ++j) {
        p[j] = exp(x[j] - m);
        z += p[j];
    }
    for (int32_t j = 0; j < vocab; ++j)
        p[j] /= z;

    /* Shannon entropy in nats */
    double h = 0.0;
    for (int32_t j = 0; j < vocab; ++j)
        if (p[j] > 0.0)
            h -= p[j] * log(p[j]);

    entropy[i] = h;
    conf[i] = p[a];
    token[i] = a;
}

int orc_row_stats(const void *logits, int dtype, int64_t row_stride, int32_t n_rows,
                  int32_t vocab, double *entropy, double *conf, int32_t *token)
{
    if (!dtype_ok(dtype))
        return ORC_BAD_DTYPE;
    if (n_rows < 0 || vocab <= 0 || row_stride < vocab)
        return ORC_BAD_ARG;
    int status = ORC_OK;
#pragma omp parallel num_threads(g_threads)
    {
        double *x = (double *)malloc((size_t)vocab * sizeof(double));
        double *p = (double *)malloc((size_t)vocab * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int32_t i = 0; i < n_rows; ++i) {
            if (!x || !p) {
#pragma omp atomic write
                status = ORC_NOMEM;
                continue;
            }
            row_stats_one(logits, dtype, row_stride, vocab, i, x, p, entropy, conf, token);
        }
        free(x);
        free(p);
    }
    return status;
}

/* ---- confidence-ranked unmasking, max entropy, gate, state update ---- */

typedef struct {
    double conf;
    int32_t pos;
    int32_t row;
} ranked_row;

/* higher confidence first; on equal confidence the lower position first */
static int by_conf_then_pos(const void *pa, const void *pb)
{
    const ranked_row *a = (const ranked_row *)pa, *b = (const ranked_row *)pb;
    if (a->conf > b->conf)
        return -1;
    if (a->conf < b->conf)
        return 1;
    if (a->pos < b->pos)
        return -1;
    if (a->pos > b->pos)
        return 1;
    return (a->row > b->row) - (a->row < b->row);
}

/*
 * One decode step for every sequence b.  [EC-it] steps 1-2; [EC-ar] phases 2-3.
 *
 *   rows of sequence b: [seq_row_offsets[b], seq_row_offsets[b+1]), row r at
 *   position row_pos[r] of that sequence.
 *   unmask:   the min(n_unmask, #rows) rows ranked first by (conf desc, pos asc),
 *             written in rank order to unmask_rows[b*n_unmask ...], rest -1.
 *   E_b:      max of entropy[r] over the unmasked rows ([EC-ar] E_{t+1}), -inf if none.
 *   refresh:  E_b > tau, compared in double against the float32 threshold
 *             ([EC-it] step 2: E > tau -> full forward; E <= tau -> partial).
 *   state:    for each unmasked row: is_masked[b,pos] = 0, tokens[b,pos] = token[r],
 *             decode_step[b,pos] = step (the decode-time log of [EC-ar] phase 3).
 */
int orc_unmask_gate(const double *conf, const double *entropy, const int32_t *token,
                    const int32_t *seq_row_offsets, const int32_t *row_pos, int32_t batch,
                    int32_t seq_len, int32_t n_unmask, float tau, int32_t step,
                    int32_t *unmask_rows, double *max_entropy, uint8_t *refresh,
                    uint8_t *is_masked, int32_t *tokens, int32_t *decode_step)
{
    if (batch < 0 || seq_len <= 0 || n_unmask <= 0)
        return ORC_BAD_ARG;
    for (int32_t b = 0; b < batch; ++b) {
        const int32_t r0 = seq_row_offsets[b], r1 = seq_row_offsets[b + 1];
        if (r1 < r0)
            return ORC_BAD_ARG;
        const int32_t cnt = r1 - r0;
        ranked_row *rows = (ranked_row *)malloc((size_t)(cnt > 0 ? cnt : 1) * sizeof(ranked_row));
        if (!rows)
            return ORC_NOMEM;
        for (int32_t i = 0; i < cnt; ++i) {
            rows[i].conf = conf[r0 + i];
            rows[i].pos = row_pos[r0 + i];
            rows[i].row = r0 + i;
            if (rows[i].pos < 0 || rows[i].pos >= seq_len) {
                free(rows);
                return ORC_BAD_ARG;
            }
        }
        qsort(rows, (size_t)cnt, sizeof(ranked_row), by_conf_then_pos);
        const int32_t take = cnt < n_unmask ? cnt : n_unmask;
        double e = -INFINITY;
        for (int32_t s = 0; s < n_unmask; ++s)
            unmask_rows[(int64_t)b * n_unmask + s] = s < take ? rows[s].row : -1;
        for (int32_t s = 0; s < take; ++s) {
            const int32_t r = rows[s].row;
            const int64_t at = (int64_t)b * seq_len + rows[s].pos;
            if (entropy[r] > e)
                e = entropy[r];
            is_masked[at] = 0;
            tokens[at] = token[r];
            decode_step[at] = step;
        }
        max_entropy[b] = e;
        refresh[b] = (uint8_t)(e > (double)tau);
        free(rows);
    }
    return ORC_OK;
}

/* ---- recompute index set ---- */

typedef struct {
    int32_t step;
    int32_t pos;
} decoded_pos;

/* latest decode step first; on equal step the lower position first */
static int by_recency(const void *pa, const void *pb)
{
    const decoded_pos *a = (const decoded_pos *)pa, *b = (const decoded_pos *)pb;
    if (a->step > b->step)
        return -1;
    if (a->step < b->step)
        return 1;
    return (a->pos > b->pos) - (a->pos < b->pos);
}

/*
 * Positions whose K/V the next forward recomputes.  [EC-it] step 2, second
 * bullet list; [EC-ar] phase 1 and phase 3 ("token selection").
 *
 *   refresh[b] set:  every position 0..L-1 (full forward).
 *   otherwise:       M_b = masked positions in the active block [block_lo, block_hi)
 *                    R_b = the min(k, #decoded) decoded, unmasked positions with
 *                          the largest decode_step (ties: lower position first)
 *                    idx[b, 0..count[b]) = M_b u R_b in ascending order.
 *   Entries idx[b, count[b]..L) are set to -1.
 */
int orc_recompute_set(const uint8_t *is_masked, const int32_t *decode_step,
                      const uint8_t *refresh, int32_t batch, int32_t seq_len, int32_t block_lo,
                      int32_t block_hi, int32_t k, int32_t *idx, int32_t *count)
{
    if (batch < 0 || seq_len <= 0 || k < 0 || block_lo < 0 || block_hi < block_lo ||
        block_hi > seq_len)
        return ORC_BAD_ARG;
    uint8_t *take = (uint8_t *)malloc((size_t)seq_len);
    decoded_pos *dec = (decoded_pos *)malloc((size_t)seq_len * sizeof(decoded_pos));
    if (!take || !dec) {
        free(take);
        free(dec);
        return ORC_NOMEM;
    }
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t row = (int64_t)b * seq_len;
        if (refresh[b]) {
            for (int32_t p = 0; p < seq_len; ++p)
                take[p] = 1;
        } else {
            memset(take, 0, (size_t)seq_len);
            for (int32_t p = block_lo; p < block_hi; ++p)
                if (is_masked[row + p])
                    take[p] = 1;
            int32_t nd = 0;
            for (int32_t p = 0; p < seq_len; ++p)
                if (decode_step[row + p] >= 0 && !is_masked[row + p]) {
                    dec[nd].step = decode_step[row + p];
                    dec[nd].pos = p;
                    ++nd;
                }
            qsort(dec, (size_t)nd, sizeof(decoded_pos), by_recency);
            const int32_t keep = nd < k ? nd : k;
            for (int32_t s = 0; s < keep; ++s)
                take[dec[s].pos] = 1;
        }
        int32_t c = 0;
        for (int32_t p = 0; p < seq_len; ++p)
            if (take[p])
                idx[row + c++] = p;
        for (int32_t s = c; s < seq_len; ++s)
            idx[row + s] = -1;
        count[b] = c;
    }
    free(take);
    free(dec);
    return ORC_OK;
}

/*
 * KV write-back of the recomputed rows: for r < count[b],
 *   cache[b, idx[b*idx_stride + r], :, :] = fresh[b, r, :, :]
 * ([EC-it] step 2: the partial forward recomputes K/V of the selected tokens and
 * reuses the cache for the rest; [EC-ar] phase 1).  Layouts: fresh
 * [batch, r_max, Hkv, d], cache [batch, L, Hkv, d]; a bitwise copy.
 */
int orc_scatter_kv(const void *k_new, const void *v_new, int dtype, const int32_t *idx,
                   int64_t idx_stride, const int32_t *count, void *k_cache, void *v_cache,
                   int32_t batch, int32_t seq_len, int32_t r_max, int32_t n_kv_heads,
                   int32_t head_dim)
{
    if (!dtype_ok(dtype))
        return ORC_BAD_DTYPE;
    const size_t row_bytes = (size_t)n_kv_heads * (size_t)head_dim * dtype_size(dtype);
    for (int32_t b = 0; b < batch; ++b) {
        if (count[b] < 0 || count[b] > r_max)
            return ORC_BAD_ARG;
        for (int32_t r = 0; r < count[b]; ++r) {
            const int32_t p = idx[(int64_t)b * idx_stride + r];
            if (p < 0 || p >= seq_len)
                return ORC_BAD_ARG;
            const size_t src = ((size_t)b * r_max + r) * row_bytes;
            const size_t dst = ((size_t)b * seq_len + p) * row_bytes;
            memcpy((char *)k_cache + dst, (const char *)k_new + src, row_bytes);
            memcpy((char *)v_cache + dst, (const char *)v_new + src, row_bytes);
        }
    }
    return ORC_OK;
}

/*
 * Bidirectional attention of the recomputed query rows over every cached key
 * ([EC-it] section 1: dLLM attention is non-causal, every position attends to all
 * others; [EC-it] step 2 and [EC-ar] phase 1: only the selected rows are
 * recomputed, all other K/V come from the cache).
 *
 * For a query row (b, r, h), r < count[b], with kv head g = h / (H / Hkv):
 *   s_j = scale * sum_e q[b,r,h,e] * K[b,j,g,e]        for every key j < L
 *   w_j = exp(s_j - max_j s_j)
 *   o_e = sum_j w_j V[b,j,g,e] / sum_j w_j
 *
 * samples == NULL: every valid row is written to out[b, r, h, :] (rows
 * r >= count[b] are left untouched).  Otherwise samples holds n_samples triples
 * (b, r, h) and out[s, :] receives the output of triple s.
 */
/* One output row (b, r, h) of the attention below, written to o[0 .. head_dim). */
static void attention_one(const void *q, const void *k_cache, const void *v_cache, int dtype,
                          int32_t seq_len, int32_t r_max, int32_t n_heads, int32_t n_kv_heads,
                          int32_t head_dim, double scale, int32_t b, int32_t r, int32_t h,
                          double *s, double *o)
{
    const int32_t group = n_heads / n_kv_heads;
    const int32_t g = h / group;
    const int64_t qoff = (((int64_t)b * r_max + r) * n_heads + h) * head_dim;

    double m = -INFINITY;
    for (int32_t j = 0; j < seq_len; ++j) {
        const int64_t koff = (((int64_t)b * seq_len + j) * n_kv_heads + g) * head_dim;
        double dot = 0.0;
        for (int32_t e = 0; e < head_dim; ++e)
            dot += load(q, dtype, qoff + e) * load(k_cache, dtype, koff + e);
        s[j] = scale * dot;
        if (s[j] > m)
            m = s[j];
    }
    double z = 0.0;
    for (int32_t j = 0; j < seq_len; ++j) {
        s[j] = exp(s[j] - m);
        z += s[j];
    }
    for (int32_t e = 0; e < head_dim; ++e)
        o[e] = 0.0;
    for (int32_t j = 0; j < seq_len; ++j) {
        const int64_t voff = (((int64_t)b * seq_len + j) * n_kv_heads + g) * head_dim;
        const double w = s[j] / z;
        for (int32_t e = 0; e < head_dim; ++e)
            o[e] += w * load(v_cache, dtype, voff + e);
    }
}

int orc_attention(const void *q, const void *k_cache, const void *v_cache, int dtype,
                  const int32_t *count, int32_t batch, int32_t seq_len, int32_t r_max,
                  int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, double scale,
                  const int32_t *samples, int64_t n_samples, double *out)
{
    if (!dtype_ok(dtype))
        return ORC_BAD_DTYPE;
    if (batch < 0 || seq_len <= 0 || r_max < 0 || n_heads <= 0 || n_kv_heads <= 0 ||
        head_dim <= 0 || n_heads % n_kv_heads != 0)
        return ORC_BAD_ARG;
    if (samples)
        for (int64_t t = 0; t < n_samples; ++t) {
            const int32_t b = samples[3 * t], r = samples[3 * t + 1], h = samples[3 * t + 2];
            if (b < 0 || b >= batch || r < 0 || r >= r_max || h < 0 || h >= n_heads)
                return ORC_BAD_ARG;
        }
    const int64_t total = samples ? n_samples : (int64_t)batch * r_max * n_heads;
    int status = ORC_OK;
#pragma omp parallel num_threads(g_threads)
    {
        double *s = (double *)malloc((size_t)seq_len * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < total; ++t) {
            int32_t b, r, h;
            if (samples) {
                b = samples[3 * t];
                r = samples[3 * t + 1];
                h = samples[3 * t + 2];
            } else {
                b = (int32_t)(t / ((int64_t)r_max * n_heads));
                r = (int32_t)((t / n_heads) % r_max);
                h = (int32_t)(t % n_heads);
                if (r >= count[b])
                    continue;
            }
            if (!s) {
#pragma omp atomic write
                status = ORC_NOMEM;
                continue;
            }
            attention_one(q, k_cache, v_cache, dtype, seq_len, r_max, n_heads, n_kv_heads,
                          head_dim, scale, b, r, h, s, out + t * head_dim);
        }
        free(s);
    }
    return status;
}

/*
 * Input rows of the first layer for the recomputed positions ([EC-it] step 2:
 * only the selected tokens go through the partial forward; [EC-it] section 1:
 * a position holds [MASK] until its token is decoded).  For b, r < count[b],
 * p = idx[b*idx_stride + r]:
 *   x[b, r, :] = table[is_masked[b, p] ? mask_id : tokens[b, p], :]
 * A bitwise row copy; x rows r >= count[b] are left untouched.
 */
int orc_embed_rows(const void *table, int dtype, int64_t table_rows, int32_t hidden,
                   const int32_t *idx, int64_t idx_stride, const int32_t *count,
                   const int32_t *tokens, const uint8_t *is_masked, int32_t mask_id,
                   int32_t batch, int32_t seq_len, int32_t r_max, void *x)
{
    if (!dtype_ok(dtype))
        return ORC_BAD_DTYPE;
    if (batch < 0 || seq_len <= 0 || r_max < 0 || hidden <= 0 || table_rows <= 0)
        return ORC_BAD_ARG;
    const size_t row_bytes = (size_t)hidden * dtype_size(dtype);
    for (int32_t b = 0; b < batch; ++b) {
        if (count[b] < 0 || count[b] > r_max)
            return ORC_BAD_ARG;
        for (int32_t r = 0; r < count[b]; ++r) {
            const int32_t p = idx[(int64_t)b * idx_stride + r];
            if (p < 0 || p >= seq_len)
                return ORC_BAD_ARG;
            const int64_t at = (int64_t)b * seq_len + p;
            const int64_t tok = is_masked[at] ? mask_id : tokens[at];
            if (tok < 0 || tok >= table_rows)
                return ORC_BAD_ARG;
            memcpy((char *)x + ((size_t)b * r_max + r) * row_bytes,
                   (const char *)table + (size_t)tok * row_bytes, row_bytes);
        }
    }
    return ORC_OK;
}

/*
 * Query, key and value projection of the recomputed rows ([EC-it] step 2: the
 * partial forward recomputes Q/K/V of the selected tokens only), in float64:
 *   y[row, j] = sum_e x[row, e] * w[j, e]       for j < n_out
 * x [n_rows, hidden] and w [n_out, hidden] (typed), y double [n_rows, n_out].
 * With rows != NULL only the n_sel listed rows of x are projected, and y is
 * [n_sel, n_out].
 */
int orc_projection(const void *x, const void *w, int dtype, int64_t n_rows, int32_t hidden,
                   int32_t n_out, const int64_t *rows, int64_t n_sel, double *y)
{
    if (!dtype_ok(dtype))
        return ORC_BAD_DTYPE;
    if (n_rows < 0 || hidden <= 0 || n_out <= 0)
        return ORC_BAD_ARG;
    const int64_t total = rows ? n_sel : n_rows;
    if (rows)
        for (int64_t s = 0; s < total; ++s)
            if (rows[s] < 0 || rows[s] >= n_rows)
                return ORC_BAD_ARG;
    int status = ORC_OK;
#pragma omp parallel num_threads(g_threads)
    {
        double *xr = (double *)malloc((size_t)hidden * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t s = 0; s < total; ++s) {
            if (!xr) {
#pragma omp atomic write
                status = ORC_NOMEM;
                continue;
            }
            const int64_t row = rows ? rows[s] : s;
            for (int32_t e = 0; e < hidden; ++e)
                xr[e] = load(x, dtype, row * hidden + e);
            for (int32_t j = 0; j < n_out; ++j) {
                double acc = 0.0;
                for (int32_t e = 0; e < hidden; ++e)
                    acc += xr[e] * load(w, dtype, (int64_t)j * hidden + e);
                y[s * n_out + j] = acc;
            }
        }
        free(xr);
    }
    return status;
}

/*
 * Attention under SimSD's token-level temporal causal mask ("SimSD - Simple
 * Speculative Decoding in Diffusion Language Models", Italian technical summary
 * (gist.science/it/paper/2606.02544), section "Metodologia: SimSD", items
 * 1 "Layout di Input" and 2 "Maschera di Attenzione Temporale").
 *
 * Each position j of a sequence lies in one section: 0 = prompt, 1 = data
 * section D (reference tokens), 2 = mask section (prediction slots); data and
 * mask positions carry a step label tau[j] >= 1 (the step map; a data position
 * and its paired mask slot share one label).  Key j is visible to the query at
 * position i when
 *   - j is in the prompt (every query), or
 *   - i is a mask slot and either j is a data position with tau[j] < tau[i]
 *     (revealed at an earlier step) or j is a mask slot with tau[j] >= tau[i]
 *     (the page's two rules), or
 *   - i is a data position and j a data position with tau[j] <= tau[i]
 *     (reading: reference tokens see the prompt and the references revealed
 *     no later than themselves, no prediction slot), or
 *   - nothing else: a prompt query sees the prompt only (reading).
 * The output is softmax over the visible keys only; a query with no visible
 * key gets a zero row (reading; the rules above never leave one empty).
 *
 * The query row r of sequence b sits at position idx[b*idx_stride + r]; the
 * caches already hold the fresh rows.  Layouts as in orc_attention; section
 * and tau are [batch, seq_len].
 */
static int simsd_visible(uint8_t sec_i, int32_t tau_i, uint8_t sec_j, int32_t tau_j)
{
    if (sec_j == 0)
        return 1;
    if (sec_i == 2)
        return sec_j == 1 ? tau_j < tau_i : tau_j >= tau_i;
    if (sec_i == 1)
        return sec_j == 1 && tau_j <= tau_i;
    return 0;
}

static void attention_simsd_one(const void *q, const void *k_cache, const void *v_cache,
                                int dtype, const uint8_t *section, const int32_t *tau,
                                int32_t pos, int32_t seq_len, int32_t r_max, int32_t n_heads,
                                int32_t n_kv_heads, int32_t head_dim, double scale, int32_t b,
                                int32_t r, int32_t h, double *s, double *o)
{
    const int32_t group = n_heads / n_kv_heads;
    const int32_t g = h / group;
    const int64_t qoff = (((int64_t)b * r_max + r) * n_heads + h) * head_dim;
    const uint8_t *sec = section + (int64_t)b * seq_len;
    const int32_t *tl = tau + (int64_t)b * seq_len;

    double m = -INFINITY;
    for (int32_t j = 0; j < seq_len; ++j) {
        s[j] = -INFINITY;
        if (!simsd_visible(sec[pos], tl[pos], sec[j], tl[j]))
            continue;
        const int64_t koff = (((int64_t)b * seq_len + j) * n_kv_heads + g) * head_dim;
        double dot = 0.0;
        for (int32_t e = 0; e < head_dim; ++e)
            dot += load(q, dtype, qoff + e) * load(k_cache, dtype, koff + e);
        s[j] = scale * dot;
        if (s[j] > m)
            m = s[j];
    }
    for (int32_t e = 0; e < head_dim; ++e)
        o[e] = 0.0;
    if (m == -INFINITY)
        return;
    double z = 0.0;
    for (int32_t j = 0; j < seq_len; ++j) {
        s[j] = s[j] == -INFINITY ? 0.0 : exp(s[j] - m);
        z += s[j];
    }
    for (int32_t j = 0; j < seq_len; ++j) {
        if (s[j] == 0.0)
            continue;
        const int64_t voff = (((int64_t)b * seq_len + j) * n_kv_heads + g) * head_dim;
        const double w = s[j] / z;
        for (int32_t e = 0; e < head_dim; ++e)
            o[e] += w * load(v_cache, dtype, voff + e);
    }
}

int orc_attention_simsd(const void *q, const void *k_cache, const void *v_cache, int dtype,
                        const int32_t *idx, int64_t idx_stride, const int32_t *count,
                        const uint8_t *section, const int32_t *tau, int32_t batch,
                        int32_t seq_len, int32_t r_max, int32_t n_heads, int32_t n_kv_heads,
                        int32_t head_dim, double scale, const int32_t *samples,
                        int64_t n_samples, double *out)
{
    if (!dtype_ok(dtype))
        return ORC_BAD_DTYPE;
    if (batch < 0 || seq_len <= 0 || r_max < 0 || idx_stride < r_max || n_heads <= 0 ||
        n_kv_heads <= 0 || head_dim <= 0 || n_heads % n_kv_heads != 0)
        return ORC_BAD_ARG;
    for (int64_t j = 0; j < (int64_t)batch * seq_len; ++j)
        if (section[j] > 2 || (section[j] != 0 && tau[j] < 1))
            return ORC_BAD_ARG;
    for (int32_t b = 0; b < batch; ++b) {
        if (count[b] < 0 || count[b] > r_max)
            return ORC_BAD_ARG;
        for (int32_t r = 0; r < count[b]; ++r) {
            const int32_t p = idx[b * idx_stride + r];
            if (p < 0 || p >= seq_len)
                return ORC_BAD_ARG;
        }
    }
    if (samples)
        for (int64_t t = 0; t < n_samples; ++t) {
            const int32_t b = samples[3 * t], r = samples[3 * t + 1], h = samples[3 * t + 2];
            if (b < 0 || b >= batch || r < 0 || r >= count[b] || h < 0 || h >= n_heads)
                return ORC_BAD_ARG;
        }
    const int64_t total = samples ? n_samples : (int64_t)batch * r_max * n_heads;
    int status = ORC_OK;
#pragma omp parallel num_threads(g_threads)
    {
        double *s = (double *)malloc((size_t)seq_len * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < total; ++t) {
            int32_t b, r, h;
            if (samples) {
                b = samples[3 * t];
                r = samples[3 * t + 1];
                h = samples[3 * t + 2];
            } else {
                b = (int32_t)(t / ((int64_t)r_max * n_heads));
                r = (int32_t)((t / n_heads) % r_max);
                h = (int32_t)(t % n_heads);
                if (r >= count[b])
                    continue;
            }
            if (!s) {
#pragma omp atomic write
                status = ORC_NOMEM;
                continue;
            }
            attention_simsd_one(q, k_cache, v_cache, dtype, section, tau,
                                idx[b * idx_stride + r], seq_len, r_max, n_heads, n_kv_heads,
                                head_dim, scale, b, r, h, s, out + t * head_dim);
        }
        free(s);
    }
    return status;
}

/*
 * COVER's dual-view attention with the KV-cache override and the diagonal
 * correction ("Stop the Flip-Flop: Verifica Preservante il Contesto per una
 * Decodifica di Diffusione Veloce e Revocabile", Italian technical summary
 * (gist.science/it/paper/2602.06161), section "Metodologia: COVER", item 1
 * "Dual-View Feed Forward tramite KV Cache Override").
 *
 * The recomputed rows r < count[b] of sequence b sit at positions
 * p_r = idx[b*idx_stride + r]; seed[b*r_max + r] != 0 marks a seed (a decoded
 * token under verification: its input was [MASK], so k_new / v_new of that row
 * are the masked-input K/V).  The cache holds the K/V of the previous step.
 *   - Cache: every non-seed row is written back, cache[p_r] = new[r]; a seed's
 *     position keeps the previous step's K/V (the override).
 *   - Attention of row r, head h (kv head g): softmax over all keys j < seq_len of
 *     the cache after that write-back, except that for a seed row the key at its
 *     own position p_r is its masked-input k_new[r] / v_new[r] (the diagonal
 *     correction: no self-leakage of the stored token).
 * Writes the caches in place (k_cache, v_cache) and the outputs to out
 * ([batch, r_max, n_heads, head_dim] float64, rows past count NaN).
 */
int orc_attention_cover(const void *q, const void *k_new, const void *v_new, void *k_cache,
                        void *v_cache, int dtype, const int32_t *idx, int64_t idx_stride,
                        const int32_t *count, const uint8_t *seed, int32_t batch,
                        int32_t seq_len, int32_t r_max, int32_t n_heads, int32_t n_kv_heads,
                        int32_t head_dim, double scale, double *out)
{
    if (!dtype_ok(dtype))
        return ORC_BAD_DTYPE;
    if (batch < 0 || seq_len <= 0 || r_max < 0 || idx_stride < r_max || n_heads <= 0 ||
        n_kv_heads <= 0 || head_dim <= 0 || n_heads % n_kv_heads != 0)
        return ORC_BAD_ARG;
    const size_t esz = dtype_size(dtype);
    const size_t row_bytes = (size_t)head_dim * esz;
    for (int32_t b = 0; b < batch; ++b) {
        if (count[b] < 0 || count[b] > r_max)
            return ORC_BAD_ARG;
        for (int32_t r = 0; r < count[b]; ++r) {
            const int32_t p = idx[b * idx_stride + r];
            if (p < 0 || p >= seq_len)
                return ORC_BAD_ARG;
        }
    }
    /* the write-back of the non-seed rows */
    for (int32_t b = 0; b < batch; ++b)
        for (int32_t r = 0; r < count[b]; ++r) {
            if (seed[(int64_t)b * r_max + r])
                continue;
            const int32_t p = idx[b * idx_stride + r];
            for (int32_t g = 0; g < n_kv_heads; ++g) {
                const int64_t src = (((int64_t)b * r_max + r) * n_kv_heads + g) * head_dim;
                const int64_t dst = (((int64_t)b * seq_len + p) * n_kv_heads + g) * head_dim;
                memcpy((char *)k_cache + dst * esz, (const char *)k_new + src * esz, row_bytes);
                memcpy((char *)v_cache + dst * esz, (const char *)v_new + src * esz, row_bytes);
            }
        }
    const int64_t total = (int64_t)batch * r_max * n_heads;
    int status = ORC_OK;
#pragma omp parallel num_threads(g_threads)
    {
        double *s = (double *)malloc((size_t)seq_len * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < total; ++t) {
            const int32_t b = (int32_t)(t / ((int64_t)r_max * n_heads));
            const int32_t r = (int32_t)((t / n_heads) % r_max);
            const int32_t h = (int32_t)(t % n_heads);
            double *o = out + t * head_dim;
            if (r >= count[b]) {
                for (int32_t e = 0; e < head_dim; ++e)
                    o[e] = NAN;
                continue;
            }
            if (!s) {
#pragma omp atomic write
                status = ORC_NOMEM;
                continue;
            }
            const int32_t g = h / (n_heads / n_kv_heads);
            const int is_seed = seed[(int64_t)b * r_max + r] != 0;
            const int32_t own = idx[b * idx_stride + r];
            const int64_t qoff = (((int64_t)b * r_max + r) * n_heads + h) * head_dim;
            const int64_t own_new = (((int64_t)b * r_max + r) * n_kv_heads + g) * head_dim;
            double m = -INFINITY;
            for (int32_t j = 0; j < seq_len; ++j) {
                const int diag = is_seed && j == own;
                const void *kb = diag ? k_new : k_cache;
                const int64_t koff =
                    diag ? own_new : (((int64_t)b * seq_len + j) * n_kv_heads + g) * head_dim;
                double dot = 0.0;
                for (int32_t e = 0; e < head_dim; ++e)
                    dot += load(q, dtype, qoff + e) * load(kb, dtype, koff + e);
                s[j] = scale * dot;
                if (s[j] > m)
                    m = s[j];
            }
            double z = 0.0;
            for (int32_t j = 0; j < seq_len; ++j) {
                s[j] = exp(s[j] - m);
                z += s[j];
            }
            for (int32_t e = 0; e < head_dim; ++e)
                o[e] = 0.0;
            for (int32_t j = 0; j < seq_len; ++j) {
                const int diag = is_seed && j == own;
                const void *vb = diag ? v_new : v_cache;
                const int64_t voff =
                    diag ? own_new : (((int64_t)b * seq_len + j) * n_kv_heads + g) * head_dim;
                const double w = s[j] / z;
                for (int32_t e = 0; e < head_dim; ++e)
                    o[e] += w * load(vb, dtype, voff + e);
            }
        }
        free(s);
    }
    return status;
}

/*
 * COVER's stability-aware seed score ("Stop the Flip-Flop: Verifica Preservante
 * il Contesto per una Decodifica di Diffusione Veloce e Revocabile", Italian
 * technical summary (gist.science/it/paper/2602.06161), section "Metodologia:
 * COVER", item 2 "Selezione dei Seed Sensibile alla Stabilità").
 *
 * The page scores a decoded token by Score = u (1 + d_in) / (1 + d_out): u the
 * entropy of its current assignment, d_in how much the still-masked positions
 * rely on it as context, d_out how strongly it attends to the positions drafted
 * at this step.  It gives no formula for the two attention terms; the plain one
 * is taken, over one layer's attention probabilities averaged over the heads:
 *   a^h_{r,j} = softmax_j(scale * q_{r,h} . k_{j,g(h)}), j < seq_len: recomputed
 *               row r's bidirectional attention on every key of the cache as it
 *               stands (g(h) = h / (n_heads / n_kv_heads));
 *   d_in(c)   = (1/H) sum_h sum_{r < count[b], role_r & 1} a^h_{r, p_c};
 *   d_out(c)  = (1/H) sum_h sum_{j : drafted[b, j] != 0} a^h_{c, j};
 *   score(c)  = u_c (1 + d_in(c)) / (1 + d_out(c)).
 * role[b*r_max + r]: bit 0 = the row's position is still masked after this step
 * (its query counts toward d_in), bit 1 = the row is a candidate (a decoded token
 * that may be verified); p_c = idx[b*idx_stride + c].  u[b*r_max + r] is the
 * candidate row's entropy.  The seed set is the n_seed candidates of highest
 * score, ties to the lower position (a NaN score ranks last), written as
 * positions to seeds[b*n_seed ...] and padded with -1.
 * Outputs d_in, d_out, score: [batch, r_max] float64, NaN except at the
 * candidate rows r < count[b].
 */
int orc_cover_seed_score(const void *q, const void *k_cache, int dtype, const int32_t *idx,
                         int64_t idx_stride, const int32_t *count, const uint8_t *role,
                         const uint8_t *drafted, const double *u, int32_t batch,
                         int32_t seq_len, int32_t r_max, int32_t n_heads, int32_t n_kv_heads,
                         int32_t head_dim, double scale, int32_t n_seed, double *d_in,
                         double *d_out, double *score, int32_t *seeds)
{
    if (!dtype_ok(dtype))
        return ORC_BAD_DTYPE;
    if (batch < 0 || seq_len <= 0 || r_max < 0 || idx_stride < r_max || n_heads <= 0 ||
        n_kv_heads <= 0 || head_dim <= 0 || n_heads % n_kv_heads != 0 || n_seed < 0)
        return ORC_BAD_ARG;
    for (int32_t b = 0; b < batch; ++b) {
        if (count[b] < 0 || count[b] > r_max)
            return ORC_BAD_ARG;
        for (int32_t r = 0; r < count[b]; ++r) {
            const int32_t p = idx[b * idx_stride + r];
            if (p < 0 || p >= seq_len)
                return ORC_BAD_ARG;
        }
    }
    /* per (sequence, head): that head's sums, in_h[(b*H + h)*r_max + c] and
       out_h[...]; then the head means, in head order */
    const int64_t n_items = (int64_t)batch * n_heads;
    double *in_h = (double *)calloc((size_t)(n_items * r_max + 1), sizeof(double));
    double *out_h = (double *)calloc((size_t)(n_items * r_max + 1), sizeof(double));
    if (!in_h || !out_h) {
        free(in_h), free(out_h);
        return ORC_NOMEM;
    }
    int status = ORC_OK;
#pragma omp parallel num_threads(g_threads)
    {
        double *a = (double *)malloc((size_t)seq_len * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < n_items; ++t) {
            if (!a) {
#pragma omp atomic write
                status = ORC_NOMEM;
                continue;
            }
            const int32_t b = (int32_t)(t / n_heads), h = (int32_t)(t % n_heads);
            const int32_t g = h / (n_heads / n_kv_heads);
            const int64_t row0 = (int64_t)b * r_max;
            double *in_sum = in_h + t * r_max, *out_sum = out_h + t * r_max;
            for (int32_t r = 0; r < count[b]; ++r) {
                const uint8_t rr = role[row0 + r];
                if (!(rr & 3))
                    continue;
                /* a^h_{r, j} for every key j */
                const int64_t qoff = ((row0 + r) * n_heads + h) * head_dim;
                double m = -INFINITY;
                for (int32_t j = 0; j < seq_len; ++j) {
                    const int64_t koff = (((int64_t)b * seq_len + j) * n_kv_heads + g) * head_dim;
                    double dot = 0.0;
                    for (int32_t e = 0; e < head_dim; ++e)
                        dot += load(q, dtype, qoff + e) * load(k_cache, dtype, koff + e);
                    a[j] = scale * dot;
                    if (a[j] > m)
                        m = a[j];
                }
                double z = 0.0;
                for (int32_t j = 0; j < seq_len; ++j) {
                    a[j] = exp(a[j] - m);
                    z += a[j];
                }
                for (int32_t j = 0; j < seq_len; ++j)
                    a[j] /= z;
                if (rr & 1) /* a still-masked query: the weight it puts on every candidate */
                    for (int32_t c = 0; c < count[b]; ++c)
                        if (role[row0 + c] & 2)
                            in_sum[c] += a[idx[b * idx_stride + c]];
                if (rr & 2) /* a candidate: its weight on the drafted positions */
                    for (int32_t j = 0; j < seq_len; ++j)
                        if (drafted[(int64_t)b * seq_len + j])
                            out_sum[r] += a[j];
            }
        }
        free(a);
    }
    ranked_row *cand = (ranked_row *)malloc(((size_t)r_max + 1) * sizeof(ranked_row));
    if (!cand)
        status = ORC_NOMEM;
    for (int32_t b = 0; b < batch && cand; ++b) {
        const int64_t row0 = (int64_t)b * r_max;
        for (int32_t r = 0; r < r_max; ++r)
            d_in[row0 + r] = d_out[row0 + r] = score[row0 + r] = NAN;
        int32_t nc = 0;
        for (int32_t c = 0; c < count[b]; ++c) {
            if (!(role[row0 + c] & 2))
                continue;
            double din = 0.0, dout = 0.0;
            for (int32_t h = 0; h < n_heads; ++h) {
                din += in_h[((int64_t)b * n_heads + h) * r_max + c];
                dout += out_h[((int64_t)b * n_heads + h) * r_max + c];
            }
            d_in[row0 + c] = din / n_heads;
            d_out[row0 + c] = dout / n_heads;
            score[row0 + c] = u[row0 + c] * (1.0 + d_in[row0 + c]) / (1.0 + d_out[row0 + c]);
            cand[nc].conf = isnan(score[row0 + c]) ? -INFINITY : score[row0 + c];
            cand[nc].pos = idx[b * idx_stride + c];
            cand[nc].row = c;
            ++nc;
        }
        qsort(cand, (size_t)nc, sizeof(ranked_row), by_conf_then_pos);
        for (int32_t s = 0; s < n_seed; ++s)
            seeds[(int64_t)b * n_seed + s] = s < nc ? cand[s].pos : -1;
    }
    free(cand), free(in_h), free(out_h);
    return status;
}
