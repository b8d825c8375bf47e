/*
 * sinkattn_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, fp64 CPU statement of grouped-query attention with a
 * per-head learned sink logit.  Only tests/, the smoke check and the CPU
 * baseline leg of bench.py load this code.  It shares nothing with the CUDA
 * library: no headers, helpers, tables or constants.
 *
 * What it computes (source: "GPT-OSS on day 0", Perplexity blog, section
 * "Kernels for GPT-OSS / Sink Attention"; the page's equation was lost in
 * extraction, so the prose around it fixes the method):
 *   - every attention head owns one learned sink parameter that takes part
 *     in the softmax (section "Attention: GQA with attention sinks");
 *   - the sink is an extra logit that enters the softmax normaliser next to
 *     the scaled Q.K products and brings no value row of its own;
 *   - query heads share key/value heads (GQA).
 *
 * For one query row with key set J, sink logit sig and scores
 * s_j = scale * <q, k_j>:
 *     M   = max(sig, max_j s_j)
 *     Z   = exp(sig - M) + sum_j exp(s_j - M)
 *     out = sum_j exp(s_j - M) / Z * v_j
 *     lse = M + ln Z                                    (natural log)
 * The sink is NOT multiplied by `scale`: it is a logit in the softmax's own
 * space.  With J empty, out = 0 and lse = sig; with J empty and sig = -inf,
 * out = 0 and lse = -inf.
 *
 * Readings taken where the page is silent:
 *   - query head h reads key/value head h / (Hq / Hkv) (contiguous groups);
 *   - causal prefill: row i of a sequence sees keys 0..i of that sequence;
 *   - a paged cache of page size PS stores token t of request b in page
 *     page_table[b][t / PS], slot t % PS.
 *
 * The split-KV step (same section: the online softmax keeps a running max m
 * and scale d; seeding m with the head's sink counts the sink once, and only
 * the first of several blocks along the sequence may hold it) is stated here
 * as per-chunk partial results (o_c, lse_c) and a log-sum-exp merge, each by
 * its plain definition, so that "split + merge == unsplit" can be checked.
 *
 * All inputs are the exact bf16 bit patterns of the tensors the GPU sees,
 * widened to double; sums are taken in index order in double precision.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG -1
#define ORACLE_BAD_PAGE -2
#define ORACLE_NO_MEM -3

static double widen_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * The definition above for one query row.  keys[j] / vals[j] point at the
 * D-element bf16 rows of key j.  `with_sink` = 0 leaves the sink out (a chunk
 * that does not hold it); `s` is caller scratch of J doubles.
 */
static void sink_row(const uint16_t *q, const uint16_t *const *keys,
                     const uint16_t *const *vals, long J, int D, double sig,
                     int with_sink, double scale, double *s, double *out,
                     double *lse) {
    double M = with_sink ? sig : -INFINITY;
    for (long j = 0; j < J; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += widen_bf16(q[d]) * widen_bf16(keys[j][d]);
        s[j] = scale * dot;
        if (s[j] > M) M = s[j];
    }
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (M == -INFINITY) { /* no key and no (finite) sink: empty softmax */
        *lse = -INFINITY;
        return;
    }
    double Z = with_sink ? exp(sig - M) : 0.0;
    for (long j = 0; j < J; ++j) {
        double w = exp(s[j] - M);
        Z += w;
        for (int d = 0; d < D; ++d) out[d] += w * widen_bf16(vals[j][d]);
    }
    for (int d = 0; d < D; ++d) out[d] /= Z;
    *lse = M + log(Z);
}

/* Address of token t of request b in a paged pool [P, Hkv, PS, D]; NULL if the page id is out of range. */
static const uint16_t *paged_row(const uint16_t *pool, const int32_t *page_table,
                                 int max_pages, int num_pages, int Hkv, int PS,
                                 int D, int b, int kvh, long t) {
    int32_t page = page_table[(long)b * max_pages + t / PS];
    if (page < 0 || page >= num_pages) return NULL;
    return pool + (((long)page * Hkv + kvh) * PS + t % PS) * D;
}

/*
 * Decode: one query token per request against its paged cache.
 *   q [B, Hq, D]; k_pages, v_pages [num_pages, Hkv, PS, D]; page_table
 *   [B, max_pages]; kv_lens [B]; sinks [Hq].
 * rows: n_rows (b, h) pairs, or NULL for every (b, h) in order.
 * out: [n_rows, D], lse: [n_rows] (n_rows = B*Hq when rows is NULL).
 */
int oracle_decode(int B, int Hq, int Hkv, int D, int PS, int max_pages, int num_pages,
                  const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                  const int32_t *page_table, const int32_t *kv_lens, const float *sinks,
                  float scale, int n_rows, const int32_t *rows, double *out, double *lse) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || PS <= 0) return ORACLE_BAD_ARG;
    const int G = Hq / Hkv;
    const long total = rows ? n_rows : (long)B * Hq;
    int status = ORACLE_OK;
#pragma omp parallel
    {
        long cap = 0;
        double *s = NULL;
        const uint16_t **kp = NULL, **vp = NULL;
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < total; ++r) {
            int b = rows ? rows[2 * r] : (int)(r / Hq);
            int h = rows ? rows[2 * r + 1] : (int)(r % Hq);
            int kvh = h / G;
            long J = kv_lens[b];
            if (J > cap) {
                cap = J;
                s = realloc(s, sizeof(double) * cap);
                kp = realloc((void *)kp, sizeof(void *) * cap);
                vp = realloc((void *)vp, sizeof(void *) * cap);
            }
            int bad = 0;
            for (long t = 0; t < J; ++t) {
                kp[t] = paged_row(k_pages, page_table, max_pages, num_pages, Hkv, PS, D, b, kvh, t);
                vp[t] = paged_row(v_pages, page_table, max_pages, num_pages, Hkv, PS, D, b, kvh, t);
                if (!kp[t]) bad = 1;
            }
            if (bad) {
#pragma omp atomic write
                status = ORACLE_BAD_PAGE;
                continue;
            }
            sink_row(q + ((long)b * Hq + h) * D, kp, vp, J, D, (double)sinks[h], 1,
                     (double)scale, s, out + r * D, lse + r);
        }
        free(s);
        free((void *)kp);
        free((void *)vp);
    }
    return status;
}

/*
 * Verification of drafted tokens (speculative decoding): q_len query tokens per
 * request whose keys and values are already the last q_len entries of the
 * request's paged cache.  Source: "Accelerating Sonar through speculation"
 * (Perplexity), sections "Speculative decoding" (the target model runs over the
 * drafted sequence and produces logits for every drafted token) and "Inference
 * with speculative decoding" (verification batches over the paged KV cache).
 * Reading where the page is silent: query token i (0-based) of request b sits
 * at cache position kv_lens[b] - q_len + i and sees cache tokens 0 .. that
 * position -- everything before the draft plus the draft up to itself; a
 * position below 0 leaves the key set empty.
 *   q [B, q_len, Hq, D]; k_pages, v_pages, page_table, kv_lens, sinks as decode.
 * rows: n_rows (b, i, h) triples, or NULL for every (b, i, h) in order.
 * out: [n_rows, D], lse: [n_rows] (n_rows = B*q_len*Hq when rows is NULL).
 */
int oracle_verify(int B, int q_len, int Hq, int Hkv, int D, int PS, int max_pages, int num_pages,
                  const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                  const int32_t *page_table, const int32_t *kv_lens, const float *sinks,
                  float scale, int n_rows, const int32_t *rows, double *out, double *lse) {
    if (B < 0 || q_len <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || PS <= 0) return ORACLE_BAD_ARG;
    const int G = Hq / Hkv;
    const long total = rows ? n_rows : (long)B * q_len * Hq;
    int status = ORACLE_OK;
#pragma omp parallel
    {
        long cap = 0;
        double *s = NULL;
        const uint16_t **kp = NULL, **vp = NULL;
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < total; ++r) {
            int b = rows ? rows[3 * r] : (int)(r / ((long)q_len * Hq));
            int i = rows ? rows[3 * r + 1] : (int)((r / Hq) % q_len);
            int h = rows ? rows[3 * r + 2] : (int)(r % Hq);
            int kvh = h / G;
            long J = (long)kv_lens[b] - q_len + i + 1; /* keys 0 .. position of token i */
            if (J < 0) J = 0;
            if (J > cap) {
                cap = J;
                s = realloc(s, sizeof(double) * cap);
                kp = realloc((void *)kp, sizeof(void *) * cap);
                vp = realloc((void *)vp, sizeof(void *) * cap);
            }
            int bad = 0;
            for (long t = 0; t < J; ++t) {
                kp[t] = paged_row(k_pages, page_table, max_pages, num_pages, Hkv, PS, D, b, kvh, t);
                vp[t] = paged_row(v_pages, page_table, max_pages, num_pages, Hkv, PS, D, b, kvh, t);
                if (!kp[t]) bad = 1;
            }
            if (bad) {
#pragma omp atomic write
                status = ORACLE_BAD_PAGE;
                continue;
            }
            sink_row(q + (((long)b * q_len + i) * Hq + h) * D, kp, vp, J, D, (double)sinks[h], 1,
                     (double)scale, s, out + r * D, lse + r);
        }
        free(s);
        free((void *)kp);
        free((void *)vp);
    }
    return status;
}

/*
 * Prefill over packed variable-length sequences.
 *   q [T, Hq, D], k and v [T, Hkv, D]; sequence n occupies tokens
 *   cu_seqlens[n] .. cu_seqlens[n+1]-1.  causal != 0: row i sees keys
 *   0..i of its own sequence; causal == 0: the whole sequence.
 * rows: n_rows (t, h) pairs, or NULL for every (t, h) in order.
 */
int oracle_prefill(int N, const int32_t *cu_seqlens, int T, int Hq, int Hkv, int D,
                   const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   const float *sinks, float scale, int causal, int n_rows,
                   const int32_t *rows, double *out, double *lse) {
    if (N < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0) return ORACLE_BAD_ARG;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T) return ORACLE_BAD_ARG;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return ORACLE_BAD_ARG;
    const int G = Hq / Hkv;
    const long total = rows ? n_rows : (long)T * Hq;
#pragma omp parallel
    {
        long cap = 0;
        double *s = NULL;
        const uint16_t **kp = NULL, **vp = NULL;
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < total; ++r) {
            long t = rows ? rows[2 * r] : r / Hq;
            int h = rows ? rows[2 * r + 1] : (int)(r % Hq);
            int n = 0;
            while (cu_seqlens[n + 1] <= t) ++n; /* sequence holding token t */
            long start = cu_seqlens[n], end = cu_seqlens[n + 1];
            long J = causal ? (t - start + 1) : (end - start);
            if (J > cap) {
                cap = J;
                s = realloc(s, sizeof(double) * cap);
                kp = realloc((void *)kp, sizeof(void *) * cap);
                vp = realloc((void *)vp, sizeof(void *) * cap);
            }
            for (long j = 0; j < J; ++j) {
                kp[j] = k + ((start + j) * Hkv + h / G) * D;
                vp[j] = v + ((start + j) * Hkv + h / G) * D;
            }
            sink_row(q + (t * Hq + h) * D, kp, vp, J, D, (double)sinks[h], 1,
                     (double)scale, s, out + r * D, lse + r);
        }
        free(s);
        free((void *)kp);
        free((void *)vp);
    }
    return ORACLE_OK;
}

/*
 * Verification of a TREE of drafted tokens.  Source: "Accelerating Sonar
 * through speculation" (Perplexity), section "EAGLE": the drafts form a tree
 * explored by the drafter, and the target model checks the tree with a custom
 * attention mask.  Reading where the page is silent: the q_len drafted tokens
 * of request b are the last q_len cache tokens, in the order given (position
 * kv_lens[b] - q_len + i for token i); token i sees every cache token before
 * the draft, and drafted token j iff bit j of tree_mask[b * q_len + i] is set
 * (its ancestors in the tree and itself).  A chain mask (bits 0..i) is the
 * linear verification above.
 *   tree_mask [B, q_len] uint64 (q_len <= 64); other arguments as oracle_verify.
 */
int oracle_verify_tree(int B, int q_len, int Hq, int Hkv, int D, int PS, int max_pages, int num_pages,
                       const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                       const int32_t *page_table, const int32_t *kv_lens, const uint64_t *tree_mask,
                       const float *sinks, float scale, int n_rows, const int32_t *rows, double *out,
                       double *lse) {
    if (B < 0 || q_len <= 0 || q_len > 64 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || PS <= 0)
        return ORACLE_BAD_ARG;
    const int G = Hq / Hkv;
    const long total = rows ? n_rows : (long)B * q_len * Hq;
    int status = ORACLE_OK;
#pragma omp parallel
    {
        long cap = 0;
        double *s = NULL;
        const uint16_t **kp = NULL, **vp = NULL;
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < total; ++r) {
            int b = rows ? rows[3 * r] : (int)(r / ((long)q_len * Hq));
            int i = rows ? rows[3 * r + 1] : (int)((r / Hq) % q_len);
            int h = rows ? rows[3 * r + 2] : (int)(r % Hq);
            long L = kv_lens[b];
            long base = L - q_len; /* first drafted position */
            if (L > cap) {
                cap = L;
                s = realloc(s, sizeof(double) * cap);
                kp = realloc((void *)kp, sizeof(void *) * cap);
                vp = realloc((void *)vp, sizeof(void *) * cap);
            }
            const uint64_t bits = tree_mask[(long)b * q_len + i];
            long J = 0;
            int bad = 0;
            for (long t = 0; t < L; ++t) {
                if (t >= base && !((bits >> (t - base)) & 1ull)) continue; /* a draft token off its path */
                kp[J] = paged_row(k_pages, page_table, max_pages, num_pages, Hkv, PS, D, b, h / G, t);
                vp[J] = paged_row(v_pages, page_table, max_pages, num_pages, Hkv, PS, D, b, h / G, t);
                if (!kp[J]) bad = 1;
                ++J;
            }
            if (bad) {
#pragma omp atomic write
                status = ORACLE_BAD_PAGE;
                continue;
            }
            sink_row(q + (((long)b * q_len + i) * Hq + h) * D, kp, vp, J, D, (double)sinks[h], 1,
                     (double)scale, s, out + r * D, lse + r);
        }
        free(s);
        free((void *)kp);
        free((void *)vp);
    }
    return status;
}

/*
 * Chunked prefill over a paged cache.  Source: "Accelerating Sonar through
 * speculation" (Perplexity), section "Inference with speculative decoding":
 * input tokens are batched, slots for them are allocated in the per-request KV
 * pages, the page metadata goes to the GPU and the batch runs as prefill,
 * decode or verification over those pages.  Reading where the page is silent:
 * the new tokens of sequence n (len_n = cu_seqlens[n+1] - cu_seqlens[n]) are
 * already in its pages at cache positions start_pos[n] .. start_pos[n] + len_n - 1;
 * new token i sees cache tokens 0 .. start_pos[n] + i (the cached prefix and the
 * new tokens up to itself).
 *   q [T, Hq, D] packed new tokens; k_pages, v_pages [num_pages, Hkv, PS, D];
 *   page_table [N, max_pages]; start_pos [N]; sinks [Hq].
 * rows: n_rows (t, h) pairs, or NULL for every (t, h) in order.
 */
int oracle_prefill_paged(int N, const int32_t *cu_seqlens, const int32_t *start_pos, int T, int Hq, int Hkv,
                         int D, int PS, int max_pages, int num_pages, const uint16_t *q,
                         const uint16_t *k_pages, const uint16_t *v_pages, const int32_t *page_table,
                         const float *sinks, float scale, int n_rows, const int32_t *rows, double *out,
                         double *lse) {
    if (N < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || PS <= 0) return ORACLE_BAD_ARG;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T) return ORACLE_BAD_ARG;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n] || start_pos[n] < 0) return ORACLE_BAD_ARG;
    const int G = Hq / Hkv;
    const long total = rows ? n_rows : (long)T * Hq;
    int status = ORACLE_OK;
#pragma omp parallel
    {
        long cap = 0;
        double *s = NULL;
        const uint16_t **kp = NULL, **vp = NULL;
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < total; ++r) {
            long t = rows ? rows[2 * r] : r / Hq;
            int h = rows ? rows[2 * r + 1] : (int)(r % Hq);
            int n = 0;
            while (cu_seqlens[n + 1] <= t) ++n; /* sequence holding token t */
            long J = (long)start_pos[n] + (t - cu_seqlens[n]) + 1; /* cache tokens 0 .. its position */
            if (J > cap) {
                cap = J;
                s = realloc(s, sizeof(double) * cap);
                kp = realloc((void *)kp, sizeof(void *) * cap);
                vp = realloc((void *)vp, sizeof(void *) * cap);
            }
            int bad = 0;
            for (long j = 0; j < J; ++j) {
                kp[j] = paged_row(k_pages, page_table, max_pages, num_pages, Hkv, PS, D, n, h / G, j);
                vp[j] = paged_row(v_pages, page_table, max_pages, num_pages, Hkv, PS, D, n, h / G, j);
                if (!kp[j]) bad = 1;
            }
            if (bad) {
#pragma omp atomic write
                status = ORACLE_BAD_PAGE;
                continue;
            }
            sink_row(q + (t * Hq + h) * D, kp, vp, J, D, (double)sinks[h], 1, (double)scale, s, out + r * D,
                     lse + r);
        }
        free(s);
        free((void *)kp);
        free((void *)vp);
    }
    return status;
}

/*
 * Split-KV partial results of decode: chunk c covers tokens
 * [c*chunk_tokens, (c+1)*chunk_tokens) of each request (possibly empty).
 *   sink_mode 0: the chunk holding token 0 (chunk 0) also holds the sink --
 *                the page's rule, "only the first block";
 *   sink_mode 1: no chunk holds it (the merge adds it once instead);
 *   sink_mode 2: every chunk holds it -- a deliberately wrong rule, kept
 *                so that a test can show the merge check catches it.
 * partial_o [S, B, Hq, D] holds o_c = (sum_j e^{s_j-M_c} v_j) / Z_c and
 * partial_lse [S, B, Hq] holds M_c + ln Z_c; an empty chunk without the
 * sink gives (0, -inf).
 */
int oracle_decode_partials(int B, int Hq, int Hkv, int D, int PS, int max_pages,
                           int num_pages, const uint16_t *q, const uint16_t *k_pages,
                           const uint16_t *v_pages, const int32_t *page_table,
                           const int32_t *kv_lens, const float *sinks, float scale,
                           int S, int chunk_tokens, int sink_mode, double *partial_o,
                           double *partial_lse) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || S <= 0 || chunk_tokens <= 0) return ORACLE_BAD_ARG;
    if (sink_mode < 0 || sink_mode > 2) return ORACLE_BAD_ARG;
    const int G = Hq / Hkv;
    int status = ORACLE_OK;
    double *s = malloc(sizeof(double) * chunk_tokens);
    const uint16_t **kp = malloc(sizeof(void *) * chunk_tokens);
    const uint16_t **vp = malloc(sizeof(void *) * chunk_tokens);
    if (!s || !kp || !vp) { free(s); free((void *)kp); free((void *)vp); return ORACLE_NO_MEM; }
    for (int c = 0; c < S; ++c)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hq; ++h) {
                long lo = (long)c * chunk_tokens, hi = lo + chunk_tokens;
                if (hi > kv_lens[b]) hi = kv_lens[b];
                long J = hi > lo ? hi - lo : 0;
                for (long j = 0; j < J; ++j) {
                    kp[j] = paged_row(k_pages, page_table, max_pages, num_pages, Hkv, PS, D, b, h / G, lo + j);
                    vp[j] = paged_row(v_pages, page_table, max_pages, num_pages, Hkv, PS, D, b, h / G, lo + j);
                    if (!kp[j]) status = ORACLE_BAD_PAGE;
                }
                if (status != ORACLE_OK) continue;
                int with_sink = sink_mode == 2 || (sink_mode == 0 && c == 0);
                long r = ((long)c * B + b) * Hq + h;
                sink_row(q + ((long)b * Hq + h) * D, kp, vp, J, D, (double)sinks[h],
                         with_sink, (double)scale, s, partial_o + r * D, partial_lse + r);
            }
    free(s);
    free((void *)kp);
    free((void *)vp);
    return status;
}

/*
 * Merge of S partial results per row by log-sum-exp (same section: the
 * split along the sequence must count the sink exactly once).
 *   partial_o [S, R, H, D], partial_lse [S, R, H]; sinks [H] or NULL.
 *   L   = log( sum_c e^{lse_c} [+ e^{sink_h} when sinks is given] )
 *   out = sum_c e^{lse_c - L} o_c,  lse = L.
 * A row whose every term is -inf gives out = 0, lse = -inf.
 */
int oracle_merge(int S, int R, int H, int D, const double *partial_o,
                 const double *partial_lse, const float *sinks, double *out,
                 double *lse) {
    if (S < 0 || R < 0 || H <= 0 || D <= 0) return ORACLE_BAD_ARG;
    for (long r = 0; r < (long)R * H; ++r) {
        int h = (int)(r % H);
        double M = sinks ? (double)sinks[h] : -INFINITY;
        for (int c = 0; c < S; ++c) {
            double l = partial_lse[(long)c * R * H + r];
            if (l > M) M = l;
        }
        for (int d = 0; d < D; ++d) out[r * D + d] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = sinks ? exp((double)sinks[h] - M) : 0.0;
        for (int c = 0; c < S; ++c) sum += exp(partial_lse[(long)c * R * H + r] - M);
        double L = M + log(sum);
        for (int c = 0; c < S; ++c) {
            double w = exp(partial_lse[(long)c * R * H + r] - L);
            if (w == 0.0) continue;
            const double *o = partial_o + ((long)c * R * H + r) * D;
            for (int d = 0; d < D; ++d) out[r * D + d] += w * o[d];
        }
        lse[r] = L;
    }
    return ORACLE_OK;
}

/* Number of OpenMP threads this build would use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the number of threads later calls use (n >= 1; ignored without OpenMP). */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
