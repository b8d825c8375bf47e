/*
 * sinkattn.h -- C ABI of libsinkattn: grouped-query attention with a
 * per-head learned sink logit, for one NVIDIA GB300 (sm_103a).
 *
 * The method (source: "GPT-OSS on day 0", Perplexity blog, sections
 * "Attention: GQA with attention sinks" and "Kernels for GPT-OSS / Sink
 * Attention"):  every query head h owns a learned logit sink[h] that joins
 * the softmax normaliser beside the scaled scores s_j = scale * <q, k_j> and
 * has no value row.  For one query row with visible keys J:
 *     M   = max(sink[h], max_j s_j)
 *     Z   = exp(sink[h] - M) + sum_j exp(s_j - M)
 *     out = sum_j exp(s_j - M) / Z * v_j,      lse = M + ln Z.
 * sink[h] is compared with the scaled scores as it is (it is not multiplied
 * by `scale`).  Query head h reads key/value head h / (Hq / Hkv).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, dense and
 *     row-major in the layout stated beside each argument.  bf16 tensors and
 *     `out` must be 16-byte aligned; int32/f32 tensors 4-byte aligned.
 *   - The library allocates no device memory, frees nothing and never
 *     synchronises on the call path: the work is enqueued on `stream` (a
 *     cudaStream_t passed as void*; NULL = the legacy default stream) on the
 *     CUDA device that is current for the calling thread.
 *   - The return value reports host-side validation and launch errors only.
 *     Problems found on the device (an out-of-range page id or length, a
 *     pipeline wait that ran out) are recorded in a per-device error word
 *     that sinkattn_get_error() reads; the kernels never trap.
 *   - head_dim must be 64 and the KV page size 16; anything else returns
 *     SINKATTN_ERR_UNSUPPORTED.
 */
#ifndef SINKATTN_H_
#define SINKATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SINKATTN_OK = 0,
    SINKATTN_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer */
    SINKATTN_ERR_UNSUPPORTED = 2,  /* head_dim != 64, page size != 16, group size > 16, ... */
    SINKATTN_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
    SINKATTN_ERR_BAD_PAGE = 4,     /* device: a page id outside [0, num_pages) was met */
    SINKATTN_ERR_TIMEOUT = 5,      /* device: a pipeline wait gave up; results are invalid */
    SINKATTN_ERR_CUDA = 6,         /* a CUDA runtime call failed */
    SINKATTN_ERR_BAD_LENGTH = 7    /* device: a kv_len outside [0, max_pages*16] was met */
} sinkattn_status_t;

/* Sizes of a paged decode call. */
typedef struct {
    int32_t batch;             /* B >= 0 requests, one query token each (B <= 32768)    */
    int32_t num_q_heads;       /* Hq                                                     */
    int32_t num_kv_heads;      /* Hkv; Hq % Hkv == 0 and Hq / Hkv <= 16                  */
    int32_t head_dim;          /* must be 64                                             */
    int32_t page_size;         /* must be 16                                             */
    int32_t num_pages;         /* P, pages in the K/V pools                              */
    int32_t max_pages;         /* row length of page_table (>= 1)                        */
    int32_t num_workers;       /* 0 = automatic (one share per resident CTA, up to four per SM);
                                  otherwise the number of equal shares the flattened
                                  (request, KV head, page) work is cut into, one CTA each.
                                  A request whose pages span several shares is split and
                                  merged; the result does not depend on this value.  Two
                                  shares per SM leave room for a prefill with share_sms
                                  on another stream.                                     */
} sinkattn_decode_dims_t;

/* Sizes of a packed variable-length prefill call. */
typedef struct {
    int32_t num_seqs;          /* N >= 0 sequences                                       */
    int32_t total_tokens;      /* T = cu_seqlens[N]                                      */
    int32_t max_seqlen;        /* an upper bound of every sequence length                */
    int32_t num_q_heads;       /* Hq                                                     */
    int32_t num_kv_heads;      /* Hkv; Hq % Hkv == 0                                     */
    int32_t head_dim;          /* must be 64                                             */
    int32_t share_sms;         /* 0: the fastest kernel for a prefill that has the GPU to
                                  itself (two query heads per CTA, a whole SM each, when
                                  Hq / Hkv is even); 1: a kernel that leaves room on every
                                  SM for another kernel on another stream (one head per CTA,
                                  two CTAs per SM at 32 K registers, ~100 KB of shared
                                  memory and 256 TMEM columns each), so that a decode
                                  launched just before it with two shares per SM
                                  (num_workers = 2 x SMs) runs beside it; other values:
                                  SINKATTN_ERR_INVALID_ARG                              */
} sinkattn_prefill_dims_t;

/* Sizes of a merge call. */
typedef struct {
    int32_t num_splits;        /* S partial results per row (>= 0)                       */
    int32_t num_rows;          /* R                                                      */
    int32_t num_heads;         /* H                                                      */
    int32_t head_dim;          /* must be 64                                             */
} sinkattn_merge_dims_t;

/*
 * Bytes of device workspace sinkattn_decode needs for `dims` on the current
 * device.  0 on invalid dims.  The workspace holds the split-KV partial
 * results and a small per-(request, KV head) table; it needs no
 * initialisation and its contents are dead after the call completes.
 */
size_t sinkattn_decode_workspace_size(const sinkattn_decode_dims_t *dims);

/*
 * Paged decode with split-KV and a merge that counts the sink once.
 * Source: "GPT-OSS on day 0", section "Kernels for GPT-OSS / Sink Attention"
 * (parallelism over heads and along the KV length; online softmax whose
 * running max is seeded from the head's sink in the first block only), and
 * "Accelerating Sonar through speculation", section "Inference with
 * speculative decoding" (KV pages allocated per request; page metadata copied
 * to the GPU before the attention kernel).
 *
 *   q          [B, Hq, 64]        bf16   one query token per request
 *   k_pages    [P, Hkv, 16, 64]   bf16   page p, KV head g, slot t: key of one token
 *   v_pages    [P, Hkv, 16, 64]   bf16   same layout for values
 *   page_table [B, max_pages]     int32  token t of request b lives in page
 *                                        page_table[b][t/16], slot t%16; entries past
 *                                        the request's last page are never read
 *   kv_lens    [B]                int32  cached tokens per request, 0..max_pages*16
 *   sinks      [Hq]               f32    learned sink logit of each query head
 *   scale      softmax scale applied to q.k (usually 1/sqrt(64))
 *   out        [B, Hq, 64]        bf16   attention output
 *   lse        [B, Hq]            f32    natural-log log-sum-exp including the sink,
 *                                        or NULL
 *   workspace  device scratch of at least sinkattn_decode_workspace_size(dims) bytes,
 *              256-byte aligned; it must not be shared by calls that may overlap.
 *
 * A request with kv_len 0 gives out = 0 and lse = sink[h].  Page ids outside
 * [0, P) are skipped (their tokens count as absent) and raise
 * SINKATTN_ERR_BAD_PAGE in the error word; kv_len outside [0, max_pages*16] is
 * clamped and raises SINKATTN_ERR_BAD_LENGTH.
 */
sinkattn_status_t sinkattn_decode(const void *q, const void *k_pages, const void *v_pages,
                                  const int32_t *page_table, const int32_t *kv_lens,
                                  const float *sinks, float scale, void *out, float *lse,
                                  const sinkattn_decode_dims_t *dims, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* Shapes of a verification call. */
typedef struct {
    int32_t batch;             /* B requests, 0..32768                                     */
    int32_t q_len;             /* drafted query tokens per request, 1..16, and
                                  q_len * (num_q_heads / num_kv_heads) <= 64              */
    int32_t num_q_heads;       /* Hq                                                      */
    int32_t num_kv_heads;      /* Hkv, divides Hq                                         */
    int32_t head_dim;          /* must be 64                                              */
    int32_t page_size;         /* must be 16                                              */
    int32_t num_pages;         /* P, pages in the K/V pools                               */
    int32_t max_pages;         /* row length of page_table (>= 1)                         */
    int32_t num_workers;       /* as in sinkattn_decode_dims_t (0 = automatic)            */
} sinkattn_verify_dims_t;

/* Bytes of device workspace sinkattn_verify needs for `dims`; 0 on invalid dims. */
size_t sinkattn_verify_workspace_size(const sinkattn_verify_dims_t *dims);

/*
 * Attention of drafted tokens over the paged cache: the verification step of
 * speculative decoding.  Source: "Accelerating Sonar through speculation",
 * sections "Speculative decoding" (the target model runs over the drafted
 * tokens and produces logits for each of them) and "Inference with
 * speculative decoding" (verification batches over the paged KV cache); the
 * attention of every token is the sink attention of sinkattn_decode.
 *
 * The q_len query tokens of request b are its last q_len cached tokens, whose
 * K and V are already in the pages: token i sits at cache position
 * kv_lens[b] - q_len + i and attends to cache tokens 0 .. that position
 * (the whole prefix and the draft up to itself).  All q_len tokens of a
 * request share one pass over its pages.  q_len = 1 is sinkattn_decode.
 *
 *   q          [B, q_len, Hq, 64]  bf16
 *   k_pages, v_pages, page_table, sinks, scale: as sinkattn_decode
 *   kv_lens    [B] int32   cached tokens per request, the q_len drafted ones included;
 *                          a request shorter than q_len leaves its earliest tokens
 *                          without keys (out = 0, lse = sink)
 *   out        [B, q_len, Hq, 64]  bf16
 *   lse        [B, q_len, Hq]      f32 natural log, or NULL
 *   workspace  at least sinkattn_verify_workspace_size(dims) bytes, 256-byte aligned;
 *              it needs no initialisation and must not be shared by overlapping calls.
 *
 * Errors and the handling of bad page ids and lengths are those of sinkattn_decode.
 */
sinkattn_status_t sinkattn_verify(const void *q, const void *k_pages, const void *v_pages,
                                  const int32_t *page_table, const int32_t *kv_lens,
                                  const float *sinks, float scale, void *out, float *lse,
                                  const sinkattn_verify_dims_t *dims, void *workspace,
                                  size_t workspace_bytes, void *stream);

/*
 * sinkattn_verify for a TREE of drafted tokens.  Source: "Accelerating Sonar
 * through speculation", section "EAGLE": the drafter explores a tree of
 * candidate continuations and the target checks the whole tree at once with a
 * custom attention mask.
 *
 * The q_len drafted tokens of request b are its last q_len cached tokens, in
 * any order that puts parents before children: token i sits at cache position
 * kv_lens[b] - q_len + i, sees every cache token before the draft, and sees
 * drafted token j iff bit j of tree_mask[b][i] is set (its ancestors and
 * itself).  A mask with bits 0..i for token i is the linear draft of
 * sinkattn_verify.
 *
 *   tree_mask  [B, q_len] uint64, 8-byte aligned, device memory (q_len <= 64)
 *   everything else as sinkattn_verify (same workspace size).
 */
sinkattn_status_t sinkattn_verify_tree(const void *q, const void *k_pages, const void *v_pages,
                                       const int32_t *page_table, const int32_t *kv_lens,
                                       const uint64_t *tree_mask, const float *sinks, float scale,
                                       void *out, float *lse, const sinkattn_verify_dims_t *dims,
                                       void *workspace, size_t workspace_bytes, void *stream);

/* Shapes of the calls over a paged cache that take new tokens packed by cu_seqlens. */
typedef struct {
    int32_t num_seqs;          /* N sequences (requests), 0..16384                        */
    int32_t total_tokens;      /* T new tokens, packed by cu_seqlens                      */
    int32_t max_seqlen;        /* >= the largest number of new tokens of one sequence     */
    int32_t num_q_heads;       /* Hq (read by sinkattn_prefill_paged only)                */
    int32_t num_kv_heads;      /* Hkv, divides Hq                                         */
    int32_t head_dim;          /* must be 64                                              */
    int32_t page_size;         /* must be 16                                              */
    int32_t num_pages;         /* P, pages in the K/V pools                               */
    int32_t max_pages;         /* row length of page_table (>= 1)                         */
    int32_t share_sms;         /* sinkattn_prefill_paged only: as in sinkattn_prefill_dims_t
                                  (0 or 1; the other calls ignore it)                      */
} sinkattn_paged_dims_t;

/*
 * Writes the keys and values of new tokens into their requests' pages.
 * Source: "Accelerating Sonar through speculation", section "Inference with
 * speculative decoding": slots for the next tokens are allocated in the
 * per-request KV pages before the batch runs.
 *
 *   k, v        [T, Hkv, 64]     bf16   new tokens of N sequences, packed by cu_seqlens
 *   cu_seqlens  [N + 1]          int32  cu_seqlens[0] = 0, non-decreasing, cu_seqlens[N] = T
 *   start_pos   [N]              int32  cache position of each sequence's first new token
 *                                       (the number of tokens already cached)
 *   page_table  [N, max_pages]   int32  token at cache position p of sequence n goes to page
 *                                       page_table[n][p / 16], slot p % 16
 *   k_pages, v_pages [P, Hkv, 16, 64] bf16, written in place (only the new tokens' slots)
 *
 * A page id outside [0, P) skips its tokens and raises SINKATTN_ERR_BAD_PAGE; a
 * position past max_pages * 16 skips the token and raises SINKATTN_ERR_BAD_LENGTH.
 */
sinkattn_status_t sinkattn_kv_append(const void *k, const void *v, const int32_t *cu_seqlens,
                                     const int32_t *start_pos, const int32_t *page_table,
                                     void *k_pages, void *v_pages, const sinkattn_paged_dims_t *dims,
                                     void *stream);

/*
 * Chunked prefill over the paged cache: new tokens of N sequences attend to
 * everything cached before them and to the new tokens up to themselves.
 * Source: "Accelerating Sonar through speculation", section "Inference with
 * speculative decoding" (batches of prefill, decode or verification run over
 * the per-request KV pages); the attention is the sink attention of
 * sinkattn_prefill ("GPT-OSS on day 0", section "Kernels for GPT-OSS / Sink
 * Attention").
 *
 * The new tokens' keys and values must already be in the pages
 * (sinkattn_kv_append): new token i of sequence n sits at cache position
 * start_pos[n] + i and sees cache tokens 0 .. start_pos[n] + i.
 *
 *   q           [T, Hq, 64]   bf16   new tokens packed by cu_seqlens
 *   k_pages, v_pages [P, Hkv, 16, 64] bf16 (P >= 1), page_table [N, max_pages] int32,
 *   cu_seqlens [N + 1], start_pos [N]: as sinkattn_kv_append
 *   sinks [Hq] f32, scale: as sinkattn_prefill
 *   out         [T, Hq, 64]   bf16;  lse [T, Hq] f32 natural log, or NULL
 *
 * dims->max_seqlen bounds the new tokens of one sequence (a longer one is cut and
 * raises SINKATTN_ERR_BAD_LENGTH, as does start_pos[n] + len_n > max_pages * 16).
 * A page id outside [0, P) raises SINKATTN_ERR_BAD_PAGE; its tokens then read as
 * zero vectors and that sequence's result is not meaningful.  Slots past a
 * sequence's last cached token may hold anything.
 */
sinkattn_status_t sinkattn_prefill_paged(const void *q, const void *k_pages, const void *v_pages,
                                         const int32_t *page_table, const int32_t *cu_seqlens,
                                         const int32_t *start_pos, const float *sinks, float scale,
                                         void *out, float *lse, const sinkattn_paged_dims_t *dims,
                                         void *stream);

/* YaRN rotary embedding parameters (sinkattn_qkv_prologue). */
typedef struct {
    float theta;                    /* base of the rotary frequencies: theta^(-2d/64) for pair d  */
    float factor;                   /* context extension factor s (>= 1; 1 = plain rotary)        */
    int32_t original_max_position;  /* context length L the model was trained with               */
    float beta_fast;                /* pairs turning more than beta_fast times over L keep their
                                       frequency ...                                             */
    float beta_slow;                /* ... pairs turning fewer than beta_slow times are slowed by s;
                                       linear in between (beta_fast > beta_slow > 0)              */
    float attn_factor;              /* multiplier of rotated q and k; 0 = 0.1 ln(s) + 1 (1 if s = 1) */
    int32_t interleaved;            /* 0: pairs (d, d + 32); 1: pairs (2d, 2d + 1)                */
} sinkattn_rope_t;

/*
 * The pre-attention step of new tokens, fused: QKV bias, YaRN rotary embedding
 * of q and k, q to `q_out`, and k / v written straight into the tokens' page
 * slots (what sinkattn_kv_append does for ready keys and values).  Source:
 * "GPT-OSS on day 0", section "Attention: GQA with attention sinks" (QKV
 * projections with a bias; YaRN positional encoding as in DeepSeek-V3).  The
 * page gives no formulas; these follow the published YaRN method: for pair d,
 * theta_d = theta^(-2d/64) and r_d = L theta_d / (2 pi) (turns over the
 * original context); gamma = clamp((r_d - beta_slow) / (beta_fast - beta_slow),
 * 0, 1); the angle per position is ((1 - gamma) / s + gamma) theta_d; rotated q
 * and k are multiplied by attn_factor.
 *
 *   qkv        [T, (Hq + 2 Hkv) * 64] bf16  projected new tokens: Hq q heads, then Hkv k
 *                                           heads, then Hkv v heads
 *   bias       [(Hq + 2 Hkv) * 64]    bf16  added before the rotation, or NULL
 *   cu_seqlens [N + 1], start_pos [N], page_table [N, max_pages]: as sinkattn_kv_append
 *                                           (new token i of sequence n is at position
 *                                           start_pos[n] + i)
 *   q_out      [T, Hq, 64]            bf16
 *   k_pages, v_pages [P, Hkv, 16, 64] bf16  the new tokens' slots are written
 *
 * bf16 buffers 16-byte aligned.  Bad page ids and positions are reported as in
 * sinkattn_kv_append (q_out is still written).
 */
sinkattn_status_t sinkattn_qkv_prologue(const void *qkv, const void *bias, const int32_t *cu_seqlens,
                                        const int32_t *start_pos, const int32_t *page_table,
                                        const sinkattn_rope_t *rope, void *q_out, void *k_pages,
                                        void *v_pages, const sinkattn_paged_dims_t *dims, void *stream);

/*
 * Causal (or full) prefill over packed variable-length sequences.
 * Source: "GPT-OSS on day 0", section "Kernels for GPT-OSS / Sink Attention"
 * (the same sink-aware kernel template serves prefill and decode).
 *
 *   q          [T, Hq, 64]   bf16   query rows of all sequences, packed
 *   k, v       [T, Hkv, 64]  bf16   keys / values, packed the same way
 *   cu_seqlens [N+1]         int32  sequence n is rows cu_seqlens[n] .. cu_seqlens[n+1]-1;
 *                                   cu_seqlens[0] = 0, non-decreasing, cu_seqlens[N] = T
 *   sinks      [Hq]          f32
 *   causal     1: row i of a sequence sees keys 0..i of that sequence;
 *              0: it sees the whole sequence
 *   out        [T, Hq, 64]   bf16
 *   lse        [T, Hq]       f32    natural log, or NULL
 *
 * A sequence longer than dims->max_seqlen is computed only up to
 * max_seqlen rows; its remaining rows are left untouched and
 * SINKATTN_ERR_BAD_LENGTH is raised in the error word.
 */
sinkattn_status_t sinkattn_prefill(const void *q, const void *k, const void *v,
                                   const int32_t *cu_seqlens, const float *sinks, float scale,
                                   int32_t causal, void *out, float *lse,
                                   const sinkattn_prefill_dims_t *dims, void *stream);

/*
 * Log-sum-exp merge of split partial results.
 * Source: "GPT-OSS on day 0", section "Kernels for GPT-OSS / Sink Attention"
 * (when attention is split into blocks along the sequence, the sink belongs to
 * one block only).
 *
 *   partial_o   [S, R, H, 64] f32   o_c = normalised output of split c
 *   partial_lse [S, R, H]     f32   natural-log lse_c of split c; -inf marks an
 *                                   empty split (its o_c is ignored)
 *   sinks       [H] f32, or NULL.  NULL: the sink is already inside one split.
 *               Given: the splits hold no sink and the merge adds exp(sink[h])
 *               exactly once.
 *   out         [R, H, 64]    bf16  sum_c exp(lse_c - L) o_c
 *   lse         [R, H]        f32   L = log(sum_c exp(lse_c) [+ exp(sink[h])]), or NULL
 * A row with no live split and no sink gives out = 0 and lse = -inf.
 */
sinkattn_status_t sinkattn_merge(const float *partial_o, const float *partial_lse,
                                 const float *sinks, void *out, float *lse,
                                 const sinkattn_merge_dims_t *dims, void *stream);

/*
 * sinkattn_decode without a workspace argument, for callers that cannot
 * allocate device memory: a framework that has reserved the whole device for
 * its own pool, a plugin interface that passes only input and output buffers,
 * or a serving loop that must not call cudaMalloc / cudaFree because they can
 * synchronise the device.  The blog posts describing the method have no
 * counterpart to this call; it is a deployment convenience.
 *
 * Arguments, layouts and results are those of sinkattn_decode.  The split-KV
 * scratch lives in a fixed array inside the library, of
 * SINKATTN_DECODE_NOALLOC_SCRATCH_BYTES, held by every device that loads the
 * library until the process exits.  The call allocates and frees nothing.
 *   - A problem needing more scratch than that (see
 *     sinkattn_decode_workspace_size) returns SINKATTN_ERR_WORKSPACE and
 *     launches nothing.
 *   - The first call on a device looks up the array's device address; make it
 *     before any stream capture begins.
 *   - Every call shares the one array, which keeps the last call's contents;
 *     no value in it needs to start at zero.  Calls that can overlap on the
 *     GPU race on the array: order them (one stream, or events).
 */
#define SINKATTN_DECODE_NOALLOC_SCRATCH_BYTES (16u << 20)
sinkattn_status_t sinkattn_decode_noalloc(const void *q, const void *k_pages, const void *v_pages,
                                          const int32_t *page_table, const int32_t *kv_lens,
                                          const float *sinks, float scale, void *out, float *lse,
                                          const sinkattn_decode_dims_t *dims, void *stream);

/*
 * Takes and clears the current device's error word in one atomic step ordered
 * on `stream` (after everything enqueued on it before), synchronises `stream`
 * and returns what it took (SINKATTN_OK when no kernel reported a problem).
 * If several problems were recorded, the one with the lowest status code is
 * returned.  A problem raised by a kernel on another stream after the step
 * stays in the word for the next call.
 */
sinkattn_status_t sinkattn_get_error(void *stream);

/*
 * Diagnostic for the failure path of the kernels' bounded waits (not for the hot path): enqueues on
 * `stream` one thread that waits, with the same bounded wait as every pipeline stage of the
 * attention kernels, on an mbarrier that nothing completes.  The wait gives up after its poll limit
 * (seconds) and raises SINKATTN_ERR_TIMEOUT in the device error word -- read it with
 * sinkattn_get_error -- and the kernel returns: no trap, and the context stays usable.  Returns
 * the status of the launch itself.
 */
sinkattn_status_t sinkattn_selftest_wait_timeout(void *stream);

/* Static English text for a status code. */
const char *sinkattn_status_string(sinkattn_status_t status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t sinkattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SINKATTN_H_ */
