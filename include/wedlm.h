/*
 * wedlm.h — C ABI of libwedlm: one WeDLM window decode step on one GB300.
 *
 * The operation is the inference step of "WeDLM: Reconciling Diffusion
 * Language Models with Standard Causal Attention for Fast Inference"
 * (bud-325 summary page, Method section; Key claims §3.2, §4.1, §5.2):
 * reorder the W-slot window so observed tokens come first (RoPE keeps each
 * token's logical position), run a causal forward of the window on top of
 * the cached, paged prefix KV, score every masked slot by the entropy of its
 * softmax, pick slots to fill with the distance-penalised entropy
 * H~_j = H_j + alpha * d_j (Eq. 11), commit the leftmost contiguous observed
 * run into the KV cache and refill the freed slots with [M].
 *
 * Conventions for every entry point
 *  - Pointers marked "device" are CUDA device pointers on the current device;
 *    "host" pointers are read during the call only.  The caller owns every
 *    buffer passed in; the library owns only its workspace (sized at
 *    wedlm_create) and its cached CUDA graphs.
 *  - `stream` is a cudaStream_t (passed as void*); work is enqueued on it and
 *    the call returns without synchronising.  Inputs and outputs of one call
 *    must not alias, except `seq_len`, which is updated in place.
 *  - Calls that share one context must not run concurrently (the workspace
 *    is shared).
 *  - Return value: WEDLM_OK or an error code; wedlm_last_error() gives a
 *    message.  Errors found on the device (bad page id, capacity, token out
 *    of range, non-finite scores) set bits of a device error word that
 *    wedlm_get_status() reads; the kernels skip the offending access.
 *  - Matrices are row-major.  Linear weights are [out_features][in_features].
 *  - Element type of weights, activations and KV pools is the context's
 *    dtype: WEDLM_BF16 (bfloat16, fp32 accumulation) or WEDLM_FP32.
 *
 * Paged KV pool (one per layer): `num_pages` pages, each
 * [2 (K, V)][n_kv_heads][page_block tokens][head_dim] values.  Inside one
 * (page, K|V, kv-head) block of page_block*head_dim values, element
 * (token t, dim d) is at ((t/8)*(head_dim/8) + d/8)*64 + (t%8)*8 + d%8:
 * 8x8 tiles ordered token-group-major.  This is the layout the tensor-core
 * attention consumes directly.  page_table[b][j] is the page holding
 * positions 16j..16j+15 of sequence b.  K is stored after RoPE.  Positions
 * at or beyond seq_len inside a sequence's last page must hold finite values
 * (zeros, say): the attention multiplies them by zero probabilities.
 *
 * Supported shapes: head_dim 64 or 128 (fp32) / 128 (bf16); window <= 64;
 * max_batch * window <= 512; bf16: G * window <= 128 or G divides 128
 * (G = n_q_heads / n_kv_heads; the G * W query rows of a kv head run in
 * blocks of 128 on the tensor cores); fp32: G * window <= 512.
 */
#ifndef WEDLM_H
#define WEDLM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  WEDLM_OK = 0,
  WEDLM_ERR_INVALID_ARG = 1, /* null/misaligned pointer, size out of range  */
  WEDLM_ERR_CAPACITY = 2,    /* page table cannot hold seq_len + W          */
  WEDLM_ERR_CUDA = 3,        /* a CUDA call or launch failed                */
  WEDLM_ERR_NUMERIC = 4,     /* non-finite softmax statistics               */
  WEDLM_ERR_TIMEOUT = 5,     /* a bounded device wait expired               */
  WEDLM_ERR_DEVICE = 6       /* device error word non-zero (see bits)       */
};

/* bits of the device error word */
enum {
  WEDLM_DEV_BAD_PAGE = 1,     /* page id outside [0, num_pages)             */
  WEDLM_DEV_CAPACITY = 2,     /* seq_len + W beyond the page table          */
  WEDLM_DEV_BAD_TOKEN = 4,    /* token id outside [0, vocab)                */
  WEDLM_DEV_NUMERIC = 8,      /* non-finite lse / entropy                   */
  WEDLM_DEV_TIMEOUT = 16,     /* bounded mbarrier / flag wait expired       */
  WEDLM_DEV_BAD_SEQLEN = 32   /* negative seq_len                           */
};

enum { WEDLM_BF16 = 0, WEDLM_FP32 = 1 };

/* Score of a masked slot in Eq. 11 (H~_j = score_j + alpha * d_j):
 * the entropy of its softmax (the Method section's formula), or the
 * confidence reading of the rule (Key claims §5.2, "distance-penalized
 * confidence rule"): -ln p_max. */
enum { WEDLM_SCORE_ENTROPY = 0, WEDLM_SCORE_NEGLOGP = 1 };

typedef struct wedlm_ctx wedlm_ctx;

/* Model and capacity, fixed at create time. */
typedef struct wedlm_config {
  int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  int32_t window;            /* W, slots per sequence (1..64)               */
  int32_t page_block;        /* tokens per page; must be 16                 */
  int32_t max_batch;         /* B_max; B_max * W <= 512                     */
  int32_t max_pages_per_seq; /* columns of page_table                       */
  int32_t dtype;             /* WEDLM_BF16 | WEDLM_FP32                     */
  int32_t qk_norm;           /* 1: per-head RMSNorm on q and k before RoPE  */
  int32_t mask_id;           /* token id of [M]                             */
  float rope_theta, rms_eps;
} wedlm_config;

/* Device pointers to the weights (dtype of the context).  Per-layer fields
 * are HOST arrays of n_layers device pointers; they are copied at create.
 * q_norm / k_norm may be NULL when qk_norm = 0.  The weights must stay alive
 * and unchanged for the context's lifetime. */
typedef struct wedlm_weights {
  const void *embed;      /* [vocab][hidden]                                */
  const void *final_norm; /* [hidden]                                       */
  const void *lm_head;    /* [vocab][hidden] (untied)                       */
  const void *const *attn_norm; /* [hidden]                                 */
  const void *const *w_q;       /* [n_q_heads*head_dim][hidden]             */
  const void *const *w_k;       /* [n_kv_heads*head_dim][hidden]            */
  const void *const *w_v;       /* [n_kv_heads*head_dim][hidden]            */
  const void *const *q_norm;    /* [head_dim]                               */
  const void *const *k_norm;    /* [head_dim]                               */
  const void *const *w_o;       /* [hidden][n_q_heads*head_dim]             */
  const void *const *ffn_norm;  /* [hidden]                                 */
  const void *const *w_gate;    /* [ffn][hidden]                            */
  const void *const *w_up;      /* [ffn][hidden]                            */
  const void *const *w_down;    /* [hidden][ffn]                            */
} wedlm_weights;

/* Per-row softmax statistics of one window row (LM-head output). */
typedef struct wedlm_slot_rec {
  int32_t argmax;  /* token id with the largest logit (lowest id on ties)  */
  float entropy;   /* H = -sum p ln p, nats                                 */
  float p_max;     /* probability of argmax                                 */
  float lse;       /* log-sum-exp of the logits                             */
} wedlm_slot_rec;

/* Inputs of one step (all device pointers unless noted). */
typedef struct wedlm_step_in {
  int32_t batch;               /* B, 1..max_batch                          */
  int32_t num_pages;           /* pages in each layer's pool               */
  const int32_t *tokens;       /* [B][W] token ids; masked slots hold [M]  */
  const int32_t *pos;          /* [B][W] logical positions                 */
  const uint8_t *observed;     /* [B][W] 1 = observed, 0 = masked          */
  int32_t *seq_len;            /* [B] committed length; += n_committed     */
  const int32_t *page_table;   /* [B][max_pages_per_seq]                   */
  void *const *kv_pools;       /* HOST array of n_layers device pools      */
  const int32_t *plant_token;  /* [B][W] token to bias per slot (-1: none), or NULL */
  float plant_bias;            /* added to that token's logit              */
  float alpha, tau;            /* Eq. 11 distance weight and threshold     */
  int32_t score_mode;          /* WEDLM_SCORE_ENTROPY | WEDLM_SCORE_NEGLOGP */
} wedlm_step_in;

/* Outputs of one step (device pointers; optional ones may be NULL). */
typedef struct wedlm_step_out {
  int32_t *new_tokens;         /* [B][W] window after fill/commit/refill   */
  int32_t *new_pos;            /* [B][W]                                   */
  uint8_t *new_observed;       /* [B][W]                                   */
  int32_t *committed;          /* [B][W] committed ids, -1 after the run   */
  int32_t *n_committed;        /* [B]                                      */
  int32_t *perm;               /* [B][W] slot at each physical index, or NULL */
  uint8_t *filled;             /* [B][W] 1 where a slot was filled, or NULL */
  wedlm_slot_rec *rows;        /* [B*W] per PHYSICAL row, or NULL.  The LM
                                  head runs on the masked rows only: an
                                  observed row's record is argmax -1 and
                                  NaN statistics                           */
  float *logits;               /* [B*W][vocab] fp32 per physical row, or NULL
                                  (debug: materialises the logits of the
                                  masked rows; observed rows are not written) */
  void *hidden;                /* [B*W][hidden] final residual stream, or NULL */
} wedlm_step_out;

/* Create a context: validates the config, copies the weight pointers,
 * allocates the workspace (window K/V scratch, activations, split-K and
 * split-KV partials, error word) and builds TMA descriptors.
 * Returns WEDLM_ERR_INVALID_ARG for unsupported shapes. */
int wedlm_create(const wedlm_config *cfg, const wedlm_weights *w,
                 wedlm_ctx **out);

void wedlm_destroy(wedlm_ctx *ctx);

/* Message for the last error on this context (never NULL). */
const char *wedlm_last_error(wedlm_ctx *ctx);

/* Synchronises the stream of the last call, returns the device error word
 * in *device_error (may be NULL) and clears it.  Returns WEDLM_ERR_DEVICE
 * when the word was non-zero. */
int wedlm_get_status(wedlm_ctx *ctx, int32_t *device_error);

/* 1 = launch each step through a cached CUDA graph (default), 0 = eager.
 * Graphs are keyed by every pointer and scalar of the call. */
int wedlm_set_graphs(wedlm_ctx *ctx, int enable);

/* Per-kernel timing with CUDA events (forces eager launches while on).
 * wedlm_get_timings synchronises and writes, for each of `n` kernel kinds
 * (see WEDLM_KIND_*), the summed milliseconds and launch counts since the
 * last reset, then resets them. */
enum {
  WEDLM_KIND_REORDER = 0, WEDLM_KIND_RMSNORM, WEDLM_KIND_GEMM_QKV,
  WEDLM_KIND_ATTN, WEDLM_KIND_ATTN_MERGE, WEDLM_KIND_GEMM_O,
  WEDLM_KIND_GEMM_GATEUP, WEDLM_KIND_GEMM_DOWN, WEDLM_KIND_LMHEAD,
  WEDLM_KIND_LMHEAD_MERGE, WEDLM_KIND_SELECT, WEDLM_KIND_COMMIT,
  WEDLM_KIND_COUNT
};
int wedlm_set_timing(wedlm_ctx *ctx, int enable);
int wedlm_get_timings(wedlm_ctx *ctx, float *ms, int32_t *launches, int n);

/* Number of kernels the most recent wedlm_step enqueued (counted while it
 * was enqueued or captured; -1 before the first step).  `batch` is unused. */
int wedlm_launches_per_step(wedlm_ctx *ctx, int32_t batch);

/* ---- the whole step (rows a1..a7) ------------------------------------- */
int wedlm_step(wedlm_ctx *ctx, const wedlm_step_in *in, wedlm_step_out *out,
               void *stream);

/* ---- prompt prefill and the streaming loop ------------------------------ */

/* Prompt prefill (bud-325 summary page, Method: the decoder runs "on top of
 * the persistent KV cache"): a causal forward of `chunk` prompt tokens per
 * sequence, at logical positions seq_len[b] .. seq_len[b]+chunk-1, on top of
 * each sequence's cached prefix; the K/V of every token of every layer are
 * written to the pages, and seq_len[b] += chunk.  This is the window step
 * with every slot observed and no selection.  tokens: [B][chunk] device;
 * hidden: [B*chunk][hidden] final residual stream, or NULL.  Limits: B *
 * chunk <= max_batch * window (the workspace rows) and B * (chunk rounded
 * up to 16) <= max_batch * (window rounded up to 16); the attention limit on
 * G * chunk as above.  Returns WEDLM_ERR_INVALID_ARG beyond them. */
int wedlm_prefill(wedlm_ctx *ctx, int32_t batch, int32_t chunk, const int32_t *tokens,
                  int32_t *seq_len, const int32_t *page_table, int32_t num_pages,
                  void *const *kv_pools, void *hidden, void *stream);

/* The streaming decode loop on the device (Key claims §5.2 and Method:
 * reorder, forward, commit, select, refill, step after step, with a fixed
 * window).  One call enqueues a CUDA graph whose conditional while-node
 * runs the whole step (as wedlm_step) until `max_steps` steps have run or
 * every sequence has stopped; no host round trip between steps.  The window
 * arrays are updated in place.  Per sequence: a stopped sequence (done[b]
 * = 1) is left unchanged; a sequence stops once its seq_len reaches
 * stop_len[b] or after committing `stop_token`.  Committed tokens are
 * written to out_tokens[b][p - out_base[b]] for logical position p when
 * that index is in [0, out_cap).  All pointers are device pointers except
 * kv_pools (host array of n_layers device pools). */
typedef struct wedlm_gen_in {
  int32_t batch;               /* B, 1..max_batch                          */
  int32_t num_pages;           /* pages in each layer's pool               */
  int32_t *tokens;             /* [B][W] window, updated in place          */
  int32_t *pos;                /* [B][W]                                   */
  uint8_t *observed;           /* [B][W]                                   */
  int32_t *seq_len;            /* [B] committed length, advanced in place  */
  const int32_t *page_table;   /* [B][max_pages_per_seq]                   */
  void *const *kv_pools;       /* HOST array of n_layers device pools      */
  const int32_t *plant_token;  /* [B][W] or NULL (as in wedlm_step_in)     */
  float plant_bias;
  float alpha, tau;            /* Eq. 11 distance weight and threshold     */
  int32_t score_mode;          /* WEDLM_SCORE_*                            */
  int32_t max_steps;           /* the loop runs at most this many steps    */
  int32_t *done;               /* [B] stop flags, read and updated         */
  const int32_t *stop_len;     /* [B] length budget, or NULL               */
  int32_t stop_token;          /* token id that stops a sequence, -1: none */
  int32_t *out_tokens;         /* [B][out_cap] committed ids, or NULL      */
  const int32_t *out_base;     /* [B] position of out_tokens[b][0]         */
  int32_t out_cap;
  int32_t *steps_run;          /* [1] steps the loop ran, or NULL          */
} wedlm_gen_in;
int wedlm_generate(wedlm_ctx *ctx, const wedlm_gen_in *in, void *stream);

/* ---- Dual-Stream Masking attention (training-time mask) ------------------ */

/* Attention under Dual-Stream Masking (bud-325 summary page, Key claims
 * §4.2, Eq. 8-10; Method): a clean memory stream of n tokens at logical
 * positions 0..n-1 and a prediction stream over the same n positions, cut
 * into blocks of `block` tokens, each block topologically reordered
 * (observed tokens first) with its tokens keeping their logical positions.
 * A memory row attends causally to the memory stream; a prediction row of
 * block j attends to the memory tokens at positions before the block
 * (0..j*block-1) and, causally in the block's physical order, to its own
 * block.  Each block of either stream runs as one sequence of the paged
 * window attention with prefix = the memory positions before the block.
 *  q:        [2][n][n_q_heads][head_dim] bf16: memory rows, then prediction
 *            rows (physical order inside each block); RoPE applied;
 *  mem_pool: the memory stream's K/V as n/16 pages in order (page p holds
 *            positions 16p..16p+15; the paged layout above, K after RoPE);
 *  win:      [2][n/block][2 (K, V)][n_kv_heads][block][head_dim] bf16 in the
 *            page tile layout: every block's own K/V, memory blocks first;
 *  o:        [2][n][n_q_heads*head_dim] bf16.
 * block a multiple of 16 dividing n; bf16 contexts only.  The partials use
 * the context's attention workspace: shapes it cannot hold (2n/block
 * blocks x n_kv_heads x row blocks units) return WEDLM_ERR_CAPACITY. */
int wedlm_dual_stream_attention(wedlm_ctx *ctx, int32_t n, int32_t block, const void *q,
                                const void *mem_pool, const void *win, void *o,
                                void *stream);

/* ---- one row of the step each (tests and composition) ------------------ */

/* Topological Reordering + embedding gather (Key claims §4.1).
 * perm/inv: [B][W] int32 (device, may be NULL); x_out: [B*W][hidden] in the
 * physical order; pos_phys: [B*W] logical position of each physical row
 * (may be NULL). */
int wedlm_reorder_embed(wedlm_ctx *ctx, int32_t batch, const int32_t *tokens,
                        const int32_t *pos, const uint8_t *observed,
                        int32_t *perm, int32_t *inv, void *x_out,
                        int32_t *pos_phys, void *stream);

/* One decoder layer over the window rows (pre-attention projections with
 * RoPE at logical positions, paged causal window attention, O projection,
 * SwiGLU FFN, residuals).  x: [B*W][hidden] (physical order), updated in
 * place; pos_phys: [B*W]; seq_len: [B] (read only); kv_pool: this layer's
 * pool.  kv_win_out: [B][2][n_kv][Wp][head_dim] in the page tile layout
 * (Wp = W rounded up to 16) receives this layer's window K/V, or NULL.
 * q_out: [B*W][n_q*head_dim], attn_out: [B*W][n_q*head_dim], or NULL. */
int wedlm_layer(wedlm_ctx *ctx, int32_t layer, int32_t batch, void *x,
                const int32_t *pos_phys, const int32_t *seq_len,
                const int32_t *page_table, int32_t num_pages,
                const void *kv_pool, void *kv_win_out, void *q_out,
                void *attn_out, void *stream);

/* Paged causal GQA window attention alone (Key claims §3.2, §5.2).
 * q: [B*W][n_q][head_dim] (RoPE applied); kv_win: [B][2][n_kv][Wp][hd]
 * tile layout; o: [B*W][n_q*head_dim].  Query row p of sequence b sees
 * prefix positions 0..seq_len[b]-1 and window rows 0..p. */
int wedlm_attention(wedlm_ctx *ctx, int32_t batch, const void *q,
                    const void *kv_pool, const int32_t *page_table,
                    const int32_t *seq_len, int32_t num_pages,
                    const void *kv_win, void *o, void *stream);

/* Final RMSNorm + LM head + streaming softmax statistics per row.
 * x: [B*W][hidden]; plant_token: [B*W] per physical row or NULL;
 * rows: [B*W] out; logits: [B*W][vocab] fp32 or NULL. */
int wedlm_lm_head(wedlm_ctx *ctx, int32_t batch, const void *x,
                  const int32_t *plant_token, float plant_bias,
                  wedlm_slot_rec *rows, float *logits, void *stream);

/* ---- attention without any device allocation --------------------------- */

/* Paged causal GQA window attention (bf16, head_dim 128) for callers that
 * cannot allocate device memory: code that runs where cudaMalloc is not
 * allowed or not wanted, such as inside a host framework that owns every
 * allocation, a memory-capped service, or a setting where an allocation
 * could stall or fail mid-run.  The WeDLM pages have no counterpart for this
 * entry point; it computes the same result as wedlm_attention (same argument
 * meanings and layouts, no context needed) but keeps its split-KV partials,
 * zero page and error word in one file-scope device array of 16 MiB, which
 * every GPU that loads this library holds until the process exits.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and zeroes its zero page; make that first call
 *    before any stream capture.
 *  - Sizes whose partials do not fit in the array ((SM count + batch *
 *    n_kv_heads) segments of (n_q_heads/n_kv_heads*window) rows x 130 floats,
 *    plus a small table) return WEDLM_ERR_CAPACITY; bad arguments
 *    WEDLM_ERR_INVALID_ARG.
 *  - Every call shares the array and it keeps the last call's contents:
 *    calls that overlap on the GPU (other streams, other threads) race.
 *  - Nothing found on the device makes the call fail: page ids outside
 *    [0, num_pages) read as zeros, and a bounded wait that expires (2 s)
 *    leaves the output partly written.  Both set bits of an error word in
 *    the array, cleared at the start of every call and read back by
 *    wedlm_attention_static_status.
 *  - q, kv_pool, kv_win and o must be 16-byte aligned; n_q_heads a positive
 *    multiple of n_kv_heads.
 *  - Calls no cudaMalloc, cudaFree or allocating library routine. */
int wedlm_attention_static(int32_t batch, int32_t window, int32_t n_q_heads,
                           int32_t n_kv_heads, int32_t max_pages_per_seq,
                           int32_t num_pages, const void *q, const void *kv_pool,
                           const int32_t *page_table, const int32_t *seq_len,
                           const void *kv_win, void *o, void *stream);

/* The device error word of the last wedlm_attention_static call on the
 * current device: WEDLM_DEV_* bits (WEDLM_DEV_BAD_PAGE for a page id outside
 * [0, num_pages), WEDLM_DEV_TIMEOUT for a bounded wait that expired), 0 when
 * the call found nothing or no call has run on this device.  Waits for
 * `stream` (the stream the call was issued on) and copies 4 bytes to the
 * host; allocates nothing.  device_error: host pointer, written on success.
 * Returns WEDLM_ERR_INVALID_ARG for a null pointer, WEDLM_ERR_CUDA if the
 * copy or the wait fails. */
int wedlm_attention_static_status(void *stream, int32_t *device_error);

/* ---- failure detection self-test ---------------------------------------- */

/* Self-test of the bounded waits every kernel uses (failure detection
 * without a GPU fault).  One thread waits on a shared-memory barrier that
 * nothing completes; after the wait limit (2 s) the wait gives up, sets
 * WEDLM_DEV_TIMEOUT in an error word and the kernel returns, leaving the CUDA
 * context usable.  Not part of WeDLM; a diagnostic of this library.
 *  - word: device int32[2], caller-owned, 4-byte aligned; cleared here, then
 *    word[0] receives the error bits and word[1] 1 if the wait gave up (2 if
 *    the barrier completed, which nothing makes happen).
 *  - device_error, gave_up: host pointers, receive word[0] and word[1].
 * Synchronises `stream` (about 2 s).  Returns WEDLM_ERR_INVALID_ARG for null
 * or misaligned pointers, WEDLM_ERR_CUDA if the launch, copy or wait fails. */
int wedlm_selftest_bounded_wait(int32_t *word, int32_t *device_error, int32_t *gave_up,
                                void *stream);

#ifdef __cplusplus
}
#endif
#endif /* WEDLM_H */
