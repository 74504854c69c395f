// libwedlm C ABI: context, workspace, step orchestration, CUDA graphs and
// per-kernel timing.  See include/wedlm.h for the contract of each call.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <memory>
#include <string>
#include <type_traits>
#include <vector>

#include "gemm_tc.h"
#include "internal.h"

using namespace wedlm;

namespace {

struct GraphEntry {
  std::vector<uint64_t> key;
  cudaGraphExec_t exec = nullptr;
  uint64_t last_use = 0;
};

constexpr int kMaxGraphs = 4;
constexpr int kMaxEvents = 8192;
constexpr int kDualMaxBlocks = 512;   // blocks of both streams (sequences of one launch)
constexpr int kDualMaxPages = 4096;   // memory stream of up to 65536 tokens

}  // namespace

struct wedlm_ctx {
  wedlm_config cfg{};
  int es = 2;                 // element size
  int Wp = 16;                // window rounded up to a page
  int M_max = 0;
  int num_sms = 0;
  int device = 0;
  const void* embed = nullptr;
  const void* final_norm = nullptr;
  const void* lm_head = nullptr;
  std::vector<LayerWeights> layers;
  // workspace
  std::vector<void*> allocs;
  int* err = nullptr;
  int32_t *perm = nullptr, *inv = nullptr, *pos_phys = nullptr,
          *seq_snap = nullptr, *plant_phys = nullptr, *ncommit = nullptr;
  double* inv_freq = nullptr;
  float *cosb = nullptr, *sinb = nullptr;
  void *x = nullptr, *xn = nullptr, *q = nullptr, *o = nullptr, *act = nullptr;
  void* kv_win = nullptr;
  size_t win_layer_stride = 0;  // elements
  float *attn_o = nullptr, *attn_ml = nullptr;
  int attn_chunk = 0, attn_max_chunks = 0;
  int* attn_unit_cnt = nullptr;   // tensor-core attention: segment counts per unit
  size_t attn_units_cap = 0;      // units the counters and partials are sized for
  int* gen_ctrl = nullptr;        // streaming loop: [0] steps left, [1] steps run
  int32_t *gen_committed = nullptr, *gen_ncommitted = nullptr;  // its per-step outputs
  size_t attn_part_rows = 0;      // rows of partial O the attention may use
  int32_t *dual_len = nullptr, *dual_pt = nullptr;  // dual-stream block lengths, page row
  float* gemm_part = nullptr;
  size_t gemm_part_elems = 0;
  int* gemm_counters = nullptr;
  int vtiles = 0;
  SoftmaxPart* lm_part = nullptr;
  wedlm_slot_rec* rows = nullptr;  // LM-head records, compact (masked rows only)
  int32_t *lm_src = nullptr, *lm_dst = nullptr, *lm_plant = nullptr;  // MaskedRows
  int* lm_count = nullptr;
  void* zero_page = nullptr;  // 4 KiB of zeros: stands in for missing KV pages
  // tensor-core GEMM plans (bf16 contexts)
  std::unique_ptr<TcPlanSet> tc;
  // runtime state
  cudaStream_t last_stream = nullptr;
  cudaStream_t cap_stream = nullptr;
  std::string last_error = "ok";
  bool use_graphs = true;
  std::vector<GraphEntry> graphs;
  std::vector<GraphEntry> gen_graphs;  // streaming loops (conditional while node)
  uint64_t graph_clock = 0;
  // timing
  bool timing = false;
  std::vector<cudaEvent_t> ev;
  std::vector<int> ev_kind;
  int ev_used = 0;
  double kind_ms[WEDLM_KIND_COUNT] = {};
  int kind_launches[WEDLM_KIND_COUNT] = {};
  // kernels enqueued by the current / last complete step
  int launch_count = 0;
  int last_step_launches = -1;
};

namespace {

int fail(wedlm_ctx* c, int code, const std::string& msg) {
  if (c) c->last_error = msg;
  return code;
}

#define CUDA_TRY(c, expr)                                                     \
  do {                                                                        \
    cudaError_t _e = (expr);                                                  \
    if (_e != cudaSuccess)                                                    \
      return fail((c), WEDLM_ERR_CUDA,                                        \
                  std::string(#expr) + ": " + cudaGetErrorString(_e));        \
  } while (0)

template <typename P>
cudaError_t walloc(wedlm_ctx* c, P** p, size_t bytes) {
  void* v = nullptr;
  cudaError_t e = cudaMalloc(&v, std::max<size_t>(bytes, 256));
  if (e != cudaSuccess) return e;
  c->allocs.push_back(v);
  *p = static_cast<P*>(v);
  return cudaMemset(v, 0, std::max<size_t>(bytes, 256));
}

// timing helpers: an event pair around each launch of a kernel kind
struct Timed {
  wedlm_ctx* c;
  int kind;
  cudaStream_t st;
  int slot = -1;
  Timed(wedlm_ctx* c_, int k, cudaStream_t s) : c(c_), kind(k), st(s) {
    if (c->timing && c->ev_used + 2 <= kMaxEvents) {
      slot = c->ev_used;
      c->ev_used += 2;
      c->ev_kind[slot] = kind;
      cudaEventRecord(c->ev[slot], st);
    }
  }
  ~Timed() {
    if (slot >= 0) cudaEventRecord(c->ev[slot + 1], st);
  }
};

int choose_splits(const wedlm_ctx* c, int tiles, int M, int N, int K, int kblk) {
  const int target = 2 * c->num_sms;
  int s = std::max(1, target / std::max(1, tiles));
  s = std::min(s, std::max(1, K / (kblk * 4)));
  while (s > 1 && (size_t)s * M * N > c->gemm_part_elems) --s;
  return s;
}

template <typename T>
int run_gemm(wedlm_ctx* c, GemmProblem P, int kind, cudaStream_t st,
             int* tiles_out = nullptr) {
  const int tiles = P.swiglu ? P.N / 128 : (P.N + 127) / 128;
  if (tiles_out) *tiles_out = tiles;
  P.partial = c->gemm_part;
  P.counters = c->gemm_counters;
  P.err = c->err;
  cudaError_t e;
  {
    Timed t(c, kind, st);
    if (c->cfg.dtype == WEDLM_BF16) {
      int nl = 1;
      e = launch_gemm_tc(*c->tc, P, kind, st, tiles_out, &nl);
      c->launch_count += nl;
    } else {
      P.splits = choose_splits(c, tiles, P.M, P.N, P.K, 16);
      e = launch_gemm_simt<T>(P, st);
      c->launch_count += 1;
    }
  }
  if (e != cudaSuccess)
    return fail(c, WEDLM_ERR_CUDA, std::string("gemm launch: ") + cudaGetErrorString(e));
  return WEDLM_OK;
}

#define LAUNCH(c, kind, st, expr)                                             \
  do {                                                                        \
    cudaError_t _e;                                                           \
    {                                                                         \
      Timed _t((c), (kind), (st));                                            \
      _e = (expr);                                                            \
      (c)->launch_count += 1;                                                 \
    }                                                                         \
    if (_e != cudaSuccess)                                                    \
      return fail((c), WEDLM_ERR_CUDA,                                        \
                  std::string(#kind) + ": " + cudaGetErrorString(_e));        \
  } while (0)

// fp32 contexts: CUDA-core attention; bf16: tensor-core attention
template <typename T>
cudaError_t run_attention(wedlm_ctx* c, const AttnArgs& A, cudaStream_t st);
template <>
cudaError_t run_attention<float>(wedlm_ctx*, const AttnArgs& A, cudaStream_t st) {
  return launch_attention<float>(A, st);
}
template <>
cudaError_t run_attention<bf16>(wedlm_ctx* c, const AttnArgs& A, cudaStream_t st) {
  return launch_attention_tc(A, c->zero_page, c->num_sms, st);
}

// Rows of one sequence in a call: the decode window (W slots) or a prefill
// chunk; Wp = W rounded up to a page.
struct Win {
  int W, Wp;
};
Win ctx_win(const wedlm_ctx* c) { return Win{c->cfg.window, c->Wp}; }
Win chunk_win(int chunk) { return Win{chunk, (chunk + kPageBlock - 1) / kPageBlock * kPageBlock}; }

// Commit of the window rows of a call into the paged cache (QKV epilogue):
// per sequence, rows 0..n[b]-1 go to positions base[b]..; n == null: none.
struct Commit {
  const int32_t* n = nullptr;
  const int32_t* base = nullptr;
  const int32_t* page_table = nullptr;
  int num_pages = 0;
};

AttnArgs attn_args(wedlm_ctx* c, int B, Win win, const void* q, const void* pool,
                   const int32_t* page_table, const int32_t* seq_len,
                   int num_pages, const void* kv_win, void* o) {
  const wedlm_config& g = c->cfg;
  AttnArgs A{};
  A.B = B; A.W = win.W; A.Wp = win.Wp; A.nq = g.n_q_heads; A.nkv = g.n_kv_heads;
  A.hd = g.head_dim; A.chunk = c->attn_chunk; A.max_chunks = c->attn_max_chunks;
  A.num_pages = num_pages; A.max_pages = g.max_pages_per_seq; A.pt_stride = g.max_pages_per_seq;
  A.scale_log2 = (float)(1.4426950408889634 / sqrt((double)g.head_dim));
  A.q = q; A.pool = pool; A.page_table = page_table; A.seq_len = seq_len;
  A.kv_win = kv_win; A.part_o = c->attn_o; A.part_ml = c->attn_ml; A.o = o;
  A.err = c->err;
  A.min_tiles = 2;
  A.unit_cost = kAttnUnitCost;
  A.unit_cnt = c->attn_unit_cnt;
  return A;
}

// The four projections of layer l on workspace activations (M rows).
GemmProblem qkv_problem(wedlm_ctx* c, int l, int M, Win win, void* kv_win_layer,
                        const Commit& cm, void* pool) {
  const wedlm_config& g = c->cfg;
  const LayerWeights& w = c->layers[l];
  const int nq = g.n_q_heads, nkv = g.n_kv_heads, hd = g.head_dim;
  GemmProblem P{};
  P.M = M; P.N = (nq + 2 * nkv) * hd; P.K = g.hidden; P.X = c->xn;
  P.A0 = w.w_q; P.A1 = w.w_k; P.A2 = w.w_v;
  P.seg1 = nq * hd; P.seg2 = (nq + nkv) * hd; P.swiglu = 0;
  GemmEpi& e = P.epi;
  e.mode = EPI_QKV; e.q_out = c->q; e.kv_win = kv_win_layer;
  e.cosb = c->cosb; e.sinb = c->sinb; e.q_norm = w.q_norm; e.k_norm = w.k_norm;
  e.qk_norm = g.qk_norm; e.W = win.W; e.Wp = win.Wp; e.nq = nq; e.nkv = nkv;
  e.hd = hd; e.eps = g.rms_eps;
  e.commit_n = cm.n; e.commit_base = cm.base; e.page_table = cm.page_table;
  e.pool = pool; e.max_pages = g.max_pages_per_seq; e.num_pages = cm.num_pages;
  e.err = c->err;
  return P;
}
GemmProblem o_problem(wedlm_ctx* c, int l, int M, void* x, bool fuse) {
  const wedlm_config& g = c->cfg;
  const LayerWeights& w = c->layers[l];
  GemmProblem P{};
  P.M = M; P.N = g.hidden; P.K = g.n_q_heads * g.head_dim; P.X = c->o;
  P.A0 = w.w_o; P.A1 = w.w_o; P.A2 = w.w_o; P.seg1 = P.N; P.seg2 = P.N;
  P.epi.mode = EPI_RESID; P.epi.x = x;
  if (fuse) {  // residual add + the FFN norm in one epilogue
    P.epi.norm_w = w.ffn_norm; P.epi.xn = c->xn; P.epi.eps = g.rms_eps;
  }
  return P;
}
GemmProblem gateup_problem(wedlm_ctx* c, int l, int M) {
  const wedlm_config& g = c->cfg;
  const LayerWeights& w = c->layers[l];
  GemmProblem P{};
  P.M = M; P.N = 2 * g.ffn; P.K = g.hidden; P.X = c->xn;
  P.A0 = w.w_gate; P.A1 = w.w_up; P.A2 = w.w_up; P.seg1 = P.N; P.seg2 = P.N;
  P.swiglu = 1;
  P.epi.mode = EPI_SWIGLU; P.epi.act = c->act;
  return P;
}
GemmProblem down_problem(wedlm_ctx* c, int l, int M, void* x, const void* next_norm,
                         const int32_t* norm_row_dst = nullptr) {
  const wedlm_config& g = c->cfg;
  const LayerWeights& w = c->layers[l];
  GemmProblem P{};
  P.M = M; P.N = g.hidden; P.K = g.ffn; P.X = c->act;
  P.A0 = w.w_down; P.A1 = w.w_down; P.A2 = w.w_down; P.seg1 = P.N; P.seg2 = P.N;
  P.epi.mode = EPI_RESID; P.epi.x = x;
  if (next_norm) {
    P.epi.norm_w = next_norm; P.epi.xn = c->xn; P.epi.eps = g.rms_eps;
    P.epi.row_dst = norm_row_dst;
  }
  return P;
}
GemmProblem lmhead_problem(wedlm_ctx* c, int M) {
  const wedlm_config& g = c->cfg;
  GemmProblem P{};
  P.M = M; P.N = g.vocab; P.K = g.hidden; P.X = c->xn;
  P.A0 = c->lm_head; P.A1 = c->lm_head; P.A2 = c->lm_head;
  P.seg1 = g.vocab; P.seg2 = g.vocab;
  P.epi.mode = EPI_LMHEAD;
  return P;
}

// rows a2..a4 for one layer, on workspace activations.  xn_ready: xn
// already holds RMSNorm(x) with this layer's attention norm (written by the
// previous layer's down projection); next_norm: when set, the down
// projection's epilogue also writes xn = RMSNorm(x) with these weights (the
// next layer's attention norm or the final norm).  Both are used on the
// tensor-core path only, where the residual epilogue can fuse the norm.
template <typename T>
int layer_impl(wedlm_ctx* c, int l, int B, Win win, T* x, const int32_t* seq_len,
               const int32_t* page_table, int num_pages, const void* pool,
               void* kv_win_layer, cudaStream_t st, bool xn_ready = false,
               const void* next_norm = nullptr, const Commit& cm = Commit(),
               const int32_t* norm_row_dst = nullptr) {
  const wedlm_config& g = c->cfg;
  const LayerWeights& w = c->layers[l];
  const int M = B * win.W, H = g.hidden;
  const bool fuse = g.dtype == WEDLM_BF16;
  int rc;
  GemmProblem Pqkv = qkv_problem(c, l, M, win, kv_win_layer, cm, const_cast<void*>(pool));
  GemmProblem Po = o_problem(c, l, M, x, fuse);
  GemmProblem Pgu = gateup_problem(c, l, M);
  GemmProblem Pd = down_problem(c, l, M, x, fuse ? next_norm : nullptr, norm_row_dst);
  if (!xn_ready)
    LAUNCH(c, WEDLM_KIND_RMSNORM, st,
           launch_rmsnorm<T>(M, H, x, (const T*)w.attn_norm, g.rms_eps, (T*)c->xn, st));
  if ((rc = run_gemm<T>(c, Pqkv, WEDLM_KIND_GEMM_QKV, st))) return rc;
  AttnArgs A = attn_args(c, B, win, c->q, pool, page_table, seq_len, num_pages,
                         kv_win_layer, c->o);
  // bf16: tensor-core attention, one kernel (the segment merge is inside);
  // fp32: CUDA-core split-KV attention and its merge kernel
  LAUNCH(c, WEDLM_KIND_ATTN, st, run_attention<T>(c, A, st));
  if constexpr (std::is_same<T, float>::value)
    LAUNCH(c, WEDLM_KIND_ATTN_MERGE, st, launch_attention_merge<float>(A, st));
  if ((rc = run_gemm<T>(c, Po, WEDLM_KIND_GEMM_O, st))) return rc;
  if (!fuse)
    LAUNCH(c, WEDLM_KIND_RMSNORM, st,
           launch_rmsnorm<T>(M, H, x, (const T*)w.ffn_norm, g.rms_eps, (T*)c->xn, st));
  if ((rc = run_gemm<T>(c, Pgu, WEDLM_KIND_GEMM_GATEUP, st))) return rc;
  if ((rc = run_gemm<T>(c, Pd, WEDLM_KIND_GEMM_DOWN, st))) return rc;
  return WEDLM_OK;
}

// xn_ready: xn already holds RMSNorm(x) with the final norm (compacted to
// the masked rows when mr is set).  mr: the LM head runs on the masked rows
// only (Method: the scores are needed for the masked slots), compacted in
// the order mr gives; records, planted tokens and xn rows are compact, the
// debug logits land on their physical rows.
template <typename T>
int lmhead_impl(wedlm_ctx* c, int B, const T* x, const int32_t* plant,
                float plant_bias, float* logits, cudaStream_t st, bool xn_ready = false,
                const MaskedRows* mr = nullptr) {
  const wedlm_config& g = c->cfg;
  const int M = B * g.window;
  int rc;
  if (!xn_ready)
    LAUNCH(c, WEDLM_KIND_RMSNORM, st,
           launch_rmsnorm<T>(M, g.hidden, x, (const T*)c->final_norm, g.rms_eps,
                             (T*)c->xn, st, mr ? mr->dst : nullptr));
  GemmProblem P = lmhead_problem(c, M);
  GemmEpi& e = P.epi;
  e.part = c->lm_part; e.mask_id = g.mask_id;
  e.vocab = g.vocab; e.plant = mr ? (plant ? mr->plant : nullptr) : plant;
  e.plant_bias = plant_bias;
  e.logits = logits;
  e.row_src = mr ? mr->src : nullptr;
  P.m_count = mr ? mr->count : nullptr;
  int tiles = 0;  // softmax records per row: one per output-feature tile
  if ((rc = run_gemm<T>(c, P, WEDLM_KIND_LMHEAD, st, &tiles))) return rc;
  LAUNCH(c, WEDLM_KIND_LMHEAD_MERGE, st,
         launch_lmhead_merge(M, tiles, c->lm_part, c->rows, c->err, st,
                             mr ? mr->count : nullptr));
  return WEDLM_OK;
}

int check_step_args(wedlm_ctx* c, const wedlm_step_in* in, const wedlm_step_out* out) {
  const wedlm_config& g = c->cfg;
  if (!in || !out) return fail(c, WEDLM_ERR_INVALID_ARG, "null in/out");
  if (in->batch < 1 || in->batch > g.max_batch)
    return fail(c, WEDLM_ERR_INVALID_ARG, "batch outside 1..max_batch");
  if (in->num_pages < 1) return fail(c, WEDLM_ERR_INVALID_ARG, "num_pages < 1");
  if (!in->tokens || !in->pos || !in->observed || !in->seq_len || !in->page_table ||
      !in->kv_pools)
    return fail(c, WEDLM_ERR_INVALID_ARG, "null input pointer");
  for (int l = 0; l < g.n_layers; ++l)
    if (!in->kv_pools[l] || ((uintptr_t)in->kv_pools[l] & 15))
      return fail(c, WEDLM_ERR_INVALID_ARG, "null or misaligned kv pool");
  if (!out->new_tokens || !out->new_pos || !out->new_observed || !out->committed ||
      !out->n_committed)
    return fail(c, WEDLM_ERR_INVALID_ARG, "null output pointer");
  if ((const void*)out->new_tokens == (const void*)in->tokens ||
      (const void*)out->new_pos == (const void*)in->pos ||
      (const void*)out->new_observed == (const void*)in->observed)
    return fail(c, WEDLM_ERR_INVALID_ARG, "outputs alias inputs");
  if (in->score_mode != WEDLM_SCORE_ENTROPY && in->score_mode != WEDLM_SCORE_NEGLOGP)
    return fail(c, WEDLM_ERR_INVALID_ARG, "unknown score_mode");
  return WEDLM_OK;
}

// Streaming-loop controls of a step (all optional; see SelArgs).
struct StepExtras {
  int score_mode = 0;
  int32_t* done = nullptr;
  const int32_t* stop_len = nullptr;
  int stop_token = -1;
  int32_t* out_tokens = nullptr;
  const int32_t* out_base = nullptr;
  int out_cap = 0;
};

template <typename T>
int step_launches(wedlm_ctx* c, const wedlm_step_in* in, wedlm_step_out* out,
                  cudaStream_t st, const StepExtras& x) {
  const wedlm_config& g = c->cfg;
  const int B = in->batch, W = g.window, M = B * W;
  int rc;
  // reorder + embed; also snapshots seq_len, counts the commit run of
  // every sequence (the QKV epilogues write the committed K/V to pages) and
  // lists the masked rows (the LM head runs on those only)
  const MaskedRows mr{c->lm_src, c->lm_dst, c->lm_plant, c->lm_count};
  LAUNCH(c, WEDLM_KIND_REORDER, st,
         launch_reorder_embed<T>(B, W, g.hidden, g.head_dim, g.vocab,
                                 g.max_pages_per_seq * kPageBlock, in->tokens,
                                 in->pos, in->observed, in->seq_len,
                                 in->plant_token, (const T*)c->embed, c->inv_freq,
                                 c->perm, c->inv, c->pos_phys, c->seq_snap, c->ncommit,
                                 x.done, nullptr, (T*)c->x, c->cosb, c->sinb,
                                 c->err, st, &mr));
  Commit cm;
  cm.n = c->ncommit; cm.base = c->seq_snap; cm.page_table = in->page_table;
  cm.num_pages = in->num_pages;
  // on the tensor-core path each down projection also normalises x for
  // the next layer (or the LM head)
  const bool fuse = g.dtype == WEDLM_BF16;
  for (int l = 0; l < g.n_layers; ++l) {
    void* win = (char*)c->kv_win + (size_t)l * c->win_layer_stride * c->es;
    const void* next_norm =
        !fuse ? nullptr : (l + 1 < g.n_layers ? c->layers[l + 1].attn_norm : c->final_norm);
    // the last layer's fused final norm writes the masked rows only, compacted
    const int32_t* row_dst = (fuse && l + 1 == g.n_layers) ? c->lm_dst : nullptr;
    if ((rc = layer_impl<T>(c, l, B, ctx_win(c), (T*)c->x, c->seq_snap, in->page_table,
                            in->num_pages, in->kv_pools[l], win, st, fuse && l > 0,
                            next_norm, cm, row_dst)))
      return rc;
  }
  if ((rc = lmhead_impl<T>(c, B, (const T*)c->x, in->plant_token, in->plant_bias, out->logits,
                           st, fuse, &mr)))
    return rc;
  SelArgs S{};
  S.B = B; S.W = W; S.mask_id = g.mask_id; S.alpha = in->alpha; S.tau = in->tau;
  S.score_mode = x.score_mode; S.done = x.done; S.stop_len = x.stop_len;
  S.stop_token = x.stop_token; S.out_tokens = x.out_tokens; S.out_base = x.out_base;
  S.out_cap = x.out_cap;
  S.tokens = in->tokens; S.pos = in->pos; S.obs = in->observed;
  S.seq_snap = c->seq_snap; S.seq_len = in->seq_len; S.inv = c->inv; S.rows = c->rows;
  S.new_tokens = out->new_tokens; S.new_pos = out->new_pos;
  S.new_obs = out->new_observed; S.committed = out->committed;
  S.n_committed = out->n_committed; S.ncommit_ws = c->ncommit; S.filled = out->filled;
  S.row_dst = c->lm_dst; S.out_rows = out->rows;
  LAUNCH(c, WEDLM_KIND_SELECT, st, launch_select(S, st));
  if (out->perm)
    CUDA_TRY(c, cudaMemcpyAsync(out->perm, c->perm, (size_t)M * 4,
                                cudaMemcpyDeviceToDevice, st));
  if (out->hidden)
    CUDA_TRY(c, cudaMemcpyAsync(out->hidden, c->x, (size_t)M * g.hidden * c->es,
                                cudaMemcpyDeviceToDevice, st));
  return WEDLM_OK;
}

int dispatch_step(wedlm_ctx* c, const wedlm_step_in* in, wedlm_step_out* out,
                  cudaStream_t st, const StepExtras& x) {
  c->launch_count = 0;
  const int rc = c->cfg.dtype == WEDLM_BF16 ? step_launches<bf16>(c, in, out, st, x)
                                            : step_launches<float>(c, in, out, st, x);
  if (rc == WEDLM_OK) c->last_step_launches = c->launch_count;
  return rc;
}

std::vector<uint64_t> graph_key(const wedlm_ctx* c, const wedlm_step_in* in,
                                const wedlm_step_out* out) {
  std::vector<uint64_t> k;
  auto P = [&](const void* p) { k.push_back((uint64_t)(uintptr_t)p); };
  auto F = [&](float f) { uint32_t u; memcpy(&u, &f, 4); k.push_back(u); };
  k.push_back((uint64_t)in->batch);
  k.push_back((uint64_t)in->num_pages);
  P(in->tokens); P(in->pos); P(in->observed); P(in->seq_len); P(in->page_table);
  P(in->plant_token); F(in->plant_bias); F(in->alpha); F(in->tau);
  k.push_back((uint64_t)(uint32_t)in->score_mode);
  for (int l = 0; l < c->cfg.n_layers; ++l) P(in->kv_pools[l]);
  P(out->new_tokens); P(out->new_pos); P(out->new_observed); P(out->committed);
  P(out->n_committed); P(out->perm); P(out->filled); P(out->rows); P(out->logits);
  P(out->hidden);
  return k;
}

// ---------------------------------------------------------------------------
// the streaming loop on the device: a conditional while node whose body is
// one step plus gen_next_kernel; the loop ends when the step budget is spent
// or every sequence has stopped
// ---------------------------------------------------------------------------
__device__ __forceinline__ int any_active(int B, const int32_t* done) {
  int any = 0;
  for (int b = 0; b < B; ++b) any |= (done[b] == 0);
  return any;
}

__global__ void gen_init_kernel(int B, int max_steps, const int32_t* done, int* ctrl,
                                int32_t* steps_run, cudaGraphConditionalHandle h) {
  if (threadIdx.x != 0) return;
  ctrl[0] = max_steps;  // steps left
  ctrl[1] = 0;          // steps run
  if (steps_run) *steps_run = 0;
  cudaGraphSetConditional(h, (max_steps > 0 && any_active(B, done)) ? 1u : 0u);
}

// after every step: one step fewer left; continue while steps are left and a
// sequence is still active (so the loop runs at most max_steps times)
__global__ void gen_next_kernel(int B, const int32_t* done, int* ctrl, int32_t* steps_run,
                                cudaGraphConditionalHandle h) {
  if (threadIdx.x != 0) return;
  const int left = ctrl[0] - 1, ran = ctrl[1] + 1;
  ctrl[0] = left;
  ctrl[1] = ran;
  if (steps_run) *steps_run = ran;
  cudaGraphSetConditional(h, (left > 0 && any_active(B, done)) ? 1u : 0u);
}

// Dual-Stream Masking as paged window attention: sequence s < nb is memory
// block s, sequence nb + j prediction block j; both have the memory
// positions 0..j*block-1 as cached prefix (one identity page-table row).
__global__ void dual_setup_kernel(int nb, int block, int n_pages, int32_t* len, int32_t* pt) {
  const int n = max(2 * nb, n_pages);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    if (i < 2 * nb) len[i] = (i % nb) * block;
    if (i < n_pages) pt[i] = i;
  }
}

int check_gen_args(wedlm_ctx* c, const wedlm_gen_in* in) {
  const wedlm_config& g = c->cfg;
  if (!in) return fail(c, WEDLM_ERR_INVALID_ARG, "null generate input");
  if (in->batch < 1 || in->batch > g.max_batch)
    return fail(c, WEDLM_ERR_INVALID_ARG, "batch outside 1..max_batch");
  if (in->num_pages < 1 || in->max_steps < 0)
    return fail(c, WEDLM_ERR_INVALID_ARG, "num_pages < 1 or max_steps < 0");
  if (!in->tokens || !in->pos || !in->observed || !in->seq_len || !in->page_table ||
      !in->kv_pools || !in->done)
    return fail(c, WEDLM_ERR_INVALID_ARG, "null input pointer");
  for (int l = 0; l < g.n_layers; ++l)
    if (!in->kv_pools[l] || ((uintptr_t)in->kv_pools[l] & 15))
      return fail(c, WEDLM_ERR_INVALID_ARG, "null or misaligned kv pool");
  if (in->out_tokens && (!in->out_base || in->out_cap < 1))
    return fail(c, WEDLM_ERR_INVALID_ARG, "out_tokens without out_base / out_cap");
  if (in->score_mode != WEDLM_SCORE_ENTROPY && in->score_mode != WEDLM_SCORE_NEGLOGP)
    return fail(c, WEDLM_ERR_INVALID_ARG, "unknown score_mode");
  return WEDLM_OK;
}

std::vector<uint64_t> gen_key(const wedlm_ctx* c, const wedlm_gen_in* in) {
  std::vector<uint64_t> k;
  auto P = [&](const void* p) { k.push_back((uint64_t)(uintptr_t)p); };
  auto F = [&](float f) { uint32_t u; memcpy(&u, &f, 4); k.push_back(u); };
  k.push_back((uint64_t)in->batch);
  k.push_back((uint64_t)in->num_pages);
  P(in->tokens); P(in->pos); P(in->observed); P(in->seq_len); P(in->page_table);
  P(in->plant_token); F(in->plant_bias); F(in->alpha); F(in->tau);
  k.push_back((uint64_t)(uint32_t)in->score_mode);
  k.push_back((uint64_t)(uint32_t)in->max_steps);
  P(in->done); P(in->stop_len); k.push_back((uint64_t)(uint32_t)in->stop_token);
  P(in->out_tokens); P(in->out_base); k.push_back((uint64_t)(uint32_t)in->out_cap);
  P(in->steps_run);
  for (int l = 0; l < c->cfg.n_layers; ++l) P(in->kv_pools[l]);
  return k;
}

// Build the loop graph: gen_init_kernel -> while (cond) { step; gen_next_kernel }.
int build_gen_graph(wedlm_ctx* c, const wedlm_gen_in* in, cudaGraphExec_t* exec_out) {
  const wedlm_config& g = c->cfg;
  cudaGraph_t graph = nullptr;
  CUDA_TRY(c, cudaGraphCreate(&graph, 0));
  struct GraphGuard {
    cudaGraph_t g;
    ~GraphGuard() { if (g) cudaGraphDestroy(g); }
  } guard{graph};
  cudaGraphConditionalHandle h;
  CUDA_TRY(c, cudaGraphConditionalHandleCreate(&h, graph, 0, 0));
  // the init kernel, then the conditional node after it
  cudaGraphNode_t init = nullptr;
  {
    cudaKernelNodeParams kp = {};
    int B = in->batch, ms = in->max_steps;
    const int32_t* done = in->done;
    int* ctrl = c->gen_ctrl;
    int32_t* sr = in->steps_run;
    void* args[] = {&B, &ms, &done, &ctrl, &sr, &h};
    kp.func = (void*)gen_init_kernel;
    kp.gridDim = dim3(1);
    kp.blockDim = dim3(32);
    kp.kernelParams = args;
    CUDA_TRY(c, cudaGraphAddKernelNode(&init, graph, nullptr, 0, &kp));
  }
  cudaGraphNodeParams cp = {};
  cp.type = cudaGraphNodeTypeConditional;
  cp.conditional.handle = h;
  cp.conditional.type = cudaGraphCondTypeWhile;
  cp.conditional.size = 1;
  cudaGraphNode_t cnode = nullptr;
  CUDA_TRY(c, cudaGraphAddNode(&cnode, graph, &init, nullptr, 1, &cp));
  cudaGraph_t body = cp.conditional.phGraph_out[0];
  // the body: one step with the window updated in place, then the control
  wedlm_step_in sin{};
  sin.batch = in->batch; sin.num_pages = in->num_pages; sin.tokens = in->tokens;
  sin.pos = in->pos; sin.observed = in->observed; sin.seq_len = in->seq_len;
  sin.page_table = in->page_table; sin.kv_pools = in->kv_pools;
  sin.plant_token = in->plant_token; sin.plant_bias = in->plant_bias;
  sin.alpha = in->alpha; sin.tau = in->tau; sin.score_mode = in->score_mode;
  wedlm_step_out sout{};
  sout.new_tokens = in->tokens; sout.new_pos = in->pos; sout.new_observed = in->observed;
  sout.committed = c->gen_committed; sout.n_committed = c->gen_ncommitted;
  StepExtras x;
  x.score_mode = in->score_mode; x.done = in->done; x.stop_len = in->stop_len;
  x.stop_token = in->stop_token; x.out_tokens = in->out_tokens; x.out_base = in->out_base;
  x.out_cap = in->out_cap;
  CUDA_TRY(c, cudaStreamBeginCaptureToGraph(c->cap_stream, body, nullptr, nullptr, 0,
                                            cudaStreamCaptureModeThreadLocal));
  // a loop body holds kernels only: no timing events inside it
  const bool timing = c->timing;
  c->timing = false;
  int rc = dispatch_step(c, &sin, &sout, c->cap_stream, x);
  c->timing = timing;
  if (rc == WEDLM_OK) {
    gen_next_kernel<<<1, 32, 0, c->cap_stream>>>(in->batch, in->done, c->gen_ctrl,
                                                 in->steps_run, h);
    c->launch_count += 1;
  }
  cudaGraph_t captured = nullptr;
  const cudaError_t ce = cudaStreamEndCapture(c->cap_stream, &captured);
  if (rc) return rc;
  if (ce != cudaSuccess)
    return fail(c, WEDLM_ERR_CUDA, std::string("loop capture: ") + cudaGetErrorString(ce));
  (void)g;
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
  if (ie != cudaSuccess)
    return fail(c, WEDLM_ERR_CUDA, std::string("loop instantiate: ") + cudaGetErrorString(ie));
  *exec_out = exec;
  return WEDLM_OK;
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

int wedlm_create(const wedlm_config* cfg, const wedlm_weights* w, wedlm_ctx** out) {
  if (!cfg || !w || !out) return WEDLM_ERR_INVALID_ARG;
  *out = nullptr;
  const wedlm_config& g = *cfg;
  auto bad = [&](bool cond) { return cond; };
  if (bad(g.n_layers < 1 || g.n_layers > kMaxLayers) ||
      bad(g.hidden < 128 || g.hidden % 128) ||
      bad(g.head_dim != 64 && g.head_dim != 128) ||
      bad(g.n_kv_heads < 1 || g.n_q_heads % g.n_kv_heads) ||
      bad((g.n_q_heads * g.head_dim) % 128 || (g.n_kv_heads * g.head_dim) % 128) ||
      bad(g.ffn < 64 || g.ffn % 64) || bad(g.vocab < 8 || g.vocab % 4) ||
      bad(g.mask_id < 0 || g.mask_id >= g.vocab) ||
      bad(g.window < 1 || g.window > kMaxWindow) || bad(g.page_block != kPageBlock) ||
      bad(g.max_batch < 1 || g.max_batch * g.window > kMaxRows) ||
      bad(g.max_pages_per_seq < 1) ||
      bad(g.dtype != WEDLM_BF16 && g.dtype != WEDLM_FP32) ||
      bad(!(g.rope_theta > 0.f) || !(g.rms_eps >= 0.f)))
    return WEDLM_ERR_INVALID_ARG;
  // bf16: tensor-core GEMMs (K multiple of 64) and attention (head_dim 128,
  // query rows of a kv head in row blocks); fp32: CUDA-core attention with
  // at most 512 query rows per kv head
  if (g.dtype == WEDLM_BF16 &&
      ((g.hidden % 64) || ((g.n_q_heads * g.head_dim) % 64) || (g.ffn % 64) ||
       g.head_dim != 128 ||
       attention_tc_row_blocks(g.n_q_heads, g.n_kv_heads, g.window, nullptr) == 0))
    return WEDLM_ERR_INVALID_ARG;
  if (g.dtype == WEDLM_FP32 && (g.n_q_heads / g.n_kv_heads) * g.window > 512)
    return WEDLM_ERR_INVALID_ARG;
  if (!w->embed || !w->final_norm || !w->lm_head || !w->attn_norm || !w->w_q ||
      !w->w_k || !w->w_v || !w->w_o || !w->ffn_norm || !w->w_gate || !w->w_up ||
      !w->w_down)
    return WEDLM_ERR_INVALID_ARG;
  if (g.qk_norm && (!w->q_norm || !w->k_norm)) return WEDLM_ERR_INVALID_ARG;

  std::unique_ptr<wedlm_ctx> c(new wedlm_ctx());
  c->cfg = g;
  c->es = g.dtype == WEDLM_BF16 ? 2 : 4;
  c->Wp = ((g.window + kPageBlock - 1) / kPageBlock) * kPageBlock;
  c->M_max = g.max_batch * g.window;
  c->embed = w->embed; c->final_norm = w->final_norm; c->lm_head = w->lm_head;
  for (int l = 0; l < g.n_layers; ++l) {
    LayerWeights lw{};
    lw.attn_norm = w->attn_norm[l]; lw.w_q = w->w_q[l]; lw.w_k = w->w_k[l];
    lw.w_v = w->w_v[l]; lw.q_norm = g.qk_norm ? w->q_norm[l] : nullptr;
    lw.k_norm = g.qk_norm ? w->k_norm[l] : nullptr; lw.w_o = w->w_o[l];
    lw.ffn_norm = w->ffn_norm[l]; lw.w_gate = w->w_gate[l]; lw.w_up = w->w_up[l];
    lw.w_down = w->w_down[l];
    const void* ptrs[] = {lw.attn_norm, lw.w_q, lw.w_k, lw.w_v, lw.w_o, lw.ffn_norm,
                          lw.w_gate, lw.w_up, lw.w_down};
    for (const void* p : ptrs)
      if (!p || ((uintptr_t)p & 15)) return WEDLM_ERR_INVALID_ARG;
    c->layers.push_back(lw);
  }
  wedlm_ctx* C = c.get();
  if (cudaGetDevice(&C->device) != cudaSuccess) return WEDLM_ERR_CUDA;
  cudaDeviceGetAttribute(&C->num_sms, cudaDevAttrMultiProcessorCount, C->device);
  if (C->num_sms <= 0) C->num_sms = 148;

  const size_t M = C->M_max, es = C->es, H = g.hidden, hd = g.head_dim;
  const size_t qd = (size_t)g.n_q_heads * hd;
  const size_t max_len = (size_t)g.max_pages_per_seq * kPageBlock;
  // key chunk per attention block: about 1/16 of the capacity, a multiple
  // of 64 keys (the tensor-core kernel's tile), at least 256
  C->attn_chunk = (int)std::max<size_t>(256, ((max_len + 15) / 16 + 63) / 64 * 64);
  C->attn_max_chunks = (int)((max_len + C->attn_chunk - 1) / C->attn_chunk) + 1;
  const size_t R = (size_t)(g.n_q_heads / g.n_kv_heads) * g.window;
  C->vtiles = (g.vocab + 127) / 128;
  C->win_layer_stride = (size_t)g.max_batch * 2 * g.n_kv_heads * C->Wp * hd;
  C->gemm_part_elems = (size_t)16 << 20;  // 64 MB of fp32 split-K partials

  cudaError_t e = cudaSuccess;
#define WA(ptr, bytes) if (e == cudaSuccess) e = walloc(C, &(ptr), (bytes))
  WA(C->err, 256);
  WA(C->perm, M * 4); WA(C->inv, M * 4); WA(C->pos_phys, M * 4);
  WA(C->plant_phys, M * 4); WA(C->seq_snap, g.max_batch * 4);
  WA(C->ncommit, g.max_batch * 4);
  WA(C->inv_freq, hd / 2 * 8);
  WA(C->cosb, M * hd / 2 * 4); WA(C->sinb, M * hd / 2 * 4);
  WA(C->x, M * H * es); WA(C->xn, M * H * es);
  WA(C->q, M * qd * es); WA(C->o, M * qd * es);
  WA(C->act, M * g.ffn * es);
  WA(C->kv_win, C->win_layer_stride * g.n_layers * es);
  // split-KV partials: per (sequence, kv head, chunk) for the CUDA-core
  // attention (rows * chunks, the same bound for a prefill chunk since
  // B * chunk <= max_batch * window); per segment for the tensor-core
  // attention: at most one per block (SM) plus one per unit (sequence x kv
  // head x row block), of at most 128 rows, where the rows of all units'
  // row blocks together stay below nkv * (G * M_max + 128 * max_batch)
  const size_t units = (size_t)g.max_batch * g.n_kv_heads;
  const size_t G = (size_t)(g.n_q_heads / g.n_kv_heads);
  const size_t simt_rows = units * C->attn_max_chunks * R;
  const size_t tc_rows = (size_t)C->num_sms * 128 +
                         (size_t)g.n_kv_heads * (G * M + 128 * (size_t)g.max_batch);
  const size_t part_rows = g.dtype == WEDLM_BF16 ? tc_rows : simt_rows;
  C->attn_units_cap = (size_t)g.n_kv_heads * M;  // B * nkv * row blocks <= nkv * B * chunk
  WA(C->attn_o, part_rows * hd * 4);
  WA(C->attn_ml, part_rows * 2 * 4);
  WA(C->attn_unit_cnt, C->attn_units_cap * 4);
  WA(C->gen_ctrl, 256);
  C->attn_part_rows = part_rows;
  WA(C->dual_len, (size_t)kDualMaxBlocks * 4); WA(C->dual_pt, (size_t)kDualMaxPages * 4);
  WA(C->gen_committed, M * 4); WA(C->gen_ncommitted, g.max_batch * 4);
  WA(C->gemm_part, C->gemm_part_elems * 4);
  WA(C->gemm_counters, (size_t)std::max(C->vtiles, 4096) * 4);
  WA(C->lm_part, (size_t)C->vtiles * M * sizeof(SoftmaxPart));
  WA(C->rows, M * sizeof(wedlm_slot_rec));
  WA(C->lm_src, M * 4); WA(C->lm_dst, M * 4); WA(C->lm_plant, M * 4); WA(C->lm_count, 256);
  WA(C->zero_page, 4096);
#undef WA
  if (e != cudaSuccess) {
    wedlm_destroy(c.release());
    return WEDLM_ERR_CUDA;
  }
  std::vector<double> inv_freq(hd / 2);
  for (size_t i = 0; i < hd / 2; ++i)
    inv_freq[i] = pow((double)g.rope_theta, -2.0 * (double)i / (double)hd);
  if (cudaMemcpy(C->inv_freq, inv_freq.data(), hd / 2 * 8, cudaMemcpyHostToDevice) !=
      cudaSuccess) {
    wedlm_destroy(c.release());
    return WEDLM_ERR_CUDA;
  }
  if (g.dtype == WEDLM_BF16) {
    std::string msg;
    C->tc = make_tc_plans(g, C->layers, C->embed, C->lm_head, C->xn, C->o, C->act,
                          C->num_sms, C->gemm_part_elems, &msg);
    if (!C->tc) {
      fprintf(stderr, "wedlm_create: %s\n", msg.c_str());
      wedlm_destroy(c.release());
      return WEDLM_ERR_CUDA;
    }
  }
  if (cudaStreamCreateWithFlags(&C->cap_stream, cudaStreamNonBlocking) != cudaSuccess) {
    wedlm_destroy(c.release());
    return WEDLM_ERR_CUDA;
  }
  const char* ng = getenv("WEDLM_NO_GRAPH");
  if (ng && ng[0] == '1') C->use_graphs = false;
  *out = c.release();
  return WEDLM_OK;
}

void wedlm_destroy(wedlm_ctx* c) {
  if (!c) return;
  cudaDeviceSynchronize();
  for (auto& g : c->graphs)
    if (g.exec) cudaGraphExecDestroy(g.exec);
  for (auto& g : c->gen_graphs)
    if (g.exec) cudaGraphExecDestroy(g.exec);
  for (auto e : c->ev) cudaEventDestroy(e);
  for (void* p : c->allocs) cudaFree(p);
  if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
  delete c;
}

const char* wedlm_last_error(wedlm_ctx* c) {
  return c ? c->last_error.c_str() : "null context";
}

int wedlm_get_status(wedlm_ctx* c, int32_t* device_error) {
  if (!c) return WEDLM_ERR_INVALID_ARG;
  CUDA_TRY(c, cudaStreamSynchronize(c->last_stream));
  int32_t word = 0;
  CUDA_TRY(c, cudaMemcpy(&word, c->err, 4, cudaMemcpyDeviceToHost));
  CUDA_TRY(c, cudaMemset(c->err, 0, 4));
  // a launch that gave up on a wait may have left segment counts behind
  if (word) CUDA_TRY(c, cudaMemset(c->attn_unit_cnt, 0, c->attn_units_cap * 4));
  if (device_error) *device_error = word;
  if (word) return fail(c, WEDLM_ERR_DEVICE, "device error word " + std::to_string(word));
  return WEDLM_OK;
}

int wedlm_set_graphs(wedlm_ctx* c, int enable) {
  if (!c) return WEDLM_ERR_INVALID_ARG;
  c->use_graphs = enable != 0;
  return WEDLM_OK;
}

int wedlm_set_timing(wedlm_ctx* c, int enable) {
  if (!c) return WEDLM_ERR_INVALID_ARG;
  if (enable && c->ev.empty()) {
    c->ev.resize(kMaxEvents);
    c->ev_kind.assign(kMaxEvents, 0);
    for (auto& e : c->ev) CUDA_TRY(c, cudaEventCreate(&e));
  }
  c->timing = enable != 0;
  return WEDLM_OK;
}

static int harvest_events(wedlm_ctx* c) {
  if (c->ev_used == 0) return WEDLM_OK;
  CUDA_TRY(c, cudaEventSynchronize(c->ev[c->ev_used - 1]));
  for (int i = 0; i + 1 < c->ev_used; i += 2) {
    float ms = 0.f;
    CUDA_TRY(c, cudaEventElapsedTime(&ms, c->ev[i], c->ev[i + 1]));
    c->kind_ms[c->ev_kind[i]] += ms;
    c->kind_launches[c->ev_kind[i]] += 1;
  }
  c->ev_used = 0;
  return WEDLM_OK;
}

int wedlm_get_timings(wedlm_ctx* c, float* ms, int32_t* launches, int n) {
  if (!c) return WEDLM_ERR_INVALID_ARG;
  int rc = harvest_events(c);
  if (rc) return rc;
  for (int k = 0; k < WEDLM_KIND_COUNT && k < n; ++k) {
    if (ms) ms[k] = (float)c->kind_ms[k];
    if (launches) launches[k] = c->kind_launches[k];
  }
  for (int k = 0; k < WEDLM_KIND_COUNT; ++k) { c->kind_ms[k] = 0; c->kind_launches[k] = 0; }
  return WEDLM_OK;
}

int wedlm_launches_per_step(wedlm_ctx* c, int32_t batch) {
  if (!c) return -1;
  (void)batch;
  return c->last_step_launches;  // counted while the last step was enqueued
}

int wedlm_step(wedlm_ctx* c, const wedlm_step_in* in, wedlm_step_out* out, void* stream) {
  if (!c) return WEDLM_ERR_INVALID_ARG;
  int rc = check_step_args(c, in, out);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  c->last_stream = st;
  StepExtras x;
  x.score_mode = in->score_mode;
  if (c->timing || !c->use_graphs) {
    if (c->timing && c->ev_used + 4 * wedlm_launches_per_step(c, in->batch) > kMaxEvents)
      if ((rc = harvest_events(c))) return rc;
    return dispatch_step(c, in, out, st, x);
  }
  std::vector<uint64_t> key = graph_key(c, in, out);
  GraphEntry* hit = nullptr;
  for (auto& g : c->graphs)
    if (g.key == key) hit = &g;
  if (!hit) {
    // capture on the library's own stream, replay on the caller's
    cudaGraph_t graph = nullptr;
    CUDA_TRY(c, cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal));
    rc = dispatch_step(c, in, out, c->cap_stream, x);
    cudaError_t ce = cudaStreamEndCapture(c->cap_stream, &graph);
    if (rc) {
      if (graph) cudaGraphDestroy(graph);
      return rc;
    }
    if (ce != cudaSuccess)
      return fail(c, WEDLM_ERR_CUDA, std::string("capture: ") + cudaGetErrorString(ce));
    cudaGraphExec_t exec = nullptr;
    ce = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ce != cudaSuccess)
      return fail(c, WEDLM_ERR_CUDA, std::string("instantiate: ") + cudaGetErrorString(ce));
    if ((int)c->graphs.size() >= kMaxGraphs) {
      auto lru = std::min_element(c->graphs.begin(), c->graphs.end(),
                                  [](const GraphEntry& a, const GraphEntry& b) {
                                    return a.last_use < b.last_use;
                                  });
      cudaGraphExecDestroy(lru->exec);
      c->graphs.erase(lru);
    }
    c->graphs.push_back(GraphEntry{key, exec, 0});
    hit = &c->graphs.back();
  }
  hit->last_use = ++c->graph_clock;
  CUDA_TRY(c, cudaGraphLaunch(hit->exec, st));
  return WEDLM_OK;
}

int wedlm_prefill(wedlm_ctx* c, int32_t batch, int32_t chunk, const int32_t* tokens,
                  int32_t* seq_len, const int32_t* page_table, int32_t num_pages,
                  void* const* kv_pools, void* hidden, void* stream) {
  if (!c) return WEDLM_ERR_INVALID_ARG;
  const wedlm_config& g = c->cfg;
  const Win win = chunk_win(chunk);
  const int G = g.n_q_heads / g.n_kv_heads;
  if (batch < 1 || batch > g.max_batch || chunk < 1 || batch * chunk > c->M_max ||
      batch * win.Wp > g.max_batch * c->Wp || !tokens || !seq_len || !page_table ||
      !kv_pools || num_pages < 1)
    return fail(c, WEDLM_ERR_INVALID_ARG, "bad prefill arguments");
  if (g.dtype == WEDLM_BF16
          ? attention_tc_row_blocks(g.n_q_heads, g.n_kv_heads, chunk, nullptr) == 0
          : G * chunk > 512)
    return fail(c, WEDLM_ERR_INVALID_ARG, "prefill chunk too large for the attention");
  for (int l = 0; l < g.n_layers; ++l)
    if (!kv_pools[l] || ((uintptr_t)kv_pools[l] & 15))
      return fail(c, WEDLM_ERR_INVALID_ARG, "null or misaligned kv pool");
  cudaStream_t st = (cudaStream_t)stream;
  c->last_stream = st;
  c->launch_count = 0;
  const int M = batch * chunk;
  const int page_cap = g.max_pages_per_seq * kPageBlock;
  if (g.dtype == WEDLM_BF16)
    LAUNCH(c, WEDLM_KIND_REORDER, st,
           launch_prefill_embed<bf16>(batch, chunk, g.hidden, g.head_dim, g.vocab, page_cap,
                                      tokens, seq_len, (const bf16*)c->embed, c->inv_freq,
                                      c->pos_phys, c->seq_snap, c->ncommit, (bf16*)c->x,
                                      c->cosb, c->sinb, c->err, st));
  else
    LAUNCH(c, WEDLM_KIND_REORDER, st,
           launch_prefill_embed<float>(batch, chunk, g.hidden, g.head_dim, g.vocab, page_cap,
                                       tokens, seq_len, (const float*)c->embed, c->inv_freq,
                                       c->pos_phys, c->seq_snap, c->ncommit, (float*)c->x,
                                       c->cosb, c->sinb, c->err, st));
  Commit cm;
  cm.n = c->ncommit; cm.base = c->seq_snap; cm.page_table = page_table;
  cm.num_pages = num_pages;
  const bool fuse = g.dtype == WEDLM_BF16;
  for (int l = 0; l < g.n_layers; ++l) {
    void* wl = (char*)c->kv_win + (size_t)l * c->win_layer_stride * c->es;
    const void* next_norm = fuse && l + 1 < g.n_layers ? c->layers[l + 1].attn_norm : nullptr;
    const int rc =
        fuse ? layer_impl<bf16>(c, l, batch, win, (bf16*)c->x, c->seq_snap, page_table,
                                num_pages, kv_pools[l], wl, st, l > 0, next_norm, cm)
             : layer_impl<float>(c, l, batch, win, (float*)c->x, c->seq_snap, page_table,
                                 num_pages, kv_pools[l], wl, st, false, nullptr, cm);
    if (rc) return rc;
  }
  LAUNCH(c, WEDLM_KIND_SELECT, st, launch_seq_advance(batch, chunk, c->seq_snap, seq_len, st));
  if (hidden)
    CUDA_TRY(c, cudaMemcpyAsync(hidden, c->x, (size_t)M * g.hidden * c->es,
                                cudaMemcpyDeviceToDevice, st));
  return WEDLM_OK;
}

int wedlm_generate(wedlm_ctx* c, const wedlm_gen_in* in, void* stream) {
  if (!c) return WEDLM_ERR_INVALID_ARG;
  int rc = check_gen_args(c, in);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  c->last_stream = st;
  if (in->max_steps == 0) return WEDLM_OK;
  std::vector<uint64_t> key = gen_key(c, in);
  GraphEntry* hit = nullptr;
  for (auto& e : c->gen_graphs)
    if (e.key == key) hit = &e;
  if (!hit) {
    cudaGraphExec_t exec = nullptr;
    if ((rc = build_gen_graph(c, in, &exec))) return rc;
    if ((int)c->gen_graphs.size() >= kMaxGraphs) {
      auto lru = std::min_element(c->gen_graphs.begin(), c->gen_graphs.end(),
                                  [](const GraphEntry& a, const GraphEntry& b) {
                                    return a.last_use < b.last_use;
                                  });
      cudaGraphExecDestroy(lru->exec);
      c->gen_graphs.erase(lru);
    }
    c->gen_graphs.push_back(GraphEntry{key, exec, 0});
    hit = &c->gen_graphs.back();
  }
  hit->last_use = ++c->graph_clock;
  CUDA_TRY(c, cudaGraphLaunch(hit->exec, st));
  return WEDLM_OK;
}

int wedlm_dual_stream_attention(wedlm_ctx* c, int32_t n, int32_t block, const void* q,
                                const void* mem_pool, const void* win, void* o, void* stream) {
  if (!c) return WEDLM_ERR_INVALID_ARG;
  const wedlm_config& g = c->cfg;
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
  if (g.dtype != WEDLM_BF16 || block < 16 || block % kPageBlock || n < block || n % block ||
      !q || !mem_pool || !win || !o || misaligned(q) || misaligned(mem_pool) ||
      misaligned(win) || misaligned(o))
    return fail(c, WEDLM_ERR_INVALID_ARG, "bad dual-stream arguments");
  int rpb = 0;
  const int nrb = attention_tc_row_blocks(g.n_q_heads, g.n_kv_heads, block, &rpb);
  if (nrb == 0) return fail(c, WEDLM_ERR_INVALID_ARG, "block too large for the attention");
  const int nb = n / block, B = 2 * nb, n_pages = n / kPageBlock;
  const size_t units = (size_t)B * g.n_kv_heads * nrb;
  if (B > kDualMaxBlocks || n_pages > kDualMaxPages || units > c->attn_units_cap ||
      ((size_t)c->num_sms + units) * rpb > c->attn_part_rows)
    return fail(c, WEDLM_ERR_CAPACITY, "dual-stream shape beyond the context's workspace");
  cudaStream_t st = (cudaStream_t)stream;
  c->last_stream = st;
  dual_setup_kernel<<<std::max(1, (std::max(B, n_pages) + 255) / 256), 256, 0, st>>>(
      nb, block, n_pages, c->dual_len, c->dual_pt);
  CUDA_TRY(c, cudaGetLastError());
  AttnArgs A = attn_args(c, B, chunk_win(block), q, mem_pool, c->dual_pt, c->dual_len, n_pages,
                         win, o);
  A.max_pages = n_pages;
  A.pt_stride = 0;  // every block reads the one identity row
  A.kv_reuse = 1;   // and every block re-reads the memory stream's pages
  // units here are short (a block and its prefix): counting their start and
  // end as six tiles balances the shares best (measured at n = 4096, blocks
  // of 32: 0.437 ms, against 0.445 ms with eight and 0.472 ms with four)
  A.unit_cost = 2 * kAttnUnitCost;
  cudaError_t e;
  {
    Timed t(c, WEDLM_KIND_ATTN, st);
    // plain launch: the lengths and the page row come from the kernel above
    e = launch_attention_tc(A, c->zero_page, c->num_sms, st, false);
  }
  if (e != cudaSuccess) return fail(c, WEDLM_ERR_CUDA, cudaGetErrorString(e));
  return WEDLM_OK;
}

int wedlm_reorder_embed(wedlm_ctx* c, int32_t batch, const int32_t* tokens,
                        const int32_t* pos, const uint8_t* observed, int32_t* perm,
                        int32_t* inv, void* x_out, int32_t* pos_phys, void* stream) {
  if (!c) return WEDLM_ERR_INVALID_ARG;
  const wedlm_config& g = c->cfg;
  if (batch < 1 || batch > g.max_batch || !tokens || !pos || !observed || !x_out)
    return fail(c, WEDLM_ERR_INVALID_ARG, "bad reorder arguments");
  cudaStream_t st = (cudaStream_t)stream;
  c->last_stream = st;
  const int M = batch * g.window;
  // the kernel reads seq_len only for the snapshot; feed it a zero array
  CUDA_TRY(c, cudaMemsetAsync(c->ncommit, 0, (size_t)batch * 4, st));
  cudaError_t e;
  if (g.dtype == WEDLM_BF16)
    e = launch_reorder_embed<bf16>(batch, g.window, g.hidden, g.head_dim, g.vocab,
                                   g.max_pages_per_seq * kPageBlock, tokens, pos,
                                   observed, c->ncommit, nullptr, (const bf16*)c->embed,
                                   c->inv_freq, c->perm, c->inv, c->pos_phys,
                                   c->seq_snap, nullptr, nullptr, nullptr, (bf16*)x_out,
                                   c->cosb, c->sinb, c->err, st);
  else
    e = launch_reorder_embed<float>(batch, g.window, g.hidden, g.head_dim, g.vocab,
                                    g.max_pages_per_seq * kPageBlock, tokens, pos,
                                    observed, c->ncommit, nullptr, (const float*)c->embed,
                                    c->inv_freq, c->perm, c->inv, c->pos_phys,
                                    c->seq_snap, nullptr, nullptr, nullptr, (float*)x_out,
                                    c->cosb, c->sinb, c->err, st);
  if (e != cudaSuccess) return fail(c, WEDLM_ERR_CUDA, cudaGetErrorString(e));
  if (perm) CUDA_TRY(c, cudaMemcpyAsync(perm, c->perm, M * 4, cudaMemcpyDeviceToDevice, st));
  if (inv) CUDA_TRY(c, cudaMemcpyAsync(inv, c->inv, M * 4, cudaMemcpyDeviceToDevice, st));
  if (pos_phys)
    CUDA_TRY(c, cudaMemcpyAsync(pos_phys, c->pos_phys, M * 4, cudaMemcpyDeviceToDevice, st));
  return WEDLM_OK;
}

int wedlm_layer(wedlm_ctx* c, int32_t layer, int32_t batch, void* x,
                const int32_t* pos_phys, const int32_t* seq_len,
                const int32_t* page_table, int32_t num_pages, const void* kv_pool,
                void* kv_win_out, void* q_out, void* attn_out, void* stream) {
  if (!c) return WEDLM_ERR_INVALID_ARG;
  const wedlm_config& g = c->cfg;
  if (layer < 0 || layer >= g.n_layers || batch < 1 || batch > g.max_batch || !x ||
      !pos_phys || !seq_len || !page_table || !kv_pool || num_pages < 1)
    return fail(c, WEDLM_ERR_INVALID_ARG, "bad layer arguments");
  cudaStream_t st = (cudaStream_t)stream;
  c->last_stream = st;
  const int M = batch * g.window;
  CUDA_TRY(c, launch_rope_table(M, g.head_dim, pos_phys, c->inv_freq, c->cosb, c->sinb, st));
  CUDA_TRY(c, cudaMemcpyAsync(c->x, x, (size_t)M * g.hidden * c->es,
                              cudaMemcpyDeviceToDevice, st));
  void* win = (char*)c->kv_win + (size_t)layer * c->win_layer_stride * c->es;
  int rc = g.dtype == WEDLM_BF16
               ? layer_impl<bf16>(c, layer, batch, ctx_win(c), (bf16*)c->x, seq_len, page_table,
                                  num_pages, kv_pool, win, st)
               : layer_impl<float>(c, layer, batch, ctx_win(c), (float*)c->x, seq_len,
                                   page_table, num_pages, kv_pool, win, st);
  if (rc) return rc;
  CUDA_TRY(c, cudaMemcpyAsync(x, c->x, (size_t)M * g.hidden * c->es,
                              cudaMemcpyDeviceToDevice, st));
  const size_t per_b = (size_t)2 * g.n_kv_heads * c->Wp * g.head_dim * c->es;
  if (kv_win_out)
    CUDA_TRY(c, cudaMemcpyAsync(kv_win_out, win, per_b * batch, cudaMemcpyDeviceToDevice, st));
  const size_t qbytes = (size_t)M * g.n_q_heads * g.head_dim * c->es;
  if (q_out) CUDA_TRY(c, cudaMemcpyAsync(q_out, c->q, qbytes, cudaMemcpyDeviceToDevice, st));
  if (attn_out)
    CUDA_TRY(c, cudaMemcpyAsync(attn_out, c->o, qbytes, cudaMemcpyDeviceToDevice, st));
  return WEDLM_OK;
}

int wedlm_attention(wedlm_ctx* c, int32_t batch, const void* q, const void* kv_pool,
                    const int32_t* page_table, const int32_t* seq_len, int32_t num_pages,
                    const void* kv_win, void* o, void* stream) {
  if (!c) return WEDLM_ERR_INVALID_ARG;
  const wedlm_config& g = c->cfg;
  if (batch < 1 || batch > g.max_batch || !q || !kv_pool || !page_table || !seq_len ||
      !kv_win || !o || num_pages < 1)
    return fail(c, WEDLM_ERR_INVALID_ARG, "bad attention arguments");
  cudaStream_t st = (cudaStream_t)stream;
  c->last_stream = st;
  AttnArgs A = attn_args(c, batch, ctx_win(c), q, kv_pool, page_table, seq_len, num_pages,
                         kv_win, o);
  cudaError_t e;
  {
    Timed t(c, WEDLM_KIND_ATTN, st);
    e = g.dtype == WEDLM_BF16 ? run_attention<bf16>(c, A, st)
                              : run_attention<float>(c, A, st);
  }
  if (e != cudaSuccess) return fail(c, WEDLM_ERR_CUDA, cudaGetErrorString(e));
  if (g.dtype != WEDLM_BF16) {  // the tensor-core launcher merges itself
    Timed t(c, WEDLM_KIND_ATTN_MERGE, st);
    e = launch_attention_merge<float>(A, st);
  }
  if (e != cudaSuccess) return fail(c, WEDLM_ERR_CUDA, cudaGetErrorString(e));
  return WEDLM_OK;
}

int wedlm_lm_head(wedlm_ctx* c, int32_t batch, const void* x, const int32_t* plant_token,
                  float plant_bias, wedlm_slot_rec* rows, float* logits, void* stream) {
  if (!c) return WEDLM_ERR_INVALID_ARG;
  const wedlm_config& g = c->cfg;
  if (batch < 1 || batch > g.max_batch || !x || !rows)
    return fail(c, WEDLM_ERR_INVALID_ARG, "bad lm_head arguments");
  cudaStream_t st = (cudaStream_t)stream;
  c->last_stream = st;
  const int M = batch * g.window;
  int rc = g.dtype == WEDLM_BF16
               ? lmhead_impl<bf16>(c, batch, (const bf16*)x, plant_token, plant_bias, logits, st)
               : lmhead_impl<float>(c, batch, (const float*)x, plant_token, plant_bias, logits, st);
  if (rc) return rc;
  CUDA_TRY(c, cudaMemcpyAsync(rows, c->rows, (size_t)M * sizeof(wedlm_slot_rec),
                              cudaMemcpyDeviceToDevice, st));
  return WEDLM_OK;
}

}  // extern "C"
