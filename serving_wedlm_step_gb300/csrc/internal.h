// Internal launch interfaces of libwedlm (host side).
#pragma once

#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <set>
#include <string>
#include <utility>
#include <vector>

#include "common.cuh"

namespace wedlm {

// Raise a kernel's dynamic shared-memory limit on the current device.  The
// attribute belongs to (kernel, device): it is set once per pair, under a
// lock, so launches on a second device (or from several threads) see it too.
inline cudaError_t ensure_dyn_smem(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({kernel, dev});
  return e;
}

// Launch with programmatic stream serialization (see pdl_wait): the kernel
// must call pdl_wait before touching the previous kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// threads of one RMSNorm block (one block per row); the fused residual +
// norm epilogue uses the same count so that both reduce in the same order
constexpr int kNormThreads = 512;

enum EpiMode { EPI_RESID = 0, EPI_SWIGLU = 1, EPI_QKV = 2, EPI_LMHEAD = 3 };

#ifdef __CUDACC__
// Element (token t % 16, dim d) of K (kv = 0) or V (kv = 1), kv head kvh,
// of the page holding position t of sequence b, for a committed window row;
// null when the position is beyond the page table or its page id is out of
// range (the error word records which).
template <typename T, typename Epi>
__device__ __forceinline__ T* commit_dst(const Epi& e, int b, int t, int kv, int kvh, int d) {
  const int pg = t / kPageBlock;
  if (pg >= e.max_pages) {
    set_err(e.err, WEDLM_DEV_CAPACITY);
    return nullptr;
  }
  const int page = e.page_table[(size_t)b * e.max_pages + pg];
  if (page < 0 || page >= e.num_pages) {
    set_err(e.err, WEDLM_DEV_BAD_PAGE);
    return nullptr;
  }
  return static_cast<T*>(e.pool) + (((size_t)page * 2 + kv) * e.nkv + kvh) * kPageBlock * e.hd +
         tile_off(t % kPageBlock, d, e.hd);
}
#endif

// Epilogue of the weight-streaming GEMM Y[m][n] = sum_k X[m][k] W[n][k].
struct GemmEpi {
  int mode;
  void* x;              // RESID: residual stream [M][N], updated in place
  const void* norm_w;   // RESID (tensor-core path): when set, also write
  void* xn;             //   xn = RMSNorm(x) * norm_w (eps below) for the next GEMM
  void* act;            // SWIGLU: out [M][N/2] = silu(gate) * up
  // QKV
  void* q_out;          // [M][nq*hd]
  void* kv_win;         // this layer's window K/V [B][2][nkv][Wp*hd] (tiled)
  const float* cosb;    // [M][hd/2]
  const float* sinb;
  const void* q_norm;   // [hd] or null
  const void* k_norm;
  int qk_norm, W, Wp, nq, nkv, hd;
  float eps;
  // QKV, commit into the paged cache: window row p of sequence b with
  // p < commit_n[b] (the leftmost observed run, physical rows 0..c-1) also
  // writes its K and V at position commit_base[b] + p of `pool`
  const int32_t* commit_n;     // [B] or null (nothing committed)
  const int32_t* commit_base;  // [B]
  const int32_t* page_table;   // [B][max_pages]
  void* pool;                  // this layer's KV pool
  int max_pages, num_pages;
  int* err;
  // LMHEAD
  SoftmaxPart* part;    // [tiles][M]
  int mask_id, vocab;
  const int32_t* plant; // [M] or null
  float plant_bias;
  float* logits;        // [M][vocab] or null
  const int32_t* row_src;  // LMHEAD on compacted rows: logits row of row m, or null
  // RESID with the next RMSNorm: normed row m goes to row row_dst[m] of xn
  // (skipped when negative), or to row m when null
  const int32_t* row_dst;
};

// One weight-streaming GEMM.  Output features come in tiles of 128 rows of
// the weight; the rows of a tile come from A0/A1/A2 (q/k/v segments) or,
// for SWIGLU, rows 0..63 from A0 (gate) and 64..127 from A1 (up).
struct GemmProblem {
  int M, N, K;
  const void* X;        // [M][K]
  const void* A0;
  const void* A1;
  const void* A2;
  int seg1, seg2;       // segment row boundaries (QKV); N otherwise
  int swiglu;
  int splits;
  const int* m_count;   // rows actually present (<= M, read on the device), or
                        // null for all M; only for splits == 1
  float* partial;       // [splits][M][N] fp32 (splits > 1)
  int* counters;        // [tiles], zero between launches
  int* err;
  GemmEpi epi;
};

// A tensor-core attention unit's start (Q, the first tile) and end (normalise
// and write, or partial and merge) cost about as much as this many of its
// 128-key tiles; the stream-K shares count them.  Swept 0..8 on GB300: 3 is
// best for the decode step (0 is the plain tile split).
constexpr int kAttnUnitCost = 3;

struct AttnArgs {
  int B, W, Wp, nq, nkv, hd, chunk, max_chunks, num_pages, max_pages;
  int pt_stride;        // page-table row of sequence b starts at b * pt_stride
                        // (max_pages; 0: every sequence reads row 0)
  int kv_reuse;         // 1: pages are read by many units (keep them in L2)
  float scale_log2;     // log2(e) / sqrt(hd)
  const void* q;        // [B*W][nq][hd]
  const void* pool;     // this layer's pool
  const int32_t* page_table;
  const int32_t* seq_len;
  const void* kv_win;   // [B][2][nkv][Wp*hd]
  float* part_o;        // [B][nkv][max_chunks][G*W][hd]
  float* part_ml;       // [B][nkv][max_chunks][G*W][2]
  void* o;              // [B*W][nq*hd]
  int* err;
  // tensor-core (stream-K) attention: partials per segment
  int min_tiles;        // fewest 64-key tiles a block is given
  int unit_cost;        // tensor-core attention: tiles' worth of time a unit's
                        // start and end cost, counted when the work is cut
                        // into the blocks' shares (0: tiles only)
  int* unit_cnt;        // [B*nkv]: segments of each unit written so far (zero
                        // between launches; the unit's merging block resets it)
};

struct LayerWeights {
  const void *attn_norm, *w_q, *w_k, *w_v, *q_norm, *k_norm, *w_o, *ffn_norm,
      *w_gate, *w_up, *w_down;
};

// host launchers (one per kernel family); each returns cudaGetLastError()
// The masked rows of a step in compact order (LM head on masked slots
// only): physical row of compact row i, compact row of physical row m (-1
// for observed rows), the planted token of compact row i, their count.
struct MaskedRows {
  int32_t* src;
  int32_t* dst;
  int32_t* plant;
  int* count;
};

template <typename T>
cudaError_t launch_reorder_embed(int B, int W, int H, int hd, int vocab,
                                 int page_cap, const int32_t* tokens,
                                 const int32_t* pos, const uint8_t* obs,
                                 const int32_t* seq_len, const int32_t* plant,
                                 const T* embed, const double* inv_freq,
                                 int32_t* perm_ws, int32_t* inv_ws,
                                 int32_t* pos_phys, int32_t* seq_snap,
                                 int32_t* ncommit, const int32_t* done,
                                 int32_t* plant_phys, T* x, float* cosb,
                                 float* sinb, int* err, cudaStream_t st,
                                 const MaskedRows* mr = nullptr);
template <typename T>
cudaError_t launch_prefill_embed(int B, int C, int H, int hd, int vocab, int page_cap,
                                 const int32_t* tokens, const int32_t* seq_len, const T* embed,
                                 const double* inv_freq, int32_t* pos_phys, int32_t* seq_snap,
                                 int32_t* ncommit, T* x, float* cosb, float* sinb, int* err,
                                 cudaStream_t st);
cudaError_t launch_seq_advance(int B, int C, const int32_t* seq_snap, int32_t* seq_len,
                               cudaStream_t st);
cudaError_t launch_rope_table(int M, int hd, const int32_t* pos_phys,
                              const double* inv_freq, float* cosb, float* sinb,
                              cudaStream_t st);
// y[row_dst[m]] = RMSNorm(x[m]) * g (rows with row_dst[m] < 0 skipped), or
// y[m] when row_dst is null
template <typename T>
cudaError_t launch_rmsnorm(int M, int H, const T* x, const T* g, float eps,
                           T* y, cudaStream_t st, const int32_t* row_dst = nullptr);
template <typename T>
cudaError_t launch_gemm_simt(const GemmProblem& P, cudaStream_t st);
template <typename T>
cudaError_t launch_attention(const AttnArgs& A, cudaStream_t st);
template <typename T>
cudaError_t launch_attention_merge(const AttnArgs& A, cudaStream_t st);
// tensor-core attention (bf16, head_dim 128; the segment merge is inside);
// grid = blocks (one per SM); zero_page: 4 KiB of zeros in device memory.
// The G*W query rows of a kv head run in row blocks of at most 128 rows
// (attention_tc_row_blocks gives their number, or 0 for an unsupported
// shape, and the rows per block); part_o / part_ml must hold
// grid + B*nkv*row_blocks segments of rows_per_block rows and unit_cnt
// B*nkv*row_blocks counters.
cudaError_t launch_attention_tc(const AttnArgs& A, const void* zero_page, int grid,
                                cudaStream_t st, bool pdl = true);
int attention_tc_row_blocks(int nq, int nkv, int W, int* rows_per_block);
cudaError_t launch_lmhead_merge(int M, int tiles, const SoftmaxPart* part,
                                wedlm_slot_rec* rows, int* err,
                                cudaStream_t st, const int* m_count = nullptr);

enum ScoreMode { SCORE_ENTROPY = 0, SCORE_NEGLOGP = 1 };

struct SelArgs {
  int B, W, mask_id;
  float alpha, tau;
  int score_mode;             // ScoreMode
  // streaming generation (all optional): done[b] = 1 marks a stopped
  // sequence (left unchanged); a sequence stops once seq_len reaches
  // stop_len[b] or after committing stop_token; committed tokens are also
  // written to out_tokens[b][pos - out_base[b]] when 0 <= that < out_cap
  int32_t* done;
  const int32_t* stop_len;
  int stop_token;
  int32_t* out_tokens;
  const int32_t* out_base;
  int out_cap;
  const int32_t* tokens;
  const int32_t* pos;
  const uint8_t* obs;
  const int32_t* seq_snap;
  int32_t* seq_len;
  const int32_t* inv;
  const wedlm_slot_rec* rows;
  int32_t* new_tokens;
  int32_t* new_pos;
  uint8_t* new_obs;
  int32_t* committed;
  int32_t* n_committed;
  const int32_t* ncommit_ws;  // commit counts found at step start (reorder)
  uint8_t* filled;
  const int32_t* row_dst;     // compact LM-head row of physical row m, or null
                              // (records indexed by physical row)
  wedlm_slot_rec* out_rows;   // [B*W] per physical row (observed: no record), or null
};
cudaError_t launch_select(const SelArgs& S, cudaStream_t st);

struct PoolPtrs {
  void* p[kMaxLayers];
};
struct CommitArgs {
  int B, W, Wp, nkv, hd, n_layers, max_pages, num_pages;
  size_t win_layer_stride;  // elements per layer of the window scratch
  const void* kv_win;
  const int32_t* inv;
  const int32_t* seq_snap;
  const int32_t* ncommit;
  const int32_t* page_table;
  int* err;
  PoolPtrs pools;
};
template <typename T>
cudaError_t launch_commit(const CommitArgs& C, cudaStream_t st);

}  // namespace wedlm
