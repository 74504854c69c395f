// LM-head record merge, Eq. 11 selection, commit and refill.
//
// WeDLM summary page, Method section: each step "commits the leftmost
// contiguous filled prefix (which is immediately cache-valid because of
// strict causality), picks additional masks to fill using
// distance-penalized entropy H~_j = H_j + alpha*d_j (where d_j is distance
// from slot j to the leftmost remaining mask), and refills the freed slots
// with new [M] tokens".  Readings: score = entropy (nats), or -ln p_max
// for the confidence reading of the rule (Key claims §5.2 calls Eq. 11 a
// "distance-penalized confidence rule"); fill every masked slot with
// H~ < tau, else the single argmin (ties: lowest slot, NaN = +inf);
// d_j = pos_j - pos_m0 for the leftmost masked slot m0 at input; commit =
// slots 0..c-1 observed at input with pos = L + i (counted by the reorder
// kernel at step start, when the K/V of those rows are written to pages).
#include "internal.h"

namespace wedlm {

// ---------------------------------------------------------------------------
// merge per-vocab-tile softmax records into (argmax, H, p_max, lse) per row
// ---------------------------------------------------------------------------
__device__ __forceinline__ void combine(SoftmaxPart& a, const SoftmaxPart& b) {
  if (b.s <= 0.f && b.m == -INFINITY) return;            // b empty
  if (a.s <= 0.f && a.m == -INFINITY) { a = b; return; }  // a empty
  const float M = fmaxf(a.m, b.m);
  const float ea = expf(a.m - M), eb = expf(b.m - M);
  const float s = a.s * ea + b.s * eb;
  // sum (z - M) e^(z - M) = e^(m - M) * (u + (m - M) s) per side
  const float u = ea * (a.u + (a.m - M) * a.s) + eb * (b.u + (b.m - M) * b.s);
  int am;
  if (a.m > b.m) am = a.a;
  else if (b.m > a.m) am = b.a;
  else am = min(a.a, b.a);
  a.m = M; a.s = s; a.u = u; a.a = am;
}

__global__ void lmhead_merge_kernel(int M, int tiles,
                                    const SoftmaxPart* __restrict__ part,
                                    wedlm_slot_rec* __restrict__ rows,
                                    int* err, const int* m_count) {
  pdl_wait();  // the previous kernel's results
  pdl_trigger();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= M || (m_count && warp >= *m_count)) return;
  SoftmaxPart acc;
  acc.m = -INFINITY; acc.a = INT32_MAX; acc.s = 0.f; acc.u = 0.f;
  // this lane's records in tile order; the loads of eight go out before
  // they are combined (one L2 round trip per eight, the order unchanged)
  for (int t0 = lane; t0 < tiles; t0 += 8 * 32) {
    SoftmaxPart r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (t0 + 32 * k < tiles) r[k] = part[(size_t)(t0 + 32 * k) * M + warp];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (t0 + 32 * k < tiles) combine(acc, r[k]);
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    SoftmaxPart b;
    b.m = __shfl_xor_sync(0xffffffffu, acc.m, o);
    b.a = __shfl_xor_sync(0xffffffffu, acc.a, o);
    b.s = __shfl_xor_sync(0xffffffffu, acc.s, o);
    b.u = __shfl_xor_sync(0xffffffffu, acc.u, o);
    // combine in lane order so every lane holds the same bits
    SoftmaxPart lo = (lane & o) ? b : acc, hi = (lane & o) ? acc : b;
    combine(lo, hi);
    acc = lo;
  }
  if (lane == 0) {
    wedlm_slot_rec r;
    const float lns = logf(acc.s);
    r.argmax = acc.a;
    r.entropy = lns - acc.u / acc.s;
    r.p_max = 1.0f / acc.s;
    r.lse = acc.m + lns;
    if (!isfinite(r.entropy) || !isfinite(r.lse)) set_err(err, WEDLM_DEV_NUMERIC);
    rows[warp] = r;
  }
}

cudaError_t launch_lmhead_merge(int M, int tiles, const SoftmaxPart* part,
                                wedlm_slot_rec* rows, int* err,
                                cudaStream_t st, const int* m_count) {
  const int threads = 128;
  const int blocks = (M * 32 + threads - 1) / threads;
  return launch_pdl(lmhead_merge_kernel, dim3(blocks), dim3(threads), 0, st, M, tiles, part, rows,
                    err, m_count);
}

// ---------------------------------------------------------------------------
// Eq. 11 selection + commit run + refill: one block of 64 threads per
// sequence, thread j = slot j
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kMaxWindow) select_kernel(SelArgs S) {
  pdl_wait();  // the previous kernel's results
  pdl_trigger();
  const int b = blockIdx.x, j = threadIdx.x, W = S.W;
  __shared__ int s_obs[kMaxWindow], s_pos[kMaxWindow], s_tok[kMaxWindow];
  __shared__ int s_sel[kMaxWindow], s_fill_tok[kMaxWindow];
  __shared__ float s_ht[kMaxWindow];
  __shared__ int s_m0, s_done;
  const int L = S.seq_snap[b];
  // the window may be updated in place (out == in): everything is read
  // into shared memory before anything is written
  if (j < W) {
    s_obs[j] = S.obs[b * W + j] != 0;
    s_pos[j] = S.pos[b * W + j];
    s_tok[j] = S.tokens[b * W + j];
  }
  if (j == 0) s_done = S.done ? S.done[b] : 0;
  __syncthreads();
  const bool stopped = s_done != 0;
  const int c = stopped ? 0 : S.ncommit_ws[b];
  if (j == 0) {
    int m0 = -1;
    for (int i = 0; i < W; ++i)
      if (!s_obs[i]) { m0 = i; break; }
    s_m0 = stopped ? -1 : m0;
  }
  __syncthreads();
  const int m0 = s_m0;
  // a row without a record (observed: the LM head ran on masked rows only)
  wedlm_slot_rec none;
  none.argmax = -1;
  none.entropy = none.p_max = none.lse = __int_as_float(0x7fc00000);
  auto record = [&](int phys) {  // the record of physical row phys of sequence b
    const int ci = S.row_dst ? S.row_dst[b * W + phys] : b * W + phys;
    return ci >= 0 ? S.rows[ci] : none;
  };
  if (j < W && S.out_rows) S.out_rows[b * W + j] = record(j);
  if (j < W) {
    const wedlm_slot_rec rec = record(S.inv[b * W + j]);
    s_fill_tok[j] = rec.argmax;
    float ht = __int_as_float(0x7fc00000);  // NaN at observed slots
    int sel = 0;
    if (!s_obs[j] && !stopped) {
      const float d = (float)(s_pos[j] - s_pos[m0]);
      const float score = S.score_mode == SCORE_NEGLOGP ? -logf(rec.p_max) : rec.entropy;
      ht = __fadd_rn(score, __fmul_rn(S.alpha, d));
      sel = ht < S.tau;
    }
    s_ht[j] = ht;
    s_sel[j] = sel;
  }
  __syncthreads();
  if (j == 0 && m0 >= 0) {
    int any = 0;
    for (int i = 0; i < W; ++i) any |= s_sel[i];
    if (!any) {
      int best = -1;
      float bv = INFINITY;
      for (int i = 0; i < W; ++i) {
        if (s_obs[i]) continue;
        const float v = isnan(s_ht[i]) ? INFINITY : s_ht[i];
        if (best < 0 || v < bv) { best = i; bv = v; }
      }
      s_sel[best] = 1;
    }
  }
  __syncthreads();
  if (j < W) {
    const int src = j + c;
    int tok, pos, ob;
    if (src < W) {
      tok = s_sel[src] ? s_fill_tok[src] : s_tok[src];
      ob = s_obs[src] | s_sel[src];
      pos = s_pos[src];
    } else {
      tok = S.mask_id;
      ob = 0;
      pos = s_pos[W - 1] + (src - W + 1);
    }
    S.new_tokens[b * W + j] = tok;
    S.new_pos[b * W + j] = pos;
    S.new_obs[b * W + j] = (uint8_t)ob;
    S.committed[b * W + j] = j < c ? s_tok[j] : -1;
    if (S.filled) S.filled[b * W + j] = (uint8_t)s_sel[j];
    if (S.out_tokens && j < c) {
      const int k = L + j - S.out_base[b];
      if (k >= 0 && k < S.out_cap) S.out_tokens[(size_t)b * S.out_cap + k] = s_tok[j];
    }
  }
  // stop after committing the stop token or on reaching the length budget
  int hit = (j < c && s_tok[j] == S.stop_token && S.stop_token >= 0) ? 1 : 0;
  hit = __syncthreads_or(hit);
  if (j == 0) {
    S.n_committed[b] = c;
    S.seq_len[b] = L + c;
    if (S.done && !stopped && (hit || (S.stop_len && L + c >= S.stop_len[b]))) S.done[b] = 1;
  }
}

cudaError_t launch_select(const SelArgs& S, cudaStream_t st) {
  return launch_pdl(select_kernel, dim3(S.B), dim3(kMaxWindow), 0, st, S);
}

// ---------------------------------------------------------------------------
// commit: copy the committed slots' window K/V (every layer) into the pages
// at positions L..L+c-1, 16-byte vectors.  Grid (B, n_layers * 2 * nkv).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(128) commit_kernel(CommitArgs C) {
  pdl_wait();  // the previous kernel's results
  pdl_trigger();
  constexpr int VN = 16 / sizeof(T);
  const int b = blockIdx.x;
  const int y = blockIdx.y;
  const int layer = y / (2 * C.nkv), rem = y % (2 * C.nkv);
  const int kv = rem / C.nkv, h = rem % C.nkv;
  const int c = C.ncommit[b], L = C.seq_snap[b], hd = C.hd;
  T* pool = static_cast<T*>(C.pools.p[layer]);
  const T* win = static_cast<const T*>(C.kv_win) + layer * C.win_layer_stride +
                 (((size_t)b * 2 + kv) * C.nkv + h) * C.Wp * hd;
  const int nvec = hd / VN;
  for (int idx = threadIdx.x; idx < c * nvec; idx += blockDim.x) {
    const int i = idx / nvec, d = (idx % nvec) * VN;
    const int phys = C.inv[b * C.W + i];
    const int t = L + i, pg = t / kPageBlock;
    if (pg >= C.max_pages) { set_err(C.err, WEDLM_DEV_CAPACITY); continue; }
    const int page = C.page_table[(size_t)b * C.max_pages + pg];
    if (page < 0 || page >= C.num_pages) { set_err(C.err, WEDLM_DEV_BAD_PAGE); continue; }
    T* dst = pool + (((size_t)page * 2 + kv) * C.nkv + h) * kPageBlock * hd +
             tile_off(t % kPageBlock, d, hd);
    st16(dst, ld16(win + tile_off(phys, d, hd)));
  }
}

template <typename T>
cudaError_t launch_commit(const CommitArgs& C, cudaStream_t st) {
  return launch_pdl(commit_kernel<T>, dim3(C.B, C.n_layers * 2 * C.nkv), dim3(128), 0, st, C);
}

template cudaError_t launch_commit<float>(const CommitArgs&, cudaStream_t);
template cudaError_t launch_commit<bf16>(const CommitArgs&, cudaStream_t);

}  // namespace wedlm
