// Paged causal GQA window attention, CUDA-core version, plus the split-KV
// merge.
//
// The step is "a small causal prefill over the active window on top of
// cached KV" (WeDLM summary page, Key claims §5.2): query row p of sequence
// b (physical order) sees every cached prefix position 0..L_b-1 and window
// rows 0..p (lower-triangular mask, §3.2).  q head h reads kv head
// h / (nq/nkv).
//
// Work unit = (sequence, kv head, key chunk).  Chunks 0..ceil(L/chunk)-1
// cover the prefix; the last chunk is the window.  Each block keeps the
// G*W query rows of its kv head (G = nq/nkv) in registers, TPR threads per
// row, each owning DPT interleaved head dims (d = sub + TPR*i), streams
// 16-token pages through shared memory, and writes an unnormalised partial
// (o, running max m, sum l) in the log2 domain.
#pragma once
#include "internal.h"

namespace wedlm {

template <typename T, int DPT>
__global__ void __launch_bounds__(512)
attn_simt_kernel(AttnArgs A) {
  constexpr int KP = kPageBlock;
  const int b = blockIdx.z, kvh = blockIdx.y, c = blockIdx.x;
  const int hd = A.hd, G = A.nq / A.nkv, R = G * A.W;
  const int TPR = hd / DPT;
  const int L = max(0, min(A.seq_len[b], A.max_pages * kPageBlock));
  const int n_pre = (L + A.chunk - 1) / A.chunk;
  if (c > n_pre) return;                      // no work for this chunk
  const bool window = (c == n_pre);

  extern __shared__ float sm[];
  float* Ks = sm;                 // [KP][hd]
  float* Vs = Ks + KP * hd;       // [KP][hd]
  __shared__ int s_valid;

  const int tid = threadIdx.x;
  const int r = tid / TPR, sub = tid % TPR;
  const bool active = r < R;
  const int g = r / A.W, p = r % A.W;
  const int h = kvh * G + g;
  const int m = b * A.W + p;

  float q[DPT], o[DPT];
  const T* qp = static_cast<const T*>(A.q) + ((size_t)m * A.nq + h) * hd;
#pragma unroll
  for (int i = 0; i < DPT; ++i) {
    q[i] = active ? to_f(qp[sub + TPR * i]) * A.scale_log2 : 0.f;
    o[i] = 0.f;
  }
  float mrun = -INFINITY, l = 0.f;

  int k0, k1;
  if (window) { k0 = 0; k1 = A.W; }
  else { k0 = c * A.chunk; k1 = min(L, k0 + A.chunk); }
  const T* pool = static_cast<const T*>(A.pool);
  const size_t blockn = (size_t)KP * hd;

  for (int t0 = k0; t0 < k1; t0 += KP) {
    // stage one 16-token page of K and V (tile layout -> row-major fp32)
    const T* kb;
    const T* vb;
    if (window) {
      const T* wb = static_cast<const T*>(A.kv_win);
      kb = wb + (((size_t)b * 2 + 0) * A.nkv + kvh) * A.Wp * hd + (size_t)(t0 / KP) * blockn;
      vb = wb + (((size_t)b * 2 + 1) * A.nkv + kvh) * A.Wp * hd + (size_t)(t0 / KP) * blockn;
      if (tid == 0) s_valid = 1;
    } else {
      const int pg_idx = t0 / KP;
      int page = (pg_idx < A.max_pages) ? A.page_table[(size_t)b * A.max_pages + pg_idx] : -1;
      const bool ok = page >= 0 && page < A.num_pages;
      if (!ok) {
        if (tid == 0) set_err(A.err, WEDLM_DEV_BAD_PAGE);
        page = 0;
      }
      if (tid == 0) s_valid = ok;
      kb = pool + (((size_t)page * 2 + 0) * A.nkv + kvh) * blockn;
      vb = pool + (((size_t)page * 2 + 1) * A.nkv + kvh) * blockn;
    }
    __syncthreads();
    const bool page_ok = s_valid;
    for (int e = tid; e < KP * hd; e += blockDim.x) {
      const int t = e / hd, d = e % hd;
      const int off = tile_off(t, d, hd);
      Ks[e] = page_ok ? to_f(kb[off]) : 0.f;
      Vs[e] = page_ok ? to_f(vb[off]) : 0.f;
    }
    __syncthreads();
    float s[KP];
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < KP; ++j) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < DPT; ++i) acc = fmaf(q[i], Ks[j * hd + sub + TPR * i], acc);
      for (int off = TPR >> 1; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
      const int key = t0 + j;
      const bool ok = page_ok && key < k1 && (!window || key <= p);
      s[j] = ok ? acc : -INFINITY;
      tmax = fmaxf(tmax, s[j]);
    }
    const float mnew = fmaxf(mrun, tmax);
    if (mnew > -INFINITY) {
      const float scale = exp2f(mrun - mnew);
      l *= scale;
#pragma unroll
      for (int i = 0; i < DPT; ++i) o[i] *= scale;
#pragma unroll
      for (int j = 0; j < KP; ++j) {
        const float pj = exp2f(s[j] - mnew);
        l += pj;
#pragma unroll
        for (int i = 0; i < DPT; ++i) o[i] = fmaf(pj, Vs[j * hd + sub + TPR * i], o[i]);
      }
      mrun = mnew;
    }
    __syncthreads();
  }
  if (!active) return;
  const size_t unit = ((size_t)b * A.nkv + kvh) * A.max_chunks + c;
  float* po = A.part_o + (unit * R + r) * hd;
#pragma unroll
  for (int i = 0; i < DPT; ++i) po[sub + TPR * i] = o[i];
  if (sub == 0) {
    A.part_ml[(unit * R + r) * 2 + 0] = mrun;
    A.part_ml[(unit * R + r) * 2 + 1] = l;
  }
}

// DPT variants compiled per element type (fp32 contexts only: bf16 runs
// the tensor-core attention)
template <typename T> struct AttnVariants;
template <> struct AttnVariants<float> {
  static cudaError_t launch(int dpt, dim3 g, int th, size_t sm, cudaStream_t st,
                            const AttnArgs& A);
};

template <typename T>
cudaError_t launch_attention(const AttnArgs& A, cudaStream_t st) {
  const int R = (A.nq / A.nkv) * A.W;
  int dpt = 4;
  while (dpt < A.hd && R * (A.hd / dpt) > 512) dpt *= 2;
  if (R * (A.hd / dpt) > 512 || A.hd / dpt > 32) return cudaErrorInvalidValue;
  const int threads = ((R * (A.hd / dpt) + 31) / 32) * 32;
  const size_t smem = 2 * kPageBlock * A.hd * sizeof(float);
  dim3 grid(A.max_chunks, A.nkv, A.B);
  return AttnVariants<T>::launch(dpt, grid, threads, smem, st, A);
}

// merge the chunk partials of one (sequence, row, q head): one block per
// (b*W + p, h), one thread per head dim
template <typename T>
__global__ void attn_merge_kernel(AttnArgs A) {
  const int mh = blockIdx.x;
  const int m = mh / A.nq, h = mh % A.nq;
  const int b = m / A.W, p = m % A.W;
  const int G = A.nq / A.nkv, kvh = h / G, g = h % G, R = G * A.W;
  const int r = g * A.W + p;
  const int L = max(0, min(A.seq_len[b], A.max_pages * kPageBlock));
  const int nc = (L + A.chunk - 1) / A.chunk + 1;
  const size_t unit0 = ((size_t)b * A.nkv + kvh) * A.max_chunks;
  float M = -INFINITY;
  for (int c = 0; c < nc; ++c) M = fmaxf(M, A.part_ml[((unit0 + c) * R + r) * 2]);
  float lsum = 0.f;
  const int d = threadIdx.x;
  float acc = 0.f;
  for (int c = 0; c < nc; ++c) {
    const float mc = A.part_ml[((unit0 + c) * R + r) * 2];
    if (mc == -INFINITY) continue;
    const float w = exp2f(mc - M);
    lsum += A.part_ml[((unit0 + c) * R + r) * 2 + 1] * w;
    if (d < A.hd) acc += A.part_o[((unit0 + c) * R + r) * A.hd + d] * w;
  }
  if (d < A.hd)
    static_cast<T*>(A.o)[(size_t)m * A.nq * A.hd + h * A.hd + d] =
        from_f<T>(lsum > 0.f ? acc / lsum : 0.f);
}

template <typename T>
cudaError_t launch_attention_merge(const AttnArgs& A, cudaStream_t st) {
  attn_merge_kernel<T><<<A.B * A.W * A.nq, A.hd, 0, st>>>(A);
  return cudaGetLastError();
}

}  // namespace wedlm
