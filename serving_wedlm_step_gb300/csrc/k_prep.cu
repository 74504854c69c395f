// Topological Reordering + embedding gather + RoPE table, and RMSNorm.
//
// Reordering follows the WeDLM summary page (Key claims, "Topological
// Reordering ... §4.1, Eq. 5-6"; Method): a stable partition of the window
// slots, observed slots first, masked slots after, each group in slot order;
// RoPE angles use each token's LOGICAL position.
#include "internal.h"

namespace wedlm {

// cos/sin of position `p` for pair i.  The angle p * inv_freq[i] is formed
// in float64 and reduced to [-pi, pi] there (subtracting the nearest
// multiple of 2 pi; with p < 2^31 and 2 pi held to 2^-53 relative, the
// reduced angle is good to ~1e-9), then sincosf of the reduced angle: cos
// and sin are stored in float32, so a float64 sine would be rounded away.
__device__ __forceinline__ void rope_row(int p, int half, const double* inv_freq,
                                         float* cos_row, float* sin_row) {
  constexpr double kTwoPi = 6.283185307179586;
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const double a = (double)p * inv_freq[i];
    const double r = fma(-rint(a / kTwoPi), kTwoPi, a);
    float s, c;
    sincosf((float)r, &s, &c);
    cos_row[i] = c;
    sin_row[i] = s;
  }
}

// grid (W, B): block (p, b) builds physical row p of sequence b.
template <typename T>
__global__ void __launch_bounds__(128)
reorder_embed_kernel(int W, int H, int hd, int vocab, int page_cap,
                     const int32_t* __restrict__ tokens,
                     const int32_t* __restrict__ pos,
                     const uint8_t* __restrict__ obs,
                     const int32_t* __restrict__ seq_len,
                     const int32_t* __restrict__ plant,
                     const T* __restrict__ embed,
                     const double* __restrict__ inv_freq,
                     int32_t* perm_ws, int32_t* inv_ws, int32_t* pos_phys,
                     int32_t* seq_snap, int32_t* ncommit,
                     const int32_t* __restrict__ done, int32_t* plant_phys, T* x,
                     float* cosb, float* sinb, int* err, MaskedRows mr) {
  pdl_wait();  // the previous kernel's results
  pdl_trigger();
  const int p = blockIdx.x, b = blockIdx.y;
  if (mr.count && b == (int)gridDim.y - 1) {
    // an extra row of blocks (b = B) builds the masked-row map beside the
    // others: the masked rows of the whole batch in compact order (the
    // masked slots of sequence bb are its physical rows n_obs..W-1 after
    // Topological Reordering, in slot order).  The window goes to shared
    // memory, one thread counts each sequence, one thread scans the counts,
    // and one thread per sequence writes its rows.
    if (p != 0) return;
    const int B = gridDim.y - 1, n = B * W;
    __shared__ uint8_t s_o[kMaxRows];
    __shared__ int s_base[kMaxRows + 1];
    for (int i = threadIdx.x; i < n; i += blockDim.x) s_o[i] = obs[i] != 0;
    __syncthreads();
    for (int bb = threadIdx.x; bb < B; bb += blockDim.x) {
      int m = 0;
      for (int j = 0; j < W; ++j) m += !s_o[bb * W + j];
      s_base[bb + 1] = m;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      s_base[0] = 0;
      for (int bb = 0; bb < B; ++bb) s_base[bb + 1] += s_base[bb];
      *mr.count = s_base[B];
    }
    __syncthreads();
    for (int bb = threadIdx.x; bb < B; bb += blockDim.x) {
      const int base = s_base[bb], n_obs = W - (s_base[bb + 1] - base);
      int k = 0;
      for (int j = 0; j < W; ++j) {
        if (s_o[bb * W + j]) continue;
        mr.src[base + k] = bb * W + n_obs + k;
        mr.plant[base + k] = plant ? plant[bb * W + j] : -1;
        ++k;
      }
      for (int q = 0; q < W; ++q) mr.dst[bb * W + q] = q < n_obs ? -1 : base + (q - n_obs);
    }
    return;
  }
  __shared__ int s_slot;
  if (threadIdx.x == 0) {
    // physical index p -> slot: the p-th observed slot, else the
    // (p - n_obs)-th masked slot
    const uint8_t* o = obs + (size_t)b * W;
    int n_obs = 0;
    for (int j = 0; j < W; ++j) n_obs += (o[j] != 0);
    int want_obs = p < n_obs;
    int rank = want_obs ? p : p - n_obs;
    int slot = 0;
    for (int j = 0; j < W; ++j) {
      if ((o[j] != 0) == (want_obs != 0)) {
        if (rank == 0) { slot = j; break; }
        --rank;
      }
    }
    s_slot = slot;
    const int m = b * W + p;
    perm_ws[m] = slot;
    inv_ws[b * W + slot] = p;
    pos_phys[m] = pos[b * W + slot];
    if (plant_phys) plant_phys[m] = plant ? plant[b * W + slot] : -1;
    if (p == 0) {
      int L = seq_len[b];
      if (L < 0) { set_err(err, WEDLM_DEV_BAD_SEQLEN); L = 0; }
      if (L + W > page_cap) set_err(err, WEDLM_DEV_CAPACITY);
      seq_snap[b] = L;
      // commit set (Method: the leftmost contiguous filled prefix): the
      // run of slots 0..c-1 observed at input whose logical positions
      // continue the committed prefix, pos = L + i.  Known before the
      // forward, so the K/V of these rows go to their pages as they are
      // computed.  A stopped sequence commits nothing.
      int c = 0;
      if (!(done && done[b])) {
        const int32_t* ps = pos + (size_t)b * W;
        while (c < W && o[c] && ps[c] == L + c) ++c;
      }
      if (ncommit) ncommit[b] = c;
    }
  }
  __syncthreads();
  const int slot = s_slot;
  const int m = b * W + p;
  int tok = tokens[b * W + slot];
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) set_err(err, WEDLM_DEV_BAD_TOKEN);
    tok = 0;
  }
  const int half = hd / 2;
  rope_row(pos[b * W + slot], half, inv_freq, cosb + (size_t)m * half,
           sinb + (size_t)m * half);
  const uint4* src = reinterpret_cast<const uint4*>(embed + (size_t)tok * H);
  uint4* dst = reinterpret_cast<uint4*>(x + (size_t)m * H);
  const int nv = H * (int)sizeof(T) / 16;
  for (int i = threadIdx.x; i < nv; i += blockDim.x) dst[i] = src[i];
}

template <typename T>
cudaError_t launch_reorder_embed(int B, int W, int H, int hd, int vocab,
                                 int page_cap, const int32_t* tokens,
                                 const int32_t* pos, const uint8_t* obs,
                                 const int32_t* seq_len, const int32_t* plant,
                                 const T* embed, const double* inv_freq,
                                 int32_t* perm_ws, int32_t* inv_ws,
                                 int32_t* pos_phys, int32_t* seq_snap, int32_t* ncommit,
                                 const int32_t* done, int32_t* plant_phys, T* x,
                                 float* cosb, float* sinb, int* err, cudaStream_t st,
                                 const MaskedRows* mr) {
  const MaskedRows none{nullptr, nullptr, nullptr, nullptr};
  const int rows = B + (mr ? 1 : 0);  // + one row of blocks for the masked-row map
  return launch_pdl(reorder_embed_kernel<T>, dim3(W, rows), dim3(128), 0, st, W, H, hd, vocab,
                    page_cap, tokens, pos, obs, seq_len, plant, embed, inv_freq, perm_ws,
                    inv_ws, pos_phys, seq_snap, ncommit, done, plant_phys, x, cosb, sinb, err,
                    mr ? *mr : none);
}

// Prompt prefill rows (all observed, identity order): row p of sequence b
// is chunk token p at logical position seq_len[b] + p; every row is
// committed.  grid (C, B).
template <typename T>
__global__ void __launch_bounds__(128)
prefill_embed_kernel(int C, int H, int hd, int vocab, int page_cap,
                     const int32_t* __restrict__ tokens,
                     const int32_t* __restrict__ seq_len, const T* __restrict__ embed,
                     const double* __restrict__ inv_freq, int32_t* pos_phys,
                     int32_t* seq_snap, int32_t* ncommit, T* x, float* cosb,
                     float* sinb, int* err) {
  pdl_wait();  // the previous kernel's results
  pdl_trigger();
  const int p = blockIdx.x, b = blockIdx.y, m = b * C + p;
  int L = seq_len[b];
  if (L < 0) {
    if (threadIdx.x == 0 && p == 0) set_err(err, WEDLM_DEV_BAD_SEQLEN);
    L = 0;
  }
  if (threadIdx.x == 0) {
    pos_phys[m] = L + p;
    if (p == 0) {
      if (L + C > page_cap) set_err(err, WEDLM_DEV_CAPACITY);
      seq_snap[b] = L;
      ncommit[b] = C;
    }
  }
  int tok = tokens[(size_t)b * C + p];
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) set_err(err, WEDLM_DEV_BAD_TOKEN);
    tok = 0;
  }
  const int half = hd / 2;
  rope_row(L + p, half, inv_freq, cosb + (size_t)m * half, sinb + (size_t)m * half);
  const uint4* src = reinterpret_cast<const uint4*>(embed + (size_t)tok * H);
  uint4* dst = reinterpret_cast<uint4*>(x + (size_t)m * H);
  const int nv = H * (int)sizeof(T) / 16;
  for (int i = threadIdx.x; i < nv; i += blockDim.x) dst[i] = src[i];
}

template <typename T>
cudaError_t launch_prefill_embed(int B, int C, int H, int hd, int vocab, int page_cap,
                                 const int32_t* tokens, const int32_t* seq_len, const T* embed,
                                 const double* inv_freq, int32_t* pos_phys, int32_t* seq_snap,
                                 int32_t* ncommit, T* x, float* cosb, float* sinb, int* err,
                                 cudaStream_t st) {
  return launch_pdl(prefill_embed_kernel<T>, dim3(C, B), dim3(128), 0, st, C, H, hd, vocab,
                    page_cap, tokens, seq_len, embed, inv_freq, pos_phys, seq_snap, ncommit, x,
                    cosb, sinb, err);
}

// seq_len[b] = seq_snap[b] + C once the chunk's K/V are in the pages
__global__ void seq_advance_kernel(int B, int C, const int32_t* __restrict__ seq_snap,
                                   int32_t* seq_len) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) seq_len[b] = seq_snap[b] + C;
}

cudaError_t launch_seq_advance(int B, int C, const int32_t* seq_snap, int32_t* seq_len,
                               cudaStream_t st) {
  return launch_pdl(seq_advance_kernel, dim3((B + 127) / 128), dim3(128), 0, st, B, C, seq_snap,
                    seq_len);
}

__global__ void rope_table_kernel(int hd, const int32_t* __restrict__ pos_phys,
                                  const double* __restrict__ inv_freq,
                                  float* cosb, float* sinb) {
  const int m = blockIdx.x, half = hd / 2;
  rope_row(pos_phys[m], half, inv_freq, cosb + (size_t)m * half,
           sinb + (size_t)m * half);
}

cudaError_t launch_rope_table(int M, int hd, const int32_t* pos_phys,
                              const double* inv_freq, float* cosb, float* sinb,
                              cudaStream_t st) {
  rope_table_kernel<<<M, 64, 0, st>>>(hd, pos_phys, inv_freq, cosb, sinb);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// RMSNorm: y = x / sqrt(mean(x^2) + eps) * g, one block per row, fp32 math.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kNormThreads)
rmsnorm_kernel(int H, const T* __restrict__ x, const T* __restrict__ g,
               float eps, T* __restrict__ y, const int32_t* __restrict__ row_dst) {
  pdl_wait();  // the previous kernel's results
  pdl_trigger();
  constexpr int N = 16 / sizeof(T);
  const int m = blockIdx.x;
  const int my = row_dst ? row_dst[m] : m;
  if (my < 0) return;  // uniform for the block
  const T* xr = x + (size_t)m * H;
  T* yr = y + (size_t)my * H;
  const int nv = H / N;
  float ss = 0.f;
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    Vec16<T> v = ld16(xr + i * N);
#pragma unroll
    for (int k = 0; k < N; ++k) {
      float f = v.get(k);
      ss = fmaf(f, f, ss);
    }
  }
  __shared__ float red[32];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    t = warp_sum(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float r = rsqrtf(red[0] / (float)H + eps);
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    Vec16<T> v = ld16(xr + i * N), gv = ld16(g + i * N), o;
#pragma unroll
    for (int k = 0; k < N; ++k) o.set(k, v.get(k) * r * gv.get(k));
    st16(yr + i * N, o);
  }
}

template <typename T>
cudaError_t launch_rmsnorm(int M, int H, const T* x, const T* g, float eps,
                           T* y, cudaStream_t st, const int32_t* row_dst) {
  return launch_pdl(rmsnorm_kernel<T>, dim3(M), dim3(kNormThreads), 0, st, H, x, g, eps, y,
                    row_dst);
}

#define INST(T)                                                               \
  template cudaError_t launch_reorder_embed<T>(                               \
      int, int, int, int, int, int, const int32_t*, const int32_t*,           \
      const uint8_t*, const int32_t*, const int32_t*, const T*, const double*, \
      int32_t*, int32_t*, int32_t*, int32_t*, int32_t*, const int32_t*,       \
      int32_t*, T*, float*, float*, int*, cudaStream_t, const MaskedRows*);   \
  template cudaError_t launch_rmsnorm<T>(int, int, const T*, const T*, float, \
                                         T*, cudaStream_t, const int32_t*);   \
  template cudaError_t launch_prefill_embed<T>(                               \
      int, int, int, int, int, int, const int32_t*, const int32_t*, const T*, \
      const double*, int32_t*, int32_t*, int32_t*, T*, float*, float*, int*,  \
      cudaStream_t);
INST(float)
INST(bf16)
#undef INST

}  // namespace wedlm
