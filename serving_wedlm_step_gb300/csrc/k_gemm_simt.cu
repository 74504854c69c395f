// Weight-streaming GEMM, CUDA-core mainloop (fp32 contexts: the tensor
// cores have no fp32 x fp32 mode that keeps 1e-4 parity).
//
// Y[m][n] = sum_k X[m][k] * Wt[n][k].  Grid (tiles of 128 weight rows,
// split-K).  Each block computes 128 features x 64 activation rows per pass,
// stages the fp32 tile in shared memory and runs the fused epilogue; with
// split-K, the last block to finish a tile sums the partials in split order
// (deterministic) and runs the epilogue.
#include "epilogue.cuh"

namespace wedlm {

namespace {
constexpr int BK = 16, BMF = 128, BNM = 64;
constexpr int AS_LD = BMF + 4, XS_LD = BNM + 4;

template <typename T>
__device__ __forceinline__ const T* a_row(const GemmProblem& P, int tile,
                                          int row) {
  if (P.swiglu) {
    const T* base = static_cast<const T*>(row < 64 ? P.A0 : P.A1);
    return base + (size_t)(tile * 64 + (row & 63)) * P.K;
  }
  int g = tile * 128 + row;
  if (g >= P.N) g = P.N - 1;  // tail rows: computed, then ignored
  if (g < P.seg1) return static_cast<const T*>(P.A0) + (size_t)g * P.K;
  if (g < P.seg2) return static_cast<const T*>(P.A1) + (size_t)(g - P.seg1) * P.K;
  return static_cast<const T*>(P.A2) + (size_t)(g - P.seg2) * P.K;
}
}  // namespace

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmProblem P) {
  extern __shared__ float smem[];
  float* As = smem;                    // [BK][AS_LD]
  float* Xs = As + BK * AS_LD;         // [BK][XS_LD]
  float* sacc = Xs + BK * XS_LD;       // [128][128] (finish pass uses 128 rows)
  const int tile = blockIdx.x, split = blockIdx.y;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int nk = P.K / BK;
  const int kb0 = (int)((long long)nk * split / P.splits);
  const int kb1 = (int)((long long)nk * (split + 1) / P.splits);
  const T* X = static_cast<const T*>(P.X);
  const int arow = tid >> 1, ak = (tid & 1) * 8;
  const T* ap = a_row<T>(P, tile, arow);
  const int xr = tid >> 2, xk = (tid & 3) * 4;
  // activation rows present (the LM head on masked rows reads their count)
  const int m_live = P.m_count ? min(P.M, max(0, *P.m_count)) : P.M;

  for (int m0 = 0; m0 < m_live; m0 += BNM) {
    const int mc = min(BNM, m_live - m0);
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int kb = kb0; kb < kb1; ++kb) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        As[(ak + j) * AS_LD + arow] = to_f(ap[kb * BK + ak + j]);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        Xs[(xk + j) * XS_LD + xr] =
            (m0 + xr < m_live) ? to_f(X[(size_t)(m0 + xr) * P.K + kb * BK + xk + j])
                            : 0.f;
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < BK; ++kk) {
        float a[8], x[4];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = As[kk * AS_LD + ty * 8 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = Xs[kk * XS_LD + tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], x[j], acc[i][j]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        sacc[(tx * 4 + j) * 128 + ty * 8 + i] = acc[i][j];
    __syncthreads();
    stage_chunk<T>(P, sacc, m0, mc, tile, split);
    __syncthreads();
  }
  if (P.splits > 1) splitk_finish<T>(P, sacc, tile);
}

template <typename T>
cudaError_t launch_gemm_simt(const GemmProblem& P, cudaStream_t st) {
  const int tiles = P.swiglu ? P.N / 128 : (P.N + 127) / 128;
  const size_t smem = (size_t)(BK * AS_LD + BK * XS_LD + 128 * 128) * sizeof(float);
  const cudaError_t ae = ensure_dyn_smem((const void*)gemm_simt_kernel<T>, (int)smem);
  if (ae != cudaSuccess) return ae;
  gemm_simt_kernel<T><<<dim3(tiles, P.splits), 256, smem, st>>>(P);
  return cudaGetLastError();
}

template cudaError_t launch_gemm_simt<float>(const GemmProblem&, cudaStream_t);
template cudaError_t launch_gemm_simt<bf16>(const GemmProblem&, cudaStream_t);

}  // namespace wedlm
