// bf16 weight-streaming GEMM on the 5th-generation tensor cores (tcgen05).
//
// Y[m][n] = sum_k X[m][k] W[n][k] with few activation rows (M = B*W <= 512)
// and many weight rows.  A block owns a tile of `ntile` (256, or 128 when
// M > 256) output features and every activation row: the activation rows
// take the MMA's M side in blocks of 128 (rows beyond M are zero-filled by
// the TMA), the tile's weight rows its N side.  Per block:
//   warp 0 / lane 0: TMA producer.  Each pipeline stage is one 64-wide K
//       slice: the activation row blocks and the tile's weight rows (boxes
//       of 64 rows, L2 evict-first), all with the 128-byte swizzle, in a ring
//       of shared-memory stages guarded by full/empty mbarriers;
//   warp 1 / lane 0: MMA issuer: per stage 4 x tcgen05.mma (K = 16) per row
//       block into TMEM; a tcgen05.commit frees the stage;
//   warp 2: TMEM allocation / release;
//   all 4 warps: epilogue, one activation row per thread (TMEM lane), read
//       straight from TMEM in 32-column chunks (epilogue_tc.cuh).  With
//       split-K every block stores its fp32 partial and the last block of
//       the tile sums them in split order and runs the epilogue.
#include <cudaTypedefs.h>

#include <mutex>
#include <unordered_map>

#include "epilogue_tc.cuh"
#include "gemm_tc.h"

namespace wedlm {

namespace {
constexpr int kMaxStages = 8;
constexpr int kBK = 64;                    // K elements per stage (128 bytes)
constexpr uint32_t kXBlockBytes = 128 * kBK * 2;  // one activation row block
constexpr uint32_t kWBoxBytes = 64 * kBK * 2;     // one 64-row weight box
constexpr int kThreads = 128;
constexpr int kMaxDynSmem = 221 * 1024;
}  // namespace

struct TcLaunch {
  int stages, ntile, nrb;
  uint32_t a_bytes, stage_bytes, tmem_cols;
};

__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap mW0, const __grid_constant__ CUtensorMap mW1,
               const __grid_constant__ CUtensorMap mW2, const __grid_constant__ CUtensorMap mX,
               GemmProblem P, TcLaunch L) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ __align__(8) uint64_t bar_full[kMaxStages];
  __shared__ __align__(8) uint64_t bar_empty[kMaxStages];
  __shared__ __align__(8) uint64_t bar_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_last;

  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tile = blockIdx.x, split = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = P.K / kBK;
  const int kb0 = (int)((long long)nkb * split / P.splits);
  const int kb1 = (int)((long long)nkb * (split + 1) / P.splits);
  const int niter = kb1 - kb0;
  const int ntile = L.ntile;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L.stages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_done, 1);
    mbar_fence_init();
    tma_prefetch_desc(&mW0);
    tma_prefetch_desc(&mX);
  }
  if (warp == 2) {
    tmem_alloc(&s_tmem, L.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    const int nbox = ntile / 64;
    const CUtensorMap* wmap[4];
    int wrow[4];
    for (int j = 0; j < nbox; ++j) {
      if (P.swiglu) {  // first half of the boxes: gate rows, second half: up rows
        const int hb = nbox / 2, half = ntile / 2;
        wmap[j] = j < hb ? &mW0 : &mW1;
        wrow[j] = tile * half + 64 * (j < hb ? j : j - hb);
      } else {
        const int g = tile * ntile;
        if (g < P.seg1) { wmap[j] = &mW0; wrow[j] = g + 64 * j; }
        else if (g < P.seg2) { wmap[j] = &mW1; wrow[j] = g - P.seg1 + 64 * j; }
        else { wmap[j] = &mW2; wrow[j] = g - P.seg2 + 64 * j; }
      }
    }
    const uint64_t pol = l2_evict_first_policy();
    for (int i = 0; i < niter; ++i) {
      const int s = i % L.stages;
      const uint32_t ph = (uint32_t)(i / L.stages) & 1u;
      if (!mbar_wait(&bar_empty[s], ph ^ 1u, P.err)) break;
      uint8_t* st = base + (size_t)s * L.stage_bytes;
      mbar_arrive_expect_tx(&bar_full[s], L.stage_bytes);
      const int kx = (kb0 + i) * kBK;
      for (int r = 0; r < L.nrb; ++r)
        tma_load_2d(st + r * kXBlockBytes, &mX, &bar_full[s], kx, r * 128);
      for (int j = 0; j < nbox; ++j)
        tma_load_2d_hint(st + L.a_bytes + j * kWBoxBytes, wmap[j], &bar_full[s], kx, wrow[j],
                         pol);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = idesc_bf16_m128(ntile);
    for (int i = 0; i < niter; ++i) {
      const int s = i % L.stages;
      const uint32_t ph = (uint32_t)(i / L.stages) & 1u;
      if (!mbar_wait(&bar_full[s], ph, P.err)) break;
      tc_fence_after();
      const uint32_t sa = smem_u32(base + (size_t)s * L.stage_bytes);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint64_t bd = sdesc_sw128(sa + L.a_bytes + kk * 32);
        for (int r = 0; r < L.nrb; ++r) {
          const uint64_t ad = sdesc_sw128(sa + r * kXBlockBytes + kk * 32);
          tc_mma_f16(tmem + (uint32_t)(r * ntile), ad, bd, idesc, (i | kk) != 0);
        }
      }
      tc_commit(&bar_empty[s]);
    }
    tc_commit(&bar_done);
  }
  __syncwarp();

  // ---------------- epilogue: thread = activation row ----------------
  const bool ok = __syncthreads_and(mbar_wait(&bar_done, 0, P.err)) != 0;
  tc_fence_after();
  if (ok) {
    for (int r = 0; r < L.nrb; ++r) {
      const int m = r * 128 + 32 * warp + lane;
      const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(r * ntile);
      if (P.splits == 1) {
        AccRow a{1, taddr, nullptr, 0, 1, tile * ntile, P.N, m < P.M};
        tc_epilogue_rows(P, a, m, tile, ntile);
      } else {
        float* dst = P.partial + (size_t)split * P.M * P.N + (size_t)m * P.N + tile * ntile;
        for (int c = 0; c < ntile; c += 32) {
          float v[32];
          tmem_ld32(taddr + (uint32_t)c, v);
          if (m < P.M) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (tile * ntile + c + 4 * i < P.N)
                __stcg(reinterpret_cast<float4*>(dst + c) + i,
                       make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, L.tmem_cols);
  if (!ok || P.splits == 1) return;

  // split-K: the last block of this tile reduces in split order
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&P.counters[tile], 1) == P.splits - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int r = 0; r < L.nrb; ++r) {
    const int m = r * 128 + 32 * warp + lane;
    const float* src = P.partial + (size_t)min(m, P.M - 1) * P.N + tile * ntile;
    AccRow a{0, 0, src, (size_t)P.M * P.N, P.splits, tile * ntile, P.N, m < P.M};
    tc_epilogue_rows(P, a, m, tile, ntile);
  }
  if (threadIdx.x == 0) P.counters[tile] = 0;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [rows][K] bf16 row-major, boxes of box_rows x 64 with the 128-byte swizzle
bool encode_2d(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t rows, uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {K, rows};
  cuuint64_t strides[1] = {K * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

struct TcMapTable {
  std::unordered_map<const void*, CUtensorMap> weight;
};

std::unique_ptr<TcPlanSet> make_tc_plans(const wedlm_config& g,
                                         const std::vector<LayerWeights>& layers,
                                         const void* embed, const void* lm_head, void* xn,
                                         void* o, void* act, int num_sms, size_t part_elems,
                                         std::string* msg) {
  (void)embed; (void)xn; (void)o; (void)act;
  std::unique_ptr<TcPlanSet> p(new TcPlanSet());
  p->num_sms = num_sms;
  p->part_elems = part_elems;
  p->maps = std::make_shared<TcMapTable>();
  auto add = [&](const void* w, uint64_t rows, uint64_t K) {
    CUtensorMap m;
    if (!encode_2d(&m, w, K, rows, 64)) return false;
    p->maps->weight[w] = m;
    return true;
  };
  const uint64_t H = g.hidden, hd = g.head_dim;
  for (const LayerWeights& l : layers) {
    bool okk = add(l.w_q, (uint64_t)g.n_q_heads * hd, H) &&
               add(l.w_k, (uint64_t)g.n_kv_heads * hd, H) &&
               add(l.w_v, (uint64_t)g.n_kv_heads * hd, H) &&
               add(l.w_o, H, (uint64_t)g.n_q_heads * hd) && add(l.w_gate, g.ffn, H) &&
               add(l.w_up, g.ffn, H) && add(l.w_down, H, g.ffn);
    if (!okk) {
      if (msg) *msg = "cuTensorMapEncodeTiled failed for a layer weight";
      return nullptr;
    }
  }
  if (!add(lm_head, g.vocab, H)) {
    if (msg) *msg = "cuTensorMapEncodeTiled failed for the LM head";
    return nullptr;
  }
  // dynamic shared memory: up to 220 KB of stages + 1 KB alignment slack
  const cudaError_t e = cudaFuncSetAttribute(
      gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (msg) *msg = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return nullptr;
  }
  return p;
}

// split-K factor: minimise waves x (k-blocks per block + a fixed per-block
// cost), plus a charge for the partial round trip; >= 4 k-blocks per block
int tc_choose_splits(int tiles, int nkb, int M, int N, int num_sms, size_t part_elems) {
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= 16; ++s) {
    if (s > 1 && (nkb / s < 4 || (size_t)s * M * N > part_elems)) break;
    const int waves = (tiles * s + num_sms - 1) / num_sms;
    const int kper = (nkb + s - 1) / s;
    const double cost = (double)waves * (kper + 3.0) + (s > 1 ? 2.0 : 0.0);
    if (cost < best_cost - 1e-9) { best_cost = cost; best = s; }
  }
  return best;
}

// output features per tile for a problem with M activation rows
int tc_tile_width(const GemmProblem& P) {
  if (P.M > 256) return 128;
  if (P.swiglu) return (P.N / 2) % 128 == 0 ? 256 : 128;
  if (P.seg1 % 256 || (P.seg2 - P.seg1) % 256) return 128;
  if (P.seg2 < P.N && (P.N - P.seg2) % 256) return 128;
  return 256;
}

cudaError_t launch_gemm_tc(const TcPlanSet& plans, GemmProblem P, int kind, cudaStream_t st,
                           int* tiles_out) {
  (void)kind;
  if (P.K % kBK || P.M < 1 || P.M > 512 || P.N % 4) return cudaErrorInvalidValue;
  auto find = [&](const void* w) -> const CUtensorMap* {
    auto it = plans.maps->weight.find(w);
    return it == plans.maps->weight.end() ? nullptr : &it->second;
  };
  const CUtensorMap* a0 = find(P.A0);
  const CUtensorMap* a1 = find(P.A1);
  const CUtensorMap* a2 = find(P.A2);
  if (!a0 || !a1 || !a2) return cudaErrorInvalidValue;
  TcLaunch L;
  L.ntile = tc_tile_width(P);
  L.nrb = (P.M + 127) / 128;
  L.a_bytes = (uint32_t)L.nrb * kXBlockBytes;
  L.stage_bytes = L.a_bytes + (uint32_t)L.ntile * 128u;
  L.stages = (int)std::min<uint32_t>(kMaxStages, (kMaxDynSmem - 1024) / L.stage_bytes);
  if (L.stages < 2) return cudaErrorInvalidValue;
  uint32_t cols = 32;
  while (cols < (uint32_t)(L.nrb * L.ntile)) cols <<= 1;
  if (cols > 512) return cudaErrorInvalidValue;
  L.tmem_cols = cols;
  CUtensorMap mx;
  if (!encode_2d(&mx, P.X, P.K, P.M, 128)) return cudaErrorInvalidValue;
  const int tiles = P.swiglu ? (P.N / 2) / (L.ntile / 2) : (P.N + L.ntile - 1) / L.ntile;
  if (tiles_out) *tiles_out = tiles;
  P.splits = tc_choose_splits(tiles, P.K / kBK, P.M, P.N, plans.num_sms, plans.part_elems);
  const size_t smem = (size_t)L.stages * L.stage_bytes + 1024;
  gemm_tc_kernel<<<dim3(tiles, P.splits), kThreads, smem, st>>>(*a0, *a1, *a2, mx, P, L);
  return cudaGetLastError();
}

}  // namespace wedlm
