// bf16 weight-streaming GEMM on the 5th-generation tensor cores (tcgen05).
//
// Y[m][n] = sum_k X[m][k] W[n][k] with few activation rows (M = B*W <= 512)
// and many weight rows.  Work unit = (tile of `ntile` output features,
// K split).  The activation rows take the MMA's M side in blocks of 128
// (rows beyond M are zero-filled by the TMA), the tile's weight rows its N
// side.  Persistent, warp-specialised: one block per SM loops over work
// units;
//   warp 0 / lane 0: TMA producer.  Each pipeline stage is one 64-wide K
//       slice: the activation row blocks and the tile's weight rows (one
//       box per tile, two for SwiGLU; L2 evict-first), 128-byte swizzle, in
//       a ring of shared-memory stages guarded by full/empty mbarriers;
//   warp 1 / lane 0: MMA issuer: 4 x tcgen05.mma (K = 16) per stage and
//       row block into one of two TMEM accumulators; a tcgen05.commit frees
//       each stage, another hands the finished accumulator to the epilogue;
//   warps 2-5: epilogue, one activation row per thread (TMEM lane quadrant
//       = warp % 4), straight from TMEM (epilogue_tc.cuh), overlapping the
//       next unit's mainloop.  With split-K they store the fp32 partial
//       (32 x 32 boxes staged in shared memory, written by TMA); a split-K
//       epilogue kernel then sums the partials in split order, consecutive
//       threads on consecutive columns, and runs the epilogue.
#include <cudaTypedefs.h>

#include <mutex>
#include <unordered_map>

#include "epilogue_tc.cuh"
#include "gemm_tc.h"

namespace wedlm {

namespace {
constexpr int kMaxStages = 8;
constexpr int kBK = 64;                           // K elements per stage (128 bytes)
constexpr uint32_t kXBlockBytes = 128 * kBK * 2;  // one activation row block
constexpr int kThreads = 192;                     // producer, MMA, 4 epilogue warps
constexpr int kMaxDynSmem = 221 * 1024;

// bounded wait that gives up at once after any wait of this block timed out
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, int* err,
                                              volatile int* abort) {
  // a phase that has already completed costs one poll (the issuing threads
  // are on the critical path); the abort flag is read only when waiting
  if (mbar_try_wait(bar, parity)) return true;
  if (*abort) return false;
  if (mbar_wait(bar, parity, err)) return true;
  *abort = 1;
  return false;
}
}  // namespace

struct TcLaunch {
  int stages, ntile, nrb, nbuf, tiles;
  int mma_n;         // pair kernel: N of one pair MMA (256, or 192 for SwiGLU tiles of 384)
  uint32_t a_bytes, stage_bytes, tmem_cols, buf_cols;
  uint32_t stg_off;  // split-K partials: 4 KB staging box per epilogue warp
};
constexpr uint32_t kStageBoxBytes = 32 * 32 * 4;  // 32 rows x 32 fp32 columns

__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap mW0, const __grid_constant__ CUtensorMap mW1,
               const __grid_constant__ CUtensorMap mW2, const __grid_constant__ CUtensorMap mX,
               const __grid_constant__ CUtensorMap mPart, GemmProblem P, TcLaunch L) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ __align__(8) uint64_t bar_full[kMaxStages];
  __shared__ __align__(8) uint64_t bar_empty[kMaxStages];
  __shared__ __align__(8) uint64_t acc_full[2];
  __shared__ __align__(8) uint64_t acc_empty[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_issued, s_consumed;

  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = P.K / kBK;
  const int ntile = L.ntile;
  const int units = L.tiles * P.splits;
  // activation rows present (the LM head on masked rows reads their count,
  // written at the start of the step); row blocks beyond them are skipped
  const int m_live = P.m_count ? min(P.M, max(0, *P.m_count)) : P.M;
  const int nrb_live = (m_live + 127) / 128;
  // with fewer live row blocks than planned, the ring is cut into stages of
  // the live size, so that more K blocks are in flight; with every block
  // live this is the plan's own ring
  const uint32_t a_bytes =
      nrb_live < L.nrb ? (uint32_t)max(nrb_live, 1) * kXBlockBytes : L.a_bytes;
  const uint32_t stage_bytes = a_bytes + (uint32_t)ntile * 128u;
  const int stages = min(kMaxStages, (int)(((uint32_t)L.stages * L.stage_bytes) / stage_bytes));

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrive per epilogue warp
    }
    s_abort = 0;
    s_issued = 0;
    s_consumed = 0;
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
  const uint32_t stage_live = (uint32_t)nrb_live * kXBlockBytes + (uint32_t)ntile * 128u;
  // the live blocks' accumulators take two buffers whenever two fit in the
  // TMEM allocation, so that the epilogue of one tile overlaps the MMAs of
  // the next (the LM head planned for 256 rows with at most 128 of them
  // masked); with every block live this is the plan's own layout
  const uint32_t buf_cols = (uint32_t)nrb_live * (uint32_t)ntile;
  const int nbuf = buf_cols * 2u <= L.tmem_cols ? 2 : 1;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      const uint64_t pol = l2_evict_first_policy();
      const int half = ntile / 2;
      int it = 0, ps = 0;
      uint32_t pph = 0;
      bool alive = true;
      // weights do not depend on the previous kernel: the first ring of
      // weight boxes goes out before waiting for it, their activation boxes
      // once it is done
      bool waited = false;
      int npend = 0, pend_s[kMaxStages], pend_kx[kMaxStages];
      auto issue_x = [&](int s, int kx) {
        uint8_t* st = base + (size_t)s * stage_bytes;
        for (int r = 0; r < nrb_live; ++r)
          tma_load_2d(st + r * kXBlockBytes, &mX, &bar_full[s], kx, r * 128);
      };
      auto wait_prev = [&]() {
        pdl_wait();
        pdl_trigger();
        waited = true;
        for (int j = 0; j < npend; ++j) issue_x(pend_s[j], pend_kx[j]);
        npend = 0;
      };
      for (int u = blockIdx.x; u < units && alive && nrb_live > 0; u += gridDim.x) {
        const int tile = u / P.splits, split = u % P.splits;
        const int kb0 = (int)((long long)nkb * split / P.splits);
        const int kb1 = (int)((long long)nkb * (split + 1) / P.splits);
        const CUtensorMap* seg = &mW0;
        int row0 = tile * ntile;
        if (!P.swiglu) {
          if (row0 >= P.seg2) { seg = &mW2; row0 -= P.seg2; }
          else if (row0 >= P.seg1) { seg = &mW1; row0 -= P.seg1; }
        }
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = ps;
          const uint32_t ph = pph;
          if (++ps == stages) {  // the ring position of the next K block
            ps = 0;
            pph ^= 1u;
          }
          if (!wait_or_abort(&bar_empty[s], ph ^ 1u, P.err, &s_abort)) { alive = false; break; }
          uint8_t* st = base + (size_t)s * stage_bytes;
          mbar_arrive_expect_tx(&bar_full[s], stage_live);
          const int kx = kb * kBK;
          // the weight tile in one box (SwiGLU: gate rows, then up rows);
          // rows of 128 bytes one after another, as the MMA descriptors expect
          if (P.swiglu) {
            tma_load_2d_hint(st + a_bytes, &mW0, &bar_full[s], kx, tile * half, pol);
            tma_load_2d_hint(st + a_bytes + half * 128, &mW1, &bar_full[s], kx, tile * half, pol);
          } else {
            tma_load_2d_hint(st + a_bytes, seg, &bar_full[s], kx, row0, pol);
          }
          if (waited) {
            issue_x(s, kx);
          } else {
            pend_s[npend] = s;
            pend_kx[npend] = kx;
            if (++npend == stages) wait_prev();
          }
        }
      }
      if (!waited) wait_prev();
      s_issued = it;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t idesc = idesc_bf16_m128(ntile);
      // as in the pair kernel: stage and phase stepped, descriptors formed
      // once per stage and stepped along K (2 = 32 bytes in 16-byte units)
      const uint64_t da0 = sdesc_sw128(smem_u32(base));
      const uint64_t dstage = (uint64_t)(stage_bytes >> 4), dw = (uint64_t)(a_bytes >> 4);
      const uint64_t dx = (uint64_t)(kXBlockBytes >> 4);
      int it = 0, ul = 0, s = 0;
      uint32_t ph = 0;
      bool alive = true;
      for (int u = blockIdx.x; u < units && alive && nrb_live > 0; u += gridDim.x, ++ul) {
        const int split = u % P.splits;
        const int kb0 = (int)((long long)nkb * split / P.splits);
        const int kb1 = (int)((long long)nkb * (split + 1) / P.splits);
        const int buf = ul % nbuf, use = ul / nbuf;
        if (!wait_or_abort(&acc_empty[buf], ((uint32_t)use & 1u) ^ 1u, P.err, &s_abort)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)buf * buf_cols;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          if (!wait_or_abort(&bar_full[s], ph, P.err, &s_abort)) { alive = false; break; }
          tc_fence_after();
          const uint64_t da = da0 + (uint64_t)s * dstage;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t bd = da + dw + (uint64_t)(2 * kk);
            for (int r = 0; r < nrb_live; ++r)
              tc_mma_f16(d0 + (uint32_t)(r * ntile), da + (uint64_t)r * dx + (uint64_t)(2 * kk), bd,
                         idesc, (kb != kb0 || kk) ? 1u : 0u);
          }
          tc_commit(&bar_empty[s]);
          if (++s == stages) {
            s = 0;
            ph ^= 1u;
          }
        }
        tc_commit(&acc_full[buf]);
      }
      s_consumed = it;
    }
  } else {
    // ---------------- epilogue warps: thread = activation row ----------------
    pdl_wait();  // outputs and partials may still be read by the previous kernel
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    int ul = 0;
    for (int u = blockIdx.x; u < units && nrb_live > 0; u += gridDim.x, ++ul) {
      const int tile = u / P.splits, split = u % P.splits;
      const int buf = ul % nbuf, use = ul / nbuf;
      // on a timeout keep going without waiting (outputs are then invalid and
      // the error word says so): the epilogue warps must stay in step at
      // their named barrier
      wait_or_abort(&acc_full[buf], (uint32_t)use & 1u, P.err, &s_abort);
      tc_fence_after();
      for (int r = 0; r < nrb_live; ++r) {
        const int m = r * 128 + 32 * q + lane;
        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)buf * buf_cols +
                               (uint32_t)(r * ntile);
        if (P.splits == 1) {
          AccRow a{ACC_TMEM, taddr, nullptr, 0, 1, tile * ntile, P.N, m < m_live};
          tc_epilogue_rows(P, a, m, tile, ntile, 0, tc_epi_items(P, ntile));
        } else if (r * 128 + 32 * q < m_live) {
          // fp32 partial [split][M][N]: the warp's 32 rows x 32 columns go
          // to its staging box in the 128-byte swizzle (16-byte chunk j of
          // row i at chunk j ^ (i % 8): the row-per-lane writes hit every
          // bank once per 8 lanes) and one lane stores the box with TMA,
          // whole 128-byte rows; rows and columns outside [M][N] are clipped
          const uint32_t stg = smem_u32(base + L.stg_off + q * kStageBoxBytes);
          for (int c = 0; c < ntile && tile * ntile + c < P.N; c += 32) {
            float v[32];
            tmem_ld32(taddr + (uint32_t)c, v);
            if (lane == 0) bulk_wait_read0();  // the previous box has left the buffer
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              st_shared_f32x4(stg + (uint32_t)(lane * 128 + ((j ^ (lane & 7)) << 4)), v[4 * j],
                              v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&mPart, stg, tile * ntile + c, r * 128 + 32 * q, split);
              bulk_commit();
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);  // accumulator free for the MMA warp
    }
    if (lane == 0) bulk_wait0();  // partials written before the block exits
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (s_abort && threadIdx.x == 0) {
    // after a timeout: wait (bounded) for this block's copies still in flight
    for (int it = s_consumed; it < s_issued; ++it)
      mbar_wait(&bar_full[it % stages], (uint32_t)(it / stages) & 1u, P.err);
  }
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, L.tmem_cols);
}

// Split-K epilogues.  The partial sums of every split are added in split
// order (deterministic), with consecutive threads on consecutive columns so
// that every partial is read once, coalesced.

// sum of the splits at float4 index i of [M][N]; the additions stay in
// split order.  NB > 1: the loads of up to NB splits are issued before the
// first addition, so that they share one L2 round trip; NB = 1: the loads of
// four splits at a time only when four remain (fewer registers)
template <int NB = 4>
__device__ __forceinline__ float4 splitk_sum4(const GemmProblem& P, size_t i) {
  const float4* p4 = reinterpret_cast<const float4*>(P.partial) + i;
  const size_t stride4 = (size_t)P.M * P.N / 4;
  float4 a = __ldcg(p4);
  if constexpr (NB > 1) {
    for (int sp = 1; sp < P.splits; sp += NB) {
      float4 t[NB];
#pragma unroll
      for (int k = 0; k < NB; ++k)
        if (sp + k < P.splits) t[k] = __ldcg(p4 + (size_t)(sp + k) * stride4);
#pragma unroll
      for (int k = 0; k < NB; ++k)
        if (sp + k < P.splits) { a.x += t[k].x; a.y += t[k].y; a.z += t[k].z; a.w += t[k].w; }
    }
  } else {
    int sp = 1;
    for (; sp + 3 < P.splits; sp += 4) {
      float4 t[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) t[k] = __ldcg(p4 + (sp + k) * stride4);
#pragma unroll
      for (int k = 0; k < 4; ++k) { a.x += t[k].x; a.y += t[k].y; a.z += t[k].z; a.w += t[k].w; }
    }
    for (; sp < P.splits; ++sp) {
      const float4 t = __ldcg(p4 + sp * stride4);
      a.x += t.x; a.y += t.y; a.z += t.z; a.w += t.w;
    }
  }
  return a;
}

// RESID: x[m][n] += acc[m][n]
__global__ void __launch_bounds__(256) splitk_resid_kernel(GemmProblem P) {
  pdl_wait();  // the previous kernel's results
  pdl_trigger();
  const size_t n4 = (size_t)P.M * P.N / 4;
  bf16* x = static_cast<bf16*>(P.epi.x);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = splitk_sum4(P, i);
    __nv_bfloat162* xp = reinterpret_cast<__nv_bfloat162*>(x + 4 * i);
    const float2 x01 = __bfloat1622float2(xp[0]), x23 = __bfloat1622float2(xp[1]);
    xp[0] = __floats2bfloat162_rn(x01.x + a.x, x01.y + a.y);
    xp[1] = __floats2bfloat162_rn(x23.x + a.z, x23.y + a.w);
  }
}

// RESID followed by the RMSNorm of the next GEMM's input: one block of
// kNormThreads threads per activation row.  x[m] += acc[m] (bf16 rounding as in the plain
// residual add), then xn[m] = x[m] * rsqrt(mean(x[m]^2) + eps) * norm_w from
// the stored bf16 x, with the same per-thread 8-element vectors and the same
// reduction order as rmsnorm_kernel, so the result is bit-identical to the
// two separate kernels.
// NB = 4: the split loads batched, at most 64 registers (two blocks per
// SM); NB = 1: fewer loads in flight (about 40 registers, three blocks per
// SM), for more rows than two blocks per SM hold: measured on GB300, the
// batched kernel saves 1-2 us per launch at 256 rows, but at 512 rows its
// second wave of blocks costs the step more than that
template <int NB>
__global__ void __launch_bounds__(kNormThreads, NB > 1 ? 2 : 3)
    splitk_resid_norm_kernel(GemmProblem P) {
  pdl_wait();  // the previous kernel's results
  pdl_trigger();
  const int m = blockIdx.x;
  const int n8 = P.N / 8;
  bf16* x = static_cast<bf16*>(P.epi.x) + (size_t)m * P.N;
  float ss = 0.f;
  for (int i = threadIdx.x; i < n8; i += blockDim.x) {
    const float4 a0 = splitk_sum4<NB>(P, ((size_t)m * P.N) / 4 + 2 * i);
    const float4 a1 = splitk_sum4<NB>(P, ((size_t)m * P.N) / 4 + 2 * i + 1);
    const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    Vec16<bf16> v = ld16(x + 8 * i);
#pragma unroll
    for (int k = 0; k < 8; ++k) v.set(k, v.get(k) + a[k]);
    st16(x + 8 * i, v);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float f = v.get(k);
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
  const float r = rsqrtf(red[0] / (float)P.N + P.epi.eps);
  const bf16* g = static_cast<const bf16*>(P.epi.norm_w);
  // the normed row goes to its compacted row (the LM head on masked rows)
  const int my = P.epi.row_dst ? P.epi.row_dst[m] : m;
  if (my < 0) return;  // uniform for the block
  bf16* xn = static_cast<bf16*>(P.epi.xn) + (size_t)my * P.N;
  for (int i = threadIdx.x; i < n8; i += blockDim.x) {  // this thread's own stores
    Vec16<bf16> v = ld16(x + 8 * i), gv = ld16(g + 8 * i), o;
#pragma unroll
    for (int k = 0; k < 8; ++k) o.set(k, v.get(k) * r * gv.get(k));
    st16(xn + 8 * i, o);
  }
}

// SWIGLU: act[m][f] = silu(gate) * up; tile t holds gate features
// [t*half, (t+1)*half) in columns [0, half) and the same up features in
// [half, ntile)
__global__ void __launch_bounds__(256) splitk_swiglu_kernel(GemmProblem P, int ntile) {
  pdl_wait();  // the previous kernel's results
  pdl_trigger();
  const int half = ntile / 2, F = P.N / 2;
  const size_t n4 = (size_t)P.M * F / 4;
  bf16* act = static_cast<bf16*>(P.epi.act);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t e = 4 * i;
    const int m = (int)(e / F), f = (int)(e % F);
    const int t = f / half, c = f % half;
    const size_t g4 = ((size_t)m * P.N + (size_t)t * ntile + c) / 4;
    const float4 g = splitk_sum4(P, g4), u = splitk_sum4(P, g4 + half / 4);
    const float gv[4] = {g.x, g.y, g.z, g.w}, uv[4] = {u.x, u.y, u.z, u.w};
    float o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = silu_fast(gv[k]) * uv[k];
    __nv_bfloat162* ap = reinterpret_cast<__nv_bfloat162*>(act + e);
    ap[0] = __floats2bfloat162_rn(o[0], o[1]);
    ap[1] = __floats2bfloat162_rn(o[2], o[3]);
  }
}

// QKV (head_dim 128): one warp per (row, head), lane l holds dims 4l..4l+3.
// q and k heads: per-head RMSNorm (when enabled), then RoPE on the pairs
// (d, d + 64), which sit in lanes l and l ^ 16; q goes to q_out, k and v
// to the layer's window scratch in the 8x8-tile layout.
// (at most 64 registers: four blocks per SM)
__global__ void __launch_bounds__(256, 4) splitk_qkv_kernel(GemmProblem P) {
  pdl_wait();  // the previous kernel's results
  pdl_trigger();
  const GemmEpi& e = P.epi;
  const int lane = threadIdx.x & 31;
  const int heads = P.N / 128;
  const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= P.M * heads) return;
  const int m = wid / heads, gh = wid % heads;
  const int kind = gh < e.nq ? 0 : (gh < e.nq + e.nkv ? 1 : 2);
  const int d0 = 4 * lane;
  // the norm weights and the RoPE table go out with the partials' loads
  // (none depends on the sum), not one L2 round trip after them
  float gw[4] = {1.f, 1.f, 1.f, 1.f}, cs[4] = {}, sn[4] = {};
  if (kind < 2) {
    if (e.qk_norm) {
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(
          static_cast<const bf16*>(kind == 0 ? e.q_norm : e.k_norm) + d0);
      const float2 g01 = __bfloat1622float2(g2[0]), g23 = __bfloat1622float2(g2[1]);
      gw[0] = g01.x; gw[1] = g01.y; gw[2] = g23.x; gw[3] = g23.y;
    }
    const int dh = d0 & 63;  // position within the rotated half
    const float4 c4 = *reinterpret_cast<const float4*>(e.cosb + (size_t)m * 64 + dh);
    const float4 s4 = *reinterpret_cast<const float4*>(e.sinb + (size_t)m * 64 + dh);
    cs[0] = c4.x; cs[1] = c4.y; cs[2] = c4.z; cs[3] = c4.w;
    sn[0] = s4.x; sn[1] = s4.y; sn[2] = s4.z; sn[3] = s4.w;
  }
  const float4 a = splitk_sum4<3>(P, ((size_t)m * P.N + (size_t)gh * 128) / 4 + lane);
  float x[4] = {a.x, a.y, a.z, a.w};
  if (kind < 2) {
    if (e.qk_norm) {
      float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
      ss = warp_sum(ss);
      const float rs = rsqrtf(ss / 128.f + e.eps);
#pragma unroll
      for (int k = 0; k < 4; ++k) x[k] = x[k] * rs * gw[k];
    }
    float y[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = __shfl_xor_sync(0xffffffffu, x[k], 16);
    if (lane < 16) {
#pragma unroll
      for (int k = 0; k < 4; ++k) x[k] = x[k] * cs[k] - y[k] * sn[k];
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) x[k] = x[k] * cs[k] + y[k] * sn[k];
    }
  }
  const __nv_bfloat162 v01 = __floats2bfloat162_rn(x[0], x[1]);
  const __nv_bfloat162 v23 = __floats2bfloat162_rn(x[2], x[3]);
  bf16* dst;
  if (kind == 0) {
    dst = static_cast<bf16*>(e.q_out) + ((size_t)m * e.nq + gh) * 128 + d0;
  } else {
    const int b = m / e.W, p = m % e.W;
    const int kvh = gh - e.nq - (kind == 2 ? e.nkv : 0);
    dst = static_cast<bf16*>(e.kv_win) + (((size_t)b * 2 + (kind - 1)) * e.nkv + kvh) * e.Wp * 128 +
          tile_off(p, d0, 128);
    // a committed row (physical rows 0..c-1) also goes to its page
    if (e.commit_n && p < e.commit_n[b]) {
      bf16* c = commit_dst<bf16>(e, b, e.commit_base[b] + p, kind - 1, kvh, d0);
      if (c) {
        __nv_bfloat162* cp = reinterpret_cast<__nv_bfloat162*>(c);
        cp[0] = v01;
        cp[1] = v23;
      }
    }
  }
  __nv_bfloat162* dp = reinterpret_cast<__nv_bfloat162*>(dst);
  dp[0] = v01;
  dp[1] = v23;
}

// any other epilogue: thread = (activation row, epilogue item)
__global__ void __launch_bounds__(128)
splitk_epilogue_kernel(GemmProblem P, int ntile, int items) {
  pdl_wait();  // the previous kernel's results
  pdl_trigger();
  const int tile = blockIdx.x / items, item = blockIdx.x % items;
  const int m = blockIdx.y * 128 + threadIdx.x;
  const float* src = P.partial + (size_t)min(m, P.M - 1) * P.N + tile * ntile;
  AccRow a{ACC_PARTIAL, 0, src, (size_t)P.M * P.N, P.splits, tile * ntile, P.N, m < P.M};
  tc_epilogue_rows(P, a, m, tile, ntile, item, item + 1);
}

// ---------------------------------------------------------------------------
// 2-SM variant for 129..512 activation rows: a cluster of two CTAs (an SM
// pair) computes one 256-row x (mma_n * nmma)-feature tile (NRB of them
// over the same weights above 256 rows) with
// tcgen05.mma.cta_group::2 (nmma MMAs of N = mma_n per K step, one per
// mma_n-column accumulator; mma_n = 256, or 192 for SwiGLU tiles of 192
// gate + 192 up features).  CTA r of the pair holds activation rows
// 128r..128r+127 and, for each MMA, half r of its mma_n weight rows in its
// shared memory, so each SM receives half the tile's activations and half
// its weights; its TMEM receives its 128 rows of the tile (rows
// 256b + 128r.. of each row block b).  Roles as in gemm_tc_kernel:
//   warp 0 / lane 0 (both CTAs): TMA producer for this CTA's halves; the
//       loads complete on the even CTA's full barrier (cta_group::2 form),
//       on which the even CTA's producer set the bytes of both;
//   warp 1 / lane 0 (even CTA only): MMA issuer; its commits arrive on the
//       empty / accumulator barriers of both CTAs (multicast);
//   warps 2-5 (both CTAs): epilogue of this CTA's rows from its own TMEM;
//       each warp arrives on the even CTA's accumulator-empty barrier.
// TMEM is allocated and freed by warp 2 of both CTAs together; a cluster
// barrier after set-up and one before the end keep each CTA's barriers and
// shared memory alive while the other may use them.  Every wait is bounded.
// ---------------------------------------------------------------------------
constexpr int kPairN = 256;                    // widest N of one pair MMA
// one CTA's half of one MMA's weights per stage: mma_n / 2 rows x 128 bytes
__host__ __device__ constexpr uint32_t pair_wbytes(int mma_n) { return (uint32_t)mma_n * 64u; }

template <int NMMA, int NRB = 1>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap mW0, const __grid_constant__ CUtensorMap mW1,
                    const __grid_constant__ CUtensorMap mW2, const __grid_constant__ CUtensorMap mX,
                    const __grid_constant__ CUtensorMap mPart, GemmProblem P, TcLaunch L) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ __align__(8) uint64_t bar_full[kMaxStages];
  __shared__ __align__(8) uint64_t bar_empty[kMaxStages];
  __shared__ __align__(8) uint64_t acc_full[2];
  __shared__ __align__(8) uint64_t acc_empty[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_issued, s_consumed;

  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: even CTA (issues the MMAs), 1: odd
  const int nkb = P.K / kBK;
  const int units = L.tiles * P.splits;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  constexpr int nmma = NMMA;
  const int mma_n = L.mma_n, ntile = NMMA * mma_n, hn = mma_n / 2;
  const uint32_t wbytes = pair_wbytes(mma_n);
  // NRB row blocks of 256 per pair (CTA r holds rows 256 * b + 128 * r of
  // block b), the weights after them in a stage; with NRB > 1 (above 256
  // rows: the projections, and the LM head on its masked rows) the blocks
  // past the live rows are skipped
  constexpr uint32_t kABytes = (uint32_t)NRB * kXBlockBytes;
  int m_live = P.M, nrb_live = 1;
  if constexpr (NRB > 1) {
    m_live = P.m_count ? min(P.M, max(0, *P.m_count)) : P.M;
    nrb_live = max(1, min(NRB, (m_live + 255) / 256));
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < L.stages; ++s) {
      mbar_init(&bar_full[s], 1);   // the even CTA's producer (bytes of both CTAs)
      mbar_init(&bar_empty[s], 1);  // one multicast commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);   // one multicast commit
      mbar_init(&acc_empty[b], 8);  // the epilogue warps of both CTAs
    }
    s_abort = 0;
    s_issued = 0;
    s_consumed = 0;
    mbar_fence_init();
    tma_prefetch_desc(&mW0);
    tma_prefetch_desc(&mX);
  }
  if (warp == 2) {
    tmem_alloc_pair(&s_tmem, L.tmem_cols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised before any remote use
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  // the even CTA's barriers, as shared::cluster addresses
  const uint32_t full0 = mapa_shared(smem_u32(&bar_full[0]), 0);
  const uint32_t accempty0 = mapa_shared(smem_u32(&acc_empty[0]), 0);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (this CTA's halves) ----------------
      const uint64_t pol = l2_evict_first_policy();
      // both CTAs
      const uint32_t stage_all =
          NRB == 1 ? 2u * L.stage_bytes
                   : 2u * ((uint32_t)nrb_live * kXBlockBytes + (uint32_t)nmma * wbytes);
      int it = 0, ps = 0;
      uint32_t pph = 0;
      bool alive = true;
      bool waited = false;
      int npend = 0, pend_s[kMaxStages], pend_kx[kMaxStages];
      auto issue_x = [&](int s, int kx) {
        for (int b = 0; b < nrb_live; ++b)
          tma_load_2d_pair_nohint(base + (size_t)s * L.stage_bytes + b * kXBlockBytes, &mX,
                                  full0 + 8u * s, kx, 256 * b + (int)rank * 128);
      };
      auto wait_prev = [&]() {
        pdl_wait();
        pdl_trigger();
        waited = true;
        for (int j = 0; j < npend; ++j) issue_x(pend_s[j], pend_kx[j]);
        npend = 0;
      };
      for (int u = pair; u < units && alive; u += npairs) {
        const int tile = u / P.splits, split = u % P.splits;
        const int kb0 = (int)((long long)nkb * split / P.splits);
        const int kb1 = (int)((long long)nkb * (split + 1) / P.splits);
        // this CTA's mma_n/2 weight rows of MMA j (D columns
        // mma_n*j..mma_n*(j+1)-1): SwiGLU tiles are [gate ntile/2 | up
        // ntile/2], so MMA j < nmma/2 takes gate rows and the rest up rows,
        // mma_n features a block (with one MMA: the even CTA gate, the odd
        // CTA up rows); other tiles take rows tile*ntile + mma_n*j of the
        // q|k|v (or single) weight; the even CTA the first half of each
        // block, the odd CTA the second
        const CUtensorMap* segj[NMMA];
        int rowj[NMMA];
        for (int j = 0; j < nmma; ++j) {
          if (P.swiglu) {
            const int half = nmma / 2;  // MMAs per gate (and up) block
            const bool up = nmma == 1 ? rank == 1 : j >= half;
            segj[j] = up ? &mW1 : &mW0;
            rowj[j] = nmma == 1 ? tile * hn
                                : tile * (ntile / 2) + (j % half) * mma_n + (int)rank * hn;
          } else {
            int r0 = tile * ntile + j * mma_n + (int)rank * hn;
            const CUtensorMap* sg = &mW0;
            if (r0 >= P.seg2) { sg = &mW2; r0 -= P.seg2; }
            else if (r0 >= P.seg1) { sg = &mW1; r0 -= P.seg1; }
            segj[j] = sg;
            rowj[j] = r0;
          }
        }
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = ps;
          const uint32_t ph = pph;
          if (++ps == L.stages) {  // the ring position of the next K block
            ps = 0;
            pph ^= 1u;
          }
          if (!wait_or_abort(&bar_empty[s], ph ^ 1u, P.err, &s_abort)) { alive = false; break; }
          uint8_t* st = base + (size_t)s * L.stage_bytes;
          if (rank == 0) mbar_arrive_expect_tx(&bar_full[s], stage_all);
          const int kx = kb * kBK;
          for (int j = 0; j < nmma; ++j)
            tma_load_2d_pair(st + kABytes + j * wbytes, segj[j], full0 + 8u * s, kx,
                             rowj[j], pol);
          if (waited) {
            issue_x(s, kx);
          } else {
            pend_s[npend] = s;
            pend_kx[npend] = kx;
            if (++npend == L.stages) wait_prev();
          }
        }
      }
      if (!waited) wait_prev();
      s_issued = it;
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (even CTA) ----------------
      // M = 256 over the pair (A: 128 rows in each CTA), N = mma_n (B:
      // mma_n/2 rows in each CTA)
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) |
                             ((uint32_t)(mma_n >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
      // This one thread feeds the tensor pipe, so its per-K-block scalar
      // work is kept small: the ring stage and phase advance by one step
      // (no division), the operand descriptors are formed once per stage
      // and stepped along K by adding the 32-byte offset (2 in the
      // descriptor's 16-byte address units).
      const uint64_t da0 = sdesc_sw128(smem_u32(base));
      const uint64_t dstage = (uint64_t)(L.stage_bytes >> 4);
      const uint64_t dw = (uint64_t)(wbytes >> 4), dx = (uint64_t)(kXBlockBytes >> 4);
      [[maybe_unused]] const uint64_t da_w = (uint64_t)(kABytes >> 4);  // weights after the blocks
      int it = 0, ul = 0, s = 0;
      uint32_t ph = 0;
      bool alive = true;
      for (int u = pair; u < units && alive; u += npairs, ++ul) {
        const int split = u % P.splits;
        const int kb0 = (int)((long long)nkb * split / P.splits);
        const int kb1 = (int)((long long)nkb * (split + 1) / P.splits);
        const int buf = ul % L.nbuf, use = ul / L.nbuf;
        if (!wait_or_abort(&acc_empty[buf], ((uint32_t)use & 1u) ^ 1u, P.err, &s_abort)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)buf * L.buf_cols;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          if (!wait_or_abort(&bar_full[s], ph, P.err, &s_abort)) { alive = false; break; }
          tc_fence_after();
          const uint64_t da = da0 + (uint64_t)s * dstage;  // this stage's activation block
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
#pragma unroll
            for (int j = 0; j < nmma; ++j) {
              if constexpr (NRB == 1) {
                tc_mma_pair_f16(d0 + (uint32_t)(j * mma_n), da + (uint64_t)(2 * kk),
                                da + dx + (uint64_t)j * dw + (uint64_t)(2 * kk), idesc,
                                (kb != kb0 || kk) ? 1u : 0u);
              } else {
                for (int b = 0; b < nrb_live; ++b)
                  tc_mma_pair_f16(d0 + (uint32_t)(b * ntile + j * mma_n),
                                  da + (uint64_t)b * dx + (uint64_t)(2 * kk),
                                  da + da_w + (uint64_t)j * dw + (uint64_t)(2 * kk), idesc,
                                  (kb != kb0 || kk) ? 1u : 0u);
              }
            }
          tc_commit_pair(&bar_empty[s], 3);
          if (++s == L.stages) {
            s = 0;
            ph ^= 1u;
          }
        }
        tc_commit_pair(&acc_full[buf], 3);
      }
      s_consumed = it;
    }
  } else {
    // ---------------- epilogue warps: thread = one of this CTA's rows ----------------
    pdl_wait();  // outputs and partials may still be read by the previous kernel
    const int q = warp & 3;
    int ul = 0;
    for (int u = pair; u < units; u += npairs, ++ul) {
      const int tile = u / P.splits, split = u % P.splits;
      const int buf = ul % L.nbuf, use = ul / L.nbuf;
      wait_or_abort(&acc_full[buf], (uint32_t)use & 1u, P.err, &s_abort);
      tc_fence_after();
      const int r = (int)rank;
      const int m = r * 128 + 32 * q + lane;
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)buf * L.buf_cols;
      if constexpr (NRB > 1) {
        // each live row block's rows straight from TMEM, or their fp32
        // split-K partials through one staging box per warp (as in
        // gemm_tc_kernel)
        for (int b = 0; b < nrb_live; ++b) {
          const int mb = 256 * b + m;
          const uint32_t tb = taddr + (uint32_t)(b * ntile);
          if (P.splits == 1) {
            AccRow a{ACC_TMEM, tb, nullptr, 0, 1, tile * ntile, P.N, mb < m_live};
            tc_epilogue_rows(P, a, mb, tile, ntile, 0, tc_epi_items(P, ntile));
          } else if (256 * b + r * 128 + 32 * q < m_live) {
            const uint32_t stg = smem_u32(base + L.stg_off + q * kStageBoxBytes);
            for (int c = 0; c < ntile && tile * ntile + c < P.N; c += 32) {
              float v[32];
              tmem_ld32(tb + (uint32_t)c, v);
              if (lane == 0) bulk_wait_read0();  // the previous box has left the buffer
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 8; ++j)
                st_shared_f32x4(stg + (uint32_t)(lane * 128 + ((j ^ (lane & 7)) << 4)), v[4 * j],
                                v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(&mPart, stg, tile * ntile + c, 256 * b + r * 128 + 32 * q, split);
                bulk_commit();
              }
            }
          }
        }
      } else if (P.splits == 1) {
        AccRow a{ACC_TMEM, taddr, nullptr, 0, 1, tile * ntile, P.N, m < P.M};
        tc_epilogue_rows(P, a, m, tile, ntile, 0, tc_epi_items(P, ntile));
      } else if (r * 128 + 32 * q < P.M) {
        // as in gemm_tc_kernel: on the pair's last unit each box of the
        // warp's strip is staged in its own slot of the idle pipeline stages
        // (the last MMA, which read both CTAs' stages, is complete)
        const bool idle = u + npairs >= units && !s_abort &&
                          4u * (uint32_t)(ntile / 32) * kStageBoxBytes <=
                              (uint32_t)L.stages * L.stage_bytes;
        const uint32_t slot0 = smem_u32(base) + (uint32_t)(q * (ntile / 32)) * kStageBoxBytes;
        for (int c = 0; c < ntile && tile * ntile + c < P.N; c += 32) {
          float v[32];
          tmem_ld32(taddr + (uint32_t)c, v);
          uint32_t stg = slot0 + (uint32_t)(c / 32) * kStageBoxBytes;
          if (!idle) {
            stg = smem_u32(base + L.stg_off + q * kStageBoxBytes);
            if (lane == 0) bulk_wait_read0();
          }
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_shared_f32x4(stg + (uint32_t)(lane * 128 + ((j ^ (lane & 7)) << 4)), v[4 * j],
                            v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&mPart, stg, tile * ntile + c, r * 128 + 32 * q, split);
            bulk_commit();
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(accempty0 + 8u * buf);  // the even CTA's barrier
    }
    if (lane == 0) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (s_abort && threadIdx.x == 0 && rank == 0) {
    // after a timeout: wait (bounded) for the loads still in flight (both
    // CTAs' loads complete on the even CTA's full barriers)
    for (int it = s_consumed; it < s_issued; ++it)
      mbar_wait(&bar_full[it % L.stages], (uint32_t)(it / L.stages) & 1u, P.err);
  }
  __syncthreads();
  cluster_sync_all();  // the pair is done with each other's barriers and TMEM
  if (warp == 2) tmem_dealloc_pair(tmem, L.tmem_cols);
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

// split-K partials [S][M][N] fp32 as a 3-D tensor for TMA stores of
// 32 x 32 boxes, 128-byte swizzle (one box row = 32 floats = 128 bytes)
bool encode_partial(CUtensorMap* m, void* ptr, uint64_t N, uint64_t M, uint64_t S) {
  auto enc = get_encode();
  if (!enc || (N * 4) % 16) return false;
  cuuint64_t dims[3] = {N, M, S};
  cuuint64_t strides[2] = {N * 4, M * N * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

// weight descriptors for boxes of 64, 96, 128 and 256 rows (x 64 K
// elements): a GEMM loads its whole weight tile (or each SwiGLU half) in one
// box
constexpr int kBoxRows[4] = {64, 96, 128, 256};
struct TcMapTable {
  std::unordered_map<const void*, CUtensorMap> weight[4];
};
namespace {
int box_slot(int rows) {
  for (int b = 0; b < 4; ++b)
    if (kBoxRows[b] == rows) return b;
  return -1;
}
}

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
    for (int b = 0; b < 4; ++b) {
      const uint32_t box = (uint32_t)kBoxRows[b];
      if (box > rows) continue;
      CUtensorMap m;
      if (!encode_2d(&m, w, K, rows, box)) return false;
      p->maps->weight[b][w] = m;
    }
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
  cudaError_t e = ensure_dyn_smem((const void*)gemm_tc_kernel, kMaxDynSmem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (msg) *msg = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return nullptr;
  }
  return p;
}

// split-K factor for the persistent kernel: units = tiles * s are dealt
// round-robin to num_sms blocks.  Modelled time: the weight stream is bound
// by the busiest block (one SM streaming one-box weight tiles with its
// activation blocks) or by the whole GPU (about 6.5 TB/s), whichever is
// slower; split-K adds a second launch (about 3 us) and the fp32 partial
// round trip (s * M * N * 8 bytes).  The per-SM and partial rates are fitted
// to forced-plan sweeps on GB300 at the Qwen3-8B shapes: with one 128-row
// activation block about 100 GB/s per SM and 4 TB/s for the partials (down
// fastest at 6 splits, O at 5), with more blocks about 65 GB/s and 2 TB/s
// (the rates that also keep 129..256 rows on the pair kernel, which measured
// faster there).  At least 4 k-blocks per unit.
int tc_choose_splits(int tiles, int nkb, int M, int N, int ntile, int num_sms,
                     size_t part_elems, double* time_out) {
  const double w_kb = (double)ntile * kBK * 2, x_kb = (double)((M + 127) / 128) * kXBlockBytes;
  const double t_all = (double)tiles * nkb * w_kb / 6.5e12;
  const double sm_rate = M <= 128 ? 100e9 : 65e9, part_rate = M <= 128 ? 4e12 : 2e12;
  int best = 1;
  double best_t = 1e30;
  for (int s = 1; s <= 16; ++s) {
    if (s > 1 && (nkb / s < 4 || (size_t)s * M * N > part_elems)) break;
    const int rounds = (tiles * s + num_sms - 1) / num_sms;
    const int kper = (nkb + s - 1) / s;
    const double t_sm = (double)rounds * kper * (w_kb + x_kb) / sm_rate;
    double t = std::max(t_sm, t_all);
    if (s > 1) t += 3e-6 + (double)s * M * N * 8.0 / part_rate;
    if (t < best_t * (1.0 - 1e-9)) { best_t = t; best = s; }
  }
  if (time_out) *time_out = best_t;
  return best;
}

// widest tile of output features: 256 while the 128-row activation blocks
// fit one 256-column TMEM accumulator each (up to 256 rows; one accumulator
// buffer instead of two above 128 rows), else 128; every segment boundary
// (q|k|v) must fall on a tile boundary
int tc_tile_width(const GemmProblem& P) {
  if (P.M > 256) return 128;
  if (P.swiglu) return (P.N / 2) % 128 == 0 ? 256 : 128;
  if (P.seg1 < P.N && (P.seg1 % 256 || (P.seg2 - P.seg1) % 256)) return 128;
  if (P.seg2 < P.N && (P.N - P.seg2) % 256) return 128;
  return 256;
}

namespace {
int tc_tiles_for(const GemmProblem& P, int ntile) {
  return P.swiglu ? (P.N / 2) / (ntile / 2) : (P.N + ntile - 1) / ntile;
}
}  // namespace

// The plan of one GEMM: tile width and split-K factor of the persistent
// kernel (split-K through fp32 partials and an epilogue kernel when
// splits > 1).
TcChoice tc_plan(const TcPlanSet& plans, const GemmProblem& P, double* t_out) {
  const int nkb = P.K / kBK;
  const int wmax = tc_tile_width(P);
  TcChoice c;
  c.ntile = wmax;
  double best_t = 0.0;
  c.splits = tc_choose_splits(tc_tiles_for(P, wmax), nkb, P.M, P.N, wmax, plans.num_sms,
                              plans.part_elems, &best_t);
  // narrower tiles spread the features over more SMs and, above 128 rows,
  // keep two TMEM accumulator buffers.  For up to 128 rows only the SwiGLU
  // projection takes them: measured on GB300 at the Qwen3-8B shapes, the
  // model's preference for narrower split-K tiles there (O, down) did not
  // hold, the extra activation traffic costing more than the partials saved.
  for (int nt : {192, 128}) {
    if (!P.swiglu && P.M <= 128) continue;
    if (nt >= wmax || (P.swiglu ? (P.N / 2) % (nt / 2) : (nt == 192 || P.N % nt))) continue;
    if (!P.swiglu && (P.seg1 % nt || P.seg2 % nt)) continue;
    double t = 0.0;
    const int s = tc_choose_splits(tc_tiles_for(P, nt), nkb, P.M, P.N, nt, plans.num_sms,
                                   plans.part_elems, &t);
    if (t < best_t * (1.0 - 1e-9)) { best_t = t; c.ntile = nt; c.splits = s; }
  }
  if (t_out) *t_out = best_t;
  return c;
}

cudaError_t launch_gemm_epilogue(const TcPlanSet& plans, const GemmProblem& P, const TcLaunch& L,
                                 cudaStream_t st);

// The 2-SM pair kernel with one row block may take the projections with
// 129..256 activation rows (two 128-row halves, one per SM of the pair); at
// that size the LM head keeps the one-SM kernel (its row count may be known
// on the device only, and is mostly under 128 there).  Above 256 rows the
// pair kernel with two row blocks is planned separately.
bool pair_possible(const GemmProblem& P) {
  if (P.M <= 128 || P.M > 256 || P.epi.mode == EPI_LMHEAD || P.m_count) return false;
  return P.swiglu ? (P.N / 2) % 128 == 0 : P.N % 128 == 0;
}

struct PairPlan {
  int ntile = 0, mma_n = kPairN, splits = 1;
  double t = 1e30;  // modelled seconds
};

// Pair tile of ntile = nmma * mma_n features (256 = one N = 256 MMA per K
// step, 512 = two; 384 = two N = 192 MMAs, SwiGLU only: 192 gate + 192 up
// features, which puts the Qwen3-8B-sized gate/up projection on 64 tiles
// instead of 48) and its split-K factor: units = tiles * s over the pairs.
// Modelled time per K block: each SM receives its halves of the activations
// (16 KB per row block) and of every MMA's weights (mma_n/2 rows x 128 B), at about
// 65 GB/s per SM as measured on GB300 inside these kernels, or runs its MMAs
// (128 cycles per M = 256, N = 256, K = 16 pair MMA, per row block), whichever is slower;
// the whole GPU streams the weights at about 6.5 TB/s at most.  Split-K adds
// the epilogue launch (about 3 us) and the fp32 partials' round trip, which
// stays in L2 (s * M * N * 8 bytes at about 4 TB/s: measured at 256 rows,
// QKV is fastest at 3 splits, O and down at 4).
PairPlan pair_plan(const GemmProblem& P, int nmma, int mma_n, int npairs, size_t part_elems,
                   int nrb) {
  PairPlan best;
  const int ntile = nmma * mma_n;
  if (npairs < 1 || (P.swiglu ? (P.N / 2) % (ntile / 2) : P.N % 128)) return best;
  if (mma_n != kPairN && !P.swiglu) return best;  // q|k|v segments fall on 128-row halves
  if (nrb * ntile > 512) return best;             // the accumulators of all row blocks in TMEM
  const int nkb = P.K / kBK;
  const int tiles = P.swiglu ? (P.N / 2) / (ntile / 2) : (P.N + ntile - 1) / ntile;
  const double per_kb = std::max(
      ((double)nrb * kXBlockBytes + nmma * (double)pair_wbytes(mma_n)) / 65e9,
      nrb * nmma * (kBK / 16) * 128.0 * mma_n / kPairN / 1.9e9);
  const double t_all = (double)tiles * nkb * 2.0 * nmma * pair_wbytes(mma_n) / 6.5e12;
  for (int s = 1; s <= 16; ++s) {
    if (s > 1 && (nkb / s < 4 || (size_t)s * P.M * P.N > part_elems)) break;
    const int rounds = (tiles * s + npairs - 1) / npairs;
    const int kper = (nkb + s - 1) / s;
    double t = std::max((double)rounds * kper * per_kb, t_all);
    if (s > 1) t += 3e-6 + (double)s * P.M * P.N * 8.0 / 4e12;
    if (t < best.t * (1.0 - 1e-9)) {
      best.t = t;
      best.splits = s;
      best.ntile = ntile;
      best.mma_n = mma_n;
    }
  }
  return best;
}

// How many SM pairs can run the pair kernel at once with `smem` bytes of
// dynamic shared memory: clusters of two need two SMs of one GPC, so on a
// chip whose GPCs have odd SM counts this is below SMs / 2.  Asked once per
// (device, shared-memory size).
int pair_capacity(size_t smem, int num_sms) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const uint64_t key = ((uint64_t)dev << 32) | (uint64_t)smem;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const void* fn = (const void*)gemm_tc_pair_kernel<1>;  // the same smem and cluster needs as <2>
  if (ensure_dyn_smem(fn, kMaxDynSmem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  n = std::min(n, num_sms / 2);
  cache[key] = n;
  return n;
}

// dynamic shared memory of a pair launch
size_t pair_smem(int nmma, int mma_n, int splits, int nrb = 1) {
  const uint32_t stage = (uint32_t)nrb * kXBlockBytes + (uint32_t)nmma * pair_wbytes(mma_n);
  const uint32_t stg = splits > 1 ? 4 * kStageBoxBytes : 0;
  const uint32_t stages = std::min<uint32_t>(kMaxStages, (kMaxDynSmem - 1024 - stg) / stage);
  return (size_t)stages * stage + stg + 1024;
}

cudaError_t launch_gemm_pair(const TcPlanSet& plans, GemmProblem P, const PairPlan& pp,
                             int npairs_max, cudaStream_t st, int* tiles_out, int* launches_out,
                             int nrb = 1) {
  const int ntile = pp.ntile, splits = pp.splits, mma_n = pp.mma_n, nmma = ntile / mma_n;
  const int tiles = P.swiglu ? (P.N / 2) / (ntile / 2) : (P.N + ntile - 1) / ntile;
  const int bslot = box_slot(mma_n / 2);
  auto find = [&](const void* w) -> const CUtensorMap* {
    auto it = plans.maps->weight[bslot].find(w);
    return it == plans.maps->weight[bslot].end() ? nullptr : &it->second;
  };
  const CUtensorMap* a0 = find(P.A0);
  const CUtensorMap* a1 = find(P.A1);
  const CUtensorMap* a2 = find(P.A2);
  if (bslot < 0 || !a0 || !a1 || !a2) return cudaErrorInvalidValue;
  if (nrb != 1 && (nrb != 2 || nmma != 1)) return cudaErrorInvalidValue;
  TcLaunch L{};
  L.ntile = ntile;
  L.mma_n = mma_n;
  L.nrb = nrb;                                 // 128-row blocks per CTA
  L.buf_cols = nrb * ntile;
  L.nbuf = nmma == 1 && nrb == 1 ? 2 : 1;      // 512 TMEM columns either way
  L.tmem_cols = 512;
  L.a_bytes = (uint32_t)nrb * kXBlockBytes;
  // 32, 40 or 48 KB: multiples of 1024, as the 128-byte swizzle wants
  L.stage_bytes = L.a_bytes + nmma * pair_wbytes(mma_n);
  const uint32_t stg_bytes = splits > 1 ? 4 * kStageBoxBytes : 0;
  L.stages = (int)std::min<uint32_t>(kMaxStages, (kMaxDynSmem - 1024 - stg_bytes) / L.stage_bytes);
  L.stg_off = (uint32_t)L.stages * L.stage_bytes;
  L.tiles = tiles;
  if (tiles_out) *tiles_out = tiles;
  P.splits = splits;
  CUtensorMap mx, mpart;
  if (!encode_2d(&mx, P.X, P.K, P.M, 128)) return cudaErrorInvalidValue;
  if (stg_bytes) {
    if (!P.partial || !encode_partial(&mpart, P.partial, P.N, P.M, splits))
      return cudaErrorInvalidValue;
  } else {
    mpart = mx;  // not read
  }
  const bool norm = P.epi.mode == EPI_RESID && P.epi.norm_w;
  const int units = tiles * splits;
  const int npairs = std::min(units, npairs_max);
  const size_t smem = (size_t)L.stages * L.stage_bytes + stg_bytes + 1024;
  auto kernel = nrb == 2 ? gemm_tc_pair_kernel<1, 2>
                         : (nmma == 1 ? gemm_tc_pair_kernel<1> : gemm_tc_pair_kernel<2>);
  cudaError_t e = ensure_dyn_smem((const void*)kernel, kMaxDynSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * npairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kernel, *a0, *a1, *a2, mx, mpart, P, L);
  if (launches_out) *launches_out = (P.splits > 1 || norm) ? 2 : 1;
  if (e != cudaSuccess) return e;
  return launch_gemm_epilogue(plans, P, L, st);
}

cudaError_t launch_gemm_tc(const TcPlanSet& plans, GemmProblem P, int kind, cudaStream_t st,
                           int* tiles_out, int* launches_out) {
  (void)kind;
  if (P.K % kBK || P.M < 1 || P.M > 512 || P.N % 4) return cudaErrorInvalidValue;
  // the LM head above 256 rows: SM pairs with two 256-row blocks and
  // 256-wide vocabulary tiles, so that an SM receives two 16 KB activation
  // blocks per 16 KB of weights (the one-SM kernel's 128-wide tiles at 512
  // rows: four per 16 KB)
  if (P.epi.mode == EPI_LMHEAD && P.M > 256 && !P.swiglu && P.N % 128 == 0) {
    const int npairs = std::min(plans.num_sms / 2,
                                pair_capacity(pair_smem(1, kPairN, 1, 2), plans.num_sms));
    if (npairs > 0) {
      PairPlan pp;
      pp.ntile = kPairN;
      pp.mma_n = kPairN;
      pp.splits = 1;
      pp.t = 0.0;
      return launch_gemm_pair(plans, P, pp, npairs, st, tiles_out, launches_out, 2);
    }
  }
  double t_one = 0.0;
  TcChoice choice = tc_plan(plans, P, &t_one);
  if (pair_possible(P)) {
    // the pair kernel when its modelled time beats the one-SM plan's, with
    // as many pairs as can be resident at once (the smallest capacity over
    // the shared-memory sizes a plan may take)
    constexpr int kShapes[3][2] = {{1, 256}, {2, 256}, {2, 192}};  // (nmma, mma_n)
    int npairs = plans.num_sms / 2;
    for (const auto& sh : kShapes)
      for (int sp : {1, 2})
        npairs = std::min(npairs, pair_capacity(pair_smem(sh[0], sh[1], sp), plans.num_sms));
    PairPlan best;
    for (const auto& sh : kShapes) {
      const PairPlan pp = pair_plan(P, sh[0], sh[1], npairs, plans.part_elems, 1);
      if (pp.t < best.t) best = pp;
    }
    if (best.ntile && best.t < t_one)
      return launch_gemm_pair(plans, P, best, npairs, st, tiles_out, launches_out);
  }
  // 257..512 rows: SM pairs with two 256-row blocks (one N = 256 MMA per
  // block and K step, 512 TMEM columns) when the model prefers them
  if (P.M > 256 && P.epi.mode != EPI_LMHEAD && !P.m_count &&
      (P.swiglu ? (P.N / 2) % 128 == 0 : P.N % 128 == 0)) {
    int npairs = plans.num_sms / 2;
    for (int sp : {1, 2})
      npairs = std::min(npairs, pair_capacity(pair_smem(1, kPairN, sp, 2), plans.num_sms));
    const PairPlan pp = pair_plan(P, 1, kPairN, npairs, plans.part_elems, 2);
    if (pp.ntile && pp.t < t_one)
      return launch_gemm_pair(plans, P, pp, npairs, st, tiles_out, launches_out, 2);
  }
  // rows counted on the device (the LM head on masked rows): no split-K, so
  // that no epilogue kernel has to learn the count
  if (P.m_count) choice.splits = 1;
  const int ntile = choice.ntile, splits = choice.splits;
  auto tiles_for = [&](int nt) { return tc_tiles_for(P, nt); };
  const int bslot = box_slot(P.swiglu ? ntile / 2 : ntile);
  if (bslot < 0) return cudaErrorInvalidValue;
  auto find = [&](const void* w) -> const CUtensorMap* {
    auto it = plans.maps->weight[bslot].find(w);
    return it == plans.maps->weight[bslot].end() ? nullptr : &it->second;
  };
  const CUtensorMap* a0 = find(P.A0);
  const CUtensorMap* a1 = find(P.A1);
  const CUtensorMap* a2 = find(P.A2);
  if (!a0 || !a1 || !a2) return cudaErrorInvalidValue;
  TcLaunch L{};
  L.ntile = ntile;
  L.nrb = (P.M + 127) / 128;
  L.buf_cols = (uint32_t)(L.nrb * L.ntile);
  L.nbuf = L.buf_cols * 2 <= 512 ? 2 : 1;
  L.a_bytes = (uint32_t)L.nrb * kXBlockBytes;
  L.stage_bytes = L.a_bytes + (uint32_t)L.ntile * 128u;
  // persistent split-K: 4 staging boxes for the partial stores after the ring
  const uint32_t stg_bytes = splits > 1 ? 4 * kStageBoxBytes : 0;
  L.stages = (int)std::min<uint32_t>(kMaxStages,
                                     (kMaxDynSmem - 1024 - stg_bytes) / L.stage_bytes);
  if (L.stages < 2) return cudaErrorInvalidValue;
  L.stg_off = (uint32_t)L.stages * L.stage_bytes;  // a multiple of 1024
  uint32_t cols = 32;
  while (cols < L.buf_cols * (uint32_t)L.nbuf) cols <<= 1;
  if (cols > 512) return cudaErrorInvalidValue;
  L.tmem_cols = cols;
  CUtensorMap mx, mpart;
  if (!encode_2d(&mx, P.X, P.K, P.M, 128)) return cudaErrorInvalidValue;
  if (stg_bytes) {
    if (!P.partial || !encode_partial(&mpart, P.partial, P.N, P.M, splits))
      return cudaErrorInvalidValue;
  } else {
    mpart = mx;  // not read
  }
  L.tiles = tiles_for(ntile);
  if (tiles_out) *tiles_out = L.tiles;
  P.splits = splits;
  const int units = L.tiles * P.splits;
  const bool norm = P.epi.mode == EPI_RESID && P.epi.norm_w;
  const int grid = std::min(units, plans.num_sms);
  const size_t smem = (size_t)L.stages * L.stage_bytes + stg_bytes + 1024;
  cudaError_t le = launch_pdl(gemm_tc_kernel, dim3(grid), dim3(kThreads), smem, st, *a0, *a1,
                              *a2, mx, mpart, P, L);
  if (launches_out) *launches_out = (P.splits > 1 || norm) ? 2 : 1;
  if (le != cudaSuccess) return le;
  return launch_gemm_epilogue(plans, P, L, st);
}

// The kernel that follows a GEMM: the RMSNorm of a fused residual without
// split-K, or the split-K sum with its epilogue.
cudaError_t launch_gemm_epilogue(const TcPlanSet& plans, const GemmProblem& P, const TcLaunch& L,
                                 cudaStream_t st) {
  const bool norm = P.epi.mode == EPI_RESID && P.epi.norm_w;
  if (P.splits == 1 && norm) {
    return launch_rmsnorm<bf16>(P.M, P.N, static_cast<const bf16*>(P.epi.x),
                                static_cast<const bf16*>(P.epi.norm_w), P.epi.eps,
                                static_cast<bf16*>(P.epi.xn), st, P.epi.row_dst);
  }
  if (P.splits > 1) {
    const int cap = plans.num_sms * 8;  // grid-stride beyond 8 blocks per SM
    if (norm) {
      if (P.M > 2 * plans.num_sms)
        return launch_pdl(splitk_resid_norm_kernel<1>, dim3(P.M), dim3(kNormThreads), 0, st, P);
      return launch_pdl(splitk_resid_norm_kernel<4>, dim3(P.M), dim3(kNormThreads), 0, st, P);
    } else if (P.epi.mode == EPI_RESID) {
      const size_t n4 = (size_t)P.M * P.N / 4;
      return launch_pdl(splitk_resid_kernel, dim3((int)std::min<size_t>((n4 + 255) / 256, cap)),
                        dim3(256), 0, st, P);
    } else if (P.epi.mode == EPI_SWIGLU) {
      const size_t n4 = (size_t)P.M * (P.N / 2) / 4;
      return launch_pdl(splitk_swiglu_kernel, dim3((int)std::min<size_t>((n4 + 255) / 256, cap)),
                        dim3(256), 0, st, P, L.ntile);
    } else if (P.epi.mode == EPI_QKV && P.epi.hd == 128) {
      const int warps = P.M * (P.N / 128);
      return launch_pdl(splitk_qkv_kernel, dim3((warps + 7) / 8), dim3(256), 0, st, P);
    } else {
      const int items = tc_epi_items(P, L.ntile);
      return launch_pdl(splitk_epilogue_kernel, dim3(L.tiles * items, (P.M + 127) / 128),
                        dim3(128), 0, st, P, L.ntile, items);
    }
  }
  return cudaGetLastError();
}

}  // namespace wedlm
