// Paged causal GQA window attention on the 5th-generation tensor cores.
//
// The step is "a small causal prefill over the active window on top of
// cached KV" (WeDLM summary page, Key claims §5.2): the G*W query rows of
// one kv head (G = nq/nkv q heads x W window rows, physical order) attend to
// every cached prefix position and, causally, to the window (§3.2).
//
// Block = (sequence b, kv head, key chunk); chunks 0..ceil(L/chunk)-1 cover
// the prefix, the last one the window.  Warp roles:
//   warp 8 / lane 0: producer: each 64-key tile is 4 pages of K and 4 of V
//       (4 KiB each, already in the 8x8-tile operand layout), copied with
//       cp.async.bulk into 4-stage K and V rings; missing or invalid pages
//       come from a zero page;
//   warp 9 / lane 0: MMA issuer: S = Q K^T (M = 128 query rows, N = 64 keys,
//       K = head_dim) into one of two TMEM score buffers, then O_tile = P V
//       (N = head_dim, K = 64 keys; V as an MN-major operand) into one of
//       two TMEM output buffers;
//   warps 0-7: online softmax.  Warps q and q+4 share TMEM lane quadrant q
//       (query rows 32q..32q+31, thread = row): warp q takes key columns
//       0-31 of each tile and head dims 0-63 of O, warp q+4 the other halves;
//       they exchange only the row max of each tile.  Scores come from TMEM,
//       the running max / sums live in the log2 domain, P goes to shared
//       memory in bf16 and O accumulates in registers with the rescale.
// The block writes an unnormalised partial (O, running max, sum) that the
// split-KV merge combines.
#include "internal.h"
#include "tc_ptx.cuh"

namespace wedlm {

namespace {
constexpr int kTile = 64;                  // keys per prefix tile (4 pages)
constexpr int kStages = 4;
constexpr int kThreads = 320;            // 8 softmax warps, producer, MMA
constexpr uint32_t kQBytes = 128 * 128 * 2;        // 128 rows x 128 dims
constexpr uint32_t kPBytes = 128 * kTile * 2;      // 128 rows x 64 keys
constexpr uint32_t kKVBytes = kTile * 128 * 2;     // one K or V tile
constexpr uint32_t kOffP = kQBytes;
constexpr uint32_t kOffK = kOffP + kPBytes;
constexpr uint32_t kOffV = kOffK + kStages * kKVBytes;
constexpr uint32_t kSmemBytes = kOffV + kStages * kKVBytes;   // 176 KB
constexpr uint32_t kPageBytes = 16 * 128 * 2;                 // 4 KiB
constexpr uint32_t kTmemCols = 512;  // S: 2 x 64 columns; O: 2 x 128 columns
}  // namespace

struct AttnTcArgs {
  AttnArgs A;
  const void* zero_page;   // 4 KiB of zeros
};

__device__ __forceinline__ uint32_t idesc_pv() {  // M=128, N=128, B MN-major
  return idesc_bf16_m128(128) | (1u << 16);
}

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(AttnTcArgs args) {
  const AttnArgs& A = args.A;
  extern __shared__ uint8_t dsm_raw[];
  __shared__ __align__(8) uint64_t k_full[kStages], k_empty[kStages];
  __shared__ __align__(8) uint64_t v_full[kStages], v_empty[kStages];
  __shared__ __align__(8) uint64_t s_full[2], s_free[2], o_full[2], o_free[2];
  __shared__ __align__(8) uint64_t p_full, p_empty;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_issued[2], s_done[2];  // K/V tiles copied / consumed
  __shared__ float s_red[2][2][128];      // [tile parity][half][row]: row max
  __shared__ float s_lsum[2][128];        // [half][row]: final row sums

  const int b = blockIdx.z, kvh = blockIdx.y, c = blockIdx.x;
  const int hd = 128, G = A.nq / A.nkv, W = A.W, R = G * W;
  const int L = max(0, min(A.seq_len[b], A.max_pages * kPageBlock));
  const int n_pre = (L + A.chunk - 1) / A.chunk;
  if (c > n_pre) return;  // no work for this chunk (uniform for the block)
  const bool window = (c == n_pre);
  const int k0 = window ? 0 : c * A.chunk;
  const int k1 = window ? W : min(L, k0 + A.chunk);
  const int ntiles = window ? 1 : (k1 - k0 + kTile - 1) / kTile;
  const int win_keys = A.Wp;  // keys of the window tile (multiple of 16)

  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1); mbar_init(&s_free[i], 8);
      mbar_init(&o_full[i], 1); mbar_init(&o_free[i], 8);
    }
    mbar_init(&p_full, 8);
    mbar_init(&p_empty, 1);
    s_abort = 0;
    s_issued[0] = s_issued[1] = s_done[0] = s_done[1] = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  // stage Q (rows >= R zero) in the K-major 8x8-core layout: core (r/8, d/8)
  // at (r/8)*2048 + (d/8)*128 + (r%8)*16 bytes
  {
    const bf16* q = static_cast<const bf16*>(A.q);
    for (int idx = threadIdx.x; idx < 128 * 16; idx += kThreads) {
      const int r = idx >> 4, d8 = idx & 15;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < R) {
        const int g = r / W, p = r % W;
        v = *reinterpret_cast<const uint4*>(q + ((size_t)(b * W + p) * A.nq + kvh * G + g) * hd +
                                            d8 * 8);
      }
      *reinterpret_cast<uint4*>(base + (r >> 3) * 2048 + d8 * 128 + (r & 7) * 16) = v;
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort = &s_abort;
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (*abort) return false;
    if (mbar_wait(bar, parity, A.err)) return true;
    *abort = 1;
    return false;
  };

  if (warp == 8) {
    if (lane == 0) {
      // ---------------- producer ----------------
      const uint64_t pol = l2_evict_first_policy();
      const bf16* pool = static_cast<const bf16*>(A.pool);
      const bf16* win = static_cast<const bf16*>(A.kv_win);
      const size_t blockn = (size_t)kPageBlock * hd;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        for (int kv = 0; kv < 2; ++kv) {
          uint64_t* full = kv ? &v_full[st] : &k_full[st];
          if (!wait(kv ? &v_empty[st] : &k_empty[st], ph ^ 1u)) break;
          uint8_t* dst = base + (kv ? kOffV : kOffK) + st * kKVBytes;
          if (window) {
            const uint32_t bytes = (uint32_t)win_keys * hd * 2;
            mbar_arrive_expect_tx(full, bytes);
            bulk_load(dst, win + (((size_t)b * 2 + kv) * A.nkv + kvh) * A.Wp * hd, bytes, full,
                      pol);
          } else {
            mbar_arrive_expect_tx(full, kKVBytes);
            for (int pg = 0; pg < kTile / kPageBlock; ++pg) {
              const int t0 = k0 + i * kTile + pg * kPageBlock;
              const void* src = args.zero_page;
              if (t0 < k1) {
                const int pidx = t0 / kPageBlock;
                const int page = A.page_table[(size_t)b * A.max_pages + pidx];
                if (page >= 0 && page < A.num_pages)
                  src = pool + (((size_t)page * 2 + kv) * A.nkv + kvh) * blockn;
                else
                  set_err(A.err, WEDLM_DEV_BAD_PAGE);
              }
              bulk_load(dst + pg * kPageBytes, src, kPageBytes, full, pol);
            }
          }
          s_issued[kv] = i + 1;
        }
      }
    }
  } else if (warp == 9) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t sq = smem_u32(base);
      const uint32_t sp = smem_u32(base + kOffP);
      const int nS = window ? win_keys : kTile;
      const uint32_t idS = idesc_bf16_m128(nS);
      const uint32_t idPV = idesc_pv();
      auto issue_s = [&](int i) -> bool {
        const int st = i % kStages, sb = i & 1;
        if (!wait(&k_full[st], (uint32_t)(i / kStages) & 1u)) return false;
        s_done[0] = i + 1;
        if (!wait(&s_free[sb], ((uint32_t)(i >> 1) & 1u) ^ 1u)) return false;
        tc_fence_after();
        const uint32_t sk = smem_u32(base + kOffK + st * kKVBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16(tmem + (uint32_t)(sb * 64), sdesc_noswz(sq + kk * 256, 128, 2048),
                     sdesc_noswz(sk + kk * 256, 128, 2048), idS, kk ? 1u : 0u);
        tc_commit(&s_full[sb]);
        tc_commit(&k_empty[st]);
        return true;
      };
      bool ok = issue_s(0);
      for (int i = 0; i < ntiles && ok; ++i) {
        if (i + 1 < ntiles && !issue_s(i + 1)) break;
        const int st = i % kStages, ob = i & 1;
        if (!wait(&v_full[st], (uint32_t)(i / kStages) & 1u)) break;
        s_done[1] = i + 1;
        if (!wait(&p_full, (uint32_t)i & 1u)) break;
        if (!wait(&o_free[ob], ((uint32_t)(i >> 1) & 1u) ^ 1u)) break;
        tc_fence_after();
        const uint32_t sv = smem_u32(base + kOffV + st * kKVBytes);
        for (int kk = 0; kk < nS / 16; ++kk)
          tc_mma_f16(tmem + 128u + (uint32_t)(ob * 128), sdesc_noswz(sp + kk * 256, 128, 1024),
                     sdesc_noswz(sv + kk * 4096, 2048, 128), idPV, kk ? 1u : 0u);
        tc_commit(&o_full[ob]);
        tc_commit(&v_empty[st]);
        tc_commit(&p_empty);
      }
    }
  } else {
    // ---------------- softmax warps ----------------
    const int q = warp & 3, h = warp >> 2;       // lane quadrant, column / dim half
    const int r = 32 * q + lane;                  // query row
    const bool valid = r < R;
    const int p_row = valid ? r % W : 0;
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    const float sc = A.scale_log2;
    float o[64];
#pragma unroll
    for (int d = 0; d < 64; ++d) o[d] = 0.f;
    float m = -INFINITY, l = 0.f, alpha_prev = 1.f;
    uint8_t* prow = base + kOffP + (r >> 3) * 1024 + (r & 7) * 16;
    auto pair_bar = [&]() {  // warps q and q+4
      asm volatile("bar.sync %0, 64;" ::"r"(1 + q) : "memory");
    };
    auto accumulate = [&](int i, float alpha) {
      const int ob = i & 1;
      wait(&o_full[ob], (uint32_t)(i >> 1) & 1u);
      tc_fence_after();
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        float v[32];
        tmem_ld32(trow + 128u + (uint32_t)(ob * 128 + h * 64 + cb * 32), v);
#pragma unroll
        for (int j = 0; j < 32; ++j) o[cb * 32 + j] = fmaf(o[cb * 32 + j], alpha, v[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[ob]);
    };
    for (int i = 0; i < ntiles; ++i) {
      const int sb = i & 1;
      wait(&s_full[sb], (uint32_t)(i >> 1) & 1u);
      tc_fence_after();
      float v[32];
      tmem_ld32(trow + (uint32_t)(sb * 64 + h * 32), v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);
      // mask + scale (log2 domain); row max over both halves of the tile
      const int kbase = window ? 0 : k0 + i * kTile;
      float hmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int jj = h * 32 + j;
        const bool ok = window ? (jj < W && jj <= p_row) : (kbase + jj < k1);
        v[j] = ok ? v[j] * sc : -INFINITY;
        hmax = fmaxf(hmax, v[j]);
      }
      s_red[i & 1][h][r] = hmax;
      pair_bar();
      const float m_new = fmaxf(m, fmaxf(hmax, s_red[i & 1][h ^ 1][r]));
      const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
      float psum = 0.f;
      uint32_t packed[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float p0 = (v[j] == -INFINITY) ? 0.f : exp2f(v[j] - m_new);
        const float p1 = (v[j + 1] == -INFINITY) ? 0.f : exp2f(v[j + 1] - m_new);
        const bf16 b0 = __float2bfloat16_rn(p0), b1 = __float2bfloat16_rn(p1);
        psum += __bfloat162float(b0) + __bfloat162float(b1);
        packed[j >> 1] = (uint32_t)__bfloat16_as_ushort(b0) |
                         ((uint32_t)__bfloat16_as_ushort(b1) << 16);
      }
      l = l * alpha + psum;  // this half's share of the row sum
      m = m_new;
      // P buffer free once the previous tile's P V has read it
      wait(&p_empty, ((uint32_t)i & 1u) ^ 1u);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8)
        *reinterpret_cast<uint4*>(prow + (h * 4 + c8) * 128) =
            make_uint4(packed[4 * c8], packed[4 * c8 + 1], packed[4 * c8 + 2], packed[4 * c8 + 3]);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full);
      if (i >= 1) accumulate(i - 1, alpha_prev);
      alpha_prev = alpha;
    }
    if (ntiles > 0) accumulate(ntiles - 1, alpha_prev);
    // the row sum is split over the two halves
    s_lsum[h][r] = l;
    pair_bar();
    const float lsum = l + s_lsum[h ^ 1][r];
    if (valid) {
      const size_t unit = ((size_t)b * A.nkv + kvh) * A.max_chunks + c;
      float* po = A.part_o + (unit * R + r) * hd + h * 64;
#pragma unroll
      for (int d4 = 0; d4 < 16; ++d4)
        reinterpret_cast<float4*>(po)[d4] =
            make_float4(o[4 * d4], o[4 * d4 + 1], o[4 * d4 + 2], o[4 * d4 + 3]);
      if (h == 0) {
        A.part_ml[(unit * R + r) * 2 + 0] = m;
        A.part_ml[(unit * R + r) * 2 + 1] = lsum;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (s_abort && threadIdx.x == 256) {
    // after a timeout: wait (bounded) for this block's copies still in flight
    for (int kv = 0; kv < 2; ++kv)
      for (int i = s_done[kv]; i < s_issued[kv]; ++i)
        mbar_wait(kv ? &v_full[i % kStages] : &k_full[i % kStages],
                  (uint32_t)(i / kStages) & 1u, A.err);
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_attention_tc(const AttnArgs& A, const void* zero_page, cudaStream_t st) {
  if (A.hd != 128 || (A.nq / A.nkv) * A.W > 128 || A.Wp > kTile || A.chunk % kTile)
    return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(
        attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes + 1024);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  AttnTcArgs args{A, zero_page};
  attn_tc_kernel<<<dim3(A.max_chunks, A.nkv, A.B), kThreads, kSmemBytes + 1024, st>>>(args);
  return cudaGetLastError();
}

}  // namespace wedlm
