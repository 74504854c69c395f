// Paged causal GQA window attention on the 5th-generation tensor cores.
//
// The step is "a small causal prefill over the active window on top of
// cached KV" (WeDLM summary page, Key claims §5.2): the G*W query rows of
// one kv head (G = nq/nkv q heads x W window rows, physical order) attend to
// every cached prefix position and, causally, to the window (§3.2).
//
// Work = unit (sequence b, kv head) x 64-key tiles: ceil(L_b/64) prefix
// tiles, then one window tile.  Stream-K: the units' tiles are laid end to
// end and every block (one per SM) takes an equal contiguous share, so a
// block processes runs ("segments") of consecutive tiles of one unit; O, the
// running max and the sum stay in registers across a segment and each
// segment writes one unnormalised partial, combined by attn_seg_merge_kernel.
// Warp roles:
//   warps 0-7: online softmax.  Warps q and q+4 share TMEM lane quadrant q
//       (query rows 32q..32q+31, thread = row): warp q takes key columns
//       0-31 of each tile and head dims 0-63 of O, warp q+4 the other halves;
//       they exchange only the row max of each tile.  They also stage Q at
//       the start of each segment.  P goes to shared memory in bf16 (double
//       buffered); O accumulates in registers with the rescale;
//   warps 8 and 10 / lane 0: copiers of K and of V: a prefix tile is 4
//       pages of K and 4 of V (4 KiB each, already in the 8x8-tile operand
//       layout), copied with cp.async.bulk into 4-stage K and V rings; each
//       ring has its own copier so that K runs ahead of the P V consumers of
//       V; missing or invalid pages come from a zero page; the window tile
//       comes from the window scratch;
//   warp 9 / lane 0: MMA issuer: S = Q K^T (M = 128 query rows, N = keys,
//       K = head_dim) into one of two TMEM score buffers, then O_tile = P V
//       (N = head_dim; V as an MN-major operand) into one of two TMEM output
//       buffers.
#include "internal.h"
#include "tc_ptx.cuh"

namespace wedlm {

namespace {
constexpr int kTile = 64;                  // keys per prefix tile (4 pages)
constexpr int kStages = 4;
constexpr int kThreads = 352;              // 8 softmax warps, K copier, MMA, V copier
constexpr uint32_t kQBytes = 128 * 128 * 2;        // 128 rows x 128 dims
constexpr uint32_t kPBytes = 128 * kTile * 2;      // 128 rows x 64 keys
constexpr uint32_t kKVBytes = kTile * 128 * 2;     // one K or V tile
constexpr uint32_t kOffP = kQBytes;
constexpr uint32_t kOffK = kOffP + 2 * kPBytes;
constexpr uint32_t kOffV = kOffK + kStages * kKVBytes;
constexpr uint32_t kSmemBytes = kOffV + kStages * kKVBytes;   // 192 KB
constexpr uint32_t kPageBytes = 16 * 128 * 2;                 // 4 KiB
constexpr uint32_t kTmemCols = 512;  // S: 2 x 64 columns; O: 2 x 128 columns
constexpr int kMaxB = kMaxRows;      // sequences (<= rows)
constexpr int kPagesPerTile = kTile / kPageBlock;
constexpr int kPrefTiles = 1024;     // tiles whose page ids are staged up front
constexpr int kMaxGrid = 256;        // blocks of one launch
}  // namespace

// Split of the flattened tile sequence over the blocks; every block and the
// segment table agree on it.
struct StreamSplit {
  long long total;  // tiles of all units
  int G;            // blocks that get work
  __device__ long long begin(int c) const { return (long long)c * total / G; }
};

// largest index i in [0, n) with a[i] <= x (a ascending, a[0] <= x)
__device__ __forceinline__ int last_le(const long long* a, int n, long long x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int seq_len_clamped(const AttnArgs& A, int b) {
  return max(0, min(A.seq_len[b], A.max_pages * kPageBlock));
}
__device__ __forceinline__ int seq_tiles(const AttnArgs& A, int b) {
  return (seq_len_clamped(A, b) + kTile - 1) / kTile + 1;
}

__device__ __forceinline__ uint32_t idesc_pv() {  // M=128, N=128, B MN-major
  return idesc_bf16_m128(128) | (1u << 16);
}

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(AttnArgs A, const void* zero_page) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ __align__(8) uint64_t k_full[kStages], k_empty[kStages];
  __shared__ __align__(8) uint64_t v_full[kStages], v_empty[kStages];
  __shared__ __align__(8) uint64_t s_full[2], s_free[2], o_full[2], o_free[2];
  __shared__ __align__(8) uint64_t p_full[2], p_empty[2], q_full, q_empty;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_issued[2], s_done[2];  // K/V tiles copied / consumed
  __shared__ float s_red[2][2][128];      // [tile parity][half][row]: row max
  __shared__ float s_lsum[2][128];        // [half][row]: segment row sums
  __shared__ long long s_tstart[kMaxB + 1];  // first global tile of sequence b
  __shared__ long long s_begin[kMaxGrid + 1];  // first global tile of block c
  __shared__ int s_T[kMaxB];                 // tiles of one unit of sequence b
  __shared__ int s_pages[kPrefTiles * kPagesPerTile];  // page ids (-1: none)
  __shared__ StreamSplit s_split;

  const int hd = 128, G = A.nq / A.nkv, W = A.W, R = G * W;
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // The plan, computed by the whole block: tiles per sequence, their
  // prefix sums, the equal split of all tiles over the blocks.  A segment
  // (the tiles of unit u inside block c) has slot u + c: along the tile
  // order neither u nor c ever decreases and one of them grows from one
  // segment to the next, so slots are distinct and fewer than units + G.
  for (int b = threadIdx.x; b < A.B; b += kThreads) s_T[b] = seq_tiles(A, b);
  __syncthreads();
  if (warp == 0) {
    const int per = (A.B + 31) / 32;
    const int b0 = min(A.B, lane * per), b1 = min(A.B, b0 + per);
    long long sum = 0;
    for (int b = b0; b < b1; ++b) sum += (long long)s_T[b] * A.nkv;
    long long incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    long long acc = incl - sum;
    for (int b = b0; b < b1; ++b) {
      s_tstart[b] = acc;
      acc += (long long)s_T[b] * A.nkv;
    }
    if (lane == 31) {
      StreamSplit sp;
      sp.total = incl;
      const long long by_min = (incl + A.min_tiles - 1) / A.min_tiles;
      sp.G = (int)min((long long)min((int)gridDim.x, kMaxGrid), max(1LL, by_min));
      s_split = sp;
      s_tstart[A.B] = incl;
    }
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1); mbar_init(&s_free[i], 8);
      mbar_init(&o_full[i], 1); mbar_init(&o_free[i], 8);
      mbar_init(&p_full[i], 8); mbar_init(&p_empty[i], 1);
    }
    mbar_init(&q_full, 8);
    mbar_init(&q_empty, 1);
    s_abort = 0;
    s_issued[0] = s_issued[1] = s_done[0] = s_done[1] = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const StreamSplit sp = s_split;
  if ((int)blockIdx.x >= sp.G) return;  // uniform for the block
  for (int c = threadIdx.x; c <= sp.G; c += kThreads) s_begin[c] = sp.begin(c);
  __syncthreads();
  if (blockIdx.x == 0) {
    // segment table: unit u's segments are slots u + c for the blocks c
    // from the owner of its first tile to the owner of its last
    for (int u = threadIdx.x; u < A.B * A.nkv; u += kThreads) {
      const int b = u / A.nkv, h = u % A.nkv, T = s_T[b];
      const long long u0 = s_tstart[b] + (long long)h * T;
      const int c0 = last_le(s_begin, sp.G, u0), c1 = last_le(s_begin, sp.G, u0 + T - 1);
      A.seg_table[u * 2 + 0] = u + c0;
      A.seg_table[u * 2 + 1] = c1 - c0 + 1;
    }
  }
  if (warp == 0) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
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

  const long long g0 = s_begin[blockIdx.x];
  const int ntiles = (int)(s_begin[blockIdx.x + 1] - g0);
  // position of a block tile: sequence, kv head, tile within the unit and
  // tiles of the unit; found once, then advanced tile by tile
  struct Cur { int b, kvh, t, T, L; };
  Cur first;
  {
    first.b = last_le(s_tstart, A.B, g0);
    first.L = seq_len_clamped(A, first.b);
    first.T = s_T[first.b];
    const long long off = g0 - s_tstart[first.b];
    first.kvh = (int)(off / first.T);
    first.t = (int)(off % first.T);
  }
  auto advance = [&](Cur& c) {
    if (++c.t == c.T) {
      c.t = 0;
      if (++c.kvh == A.nkv) {
        c.kvh = 0;
        if (c.b + 1 < A.B) {
          c.L = seq_len_clamped(A, ++c.b);
          c.T = s_T[c.b];
        }
      }
    }
  };

  // page ids of the block's first kPrefTiles tiles, loaded and checked by
  // every thread at once so the producer never waits on a global load
  for (int e = threadIdx.x; e < min(ntiles, kPrefTiles) * kPagesPerTile; e += kThreads) {
    const long long g = g0 + e / kPagesPerTile;
    const int b = last_le(s_tstart, A.B, g);
    const int L = seq_len_clamped(A, b), T = s_T[b];
    const int t = (int)((g - s_tstart[b]) % T);
    const int t0 = t * kTile + (e % kPagesPerTile) * kPageBlock;
    int pid = -1;
    if (t != T - 1 && t0 < L) {
      pid = A.page_table[(size_t)b * A.max_pages + t0 / kPageBlock];
      if (pid < 0 || pid >= A.num_pages) {
        set_err(A.err, WEDLM_DEV_BAD_PAGE);
        pid = -1;
      }
    }
    s_pages[e] = pid;
  }
  __syncthreads();

  if (warp == 8 || warp == 10) {
    if (lane == 0) {
      // ---------------- copiers: K (warp 8), V (warp 10) ----------------
      const int kv = (warp == 10);
      const uint64_t pol = l2_evict_first_policy();
      const bf16* pool = static_cast<const bf16*>(A.pool);
      const bf16* win = static_cast<const bf16*>(A.kv_win);
      const size_t blockn = (size_t)kPageBlock * hd;
      constexpr int kPg = kPagesPerTile;
      // page ids of a tile (-1: no page there): staged in shared memory for
      // the first kPrefTiles tiles, loaded directly beyond that
      auto tile_pages = [&](int i, const Cur& c, int (&pid)[kPg]) {
#pragma unroll
        for (int pg = 0; pg < kPg; ++pg) {
          if (i < kPrefTiles) {
            pid[pg] = s_pages[i * kPg + pg];
          } else {
            const int t0 = c.t * kTile + pg * kPageBlock;
            int v = -1;
            if (c.t != c.T - 1 && t0 < c.L) {
              v = A.page_table[(size_t)c.b * A.max_pages + t0 / kPageBlock];
              if (v < 0 || v >= A.num_pages) {
                set_err(A.err, WEDLM_DEV_BAD_PAGE);
                v = -1;
              }
            }
            pid[pg] = v;
          }
        }
      };
      Cur cur = first;
      for (int i = 0; i < ntiles; ++i, advance(cur)) {
        int pid[kPg];
        tile_pages(i, cur, pid);
        const int b = cur.b, kvh = cur.kvh, t = cur.t, T = cur.T;
        const bool window = (t == T - 1);
        const int st = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        uint64_t* full = kv ? &v_full[st] : &k_full[st];
        if (!wait(kv ? &v_empty[st] : &k_empty[st], ph ^ 1u)) break;
        uint8_t* dst = base + (kv ? kOffV : kOffK) + st * kKVBytes;
        if (window) {
          const uint32_t bytes = (uint32_t)A.Wp * hd * 2;
          mbar_arrive_expect_tx(full, bytes);
          bulk_load(dst, win + (((size_t)b * 2 + kv) * A.nkv + kvh) * A.Wp * hd, bytes, full,
                    pol);
        } else {
          mbar_arrive_expect_tx(full, kKVBytes);
#pragma unroll
          for (int pg = 0; pg < kPg; ++pg) {
            const void* src =
                pid[pg] >= 0
                    ? (const void*)(pool + (((size_t)pid[pg] * 2 + kv) * A.nkv + kvh) * blockn)
                    : zero_page;
            bulk_load(dst + pg * kPageBytes, src, kPageBytes, full, pol);
          }
        }
        s_issued[kv] = i + 1;
      }
    }
  } else if (warp == 9) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t sq = smem_u32(base);
      const uint32_t idPV = idesc_pv();
      int seg = -1;  // segment counter (Q buffer phases)
      Cur cs = first;  // position of the next S to issue
      auto issue_s = [&](int i) -> bool {
        const int t = cs.t, T = cs.T;
        advance(cs);
        if (i == 0 || t == 0) {  // a new segment: wait for its Q
          ++seg;
          if (!wait(&q_full, (uint32_t)seg & 1u)) return false;
        }
        const int st = i % kStages, sb = i & 1;
        if (!wait(&k_full[st], (uint32_t)(i / kStages) & 1u)) return false;
        s_done[0] = i + 1;
        if (!wait(&s_free[sb], ((uint32_t)(i >> 1) & 1u) ^ 1u)) return false;
        tc_fence_after();
        const uint32_t sk = smem_u32(base + kOffK + st * kKVBytes);
        const uint32_t idS = idesc_bf16_m128(t == T - 1 ? A.Wp : kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16(tmem + (uint32_t)(sb * 64), sdesc_noswz(sq + kk * 256, 128, 2048),
                     sdesc_noswz(sk + kk * 256, 128, 2048), idS, kk ? 1u : 0u);
        tc_commit(&s_full[sb]);
        tc_commit(&k_empty[st]);
        if (i == ntiles - 1 || t == T - 1) tc_commit(&q_empty);  // segment's last S
        return true;
      };
      bool ok = issue_s(0);
      Cur cur = first;
      for (int i = 0; i < ntiles && ok; ++i, advance(cur)) {
        const int t = cur.t, T = cur.T;
        // within a segment the next S goes ahead of this P V; across a
        // segment boundary it must wait for the next Q, which the softmax
        // warps stage only after this tile's P V
        const bool next_same = (i + 1 < ntiles) && (t != T - 1);
        if (next_same && !issue_s(i + 1)) break;
        const int st = i % kStages, ob = i & 1, pb = i & 1;
        if (!wait(&v_full[st], (uint32_t)(i / kStages) & 1u)) break;
        s_done[1] = i + 1;
        if (!wait(&p_full[pb], (uint32_t)(i >> 1) & 1u)) break;
        if (!wait(&o_free[ob], ((uint32_t)(i >> 1) & 1u) ^ 1u)) break;
        tc_fence_after();
        const uint32_t sv = smem_u32(base + kOffV + st * kKVBytes);
        const uint32_t spp = smem_u32(base + kOffP + pb * kPBytes);
        const int nk = (t == T - 1) ? A.Wp : kTile;
        for (int kk = 0; kk < nk / 16; ++kk)
          tc_mma_f16(tmem + 128u + (uint32_t)(ob * 128), sdesc_noswz(spp + kk * 256, 128, 1024),
                     sdesc_noswz(sv + kk * 4096, 2048, 128), idPV, kk ? 1u : 0u);
        tc_commit(&o_full[ob]);
        tc_commit(&v_empty[st]);
        tc_commit(&p_empty[pb]);
        if (i + 1 < ntiles && !next_same && !issue_s(i + 1)) break;
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
    const int tid = threadIdx.x;                  // 0..255
    float o[64];
#pragma unroll
    for (int d = 0; d < 64; ++d) o[d] = 0.f;
    float m = -INFINITY, l = 0.f, alpha_prev = 1.f;
    int seg = -1;
    auto pair_bar = [&]() {  // warps q and q+4
      asm volatile("bar.sync %0, 64;" ::"r"(1 + q) : "memory");
    };
    auto softmax_bar = [&]() {  // the 8 softmax warps
      asm volatile("bar.sync 5, 256;" ::: "memory");
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
    Cur cur = first;
    for (int i = 0; i < ntiles; ++i, advance(cur)) {
      const int b = cur.b, kvh = cur.kvh, t = cur.t, T = cur.T;
      if (i == 0 || t == 0) {
        // new segment: stage its Q once the previous segment's S MMAs are done
        ++seg;
        wait(&q_empty, ((uint32_t)seg & 1u) ^ 1u);
        const bf16* qg = static_cast<const bf16*>(A.q);
        for (int idx = tid; idx < 128 * 16; idx += 256) {
          const int rr = idx >> 4, d8 = idx & 15;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (rr < R) {
            const int g = rr / W, p = rr % W;
            v = *reinterpret_cast<const uint4*>(
                qg + ((size_t)(b * W + p) * A.nq + kvh * G + g) * hd + d8 * 8);
          }
          *reinterpret_cast<uint4*>(base + (rr >> 3) * 2048 + d8 * 128 + (rr & 7) * 16) = v;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        softmax_bar();
        if (lane == 0) mbar_arrive(&q_full);
#pragma unroll
        for (int d = 0; d < 64; ++d) o[d] = 0.f;
        m = -INFINITY;
        l = 0.f;
      }
      const bool window = (t == T - 1);
      const int L = cur.L;
      const int sb = i & 1, pb = i & 1;
      wait(&s_full[sb], (uint32_t)(i >> 1) & 1u);
      tc_fence_after();
      float v[32];
      tmem_ld32(trow + (uint32_t)(sb * 64 + h * 32), v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);
      // mask (only the partial last prefix tile and the window tile need
      // one), row max over both halves of the tile, scale applied once
      const int kbase = t * kTile;
      if (window || kbase + kTile > L) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int jj = h * 32 + j;
          const bool ok = window ? (jj < W && jj <= p_row) : (kbase + jj < L);
          if (!ok) v[j] = -INFINITY;
        }
      }
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mx[k] = fmaxf(fmaxf(v[4 * k], v[4 * k + 1]), fmaxf(v[4 * k + 2], v[4 * k + 3]));
      const float hmax =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sc;
      s_red[i & 1][h][r] = hmax;
      pair_bar();
      const float m_new = fmaxf(m, fmaxf(hmax, s_red[i & 1][h ^ 1][r]));
      const float alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_new);
      // p = 2^(s*scale - m_new); masked scores are -inf and give 0
      const float nm = (m_new == -INFINITY) ? 0.f : -m_new;
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t packed[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float p0 = ex2_approx(fmaf(v[j], sc, nm));
        const float p1 = ex2_approx(fmaf(v[j + 1], sc, nm));
        ps[(j >> 1) & 3] += p0 + p1;
        const __nv_bfloat162 pk = __floats2bfloat162_rn(p0, p1);
        packed[j >> 1] = *reinterpret_cast<const uint32_t*>(&pk);
      }
      const float psum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
      // P buffer pb is free once the P V of two tiles back has read it
      wait(&p_empty[pb], ((uint32_t)(i >> 1) & 1u) ^ 1u);
      uint8_t* prow = base + kOffP + pb * kPBytes + (r >> 3) * 1024 + (r & 7) * 16;
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8)
        *reinterpret_cast<uint4*>(prow + (h * 4 + c8) * 128) =
            make_uint4(packed[4 * c8], packed[4 * c8 + 1], packed[4 * c8 + 2], packed[4 * c8 + 3]);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[pb]);
      // fold in the previous tile's P V (same segment)
      if (i >= 1 && t != 0) accumulate(i - 1, alpha_prev);
      l = l * alpha + psum;  // this half's share of the row sum
      m = m_new;
      alpha_prev = alpha;
      if (i == ntiles - 1 || t == T - 1) {
        // segment end: fold in this tile, write the unnormalised partial
        accumulate(i, alpha_prev);
        s_lsum[h][r] = l;
        pair_bar();
        const float lsum = l + s_lsum[h ^ 1][r];
        if (valid) {
          const size_t sid = (size_t)b * A.nkv + kvh + blockIdx.x;
          const size_t row = sid * R + r;
          float* po = A.part_o + row * hd + h * 64;
#pragma unroll
          for (int d4 = 0; d4 < 16; ++d4)
            reinterpret_cast<float4*>(po)[d4] =
                make_float4(o[4 * d4], o[4 * d4 + 1], o[4 * d4 + 2], o[4 * d4 + 3]);
          if (h == 0) {
            A.part_ml[row * 2 + 0] = m;
            A.part_ml[row * 2 + 1] = lsum;
          }
        }
        pair_bar();  // s_lsum is reused by the next segment
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

// Merge the segment partials of every (sequence, row, q head): one block per
// (b*W + p, h), one thread per head dim.  seg_table holds each unit's first
// segment id and segment count (written by block 0 of the attention kernel).
__global__ void attn_seg_merge_kernel(AttnArgs A) {
  const int mh = blockIdx.x;
  const int m = mh / A.nq, h = mh % A.nq;
  const int b = m / A.W, p = m % A.W;
  const int G = A.nq / A.nkv, kvh = h / G, g = h % G, R = G * A.W;
  const int r = g * A.W + p;
  const int u = b * A.nkv + kvh;
  const int s0 = A.seg_table[u * 2 + 0], ns = A.seg_table[u * 2 + 1];
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, A.part_ml[((size_t)(s0 + s) * R + r) * 2]);
  float lsum = 0.f, acc = 0.f;
  const int d = threadIdx.x;
  for (int s = 0; s < ns; ++s) {
    const size_t row = (size_t)(s0 + s) * R + r;
    const float ms = A.part_ml[row * 2];
    if (ms == -INFINITY) continue;
    const float w = exp2f(ms - M);
    lsum += A.part_ml[row * 2 + 1] * w;
    acc += A.part_o[row * A.hd + d] * w;
  }
  static_cast<bf16*>(A.o)[(size_t)m * A.nq * A.hd + h * A.hd + d] =
      __float2bfloat16_rn(lsum > 0.f ? acc / lsum : 0.f);
}

cudaError_t launch_attention_tc(const AttnArgs& A, const void* zero_page, int grid,
                                cudaStream_t st) {
  if (A.hd != 128 || (A.nq / A.nkv) * A.W > 128 || A.Wp > kTile || A.B > kMaxB ||
      A.min_tiles < 1 || !A.seg_table || grid < 1)
    return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(
        attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes + 1024);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  attn_tc_kernel<<<min(grid, kMaxGrid), kThreads, kSmemBytes + 1024, st>>>(A, zero_page);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_seg_merge_kernel<<<A.B * A.W * A.nq, A.hd, 0, st>>>(A);
  return cudaGetLastError();
}

}  // namespace wedlm
