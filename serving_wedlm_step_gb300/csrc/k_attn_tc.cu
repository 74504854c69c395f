// Paged causal GQA window attention on the 5th-generation tensor cores.
//
// In a WeDLM decode step the window is attended to like a short causal
// prefill on top of the cached prefix (WeDLM summary page, Key claims §5.2):
// the G*W query rows of one kv head (G = nq/nkv q heads x W window rows,
// physical order) attend to every cached prefix position and, causally, to
// the window (§3.2).
//
// The G*W query rows of a kv head (row r = p*G + g for window row p, q head
// g: the order in which one TMA box {8 dims, G heads, tokens} of q lands in
// shared memory) are cut into row blocks of at most 128 rows, the MMA's M:
// one block of all G*W rows when they fit, else blocks of TPB = 128/G window
// rows (prefill chunks, W = 64 at G = 4).
//
// Work = unit (sequence b, kv head, row block rb) x 128-key tiles:
// ceil(L_b/128) prefix tiles, then the window tiles the row block's causal
// extent reaches (window rows < (rb+1)*TPB).  Stream-K: the units' tiles are
// laid end to end and every block (one per SM) takes an equal contiguous
// share, so a block processes runs ("segments") of consecutive tiles of one
// unit; the row blocks of one kv head are adjacent, so blocks running side
// by side read the same cached pages and the second read hits L2.  A unit
// inside one block is normalised and written out directly; otherwise each
// segment writes an unnormalised partial (O, running max, row sum) and the
// block that finishes a unit's last segment (a per-unit counter) merges the
// partials and writes the output.
//
// Data path of one tile i (everything the softmax warps and the MMA issuers
// hand each other lives in TMEM):
//   S_i = Q K_i^T   (tcgen05.mma, M = 128 query rows, N = 128 keys, K = 128
//                    dims; A = Q, B = K_i from shared memory) -> TMEM S[i%3]
//   P_i = 2^(S_i * scale - m)   (softmax warps, bf16, written over the first
//                    64 columns of S[i%3])
//   O  += P_i V_i   (tcgen05.mma with A = P_i read from TMEM, B = V_i from
//                    shared memory, N = 128 dims)             -> TMEM O
// S buffer i%3 is free again once P_i V_i is done.
// The running max m of a row is raised only when a tile's max exceeds it by
// more than 2^8; then O (once the previous P V is done) and the row sum are
// rescaled.  Between raises the exponentials are taken against the stale
// max, which is exact after the final division because O and the row sum
// share it, and keeps every P value below 2^8.
//
// Warp roles (384 threads):
//   warps 0-7: softmax.  Warps q and q+4 share TMEM lane quadrant q (query
//       rows 32q..32q+31, thread = row): warp q takes keys 0-63 of each tile
//       and head dims 0-63 of O, warp q+4 the other halves; they exchange
//       the row max of each tile through shared memory;
//   warp 8 / lane 0: K copier: Q of each segment (16 TMA boxes into one of
//       two Q buffers) and the K tiles (8 pages of 4 KiB, already in the
//       8x8-tile operand layout, by cp.async.bulk) into the K ring;
//   warp 9 / lane 0: S issuer (S = Q K^T);
//   warp 10 / lane 0: V copier: the V tiles into the V ring;
//   warp 11 / lane 0: P V issuer.  Each issuer's commits track only its own
//       MMAs; S and P V touch disjoint TMEM columns, so the two streams run
//       independently and neither waits behind the other's operands.
// Missing or invalid pages come from a zero page; the window tile comes from
// the window scratch.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "tc_ptx.cuh"

namespace wedlm {

namespace {
constexpr int kTile = 128;                 // keys per prefix tile (8 pages)
constexpr int kPagesPerTile = kTile / kPageBlock;
constexpr int kMaxStages = 4;              // per ring
constexpr int kThreads = 384;
constexpr uint32_t kKVBytes = kTile * 128 * 2;         // one K or V tile: 32 KiB
constexpr uint32_t kPageBytes = kPageBlock * 128 * 2;  // 4 KiB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;      // S[0..2]: 128 fp32 columns each; P over the first 64
constexpr uint32_t kColO = 384;    // O: 128 fp32 columns
constexpr int kSBuf = 3;
constexpr float kRescaleLog2 = 8.f;        // raise the running max beyond 2^8
constexpr int kMaxB = kMaxRows;            // sequences (<= rows)
constexpr int kPrefTiles = 256;            // tiles whose page ids are staged
constexpr int kMaxGrid = 256;              // blocks of one launch
constexpr uint32_t kDynBytes = 205 * 1024; // dynamic shared memory (+1 KiB align)
}  // namespace

constexpr int kMaxRB = 32;  // row blocks per kv head

// ring depths, row blocks and shared-memory carve-up of one launch
// (host-chosen)
struct AttnLayout {
  int R, Rpad;          // rows of a row block (<= 128), rounded up to 8
  int KS, VS;           // K and V ring depths
  uint32_t q_bytes;     // one Q buffer: 16 dim groups x Rpad rows x 16 B
  uint32_t off_k, off_v;
  int TPB, NRB;         // window rows per row block, row blocks per kv head
  int wt[kMaxRB];       // window tiles of row block rb
  int cwt[kMaxRB + 1];  // their prefix sums
};

// Split of the flattened tile sequence over the blocks; every block and the
// segment table agree on it.  The shares are equal in weighted length: a
// unit weighs its tiles plus unit_cost, the time its start (Q, first tile)
// and end (normalise and write, or partial and merge) take, so that a block
// of many short units gets fewer tiles.
struct StreamSplit {
  long long total;    // tiles of all units
  long long total_w;  // their weighted length
  int G;              // blocks that get work
  __device__ long long begin_w(int c) const { return (long long)c * total_w / G; }
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
// prefix tiles of sequence b
__device__ __forceinline__ int prefix_tiles(const AttnArgs& A, int b) {
  return (seq_len_clamped(A, b) + kTile - 1) / kTile;
}

__device__ __forceinline__ uint32_t idesc_pv() {  // M=128, N=128, B MN-major
  return idesc_bf16_m128(128) | (1u << 16);
}

// 3-D tiled TMA load (tensor map in kernel-parameter space)
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16; A (M x K) is read from
// TMEM: lane = row, each 32-bit column holds two consecutive K elements
// (the lower K index in the low half)
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns from registers into TMEM
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 32 lanes x 64 consecutive fp32 columns of TMEM into 64 registers per thread
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, "
      "[%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]),
        "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]),
        "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
        "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]),
        "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]),
        "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap mq, AttnArgs A, AttnLayout Ly,
               const void* zero_page) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ __align__(8) uint64_t k_full[kMaxStages], k_empty[kMaxStages];
  __shared__ __align__(8) uint64_t v_full[kMaxStages], v_empty[kMaxStages];
  __shared__ __align__(8) uint64_t q_full[2], q_empty[2];
  __shared__ __align__(8) uint64_t s_full[kSBuf], s_free[kSBuf], p_full[kSBuf], o_free;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_merge;
  __shared__ int s_issued[3], s_done[3];  // K, V, Q copies issued / consumed
  __shared__ float s_red[2][2][128];      // [tile parity][half][row]: row max
  __shared__ float s_lsum[2][128];        // [half][row]: segment row sums
  __shared__ long long s_tstart[kMaxB + 1];    // first global tile of sequence b
  __shared__ long long s_begin[kMaxGrid + 1];  // first global tile of block c
  __shared__ int s_P[kMaxB];                   // prefix tiles of sequence b
  // page ids (-1: none); before they are loaded, the same bytes hold the
  // first weighted position of each sequence (the plan's split)
  __shared__ __align__(8) int s_pages[kPrefTiles * kPagesPerTile];
  static_assert(sizeof(int) * kPrefTiles * kPagesPerTile >= sizeof(long long) * (kMaxB + 1),
                "the weighted starts must fit the page-id table");
  long long* s_wstart = reinterpret_cast<long long*>(s_pages);
  __shared__ StreamSplit s_split;

  const int hd = 128, G = A.nq / A.nkv, W = A.W, R = Ly.R;
  const int KS = Ly.KS, VS = Ly.VS, NRB = Ly.NRB, TPB = Ly.TPB;
  // tiles of all row blocks of one kv head of a sequence with P prefix tiles
  auto head_tiles = [&](int P) { return NRB * P + Ly.cwt[NRB]; };
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // The plan, computed by the whole block: tiles per sequence, their
  // prefix sums, the equal split of all tiles over the blocks.  A segment
  // (the tiles of unit u inside block c) has slot u + c: along the tile
  // order neither u nor c ever decreases and one of them grows from one
  // segment to the next, so slots are distinct and fewer than units + G.
  for (int b = threadIdx.x; b < A.B; b += kThreads) s_P[b] = prefix_tiles(A, b);
  __syncthreads();
  const int ucost = max(0, A.unit_cost);
  // weighted length of the units of one kv head of a sequence with P prefix tiles
  auto head_weight = [&](int P) { return (long long)NRB * (P + ucost) + Ly.cwt[NRB]; };
  if (warp == 0) {
    const int per = (A.B + 31) / 32;
    const int b0 = min(A.B, lane * per), b1 = min(A.B, b0 + per);
    long long sum = 0, sumw = 0;
    for (int b = b0; b < b1; ++b) {
      sum += (long long)head_tiles(s_P[b]) * A.nkv;
      sumw += head_weight(s_P[b]) * A.nkv;
    }
    long long incl = sum, inclw = sumw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long x = __shfl_up_sync(0xffffffffu, incl, o);
      const long long xw = __shfl_up_sync(0xffffffffu, inclw, o);
      if (lane >= o) {
        incl += x;
        inclw += xw;
      }
    }
    long long acc = incl - sum, accw = inclw - sumw;
    for (int b = b0; b < b1; ++b) {
      s_tstart[b] = acc;
      s_wstart[b] = accw;
      acc += (long long)head_tiles(s_P[b]) * A.nkv;
      accw += head_weight(s_P[b]) * A.nkv;
    }
    if (lane == 31) {
      StreamSplit sp;
      sp.total = incl;
      sp.total_w = inclw;
      const long long by_min = (incl + A.min_tiles - 1) / A.min_tiles;
      sp.G = (int)min((long long)min((int)gridDim.x, kMaxGrid), max(1LL, by_min));
      s_split = sp;
      s_tstart[A.B] = incl;
      s_wstart[A.B] = inclw;
    }
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < kSBuf; ++i) {
      mbar_init(&s_full[i], 1); mbar_init(&s_free[i], 1); mbar_init(&p_full[i], 8);
    }
    mbar_init(&o_free, 8);
    s_abort = 0;
    for (int k = 0; k < 3; ++k) s_issued[k] = s_done[k] = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const StreamSplit sp = s_split;
  if ((int)blockIdx.x >= sp.G) return;  // uniform for the block
  // first tile of each block: its weighted start mapped to the tile it
  // falls on (a start inside a unit's cost lands on the unit's first tile,
  // so a block may be given no tiles, only ever at a unit's start)
  for (int c = threadIdx.x; c <= sp.G; c += kThreads) {
    const long long w = sp.begin_w(c);
    long long g = sp.total;
    if (w < sp.total_w) {
      const int b = last_le(s_wstart, A.B, w);
      const int P = s_P[b];
      const long long off = w - s_wstart[b], H = head_weight(P);
      const int kvh = (int)(off / H);
      const long long r = off % H;
      int rb = 0;
      while (rb + 1 < NRB && (long long)(rb + 1) * (P + ucost) + Ly.cwt[rb + 1] <= r) ++rb;
      const long long x = r - ((long long)rb * (P + ucost) + Ly.cwt[rb]);
      const long long t = max(0LL, x - ucost);  // < P + wt[rb]
      g = s_tstart[b] + (long long)kvh * head_tiles(P) + (long long)rb * P + Ly.cwt[rb] + t;
    }
    s_begin[c] = g;
  }
  __syncthreads();
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
    if (mbar_try_wait(bar, parity)) return true;  // completed: one poll, no flag read
    if (*abort) return false;
    if (mbar_wait(bar, parity, A.err)) return true;
    *abort = 1;
    return false;
  };

  const long long g0 = s_begin[blockIdx.x];
  const int ntiles = (int)(s_begin[blockIdx.x + 1] - g0);
  // position of a tile: sequence, kv head, row block, tile within the unit
  // (prefix tiles 0..P-1, then window tiles), tiles of the unit, cached
  // length and prefix tiles of the sequence; found by search for a block's
  // first tile, then advanced tile by tile
  struct Cur { int b, kvh, rb, t, T, L, P; };
  auto locate = [&](long long g) {
    Cur c;
    c.b = last_le(s_tstart, A.B, g);
    c.L = seq_len_clamped(A, c.b);
    c.P = s_P[c.b];
    const long long off = g - s_tstart[c.b];
    const int TS = head_tiles(c.P);
    c.kvh = (int)(off / TS);
    const int r = (int)(off % TS);
    c.rb = 0;
    while (c.rb + 1 < NRB && (c.rb + 1) * c.P + Ly.cwt[c.rb + 1] <= r) ++c.rb;
    c.t = r - (c.rb * c.P + Ly.cwt[c.rb]);
    c.T = c.P + Ly.wt[c.rb];
    return c;
  };
  const Cur first = locate(g0);
  auto advance = [&](Cur& c) {
    if (++c.t == c.T) {
      c.t = 0;
      if (++c.rb == NRB) {
        c.rb = 0;
        if (++c.kvh == A.nkv) {
          c.kvh = 0;
          if (c.b + 1 < A.B) {
            c.L = seq_len_clamped(A, ++c.b);
            c.P = s_P[c.b];
          }
        }
      }
      c.T = c.P + Ly.wt[c.rb];
    }
  };
  // keys of window tile w (the last one may be partial: Wp is a multiple of 16)
  auto window_keys = [&](int w) { return min(kTile, A.Wp - w * kTile); };

  // page ids of the block's first kPrefTiles tiles, loaded and checked by
  // every thread at once so the copiers never wait on a global load
  for (int e = threadIdx.x; e < min(ntiles, kPrefTiles) * kPagesPerTile; e += kThreads) {
    const Cur c = locate(g0 + e / kPagesPerTile);
    const int b = c.b, L = c.L, t = c.t;
    const int t0 = t * kTile + (e % kPagesPerTile) * kPageBlock;
    int pid = -1;
    if (t < c.P && t0 < L) {
      pid = A.page_table[(size_t)b * A.pt_stride + t0 / kPageBlock];
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
      // ---------------- copiers: K (+ Q) (warp 8), V (warp 10) ----------------
      const int kv = (warp == 10);
      const int NS = kv ? VS : KS;
      // decode reads each cached page once (evict first); Dual-Stream blocks
      // all re-read the memory stream's pages (keep them)
      const uint64_t pol = A.kv_reuse ? l2_evict_last_policy() : l2_evict_first_policy();
      const bf16* pool = static_cast<const bf16*>(A.pool);
      const bf16* win = static_cast<const bf16*>(A.kv_win);
      const size_t blockn = (size_t)kPageBlock * hd;
      constexpr int kPg = kPagesPerTile;
      if (!kv) tma_prefetch_desc(&mq);
      // a new segment's Q goes into buffer seg & 1 once the S MMAs of the
      // segment two back are done with it
      auto issue_q = [&](int sg, int b, int kvh, int rb) -> bool {
        const int qb = sg & 1;
        if (!wait(&q_empty[qb], ((uint32_t)(sg >> 1) & 1u) ^ 1u)) return false;
        uint8_t* qdst = base + qb * Ly.q_bytes;
        mbar_arrive_expect_tx(&q_full[qb], (uint32_t)(16 * R * 16));
#pragma unroll 1
        for (int c = 0; c < 16; ++c)
          tma_load_3d(qdst + c * Ly.Rpad * 16, &mq, &q_full[qb], 8 * c, kvh * G,
                      b * W + rb * TPB);
        s_issued[2] = sg + 1;
        return true;
      };
      // Cached K/V pages do not depend on the previous kernel (the QKV
      // projection): the first ring of prefix tiles is copied before
      // waiting for it; Q and the window tile (both its outputs) after.
      bool waited = false;
      int nq_def = 0, qdef_seg[kMaxStages], qdef_b[kMaxStages], qdef_h[kMaxStages],
          qdef_rb[kMaxStages];
      auto wait_prev = [&]() -> bool {
        pdl_wait();
        if (!kv) pdl_trigger();
        waited = true;
        for (int j = 0; j < nq_def; ++j)
          if (!issue_q(qdef_seg[j], qdef_b[j], qdef_h[j], qdef_rb[j])) return false;
        nq_def = 0;
        return true;
      };
      int seg = -1;
      int cst = 0;        // ring stage of tile i (i % NS, stepped)
      uint32_t cph = 0;   // and its phase ((i / NS) & 1)
      Cur cur = first;
      for (int i = 0; i < ntiles; ++i, advance(cur)) {
        const int b = cur.b, kvh = cur.kvh, t = cur.t;
        const bool window = t >= cur.P;
        if (!waited && (i == NS || window) && !wait_prev()) break;
        if (!kv && (i == 0 || t == 0)) {
          ++seg;
          if (waited) {
            if (!issue_q(seg, b, kvh, cur.rb)) break;
          } else {
            qdef_seg[nq_def] = seg;
            qdef_b[nq_def] = b;
            qdef_h[nq_def] = kvh;
            qdef_rb[nq_def] = cur.rb;
            ++nq_def;
          }
        }
        int pid[kPg];
#pragma unroll
        for (int pg = 0; pg < kPg; ++pg) {
          if (i < kPrefTiles) {
            pid[pg] = s_pages[i * kPg + pg];
          } else {
            const int t0 = t * kTile + pg * kPageBlock;
            int v = -1;
            if (!window && t0 < cur.L) {
              v = A.page_table[(size_t)b * A.pt_stride + t0 / kPageBlock];
              if (v < 0 || v >= A.num_pages) {
                set_err(A.err, WEDLM_DEV_BAD_PAGE);
                v = -1;
              }
            }
            pid[pg] = v;
          }
        }
        const int st = cst;
        const uint32_t ph = cph;
        if (++cst == NS) {
          cst = 0;
          cph ^= 1u;
        }
        uint64_t* full = kv ? &v_full[st] : &k_full[st];
        if (!wait(kv ? &v_empty[st] : &k_empty[st], ph ^ 1u)) break;
        uint8_t* dst = base + (kv ? Ly.off_v : Ly.off_k) + st * kKVBytes;
        if (window) {
          const int w = t - cur.P;
          const uint32_t bytes = (uint32_t)window_keys(w) * hd * 2;
          mbar_arrive_expect_tx(full, bytes);
          bulk_load(dst, win + ((((size_t)b * 2 + kv) * A.nkv + kvh) * A.Wp + (size_t)w * kTile) * hd,
                    bytes, full, pol);
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
      if (!waited) wait_prev();
    }
  } else if (warp == 9) {
    if (lane == 0) {
      // ---------------- S issuer ----------------
      const uint32_t qlbo = (uint32_t)Ly.Rpad * 16;  // next 8-dim group of Q
      const uint64_t dq0 = sdesc_noswz(smem_u32(base), qlbo, 128);
      const uint64_t dq1 = sdesc_noswz(smem_u32(base + Ly.q_bytes), qlbo, 128);
      const uint64_t dk0 = sdesc_noswz(smem_u32(base + Ly.off_k), 128, 2048);
      const uint64_t dq_step = (uint64_t)((2 * qlbo) >> 4);  // 16 dims, in 16-byte units
      int seg = -1;
      int kst = 0, sbi = 0;       // K stage (i % KS) and S buffer (i % 3), stepped
      uint32_t kph = 0, sph = 0;  // their phases
      Cur cs = first;
      for (int i = 0; i < ntiles; ++i, advance(cs)) {
        const int t = cs.t, T = cs.T;
        const bool seg_first = (i == 0 || t == 0), seg_last = (i == ntiles - 1 || t == T - 1);
        const int keys = t >= cs.P ? window_keys(t - cs.P) : kTile;
        if (seg_first) {
          ++seg;
          if (!wait(&q_full[seg & 1], (uint32_t)(seg >> 1) & 1u)) break;
          s_done[2] = seg + 1;
        }
        const int st = kst, sb = sbi;
        const uint32_t kp = kph, spp = sph;
        if (++kst == KS) {
          kst = 0;
          kph ^= 1u;
        }
        if (++sbi == kSBuf) {
          sbi = 0;
          sph ^= 1u;
        }
        if (!wait(&k_full[st], kp)) break;
        s_done[0] = i + 1;
        // S buffer sb is free once P V of tile i - 3 is done
        if (!wait(&s_free[sb], spp ^ 1u)) break;
        tc_fence_after();
        const uint64_t aq = (seg & 1) ? dq1 : dq0;
        const uint64_t bk = dk0 + (uint64_t)((st * kKVBytes) >> 4);
        const uint32_t idS = idesc_bf16_m128(keys);
        const uint32_t dS = tmem + kColS + (uint32_t)(sb * 128);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // 16 dims a step: two 8-dim groups
          tc_mma_f16(dS, aq + kk * dq_step, bk + (uint64_t)(kk * 16), idS, kk ? 1u : 0u);
        tc_commit(&s_full[sb]);
        tc_commit(&k_empty[st]);
        if (seg_last) tc_commit(&q_empty[seg & 1]);
      }
    }
  } else if (warp == 11) {
    if (lane == 0) {
      // ---------------- P V issuer ----------------
      const uint32_t idPV = idesc_pv();
      const uint64_t dv0 = sdesc_noswz(smem_u32(base + Ly.off_v), 2048, 128);
      int seg = -1;
      int vst = 0, pbi = 0;       // V stage (i % VS) and P buffer (i % 3), stepped
      uint32_t vph = 0, pph = 0;  // their phases
      Cur cp = first;
      for (int i = 0; i < ntiles; ++i, advance(cp)) {
        const int t = cp.t;
        const bool seg_first = (i == 0 || t == 0);
        const int st = vst, pb = pbi;
        const uint32_t vp = vph, pp = pph;
        if (++vst == VS) {
          vst = 0;
          vph ^= 1u;
        }
        if (++pbi == kSBuf) {
          pbi = 0;
          pph ^= 1u;
        }
        if (!wait(&v_full[st], vp)) break;
        s_done[1] = i + 1;
        if (!wait(&p_full[pb], pp)) break;
        if (seg_first) {
          // O is overwritten: the previous segment's O must have been read
          ++seg;
          if (seg > 0 && !wait(&o_free, (uint32_t)(seg - 1) & 1u)) break;
        }
        tc_fence_after();
        const uint64_t bv = dv0 + (uint64_t)((st * kKVBytes) >> 4);
        const uint32_t ap = tmem + kColS + (uint32_t)(pb * 128);
        const int steps = (t >= cp.P ? window_keys(t - cp.P) : kTile) / 16;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)  // 16 keys a step: 8 TMEM columns of P
          if (kk < steps)
            tc_mma_f16_ts(tmem + kColO, ap + (uint32_t)(kk * 8), bv + (uint64_t)(kk * 256),
                          idPV, (seg_first && kk == 0) ? 0u : 1u);
        tc_commit(&s_free[pb]);
        tc_commit(&v_empty[st]);
      }
    }
  } else {
    // ---------------- softmax warps ----------------
    pdl_wait();  // they write the outputs (and read nothing else of the previous kernel)
    const int q = warp & 3, h = warp >> 2;       // lane quadrant, key / dim half
    const int r = 32 * q + lane;                  // query row within the row block
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    const float sc = A.scale_log2;
    float m = -INFINITY, l = 0.f;
    auto pair_bar = [&]() {  // warps q and q+4
      asm volatile("bar.sync %0, 64;" ::"r"(1 + q) : "memory");
    };
    auto softmax_bar = [&]() {  // the 8 softmax warps
      asm volatile("bar.sync 5, 256;" ::: "memory");
    };
    Cur cur = first;
    for (int i = 0; i < ntiles; ++i, advance(cur)) {
      const int b = cur.b, kvh = cur.kvh, t = cur.t, T = cur.T, rb = cur.rb;
      const bool seg_first = (i == 0 || t == 0), seg_last = (i == ntiles - 1 || t == T - 1);
      if (seg_first) {
        m = -INFINITY;
        l = 0.f;
      }
      // rows of this row block: window rows rb*TPB .. min(W, (rb+1)*TPB) - 1
      const int rows_valid = (min(W, (rb + 1) * TPB) - rb * TPB) * G;
      const bool valid = r < rows_valid;
      const int p_row = rb * TPB + (valid ? r / G : 0);  // window row of this query row
      const bool window = t >= cur.P;
      const int L = cur.L;
      const int sb = i % kSBuf;
      const uint32_t sph = (uint32_t)(i / kSBuf) & 1u;  // phase of this tile on buffer sb
      wait(&s_full[sb], sph);
      tc_fence_after();
      float v[64];
      tmem_ld64(trow + kColS + (uint32_t)(sb * 128 + h * 64), v);
      // mask (only the partial last prefix tile and the window tile need
      // one), row max over both halves of the tile, scale applied once
      const int kbase = window ? (t - cur.P) * kTile : t * kTile;
      if (window || kbase + kTile > L) {
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const int kk = kbase + h * 64 + j;
          const bool ok = window ? (kk < W && kk <= p_row) : (kk < L);
          if (!ok) v[j] = -INFINITY;
        }
      }
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        mx[k] = fmaxf(fmaxf(v[8 * k], v[8 * k + 1]), fmaxf(v[8 * k + 2], v[8 * k + 3]));
        mx[k] = fmaxf(mx[k], fmaxf(fmaxf(v[8 * k + 4], v[8 * k + 5]),
                                   fmaxf(v[8 * k + 6], v[8 * k + 7])));
      }
      const float hmax =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sc;
      s_red[i & 1][h][r] = hmax;
      pair_bar();
      const float m_tile = fmaxf(hmax, s_red[i & 1][h ^ 1][r]);
      // both halves take the same decision for a row (same m_tile, same
      // history); the TMEM loads and stores below are warp-collective, so a
      // warp enters when any of its rows raises and the other rows scale by 1
      const bool raise = m_tile > m + kRescaleLog2;
      if (__any_sync(0xffffffffu, raise)) {
        const float alpha = !raise ? 1.f : (m == -INFINITY) ? 0.f : ex2_approx(m - m_tile);
        if (!seg_first) {
          // O holds this segment's earlier tiles: wait for the last P V
          // (tile i-1) and scale this thread's half row of O in TMEM
          wait(&s_free[(i - 1) % kSBuf], (uint32_t)((i - 1) / kSBuf) & 1u);
          tc_fence_after();
#pragma unroll
          for (int cb = 0; cb < 2; ++cb) {
            float o[32];
            uint32_t u[32];
            const uint32_t ta = trow + kColO + (uint32_t)(h * 64 + cb * 32);
            tmem_ld32(ta, o);
#pragma unroll
            for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(o[j] * alpha);
            tmem_st32(ta, u);
          }
          tmem_wait_st();
        }
        if (raise) {
          l *= alpha;
          m = m_tile;
        }
      }
      // p = 2^(s*scale - m); masked scores are -inf and give 0
      const float nm = (m == -INFINITY) ? 0.f : -m;
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t packed[32];
#pragma unroll
      for (int j = 0; j < 64; j += 2) {
        const float p0 = ex2_approx(fmaf(v[j], sc, nm));
        const float p1 = ex2_approx(fmaf(v[j + 1], sc, nm));
        ps[(j >> 1) & 3] += p0 + p1;
        const __nv_bfloat162 pk = __floats2bfloat162_rn(p0, p1);
        packed[j >> 1] = *reinterpret_cast<const uint32_t*>(&pk);
      }
      const float psum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
      // P over the first 64 columns of S: both halves have read their S
      // columns before the row-max exchange above
      tmem_st32(trow + kColS + (uint32_t)(sb * 128 + h * 32), packed);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
      l += psum;  // this half's share of the row sum
      if (seg_last) {
        // segment end: once this tile's P V is done, read O and write the
        // unnormalised partial
        wait(&s_free[sb], sph);
        tc_fence_after();
        float o[64];
        tmem_ld64(trow + kColO + (uint32_t)(h * 64), o);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&o_free);
        s_lsum[h][r] = l;
        pair_bar();
        const float lsum = l + s_lsum[h ^ 1][r];
        // the unit's segments: slots u + c for the blocks c from the owner
        // of its first tile to the owner of its last
        const int u = (b * A.nkv + kvh) * NRB + rb;
        const long long u0 = s_tstart[b] + (long long)kvh * head_tiles(cur.P) +
                             (long long)rb * cur.P + Ly.cwt[rb];
        const int c0 = last_le(s_begin, sp.G, u0), c1 = last_le(s_begin, sp.G, u0 + T - 1);
        if (c0 == c1) {
          // the whole unit is in this block: normalise and write the output
          if (valid) {
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            bf16* dst = static_cast<bf16*>(A.o) +
                        ((size_t)(b * W + p_row) * A.nq + kvh * G + r % G) * hd + h * 64;
#pragma unroll
            for (int j8 = 0; j8 < 8; ++j8) {
              uint32_t w4[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const __nv_bfloat162 t2 =
                    __floats2bfloat162_rn(o[8 * j8 + 2 * k] * inv, o[8 * j8 + 2 * k + 1] * inv);
                w4[k] = *reinterpret_cast<const uint32_t*>(&t2);
              }
              reinterpret_cast<uint4*>(dst)[j8] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
        } else {
          if (valid) {
            // partial O as [slot][half][dim/4][row] float4s: a warp's rows
            // are consecutive, so every store is one contiguous 512 bytes
            const size_t sid = (size_t)u + blockIdx.x, row = sid * R + r;
            float4* po = reinterpret_cast<float4*>(A.part_o) + (sid * 2 + h) * 16 * R + r;
#pragma unroll
            for (int d4 = 0; d4 < 16; ++d4)
              po[(size_t)d4 * R] =
                  make_float4(o[4 * d4], o[4 * d4 + 1], o[4 * d4 + 2], o[4 * d4 + 3]);
            if (h == 0) {
              A.part_ml[row * 2 + 0] = m;
              A.part_ml[row * 2 + 1] = lsum;
            }
          }
          __threadfence();
          softmax_bar();
          if (threadIdx.x == 0) s_merge = (atomicAdd(&A.unit_cnt[u], 1) == c1 - c0);
          softmax_bar();
          if (s_merge) {
            // every segment of the unit is written: merge them in slot
            // order (the same sum whichever block merges) and reset the
            // count for the next launch.  The 8 softmax warps split the
            // unit into (32 rows, 32 dims) tasks; the (max, sum) and the
            // partial O of two segments are loaded in one round trip, and
            // the running result is rescaled when a pair raises the max.
            __threadfence();
            const int ns = c1 - c0 + 1;
            const size_t s0 = (size_t)u + c0;
            const int nrg = (R + 31) / 32;
            for (int task = warp; task < nrg * 4; task += 8) {
              const int mr = 32 * (task % nrg) + lane, qd = task / nrg;
              if (mr >= rows_valid) continue;
              const int hh = qd >> 1, d40 = (qd & 1) * 8;
              float M = -INFINITY, ls = 0.f, acc[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) acc[j] = 0.f;
              for (int sb0 = 0; sb0 < ns; sb0 += 2) {
                float mk[2], lk[2];
                float4 t4[2][8];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                  mk[k] = -INFINITY;
                  lk[k] = 0.f;
                  if (sb0 + k < ns) {
                    const size_t sid = s0 + sb0 + k;
                    mk[k] = __ldcg(A.part_ml + (sid * R + mr) * 2);
                    lk[k] = __ldcg(A.part_ml + (sid * R + mr) * 2 + 1);
                    const float4* src = reinterpret_cast<const float4*>(A.part_o) +
                                        ((sid * 2 + hh) * 16 + d40) * R + mr;
#pragma unroll
                    for (int j = 0; j < 8; ++j) t4[k][j] = __ldcg(src + (size_t)j * R);
                  } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) t4[k][j] = make_float4(0.f, 0.f, 0.f, 0.f);
                  }
                }
                const float Mn = fmaxf(M, fmaxf(mk[0], mk[1]));
                if (Mn == -INFINITY) continue;  // no key seen yet for this row
                if (Mn != M) {
                  const float a = exp2f(M - Mn);  // 0 while M is -inf
                  ls *= a;
#pragma unroll
                  for (int j = 0; j < 32; ++j) acc[j] *= a;
                  M = Mn;
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                  if (mk[k] == -INFINITY) continue;
                  const float wgt = exp2f(mk[k] - M);
                  ls += lk[k] * wgt;
#pragma unroll
                  for (int j = 0; j < 8; ++j) {
                    acc[4 * j] += t4[k][j].x * wgt; acc[4 * j + 1] += t4[k][j].y * wgt;
                    acc[4 * j + 2] += t4[k][j].z * wgt; acc[4 * j + 3] += t4[k][j].w * wgt;
                  }
                }
              }
              const float inv = ls > 0.f ? 1.f / ls : 0.f;
              bf16* dst = static_cast<bf16*>(A.o) +
                          ((size_t)(b * W + rb * TPB + mr / G) * A.nq + kvh * G + mr % G) * hd +
                          qd * 32;
#pragma unroll
              for (int j8 = 0; j8 < 4; ++j8) {
                uint32_t w4[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const __nv_bfloat162 t2 = __floats2bfloat162_rn(acc[8 * j8 + 2 * k] * inv,
                                                                  acc[8 * j8 + 2 * k + 1] * inv);
                  w4[k] = *reinterpret_cast<const uint32_t*>(&t2);
                }
                reinterpret_cast<uint4*>(dst)[j8] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
              }
            }
            if (threadIdx.x == 0) A.unit_cnt[u] = 0;
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
    for (int kv = 0; kv < 2; ++kv) {
      const int NS = kv ? VS : KS;
      for (int i = s_done[kv]; i < s_issued[kv]; ++i)
        mbar_wait(kv ? &v_full[i % NS] : &k_full[i % NS], (uint32_t)(i / NS) & 1u, A.err);
    }
    for (int s = s_done[2]; s < s_issued[2]; ++s)
      mbar_wait(&q_full[s & 1], (uint32_t)(s >> 1) & 1u, A.err);
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 attn_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}
}  // namespace

// Row blocks of a launch: all G*W rows in one block when they fit the MMA's
// 128 rows, else blocks of 128/G window rows (G must divide 128).  False for
// shapes the kernel does not take.
bool attention_tc_plan(const AttnArgs& A, AttnLayout* Ly) {
  if (A.hd != 128 || A.nkv < 1 || A.nq % A.nkv || A.W < 1 ||
      A.Wp != (A.W + kPageBlock - 1) / kPageBlock * kPageBlock)
    return false;
  const int G = A.nq / A.nkv;
  if (G > 128) return false;
  if (G * A.W <= 128) {
    Ly->TPB = A.W;
  } else {
    if (128 % G) return false;
    Ly->TPB = 128 / G;
  }
  Ly->NRB = (A.W + Ly->TPB - 1) / Ly->TPB;
  if (Ly->NRB > kMaxRB) return false;
  Ly->R = G * Ly->TPB;
  Ly->Rpad = (Ly->R + 7) / 8 * 8;
  Ly->cwt[0] = 0;
  for (int rb = 0; rb < Ly->NRB; ++rb) {
    const int last = std::min(A.W, (rb + 1) * Ly->TPB) - 1;  // last window row of the block
    Ly->wt[rb] = last / kTile + 1;
    Ly->cwt[rb + 1] = Ly->cwt[rb] + Ly->wt[rb];
  }
  return true;
}

int attention_tc_row_blocks(int nq, int nkv, int W, int* rows_per_block) {
  AttnArgs A{};
  A.hd = 128; A.nq = nq; A.nkv = nkv; A.W = W;
  A.Wp = (W + kPageBlock - 1) / kPageBlock * kPageBlock;
  AttnLayout Ly;
  if (!attention_tc_plan(A, &Ly)) return 0;
  if (rows_per_block) *rows_per_block = Ly.R;
  return Ly.NRB;
}

cudaError_t launch_attention_tc(const AttnArgs& A, const void* zero_page, int grid,
                                cudaStream_t st, bool pdl) {
  AttnLayout Ly;
  if (!attention_tc_plan(A, &Ly) || A.B > kMaxB || A.min_tiles < 1 || !A.unit_cnt || grid < 1 ||
      (reinterpret_cast<uintptr_t>(A.q) & 15))
    return cudaErrorInvalidValue;
  const int G = A.nq / A.nkv;
  Ly.q_bytes = 256u * (uint32_t)Ly.Rpad;
  const int stages = (int)((kDynBytes - 2 * Ly.q_bytes) / kKVBytes);
  Ly.KS = stages >= 6 ? 3 : 2;
  Ly.VS = std::min(kMaxStages, stages - Ly.KS);
  if (Ly.VS < 2) return cudaErrorInvalidValue;
  Ly.off_k = 2 * Ly.q_bytes;
  Ly.off_v = Ly.off_k + (uint32_t)Ly.KS * kKVBytes;
  // q as a 3-D tensor {dim, head, token}; a box {8, G, W} is one 8-dim
  // group of the G*W rows of one unit
  auto enc = attn_encoder();
  if (!enc) return cudaErrorInvalidValue;
  CUtensorMap mq;
  cuuint64_t dims[3] = {128, (cuuint64_t)A.nq, (cuuint64_t)A.B * A.W};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)A.nq * 128 * 2};
  cuuint32_t box[3] = {8, (cuuint32_t)G, (cuuint32_t)Ly.TPB};
  cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(A.q), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const cudaError_t ae = ensure_dyn_smem((const void*)attn_tc_kernel, (int)kDynBytes + 1024);
  if (ae != cudaSuccess) return ae;
  const uint32_t smem = Ly.off_v + (uint32_t)Ly.VS * kKVBytes + 1024;
  if (!pdl) {
    attn_tc_kernel<<<std::min(grid, kMaxGrid), kThreads, smem, st>>>(mq, A, Ly, zero_page);
    return cudaGetLastError();
  }
  return launch_pdl(attn_tc_kernel, dim3(std::min(grid, kMaxGrid)), dim3(kThreads), smem, st, mq,
                    A, Ly, zero_page);
}

}  // namespace wedlm
