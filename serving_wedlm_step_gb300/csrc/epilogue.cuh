// Fused epilogues of the weight-streaming GEMM.  Every mainloop ends with an
// fp32 tile staged in shared memory as sacc[r][f] (r = activation row in
// the chunk, f = 0..127 output feature inside the 128-row weight tile); the
// whole block then runs one of these.
#pragma once

#include <float.h>
#include <limits.h>

#include "internal.h"

namespace wedlm {

template <typename T>
__device__ void run_epilogue(const GemmEpi& e, const float* sacc, int m0,
                             int mc, int tile, int N, int M) {
  const int tid = threadIdx.x, nth = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nth >> 5;
  if (e.mode == EPI_RESID) {
    // x[m][n] += acc  (pre-norm residual after O-proj / down-proj), 16-byte
    // vectors, several loads in flight per thread
    constexpr int VN = 16 / sizeof(T);
    T* x = static_cast<T*>(e.x);
    const int nvec = mc * (128 / VN);
#pragma unroll 4
    for (int idx = tid; idx < nvec; idx += nth) {
      const int r = idx / (128 / VN), f = (idx % (128 / VN)) * VN;
      T* p = x + (size_t)(m0 + r) * N + tile * 128 + f;
      Vec16<T> v = ld16(p);
#pragma unroll
      for (int k = 0; k < VN; ++k) v.set(k, v.get(k) + sacc[r * 128 + f + k]);
      st16(p, v);
    }
  } else if (e.mode == EPI_SWIGLU) {
    // rows 0..63: gate features 64t..64t+63; rows 64..127: up, same features
    T* a = static_cast<T*>(e.act);
    const int F = N / 2;
    for (int idx = tid; idx < mc * 64; idx += nth) {
      const int r = idx >> 6, f = idx & 63;
      const float g = sacc[r * 128 + f], u = sacc[r * 128 + 64 + f];
      const float silu = g / (1.0f + expf(-g));
      a[(size_t)(m0 + r) * F + tile * 64 + f] = from_f<T>(silu * u);
    }
  } else if (e.mode == EPI_QKV) {
    // per (row, head): optional QK-RMSNorm, rotate-half RoPE at the row's
    // logical position, store q (row-major) or window K/V (page tile layout)
    const int hd = e.hd, hpt = 128 / hd, per = hd / 32, halfp = per / 2;
    const int npairs = mc * hpt;
    float qn[4], kn[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qn[i] = (e.qk_norm && i < per) ? to_f(static_cast<const T*>(e.q_norm)[lane + 32 * i]) : 1.f;
      kn[i] = (e.qk_norm && i < per) ? to_f(static_cast<const T*>(e.k_norm)[lane + 32 * i]) : 1.f;
    }
    constexpr int PB = 4;  // pairs per batch: their table loads overlap
    for (int pb = warp * PB; pb < npairs; pb += nwarps * PB) {
      float cs[PB][2], sn[PB][2];
#pragma unroll
      for (int u = 0; u < PB; ++u) {
        const int m = m0 + min(pb + u, npairs - 1) / hpt;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int j = min(lane + 32 * i, hd / 2 - 1);
          cs[u][i] = e.cosb[(size_t)m * (hd / 2) + j];
          sn[u][i] = e.sinb[(size_t)m * (hd / 2) + j];
        }
      }
#pragma unroll
      for (int u = 0; u < PB; ++u) {
        const int pr = pb + u;
        if (pr >= npairs) break;
        const int r = pr / hpt, lh = pr % hpt, m = m0 + r;
        const int gh = tile * hpt + lh;
        const int kind = gh < e.nq ? 0 : (gh < e.nq + e.nkv ? 1 : 2);
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          v[i] = (i < per) ? sacc[r * 128 + lh * hd + lane + 32 * i] : 0.f;
        if (kind < 2) {
          if (e.qk_norm) {
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) ss = fmaf(v[i], v[i], ss);
            ss = warp_sum(ss);
            const float rs = rsqrtf(ss / (float)hd + e.eps);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = v[i] * rs * (kind == 0 ? qn[i] : kn[i]);
          }
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (i < halfp) {
              const float c = cs[u][i], sv = sn[u][i];
              const float a = v[i], b = v[i + halfp];
              v[i] = a * c - b * sv;
              v[i + halfp] = b * c + a * sv;
            }
          }
        }
        if (kind == 0) {
          T* q = static_cast<T*>(e.q_out) + ((size_t)m * e.nq + gh) * hd;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < per) q[lane + 32 * i] = from_f<T>(v[i]);
        } else {
          const int b = m / e.W, p = m % e.W;
          const int kvh = gh - e.nq - (kind == 2 ? e.nkv : 0);
          T* blk = static_cast<T*>(e.kv_win) +
                   (((size_t)b * 2 + (kind - 1)) * e.nkv + kvh) * e.Wp * hd;
          // a committed row (physical rows 0..c-1) also goes to its page
          const bool commit = e.commit_n && p < e.commit_n[b];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < per) {
              blk[tile_off(p, lane + 32 * i, hd)] = from_f<T>(v[i]);
              if (commit) {
                T* c = commit_dst<T>(e, b, e.commit_base[b] + p, kind - 1, kvh, lane + 32 * i);
                if (c) *c = from_f<T>(v[i]);
              }
            }
        }
      }
    }
  } else {  // EPI_LMHEAD: streaming softmax record of this vocab tile
    // lane i holds the planted token of row warp + i*nwarps (rows per warp
    // <= 32 since mc <= 128 and nwarps >= 4)
    const int rl = warp + lane * nwarps;
    const int my_plant = (e.plant && rl < mc) ? e.plant[m0 + rl] : -1;
    for (int r = warp, it = 0; r < mc; r += nwarps, ++it) {
      const int m = m0 + r;
      const int pt = __shfl_sync(0xffffffffu, my_plant, it);
      float z[4];
      float mx = -INFINITY;
      int am = INT_MAX;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int f = lane + 32 * i, v = tile * 128 + f;
        float zz = sacc[r * 128 + f];
        if (v == pt) zz += e.plant_bias;
        if (v >= e.vocab || v == e.mask_id) zz = -INFINITY;
        if (e.logits && v < e.vocab)
          e.logits[(size_t)(e.row_src ? e.row_src[m] : m) * e.vocab + v] = zz;
        z[i] = zz;
        if (zz > mx) { mx = zz; am = v; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, mx, o);
        const int oa = __shfl_xor_sync(0xffffffffu, am, o);
        if (om > mx || (om == mx && oa < am)) { mx = om; am = oa; }
      }
      float s = 0.f, u = 0.f;
      if (mx > -INFINITY) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (z[i] > -INFINITY) {
            const float d = z[i] - mx;
            const float ex = expf(d);
            s += ex;
            u = fmaf(d, ex, u);
          }
        }
      }
      s = warp_sum(s);
      u = warp_sum(u);
      if (lane == 0) {
        SoftmaxPart pp;
        pp.m = mx; pp.a = am; pp.s = s; pp.u = u;
        e.part[(size_t)tile * M + m] = pp;
      }
    }
  }
}

// A chunk of the tile (rows m0..m0+mc-1, all 128 features) sits in sacc:
// run the epilogue (one split) or store the fp32 partial of this split.
template <typename T>
__device__ void stage_chunk(const GemmProblem& P, const float* sacc, int m0, int mc,
                            int tile, int split) {
  if (P.splits == 1) {
    run_epilogue<T>(P.epi, sacc, m0, mc, tile, P.N, P.M);
    return;
  }
  float* dst = P.partial + (size_t)split * P.M * P.N;
  for (int idx = threadIdx.x; idx < mc * 32; idx += blockDim.x) {
    const int r = idx >> 5, f = (idx & 31) * 4;
    if (tile * 128 + f < P.N)
      __stcg(reinterpret_cast<float4*>(dst + (size_t)(m0 + r) * P.N + tile * 128 + f),
             *reinterpret_cast<const float4*>(sacc + r * 128 + f));
  }
}

// Split-K: the last block to finish a tile sums the partials in split order
// (deterministic) and runs the epilogue; it then re-arms the tile counter.
template <typename T>
__device__ void splitk_finish(const GemmProblem& P, float* sacc, int tile) {
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&P.counters[tile], 1) == P.splits - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int m_live = P.m_count ? min(P.M, max(0, *P.m_count)) : P.M;
  for (int m0 = 0; m0 < m_live; m0 += 128) {
    const int mc = min(128, m_live - m0);
    // N is a multiple of 4 and the tile start a multiple of 128, so every
    // float4 lies entirely inside or outside the matrix
#pragma unroll 4
    for (int idx = threadIdx.x; idx < mc * 32; idx += blockDim.x) {
      const int r = idx >> 5, f = (idx & 31) * 4;
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      if (tile * 128 + f < P.N) {
        const float* src = P.partial + (size_t)(m0 + r) * P.N + tile * 128 + f;
        for (int sp = 0; sp < P.splits; ++sp) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(src + (size_t)sp * P.M * P.N));
          s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
        }
      }
      *reinterpret_cast<float4*>(sacc + r * 128 + f) = s;
    }
    __syncthreads();
    run_epilogue<T>(P.epi, sacc, m0, mc, tile, P.N, P.M);
    __syncthreads();
  }
  if (threadIdx.x == 0) P.counters[tile] = 0;
}

}  // namespace wedlm
