// Row-per-thread epilogues of the tensor-core GEMM.
//
// The accumulator tile lives in TMEM with one activation row per lane and
// the tile's output features along the columns, so each thread owns one row
// and every epilogue (residual add, SwiGLU, per-head QK-RMSNorm + RoPE,
// streaming softmax over the vocabulary) runs inside a thread on 32-column
// chunks read with tcgen05.ld.  With split-K, the same epilogue reads the
// fp32 partial sums (summed in split order) instead of TMEM.
#pragma once

#include <limits.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace wedlm {

// where one thread's accumulator row comes from
enum AccFrom { ACC_PARTIAL = 0, ACC_TMEM = 1 };
struct AccRow {
  int from;             // AccFrom (warp-uniform)
  uint32_t taddr;       // ACC_TMEM: TMEM address of column 0 (this warp's lanes)
  const float* part;    // ACC_PARTIAL: partial[0][m][tile*ntile] (global)
  size_t split_stride;  // floats from one split's row to the next split's
  int splits;
  int col0;             // tile * ntile (first global column of the tile)
  int N;                // global columns
  bool valid;           // m < M
};

// 32 consecutive accumulator columns c..c+31 of this thread's row.  The
// TMEM path is warp-collective: every lane calls it.  With split-K the
// splits' values are added in split order, starting from zero.
__device__ __forceinline__ void acc_chunk(const AccRow& a, int c, float (&v)[32]) {
  if (a.from == ACC_TMEM) {
    tmem_ld32(a.taddr + (uint32_t)c, v);
    return;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = 0.f;
  if (!a.valid) return;
  for (int sp = 0; sp < a.splits; ++sp) {
    const float* p = a.part + (size_t)sp * a.split_stride + c;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (a.col0 + c + 4 * i < a.N) {  // N % 4 == 0: a float4 is all in or all out
        const float4 t = __ldcg(reinterpret_cast<const float4*>(p) + i);
        v[4 * i] += t.x; v[4 * i + 1] += t.y; v[4 * i + 2] += t.z; v[4 * i + 3] += t.w;
      }
    }
  }
}

__device__ __forceinline__ void st_bf16x32(bf16* dst, const float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    Vec16<bf16> o;
#pragma unroll
    for (int k = 0; k < 8; ++k) o.set(k, v[8 * i + k]);
    st16(dst + 8 * i, o);
  }
}

// SiLU x / (1 + e^-x) without branches: __expf and __fdividef (a few ulp,
// far below the bf16 rounding of the result; for x below about -87 the
// denominator overflows and the result is 0, the limit)
__device__ __forceinline__ float silu_fast(float x) {
  return __fdividef(x, 1.0f + __expf(-x));
}

// Epilogue items of a tile: independent pieces of one row's work.
// RESID: 32-column chunks; SWIGLU: 32-feature chunks (gate + up columns);
// QKV: heads; LMHEAD: the whole tile (one item).
__host__ __device__ inline int tc_epi_items(const GemmProblem& P, int ntile) {
  switch (P.epi.mode) {
    case EPI_RESID: return ntile / 32;
    case EPI_SWIGLU: return ntile / 64;
    case EPI_QKV: return ntile / P.epi.hd;
    default: return 1;
  }
}

// Run the epilogue items [i0, i1) of one row of a tile (thread = row m).
__device__ void tc_epilogue_rows(const GemmProblem& P, const AccRow& a, int m, int tile,
                                 int ntile, int i0, int i1) {
  const GemmEpi& e = P.epi;
  if (e.mode == EPI_RESID) {
    bf16* x = static_cast<bf16*>(e.x) + (size_t)m * P.N + tile * ntile;
    for (int c = 32 * i0; c < 32 * i1; c += 32) {
      float v[32];
      acc_chunk(a, c, v);
      if (!a.valid) continue;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        Vec16<bf16> r = ld16(x + c + 8 * i);
#pragma unroll
        for (int k = 0; k < 8; ++k) r.set(k, r.get(k) + v[8 * i + k]);
        st16(x + c + 8 * i, r);
      }
    }
  } else if (e.mode == EPI_SWIGLU) {
    // columns [0, ntile/2): gate; [ntile/2, ntile): up, same features
    const int half = ntile / 2, F = P.N / 2;
    bf16* out = static_cast<bf16*>(e.act) + (size_t)m * F + tile * half;
    for (int c = 32 * i0; c < 32 * i1; c += 32) {
      float g[32], u[32];
      acc_chunk(a, c, g);
      acc_chunk(a, half + c, u);
#pragma unroll
      for (int j = 0; j < 32; ++j) g[j] = silu_fast(g[j]) * u[j];
      if (a.valid) st_bf16x32(out + c, g);
    }
  } else if (e.mode == EPI_QKV) {
    // per head: pass 1 sums squares (QK-RMSNorm), pass 2 rotates the chunk
    // pairs (d, d + hd/2) and stores; at most 64 values live per thread
    const int hd = e.hd, heads = ntile / hd, hh = hd / 2;
    const int b = m / e.W, p = m % e.W;
    for (int lh = i0; lh < i1 && lh < heads; ++lh) {
      const int gh = (tile * ntile) / hd + lh;
      const int kind = gh < e.nq ? 0 : (gh < e.nq + e.nkv ? 1 : 2);
      float rs = 1.f;
      if (kind < 2 && e.qk_norm) {
        float ss = 0.f;
        for (int c = 0; c < hd; c += 32) {
          float v[32];
          acc_chunk(a, lh * hd + c, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) ss = fmaf(v[j], v[j], ss);
        }
        rs = rsqrtf(ss / (float)hd + e.eps);
      }
      const bf16* gw = static_cast<const bf16*>(kind == 0 ? e.q_norm : e.k_norm);
      bf16* dst;
      const int kvh = kind == 0 ? 0 : gh - e.nq - (kind == 2 ? e.nkv : 0);
      // committed rows (physical rows 0..c-1) also go to their page
      const bool commit = kind > 0 && a.valid && e.commit_n && p < e.commit_n[b];
      const int t_commit = commit ? e.commit_base[b] + p : 0;
      if (kind == 0) {
        dst = static_cast<bf16*>(e.q_out) + ((size_t)m * e.nq + gh) * hd;
      } else {
        dst = static_cast<bf16*>(e.kv_win) +
              (((size_t)b * 2 + (kind - 1)) * e.nkv + kvh) * e.Wp * hd;
      }
      for (int c = 0; c < hh; c += 32) {
        float x1[32], x2[32];
        acc_chunk(a, lh * hd + c, x1);
        acc_chunk(a, lh * hd + hh + c, x2);
        if (!a.valid) continue;
        if (kind < 2) {
          if (e.qk_norm) {
#pragma unroll
            for (int j8 = 0; j8 < 4; ++j8) {
              const Vec16<bf16> g1 = ld16(gw + c + 8 * j8), g2 = ld16(gw + hh + c + 8 * j8);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                x1[8 * j8 + k] = x1[8 * j8 + k] * rs * g1.get(k);
                x2[8 * j8 + k] = x2[8 * j8 + k] * rs * g2.get(k);
              }
            }
          }
          const float4* c4 = reinterpret_cast<const float4*>(e.cosb + (size_t)m * hh + c);
          const float4* s4 = reinterpret_cast<const float4*>(e.sinb + (size_t)m * hh + c);
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const float4 cc = c4[i4], sv = s4[i4];
            const float cs[4] = {cc.x, cc.y, cc.z, cc.w}, sn[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int j = 4 * i4 + k;
              const float a1 = x1[j], a2 = x2[j];
              x1[j] = a1 * cs[k] - a2 * sn[k];
              x2[j] = a2 * cs[k] + a1 * sn[k];
            }
          }
        }
        if (kind == 0) {
          st_bf16x32(dst + c, x1);
          st_bf16x32(dst + hh + c, x2);
        } else {
#pragma unroll
          for (int j8 = 0; j8 < 4; ++j8) {
            Vec16<bf16> o1, o2;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              o1.set(k, x1[8 * j8 + k]);
              o2.set(k, x2[8 * j8 + k]);
            }
            st16(dst + tile_off(p, c + 8 * j8, hd), o1);
            st16(dst + tile_off(p, hh + c + 8 * j8, hd), o2);
            if (commit) {
              bf16* c1 = commit_dst<bf16>(e, b, t_commit, kind - 1, kvh, c + 8 * j8);
              bf16* c2 = commit_dst<bf16>(e, b, t_commit, kind - 1, kvh, hh + c + 8 * j8);
              if (c1) st16(c1, o1);
              if (c2) st16(c2, o2);
            }
          }
        }
      }
    }
  } else {  // EPI_LMHEAD: streaming softmax record of this row over the tile
    const int pt = (e.plant && a.valid) ? e.plant[m] : -1;
    float mx = -INFINITY, s = 0.f, u = 0.f;
    int am = INT_MAX;
    for (int c = 0; c < ntile; c += 32) {
      float v[32];
      acc_chunk(a, c, v);
      float cm = -INFINITY;
      int ca = INT_MAX;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int f = tile * ntile + c + j;
        float z = v[j];
        if (f == pt) z += e.plant_bias;
        if (f >= e.vocab || f == e.mask_id) z = -INFINITY;
        v[j] = z;
        if (z > cm) { cm = z; ca = f; }
      }
      if (e.logits && a.valid && tile * ntile + c < e.vocab) {
        const int lrow = e.row_src ? e.row_src[m] : m;
        float* lg = e.logits + (size_t)lrow * e.vocab + tile * ntile + c;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (tile * ntile + c + 4 * i < e.vocab)
            reinterpret_cast<float4*>(lg)[i] =
                make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
      if (cm > mx) {  // strict: equal maxima keep the lower id of an earlier chunk
        if (mx > -INFINITY) {
          const float d = mx - cm, ex = expf(d);
          u = ex * (u + d * s);
          s *= ex;
        }
        mx = cm;
        am = ca;
      }
      if (mx > -INFINITY) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (v[j] > -INFINITY) {
            const float d = v[j] - mx, ex = expf(d);
            s += ex;
            u = fmaf(d, ex, u);
          }
        }
      }
    }
    if (a.valid) {
      SoftmaxPart pp;
      pp.m = mx; pp.a = am; pp.s = s; pp.u = u;
      e.part[(size_t)tile * P.M + m] = pp;
    }
  }
}

}  // namespace wedlm
