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
    // x[m][n] += acc  (pre-norm residual after O-proj / down-proj)
    T* x = static_cast<T*>(e.x);
    for (int idx = tid; idx < mc * 128; idx += nth) {
      const int r = idx >> 7, f = idx & 127;
      const size_t o = (size_t)(m0 + r) * N + tile * 128 + f;
      x[o] = from_f<T>(to_f(x[o]) + sacc[r * 128 + f]);
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
    for (int pr = warp; pr < npairs; pr += nwarps) {
      const int r = pr / hpt, lh = pr % hpt, m = m0 + r;
      const int gh = tile * hpt + lh;
      const int kind = gh < e.nq ? 0 : (gh < e.nq + e.nkv ? 1 : 2);
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (i < per) v[i] = sacc[r * 128 + lh * hd + lane + 32 * i];
      if (kind < 2) {
        if (e.qk_norm) {
          float ss = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < per) ss = fmaf(v[i], v[i], ss);
          ss = warp_sum(ss);
          const float rs = rsqrtf(ss / (float)hd + e.eps);
          const T* g = static_cast<const T*>(kind == 0 ? e.q_norm : e.k_norm);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < per) v[i] = v[i] * rs * to_f(g[lane + 32 * i]);
        }
        const float* cr = e.cosb + (size_t)m * (hd / 2);
        const float* sr = e.sinb + (size_t)m * (hd / 2);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (i < halfp) {
            const int j = lane + 32 * i;
            const float c = cr[j], s = sr[j];
            const float a = v[i], b = v[i + halfp];
            v[i] = a * c - b * s;
            v[i + halfp] = b * c + a * s;
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
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (i < per) blk[tile_off(p, lane + 32 * i, hd)] = from_f<T>(v[i]);
      }
    }
  } else {  // EPI_LMHEAD: streaming softmax record of this vocab tile
    for (int r = warp; r < mc; r += nwarps) {
      const int m = m0 + r;
      const int pt = e.plant ? e.plant[m] : -1;
      float z[4];
      float mx = -INFINITY;
      int am = INT_MAX;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int f = lane + 32 * i, v = tile * 128 + f;
        float zz = sacc[r * 128 + f];
        if (v == pt) zz += e.plant_bias;
        if (v >= e.vocab || v == e.mask_id) zz = -INFINITY;
        if (e.logits && v < e.vocab) e.logits[(size_t)m * e.vocab + v] = zz;
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

}  // namespace wedlm
