// Device helpers shared by the libwedlm kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/wedlm.h"

namespace wedlm {

using bf16 = __nv_bfloat16;

constexpr int kPageBlock = 16;   // tokens per KV page
constexpr int kMaxLayers = 64;
constexpr int kMaxWindow = 64;
constexpr int kMaxRows = 512;    // B * W

// ---- element conversions --------------------------------------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) {
  return __float2bfloat16_rn(x);
}

// ---- 16-byte vector of elements ---------------------------------------------
template <typename T> struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
  uint4 raw;
  __device__ __forceinline__ float get(int i) const {
    const T* p = reinterpret_cast<const T*>(&raw);
    return to_f(p[i]);
  }
  __device__ __forceinline__ void set(int i, float v) {
    T* p = reinterpret_cast<T*>(&raw);
    p[i] = from_f<T>(v);
  }
};

template <typename T>
__device__ __forceinline__ Vec16<T> ld16(const T* p) {
  Vec16<T> v;
  v.raw = *reinterpret_cast<const uint4*>(p);
  return v;
}
template <typename T>
__device__ __forceinline__ void st16(T* p, const Vec16<T>& v) {
  *reinterpret_cast<uint4*>(p) = v.raw;
}

// ---- reductions --------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Offset of (token t, dim d) inside one (page, K|V, head) block: 8x8 tiles,
// token-group-major.  Same formula for the window K/V scratch blocks.
__device__ __forceinline__ int tile_off(int t, int d, int hd) {
  return (((t >> 3) * (hd >> 3) + (d >> 3)) << 6) + ((t & 7) << 3) + (d & 7);
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may
// start while the previous kernel on the stream is still running: before
// reading anything that kernel wrote, and before writing anything, it calls
// pdl_wait (which returns once the previous kernel has completed and its
// memory is visible), then pdl_trigger lets the next kernel start early in
// turn.  Work on data no kernel of the step writes (weights, cached KV pages,
// page tables) may go before pdl_wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void set_err(int* err, int bits) {
  if (err) atomicOr(err, bits);
}

// streaming softmax record of one vocab tile for one row
struct SoftmaxPart {
  float m;     // max logit in the tile
  int32_t a;   // its token id (lowest on ties)
  float s;     // sum exp(z - m)
  float u;     // sum (z - m) exp(z - m)
};

}  // namespace wedlm
