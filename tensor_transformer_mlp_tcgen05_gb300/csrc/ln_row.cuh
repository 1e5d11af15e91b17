// One LayerNorm row by one warp, bf16 in and out, with the row held in
// registers (pre-LN placement: Megatron-LM explainer, section "Fixing BERT:
// reordering layer normalisation for scaling").  The stand-alone LayerNorm
// forward kernel and the GEMM's fused LayerNorm prologue both call it, so the
// two paths produce the same bits.
#pragma once
#include "common.cuh"

namespace tpmlp {
namespace lnrow {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void unpack8(const uint4 u, float (&v)[8]) {
  unpack_bf16x2(u.x, v[0], v[1]);
  unpack_bf16x2(u.y, v[2], v[3]);
  unpack_bf16x2(u.z, v[4], v[5]);
  unpack_bf16x2(u.w, v[6], v[7]);
}

// Eight fp32 values: through the read-only data path (global memory), or
// by generic loads (parameters staged in shared memory).
template <bool GLOBAL>
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  float4 a, b;
  if constexpr (GLOBAL) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p + 4));
  } else {
    a = reinterpret_cast<const float4*>(p)[0];
    b = reinterpret_cast<const float4*>(p)[1];
  }
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Keeps the compiler from carrying unpacked copies of the row from one pass
// to the next (the raw vectors are all that stays live between passes).
template <int VMAX>
__device__ __forceinline__ void opaque(uint4 (&raw)[VMAX]) {
#pragma unroll
  for (int j = 0; j < VMAX; ++j)
    asm volatile("" : "+r"(raw[j].x), "+r"(raw[j].y), "+r"(raw[j].z),
                 "+r"(raw[j].w));
}

// Loads lane l's 16-byte vectors l, l + 32, ... of the row x[0, 256 vpl)
// (vpl <= VMAX) at once: one DRAM round trip per row.
template <int VMAX>
__device__ __forceinline__ void load_row(const __nv_bfloat16* __restrict__ x,
                                         int vpl, int lane,
                                         uint4 (&raw)[VMAX]) {
  const uint4* xr = reinterpret_cast<const uint4*>(x);
#pragma unroll
  for (int j = 0; j < VMAX; ++j)
    raw[j] = j < vpl ? xr[lane + 32 * j] : make_uint4(0u, 0u, 0u, 0u);
}

// Normalises a row loaded by load_row into xn, h = 256 vpl: the mean, then
// the mean of the squared deviations about it (biased variance, two passes
// over the registers), each summed per lane in vector order and then by
// butterfly, all in fp32; xn = (x - mean) * rstd * gamma + beta rounded to
// bf16, rstd = 1 / sqrt(var + eps).  Returns mean and rstd (every lane).
// The arithmetic depends on vpl only, not on VMAX or on where gamma and
// beta are read from (GB_GLOBAL: global memory, else staged in shared
// memory by the caller).
template <int VMAX, bool GB_GLOBAL = true>
__device__ __forceinline__ void norm_row(uint4 (&raw)[VMAX],
                                         const float* __restrict__ gamma,
                                         const float* __restrict__ beta,
                                         __nv_bfloat16* __restrict__ xn,
                                         int vpl, int h, float eps, int lane,
                                         float& mu_out, float& rs_out) {
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < VMAX; ++j) {
    if (j < vpl) {
      float v[8];
      unpack8(raw[j], v);
#pragma unroll
      for (int k = 0; k < 8; ++k) s += v[k];
    }
  }
  const float inv_h = 1.0f / static_cast<float>(h);
  const float mu = warp_sum(s) * inv_h;
  opaque(raw);
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < VMAX; ++j) {
    if (j < vpl) {
      float v[8];
      unpack8(raw[j], v);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float d = v[k] - mu;
        ss += d * d;
      }
    }
  }
  const float rs = rsqrtf(warp_sum(ss) * inv_h + eps);
  opaque(raw);
  uint4* yr = reinterpret_cast<uint4*>(xn);
#pragma unroll
  for (int j = 0; j < VMAX; ++j) {
    if (j < vpl) {
      const int i = lane + 32 * j;
      float v[8], g[8], b[8];
      unpack8(raw[j], v);
      load8<GB_GLOBAL>(gamma + 8 * i, g);
      load8<GB_GLOBAL>(beta + 8 * i, b);
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = (v[k] - mu) * rs * g[k] + b[k];
      yr[i] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                         pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
      // gamma / beta are L1 hits: no need to load them ahead of this store
      asm volatile("" ::: "memory");
    }
  }
  mu_out = mu;
  rs_out = rs;
}

// One row, loaded and normalised.
template <int VMAX, bool GB_GLOBAL = true>
__device__ __forceinline__ void row_bf16(const __nv_bfloat16* __restrict__ x,
                                         const float* __restrict__ gamma,
                                         const float* __restrict__ beta,
                                         __nv_bfloat16* __restrict__ xn,
                                         int vpl, int h, float eps, int lane,
                                         float& mu_out, float& rs_out) {
  uint4 raw[VMAX];
  load_row<VMAX>(x, vpl, lane, raw);
  norm_row<VMAX, GB_GLOBAL>(raw, gamma, beta, xn, vpl, h, eps, lane, mu_out,
                            rs_out);
}

}  // namespace lnrow
}  // namespace tpmlp
