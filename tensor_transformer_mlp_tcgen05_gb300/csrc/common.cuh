// Definitions shared by the kernels of libtpmlp.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tp_mlp.h"

namespace tpmlp {

// Epilogues of the GEMM kernels.
enum Epilogue : int {
  // H = acc + b1; Y = GeLU(H); writes Y (out) and, if out2 != null, H.
  EPI_GELU_FWD = 0,
  // fixed-order sum over shard segments of fresh fp32 partials, + bias,
  // one rounding to the output type (bf16 or fp32).
  EPI_SHARDSUM = 1,
  // dH = acc * GeLU'(H) with H read from `aux`; writes dH (out).
  EPI_GELU_BWD = 2,
  // plain fp32 store (weight gradients).
  EPI_STORE_F32 = 3,
};

// Arguments of one GEMM launch: D[M,N] = sum over K of Aop[m,k] * Bop[k,n],
// K split into `num_seg` equal segments of `kb_per_seg` k-blocks; each
// segment accumulates into a fresh accumulator (used for the shard sum).
// (The fp32 CUDA-core GEMM reads kb_per_seg as the segment length in K.)
struct GemmArgs {
  int M, N, K;
  int kb_per_seg;
  int num_seg;
  int group_m;            // tile rasterisation: m-tiles per group
  int gelu_mode;
  int out_f32;            // EPI_SHARDSUM output type: 1 fp32, 0 bf16
  void* out;              // [M, N] row-major, leading dimension ldo
  long long ldo;
  void* out2;             // EPI_GELU_FWD: H (nullable)
  const void* aux;        // EPI_GELU_BWD: H; EPI_SHARDSUM: residual added
                          // before the rounding (nullable); leading dim ldaux
  long long ldaux;
  const float* bias;      // [N] fp32 (nullable)
  int* status;            // device status word: [0] code, [1] role, [2] block
  unsigned long long budget_ns;
};

// Roles recorded in status[1] when a bounded wait gives up.
enum WaitRole : int { ROLE_PRODUCER = 1, ROLE_MMA = 2, ROLE_EPILOGUE = 3 };

// GeLU and its derivative in fp32.  Exact form: GeLU(x) = x Phi(x) with
// Phi(x) = (1 + erf(x / sqrt 2)) / 2, GeLU'(x) = Phi(x) + x phi(x).  Tanh form
// (Hendrycks & Gimpel): 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
__device__ __forceinline__ float gelu_f32(float x, int mode) {
  if (mode == TPMLP_GELU_ERF) {
    return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
  }
  const float u = 0.79788456080286536f * (x + 0.044715f * x * x * x);
  return 0.5f * x * (1.0f + tanhf(u));
}

__device__ __forceinline__ float gelu_grad_f32(float x, int mode) {
  if (mode == TPMLP_GELU_ERF) {
    const float cdf = 0.5f * (1.0f + erff(x * 0.70710678118654752f));
    const float pdf = 0.39894228040143268f * expf(-0.5f * x * x);
    return cdf + x * pdf;
  }
  const float u = 0.79788456080286536f * (x + 0.044715f * x * x * x);
  const float th = tanhf(u);
  const float du = 0.79788456080286536f * (1.0f + 3.0f * 0.044715f * x * x);
  return 0.5f * (1.0f + th) + 0.5f * x * (1.0f - th * th) * du;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void unpack_bf16x2(uint32_t u, float& lo,
                                              float& hi) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  lo = __low2float(v);
  hi = __high2float(v);
}

}  // namespace tpmlp
