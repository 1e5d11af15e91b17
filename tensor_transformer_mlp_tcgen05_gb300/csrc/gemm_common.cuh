// Device helpers shared by the tensor-core GEMM kernels: bounded mbarrier
// waits, tile rasterisation and the fused epilogue stores.
#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace tpmlp {
namespace gemm {

// Budget for waits during teardown after an abort (copies already in flight).
constexpr unsigned long long TEARDOWN_BUDGET_NS = 200000000ull;

struct Ctl {
  volatile int* abort_flag;
  int* status;
  unsigned long long budget;
};

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             const Ctl& c, int role) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*c.abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > c.budget) {
      *c.abort_flag = 1;
      if (atomicCAS(c.status, 0, TPMLP_ERR_TIMEOUT) == 0) {
        c.status[1] = role;
        c.status[2] = static_cast<int>(blockIdx.x);
      }
      __threadfence();
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_teardown(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > TEARDOWN_BUDGET_NS) return false;
  }
  return true;
}

// Tile rasterisation: groups of `group_m` m-tiles, m fastest inside a group,
// so CTAs running at the same time share A row-panels and B column-panels.
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n,
                                            int group_m, int& mb, int& nb) {
  const int per_group = group_m * num_n;
  const int g = tile / per_group;
  const int first_m = g * group_m;
  const int gm = min(num_m - first_m, group_m);
  const int r = tile - g * per_group;
  mb = first_m + r % gm;
  nb = r / gm;
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* p,
                                              const float (&v)[32]) {
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    q[i] = make_uint4(pack_bf16x2(v[8 * i + 0], v[8 * i + 1]),
                      pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                      pack_bf16x2(v[8 * i + 4], v[8 * i + 5]),
                      pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
  }
}

__device__ __forceinline__ void store_f32x32(float* p, const float (&v)[32]) {
  float4* q = reinterpret_cast<float4*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    q[i] = make_float4(v[4 * i + 0], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

__device__ __forceinline__ void add_bias32(const float* bias, int c0,
                                           float (&v)[32]) {
  if (bias == nullptr) return;
  const float4* b = reinterpret_cast<const float4*>(bias + c0);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 t = __ldg(b + i);
    v[4 * i + 0] += t.x;
    v[4 * i + 1] += t.y;
    v[4 * i + 2] += t.z;
    v[4 * i + 3] += t.w;
  }
}

// Epilogue of one 32-column chunk of one row (non-shard-sum epilogues).
template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const GemmArgs& a, int row,
                                               int c0, float (&v)[32]) {
  const size_t off = static_cast<size_t>(row) * a.ldo + c0;
  if constexpr (EPI == EPI_GELU_FWD) {
    add_bias32(a.bias, c0, v);
    if (a.out2 != nullptr) {
      store_bf16x32(static_cast<__nv_bfloat16*>(a.out2) + off, v);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = gelu_f32(v[i], a.gelu_mode);
    store_bf16x32(static_cast<__nv_bfloat16*>(a.out) + off, v);
  } else if constexpr (EPI == EPI_GELU_BWD) {
    const uint4* hp = reinterpret_cast<const uint4*>(
        static_cast<const __nv_bfloat16*>(a.aux) +
        static_cast<size_t>(row) * a.ldaux + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 u = hp[i];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float h0, h1;
        unpack_bf16x2(w[j], h0, h1);
        v[8 * i + 2 * j + 0] *= gelu_grad_f32(h0, a.gelu_mode);
        v[8 * i + 2 * j + 1] *= gelu_grad_f32(h1, a.gelu_mode);
      }
    }
    store_bf16x32(static_cast<__nv_bfloat16*>(a.out) + off, v);
  } else if constexpr (EPI == EPI_STORE_F32) {
    store_f32x32(static_cast<float*>(a.out) + off, v);
  }
}

}  // namespace gemm
}  // namespace tpmlp
