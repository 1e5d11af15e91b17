// Device helpers shared by the tensor-core GEMM kernels: bounded mbarrier
// waits, tile rasterisation and the fused epilogue stores.
#pragma once
#include "internal.h"
#include "ln_row.cuh"
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

// Bounded wait until the counter reaches `target` (gpu-scope acquire), then
// a proxy fence so that this thread's later TMA reads of global memory see
// what the counted writers released.  Same time budget and abort protocol
// as wait_bounded.
__device__ __forceinline__ bool wait_count(const unsigned int* count,
                                           uint32_t target, const Ctl& c,
                                           int role) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (ptx::ld_acquire_gpu(count) < target) {
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
  ptx::fence_proxy_async_global();
  return true;
}

// Fused LayerNorm prologue (GemmArgs::ln_x), run by one warp: claims rows
// from a shared counter until every row is taken (two at a time when a row
// fits in half the register budget, both loaded before either is
// normalised, so that a warp keeps two rows in flight; else one),
// normalises each (lnrow::norm_row, the stand-alone kernel's arithmetic)
// into ln_xn with its mean and rstd, then publishes the claim's row count on
// its 128-row block: every lane fences its stores for the async proxy (the
// TMA loads that read them), the warp synchronises, and one lane adds the
// count with gpu-scope release semantics.  A warp never waits here, and rows
// go to whichever warps are running, so the producers' waits on these counts
// end whatever CTAs are resident.
__device__ __forceinline__ void ln_publish(unsigned int* ready, uint32_t r0,
                                           int n, int lane) {
  ptx::fence_proxy_async_global();
  __syncwarp();
  if (lane == 0) ptx::red_release_gpu_add(ready + r0 / 128, n);
}

// gamma / beta: the LayerNorm parameters staged in shared memory by the
// caller.
__device__ __forceinline__ void ln_prologue(const GemmArgs& a,
                                            const float* gamma,
                                            const float* beta, int lane) {
  const int vpl = a.K / 256;
  unsigned int* claim = a.ln_sync;
  unsigned int* ready = a.ln_sync + 1;
  const bool two = vpl <= LN_VMAX / 2;
  const uint32_t step = two ? 2u : 1u;
  while (true) {
    uint32_t r0 = 0;
    if (lane == 0) r0 = atomicAdd(claim, step);
    r0 = __shfl_sync(0xffffffffu, r0, 0);
    if (r0 >= static_cast<uint32_t>(a.M)) break;
    const size_t row = r0;
    float mu, rs;
    if (two) {
      const bool second = r0 + 1 < static_cast<uint32_t>(a.M);
      uint4 ra[LN_VMAX / 2], rb[LN_VMAX / 2];
      lnrow::load_row<LN_VMAX / 2>(a.ln_x + row * a.K, vpl, lane, ra);
      if (second)
        lnrow::load_row<LN_VMAX / 2>(a.ln_x + (row + 1) * a.K, vpl, lane, rb);
      lnrow::norm_row<LN_VMAX / 2, false>(ra, gamma, beta,
                                   a.ln_xn + row * a.K, vpl, a.K, a.ln_eps,
                                   lane, mu, rs);
      if (lane == 0) {
        a.ln_mean[row] = mu;
        a.ln_rstd[row] = rs;
      }
      if (second) {
        lnrow::norm_row<LN_VMAX / 2, false>(rb, gamma, beta,
                                     a.ln_xn + (row + 1) * a.K, vpl, a.K,
                                     a.ln_eps, lane, mu, rs);
        if (lane == 0) {
          a.ln_mean[row + 1] = mu;
          a.ln_rstd[row + 1] = rs;
        }
      }
      ln_publish(ready, r0, second ? 2 : 1, lane);
    } else {
      lnrow::row_bf16<LN_VMAX, false>(a.ln_x + row * a.K, gamma, beta,
                               a.ln_xn + row * a.K, vpl, a.K, a.ln_eps, lane,
                               mu, rs);
      if (lane == 0) {
        a.ln_mean[row] = mu;
        a.ln_rstd[row] = rs;
      }
      ln_publish(ready, r0, 1, lane);
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

__device__ __forceinline__ void store_bf16x16(__nv_bfloat16* p,
                                              const float (&v)[16]) {
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
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

// Add n bf16 values of a residual row (row, c0 .. c0+n) to v (n % 8 == 0).
__device__ __forceinline__ void add_residual_bf16(const void* res, long long ld,
                                                  int row, int M, int c0,
                                                  float* v, int n) {
  if (res == nullptr || row >= M) return;
  const uint4* p = reinterpret_cast<const uint4*>(
      static_cast<const __nv_bfloat16*>(res) + static_cast<size_t>(row) * ld +
      c0);
#pragma unroll
  for (int i = 0; i < n / 8; ++i) {
    const uint4 u = p[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float a, b;
      unpack_bf16x2(w[k], a, b);
      v[8 * i + 2 * k] += a;
      v[8 * i + 2 * k + 1] += b;
    }
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

// ---------------------------------------------- TMA-store epilogue ----
// Each epilogue warp owns 32 output rows (its TMEM lanes) and stages one
// 32-row x 128-byte chunk at a time in shared memory, laid out as the
// 128-byte-swizzled box of the output's tensor map (16-byte unit c of row r
// at unit c ^ (r % 8)), so the 32 lanes' 16-byte writes hit distinct banks.
// Lane 0 then issues one asynchronous TMA store of the chunk; two staging
// buffers per warp alternate.
constexpr uint32_t STAGE_CHUNK_BYTES = 32 * 128;

struct ChunkStager {
  uint32_t base;   // this warp's two buffers (1024-byte aligned)
  uint32_t count;  // chunks issued so far (lane 0's bulk groups)

  // Write this lane's 128-byte row `w` and store the chunk at element
  // coordinates (c0, r0) of `map`; returns the staging buffer used (it holds
  // the chunk until the next-but-one put).
  __device__ __forceinline__ uint32_t put(const CUtensorMap* map, int c0,
                                          int r0, const uint32_t (&w)[32],
                                          int lane) {
    const uint32_t buf = base + (count & 1u) * STAGE_CHUNK_BYTES;
    if (lane == 0) ptx::bulk_wait_read<1>();  // buffer used two chunks ago
    __syncwarp();
    const uint32_t row = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t u = static_cast<uint32_t>(c ^ (lane & 7));
      ptx::st_shared_v4(row + u * 16u, w[4 * c], w[4 * c + 1], w[4 * c + 2],
                        w[4 * c + 3]);
    }
    ptx::fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      ptx::tma_store_2d(map, buf, c0, r0);
      ptx::bulk_commit();
    }
    ++count;
    return buf;
  }

  // The buffer the k-th next put will use.
  __device__ __forceinline__ uint32_t buffer(uint32_t k) const {
    return base + ((count + k) & 1u) * STAGE_CHUNK_BYTES;
  }

  __device__ __forceinline__ void drain(int lane) {
    if (lane == 0) ptx::bulk_wait_all();
    __syncwarp();
  }
};

// Column sums of a staged 32-row x 64-column bf16 chunk (128-byte-swizzled
// rows): lane l gets the fp32 sums of columns 2l and 2l + 1 over the rows in
// order.  Each row read is 32 consecutive words, one per lane.
__device__ __forceinline__ float2 chunk_colsum_bf16(uint32_t buf, int lane) {
  float s0 = 0.f, s1 = 0.f;
  const uint32_t off = static_cast<uint32_t>(lane & 3) * 4u;
#pragma unroll 8
  for (int r = 0; r < 32; ++r) {
    const uint32_t u = static_cast<uint32_t>((lane >> 2) ^ (r & 7));
    const uint32_t word =
        ptx::ld_shared_u32(buf + static_cast<uint32_t>(r) * 128u + u * 16u + off);
    float a, b;
    unpack_bf16x2(word, a, b);
    s0 += a;
    s1 += b;
  }
  return make_float2(s0, s1);
}

__device__ __forceinline__ void pack_bf16x64(const float* v, uint32_t (&w)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
}

__device__ __forceinline__ void add_bias_n(const float* bias, int c0, float* v,
                                           int n) {
  if (bias == nullptr) return;
  const float4* b = reinterpret_cast<const float4*>(bias + c0);
#pragma unroll
  for (int i = 0; i < n / 4; ++i) {
    const float4 t = __ldg(b + i);
    v[4 * i + 0] += t.x;
    v[4 * i + 1] += t.y;
    v[4 * i + 2] += t.z;
    v[4 * i + 3] += t.w;
  }
}

}  // namespace gemm
}  // namespace tpmlp
