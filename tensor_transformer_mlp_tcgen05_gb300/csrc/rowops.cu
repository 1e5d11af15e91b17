// Bandwidth-bound kernels around the GEMMs: LayerNorm forward/backward and
// the fixed-order column sums behind db1, db2, dgamma and dbeta.
//
// LayerNorm (pre-LN placement: Megatron-LM explainer, section "Fixing BERT:
// reordering layer normalisation for scaling"): one warp per token row,
// 16-byte vector loads, warp-shuffle (butterfly) reductions in fp32, mean
// and biased variance in two passes over the row (the second pass hits L1).
//
// Column sums are deterministic by construction (the Megatron Core
// determinism article: fixed-order reductions, private output per writer):
// stage 1 gives every block a fixed chunk of COLSUM_CHUNK_ROWS rows and a
// fixed 128-column strip; inside the block warp w takes rows w, w+8, ... of
// the chunk in order and the 8 warp partials are added in warp order; stage
// 2 adds the chunk partials in chunk order.  No atomics anywhere.
#include "internal.h"
#include "ln_row.cuh"

namespace tpmlp {
namespace {

constexpr int LN_WARPS = 8;  // rows per LayerNorm block

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 16-byte vectors: 8 bf16 or 4 fp32.
template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    unpack_bf16x2(u.x, v[0], v[1]);
    unpack_bf16x2(u.y, v[2], v[3]);
    unpack_bf16x2(u.z, v[4], v[5]);
    unpack_bf16x2(u.w, v[6], v[7]);
  }
  __device__ static void store(__nv_bfloat16* p, const float (&v)[8]) {
    *reinterpret_cast<uint4*>(p) =
        make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                   pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
  }
};
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void load(const float* p, float (&v)[4]) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    v[0] = u.x;
    v[1] = u.y;
    v[2] = u.z;
    v[3] = u.w;
  }
  __device__ static void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};

template <int N>
__device__ __forceinline__ void load_f32(const float* p, float (&v)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    const float4 u = __ldg(reinterpret_cast<const float4*>(p + i));
    v[i] = u.x;
    v[i + 1] = u.y;
    v[i + 2] = u.z;
    v[i + 3] = u.w;
  }
}

template <typename T>
__global__ void __launch_bounds__(LN_WARPS * 32)
    ln_fwd_kernel(const T* __restrict__ X, const float* __restrict__ gamma,
                  const float* __restrict__ beta, T* __restrict__ Xn,
                  float* __restrict__ mean_out, float* __restrict__ rstd_out,
                  int rows, int h, float eps) {
  constexpr int V = Vec<T>::N;
  const int row = blockIdx.x * LN_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const T* x = X + static_cast<size_t>(row) * h;
  const int nv = h / V;
  float s = 0.f;
  for (int i = lane; i < nv; i += 32) {
    float v[V];
    Vec<T>::load(x + i * V, v);
#pragma unroll
    for (int k = 0; k < V; ++k) s += v[k];
  }
  const float mu = warp_sum(s) / static_cast<float>(h);
  float ss = 0.f;
  for (int i = lane; i < nv; i += 32) {
    float v[V];
    Vec<T>::load(x + i * V, v);
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const float d = v[k] - mu;
      ss += d * d;
    }
  }
  const float rs = rsqrtf(warp_sum(ss) / static_cast<float>(h) + eps);
  T* y = Xn + static_cast<size_t>(row) * h;
  for (int i = lane; i < nv; i += 32) {
    float v[V], g[V], b[V];
    Vec<T>::load(x + i * V, v);
    load_f32<V>(gamma + i * V, g);
    load_f32<V>(beta + i * V, b);
#pragma unroll
    for (int k = 0; k < V; ++k) v[k] = (v[k] - mu) * rs * g[k] + b[k];
    Vec<T>::store(y + i * V, v);
  }
  if (lane == 0) {
    mean_out[row] = mu;
    rstd_out[row] = rs;
  }
}

// dX = rstd * (g - mean(g) - xhat * mean(g * xhat)) [+ dres], g = gamma * dXn.
template <typename T>
__global__ void __launch_bounds__(LN_WARPS * 32)
    ln_bwd_kernel(const float* __restrict__ dXn, const T* __restrict__ X,
                  const float* __restrict__ mean, const float* __restrict__ rstd,
                  const float* __restrict__ gamma, const T* __restrict__ dres,
                  T* __restrict__ dX, int rows, int h) {
  constexpr int V = Vec<T>::N;
  const int row = blockIdx.x * LN_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const size_t base = static_cast<size_t>(row) * h;
  const float mu = mean[row], rs = rstd[row];
  const int nv = h / V;
  float sg = 0.f, sgx = 0.f;
  for (int i = lane; i < nv; i += 32) {
    float x[V], d[V], g[V];
    Vec<T>::load(X + base + i * V, x);
    load_f32<V>(dXn + base + i * V, d);
    load_f32<V>(gamma + i * V, g);
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const float gg = g[k] * d[k];
      sg += gg;
      sgx += gg * (x[k] - mu) * rs;
    }
  }
  const float inv_h = 1.0f / static_cast<float>(h);
  const float c_g = warp_sum(sg) * inv_h;
  const float c_gx = warp_sum(sgx) * inv_h;
  for (int i = lane; i < nv; i += 32) {
    float x[V], d[V], g[V], o[V];
    Vec<T>::load(X + base + i * V, x);
    load_f32<V>(dXn + base + i * V, d);
    load_f32<V>(gamma + i * V, g);
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const float xhat = (x[k] - mu) * rs;
      o[k] = rs * (g[k] * d[k] - c_g - xhat * c_gx);
    }
    if (dres != nullptr) {
      float r[V];
      Vec<T>::load(dres + base + i * V, r);
#pragma unroll
      for (int k = 0; k < V; ++k) o[k] += r[k];
    }
    Vec<T>::store(dX + base + i * V, o);
  }
}

// The backward with the row held in registers (h = 32 * VPL * V): X and dXn
// are read once and both passes run from registers, with all of a lane's
// loads in flight together.  Same per-lane accumulation order as
// ln_bwd_kernel, so the same results.
template <typename T>
__device__ __forceinline__ void unpack_vec(const uint4 u, float (&v)[Vec<T>::N]);
template <>
__device__ __forceinline__ void unpack_vec<__nv_bfloat16>(const uint4 u,
                                                          float (&v)[8]) {
  unpack_bf16x2(u.x, v[0], v[1]);
  unpack_bf16x2(u.y, v[2], v[3]);
  unpack_bf16x2(u.z, v[4], v[5]);
  unpack_bf16x2(u.w, v[6], v[7]);
}
template <>
__device__ __forceinline__ void unpack_vec<float>(const uint4 u, float (&v)[4]) {
  v[0] = __uint_as_float(u.x);
  v[1] = __uint_as_float(u.y);
  v[2] = __uint_as_float(u.z);
  v[3] = __uint_as_float(u.w);
}

template <typename T, int VPL>
__global__ void __launch_bounds__(LN_WARPS * 32)
    ln_bwd_reg_kernel(const float* __restrict__ dXn, const T* __restrict__ X,
                      const float* __restrict__ mean,
                      const float* __restrict__ rstd,
                      const float* __restrict__ gamma,
                      const T* __restrict__ dres, T* __restrict__ dX, int rows,
                      int h) {
  constexpr int V = Vec<T>::N;
  const int row = blockIdx.x * LN_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const size_t base = static_cast<size_t>(row) * h;
  const float mu = mean[row], rs = rstd[row];
  const uint4* xr = reinterpret_cast<const uint4*>(X + base);
  uint4 raw[VPL];
  float d[VPL][V];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int i = lane + 32 * j;
    raw[j] = xr[i];
    load_f32<V>(dXn + base + i * V, d[j]);
  }
  float sg = 0.f, sgx = 0.f;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    float x[V], g[V];
    unpack_vec<T>(raw[j], x);
    load_f32<V>(gamma + (lane + 32 * j) * V, g);
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const float gg = g[k] * d[j][k];
      sg += gg;
      sgx += gg * (x[k] - mu) * rs;
    }
  }
  const float inv_h = 1.0f / static_cast<float>(h);
  const float c_g = warp_sum(sg) * inv_h;
  const float c_gx = warp_sum(sgx) * inv_h;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int i = lane + 32 * j;
    float x[V], g[V], o[V];
    unpack_vec<T>(raw[j], x);
    load_f32<V>(gamma + i * V, g);
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const float xhat = (x[k] - mu) * rs;
      o[k] = rs * (g[k] * d[j][k] - c_g - xhat * c_gx);
    }
    if (dres != nullptr) {
      float r[V];
      Vec<T>::load(dres + base + i * V, r);
#pragma unroll
      for (int k = 0; k < V; ++k) o[k] += r[k];
    }
    Vec<T>::store(dX + base + i * V, o);
  }
}

// LayerNorm forward with the row in registers (h = 256 VPL, bf16): one warp
// per row, the row's arithmetic in lnrow::row_bf16 (ln_row.cuh), shared with
// the GEMM's fused LayerNorm prologue.  VPL = 0: any vpl up to LN_VMAX, read
// at run time (same arithmetic for the same vpl).
template <int VPL>
__global__ void __launch_bounds__(LN_WARPS * 32, 2)
    ln_fwd_reg_kernel(const __nv_bfloat16* __restrict__ X,
                      const float* __restrict__ gamma,
                      const float* __restrict__ beta,
                      __nv_bfloat16* __restrict__ Xn,
                      float* __restrict__ mean_out,
                      float* __restrict__ rstd_out, int rows, int h,
                      float eps) {
  const int row = blockIdx.x * LN_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const size_t base = static_cast<size_t>(row) * h;
  float mu, rs;
  constexpr int VMAX = VPL > 0 ? VPL : LN_VMAX;
  lnrow::row_bf16<VMAX>(X + base, gamma, beta, Xn + base,
                        VPL > 0 ? VPL : h / 256, h, eps, lane, mu, rs);
  if (lane == 0) {
    mean_out[row] = mu;
    rstd_out[row] = rs;
  }
}

// ------------------------------------------------------- column sums --

constexpr int CS_WARPS = 8;
constexpr int CS_COLS = 128;  // columns per block: 4 per lane

template <typename T>
__device__ __forceinline__ void load4(const T* p, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4]) {
  const float4 u = *reinterpret_cast<const float4*>(p);
  v[0] = u.x;
  v[1] = u.y;
  v[2] = u.z;
  v[3] = u.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p,
                                                     float (&v)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  unpack_bf16x2(u.x, v[0], v[1]);
  unpack_bf16x2(u.y, v[2], v[3]);
}

template <typename T>
__device__ __forceinline__ void store4(T* p, const float (&v)[4]);
template <>
__device__ __forceinline__ void store4<float>(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p,
                                                      const float (&v)[4]) {
  *reinterpret_cast<uint2*>(p) =
      make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
}

// MODE 0: part1 = sum src, and, when amax is not null, *amax raised to the
// largest |src| (fp32 bits; a maximum is order-free, so deterministic).
// MODE 1 (LayerNorm parameters): part1 = sum dXn * xhat, part2 = sum dXn,
// with xhat recomputed from X, mean, rstd.
template <typename T, int MODE>
__global__ void __launch_bounds__(CS_WARPS * 32)
    colsum_partial_kernel(const T* __restrict__ src,
                          const float* __restrict__ dxn,
                          const float* __restrict__ mean,
                          const float* __restrict__ rstd,
                          float* __restrict__ part1, float* __restrict__ part2,
                          int rows, int cols, unsigned int* amax) {
  __shared__ float red[2][CS_WARPS][CS_COLS];
  float mx = 0.f;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * CS_COLS + lane * 4;
  const int chunk = blockIdx.y;
  const int r0 = chunk * COLSUM_CHUNK_ROWS;
  const int r1 = min(rows, r0 + COLSUM_CHUNK_ROWS);
  float a1[4] = {0.f, 0.f, 0.f, 0.f}, a2[4] = {0.f, 0.f, 0.f, 0.f};
  if (c < cols) {
    for (int r = r0 + w; r < r1; r += CS_WARPS) {
      const size_t off = static_cast<size_t>(r) * cols + c;
      if constexpr (MODE == 0) {
        float v[4];
        load4<T>(src + off, v);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          a1[k] += v[k];
          mx = fmaxf(mx, fabsf(v[k]));
        }
      } else {
        float x[4], d[4];
        load4<T>(src + off, x);
        load4<float>(dxn + off, d);
        const float mu = mean[r], rs = rstd[r];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          a1[k] += d[k] * ((x[k] - mu) * rs);
          a2[k] += d[k];
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    red[0][w][lane * 4 + k] = a1[k];
    red[1][w][lane * 4 + k] = a2[k];
  }
  if (MODE == 0 && amax != nullptr) {
    const unsigned int wm = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
    if (lane == 0) atomicMax(amax, wm);
  }
  __syncthreads();
  const int nout = (MODE == 0) ? 1 : 2;
  for (int idx = threadIdx.x; idx < nout * CS_COLS; idx += blockDim.x) {
    const int which = idx / CS_COLS, cc = idx % CS_COLS;
    const int col = blockIdx.x * CS_COLS + cc;
    if (col >= cols) continue;
    float s = 0.f;
#pragma unroll
    for (int ww = 0; ww < CS_WARPS; ++ww) s += red[which][ww][cc];
    float* dst = which == 0 ? part1 : part2;
    dst[static_cast<size_t>(chunk) * cols + col] = s;
  }
}

// MODE 0 for bf16 with cols % 8 == 0: the same sums in the same order (per
// column: warp w adds rows w, w + 8, ... of the chunk in row order, then the
// eight warp sums in warp order, so the results equal colsum_partial_kernel's
// bit for bit), 8 columns per lane from one 16-byte load, four rows' loads
// in flight, 256 columns per block.
constexpr int CS8_COLS = 256;
__global__ void __launch_bounds__(CS_WARPS * 32)
    colsum_partial_bf16x8_kernel(const __nv_bfloat16* __restrict__ src,
                                 float* __restrict__ part, int rows, int cols,
                                 unsigned int* amax) {
  __shared__ float red[CS_WARPS][CS8_COLS];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * CS8_COLS + lane * 8;
  const int chunk = blockIdx.y;
  const int r0 = chunk * COLSUM_CHUNK_ROWS;
  const int r1 = min(rows, r0 + COLSUM_CHUNK_ROWS);
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float mx = 0.f;
  if (c < cols) {
    int r = r0 + w;
    for (; r + 3 * CS_WARPS < r1; r += 4 * CS_WARPS) {
      uint4 u[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        u[k] = *reinterpret_cast<const uint4*>(
            src + static_cast<size_t>(r + k * CS_WARPS) * cols + c);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t q[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float lo, hi;
          unpack_bf16x2(q[j], lo, hi);
          a[2 * j] += lo;
          a[2 * j + 1] += hi;
          mx = fmaxf(mx, fmaxf(fabsf(lo), fabsf(hi)));
        }
      }
    }
    for (; r < r1; r += CS_WARPS) {
      const uint4 u = *reinterpret_cast<const uint4*>(
          src + static_cast<size_t>(r) * cols + c);
      const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float lo, hi;
        unpack_bf16x2(q[j], lo, hi);
        a[2 * j] += lo;
        a[2 * j + 1] += hi;
        mx = fmaxf(mx, fmaxf(fabsf(lo), fabsf(hi)));
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) red[w][lane * 8 + k] = a[k];
  if (amax != nullptr) {
    const unsigned int wm = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
    if (lane == 0) atomicMax(amax, wm);
  }
  __syncthreads();
  for (int cc = threadIdx.x; cc < CS8_COLS; cc += blockDim.x) {
    const int col = blockIdx.x * CS8_COLS + cc;
    if (col >= cols) continue;
    float t = 0.f;
#pragma unroll
    for (int ww = 0; ww < CS_WARPS; ++ww) t += red[ww][cc];
    part[static_cast<size_t>(chunk) * cols + col] = t;
  }
}

// MODE 1 for bf16 X with h % 8 == 0: the same sums in the same order as
// colsum_partial_kernel<bf16, 1> (per column: warp w adds rows w, w + 8, ...
// of the chunk in row order, then the eight warp sums in warp order), 8
// columns per lane from one 16-byte load of X and two of dXn, four rows'
// loads in flight, 256 columns per block.  Chunks run last first
// (blockIdx.y = 0 takes the last chunk): the LayerNorm backward has just
// read the last rows, which are then still in L2.
__global__ void __launch_bounds__(CS_WARPS * 32)
    ln_param_partial_bf16x8_kernel(const __nv_bfloat16* __restrict__ X,
                                   const float* __restrict__ dxn,
                                   const float* __restrict__ mean,
                                   const float* __restrict__ rstd,
                                   float* __restrict__ part_g,
                                   float* __restrict__ part_b, int rows,
                                   int cols) {
  __shared__ float red[2][CS_WARPS][CS8_COLS];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * CS8_COLS + lane * 8;
  const int chunk = static_cast<int>(gridDim.y - 1 - blockIdx.y);
  const int r0 = chunk * COLSUM_CHUNK_ROWS;
  const int r1 = min(rows, r0 + COLSUM_CHUNK_ROWS);
  float ag[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float ab[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  auto accumulate = [&](const uint4 xu, const float4 d0, const float4 d1,
                        float mu, float rs) {
    const uint32_t q[4] = {xu.x, xu.y, xu.z, xu.w};
    const float d[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float lo, hi;
      unpack_bf16x2(q[j], lo, hi);
      ag[2 * j] += d[2 * j] * ((lo - mu) * rs);
      ag[2 * j + 1] += d[2 * j + 1] * ((hi - mu) * rs);
      ab[2 * j] += d[2 * j];
      ab[2 * j + 1] += d[2 * j + 1];
    }
  };
  if (c < cols) {
    int r = r0 + w;
    for (; r + 3 * CS_WARPS < r1; r += 4 * CS_WARPS) {
      uint4 xu[4];
      float4 d0[4], d1[4];
      float mu[4], rs[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const size_t off = static_cast<size_t>(r + k * CS_WARPS) * cols + c;
        xu[k] = *reinterpret_cast<const uint4*>(X + off);
        d0[k] = *reinterpret_cast<const float4*>(dxn + off);
        d1[k] = *reinterpret_cast<const float4*>(dxn + off + 4);
        mu[k] = mean[r + k * CS_WARPS];
        rs[k] = rstd[r + k * CS_WARPS];
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) accumulate(xu[k], d0[k], d1[k], mu[k], rs[k]);
    }
    for (; r < r1; r += CS_WARPS) {
      const size_t off = static_cast<size_t>(r) * cols + c;
      accumulate(*reinterpret_cast<const uint4*>(X + off),
                 *reinterpret_cast<const float4*>(dxn + off),
                 *reinterpret_cast<const float4*>(dxn + off + 4), mean[r],
                 rstd[r]);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    red[0][w][lane * 8 + k] = ag[k];
    red[1][w][lane * 8 + k] = ab[k];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < 2 * CS8_COLS; idx += blockDim.x) {
    const int which = idx / CS8_COLS, cc = idx % CS8_COLS;
    const int col = blockIdx.x * CS8_COLS + cc;
    if (col >= cols) continue;
    float t = 0.f;
#pragma unroll
    for (int ww = 0; ww < CS_WARPS; ++ww) t += red[which][ww][cc];
    (which == 0 ? part_g : part_b)[static_cast<size_t>(chunk) * cols + col] = t;
  }
}

// out[c] = sum_k part[k][c] in a fixed order: 32 columns per block, warp y
// sums the y-th eighth of the chunks in chunk order, then the eight warp
// sums are added in warp order.  Coalesced 128-byte rows, any chunk count.
__global__ void __launch_bounds__(256)
    colsum_finalize_kernel(const float* __restrict__ part,
                           float* __restrict__ out, int chunks, int cols) {
  __shared__ float red[8][33];
  const int tx = threadIdx.x, y = threadIdx.y;
  const int c = blockIdx.x * 32 + tx;
  const int per = (chunks + 7) / 8;
  const int k0 = y * per;
  const int k1 = min(chunks, k0 + per);
  float s = 0.f;
  if (c < cols) {
#pragma unroll 4
    for (int k = k0; k < k1; ++k) s += part[static_cast<size_t>(k) * cols + c];
  }
  red[y][tx] = s;
  __syncthreads();
  if (y == 0 && c < cols) {
    float t = red[0][tx];
#pragma unroll
    for (int i = 1; i < 8; ++i) t += red[i][tx];
    out[c] = t;
  }
}

// Backward of the output dropout: out = mask * scale * dZ, four columns per
// thread (one Philox draw), grid-stride over the [rows, cols] matrix.
template <typename T>
__global__ void __launch_bounds__(256)
    dropout_grad_kernel(const T* __restrict__ dZ, T* __restrict__ out, int rows,
                        int cols, uint32_t threshold, float scale,
                        unsigned long long seed, unsigned long long offset) {
  const long long groups = static_cast<long long>(rows) * (cols / 4);
  for (long long gi = blockIdx.x * static_cast<long long>(blockDim.x) +
                      threadIdx.x;
       gi < groups; gi += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(gi / (cols / 4));
    const int c0 = static_cast<int>(gi % (cols / 4)) * 4;
    const size_t off = static_cast<size_t>(r) * cols + c0;
    float v[4];
    load4<T>(dZ + off, v);
    apply_dropout(threshold, scale, seed, offset, r, c0, v, 4);
    store4<T>(out + off, v);
  }
}

}  // namespace

cudaError_t launch_dropout_grad(bool bf16, const void* dZ, void* out, int rows,
                                int cols, uint32_t threshold, float scale,
                                unsigned long long seed,
                                unsigned long long offset,
                                cudaStream_t stream) {
  const long long groups = static_cast<long long>(rows) * (cols / 4);
  const int threads = 256;
  long long blocks = (groups + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  if (bf16) {
    dropout_grad_kernel<__nv_bfloat16><<<static_cast<int>(blocks), threads, 0,
                                          stream>>>(
        static_cast<const __nv_bfloat16*>(dZ), static_cast<__nv_bfloat16*>(out),
        rows, cols, threshold, scale, seed, offset);
  } else {
    dropout_grad_kernel<float><<<static_cast<int>(blocks), threads, 0, stream>>>(
        static_cast<const float*>(dZ), static_cast<float*>(out), rows, cols,
        threshold, scale, seed, offset);
  }
  return cudaGetLastError();
}

cudaError_t launch_ln_fwd(bool bf16, const void* X, const float* gamma,
                          const float* beta, void* Xn, float* mean,
                          float* rstd, int rows, int h, float eps,
                          cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int grid = (rows + LN_WARPS - 1) / LN_WARPS;
  const int vpl = h % 256 == 0 ? h / 256 : 0;
#define TPMLP_LN_FWD_REG(N)                                                  \
  ln_fwd_reg_kernel<N><<<grid, LN_WARPS * 32, 0, stream>>>(                  \
      static_cast<const __nv_bfloat16*>(X), gamma, beta,                     \
      static_cast<__nv_bfloat16*>(Xn), mean, rstd, rows, h, eps)
  if (bf16 && vpl >= 1 && vpl <= LN_VMAX) {
    switch (vpl) {
      case 1: TPMLP_LN_FWD_REG(1); break;
      case 2: TPMLP_LN_FWD_REG(2); break;
      case 3: TPMLP_LN_FWD_REG(3); break;
      case 4: TPMLP_LN_FWD_REG(4); break;
      case 6: TPMLP_LN_FWD_REG(6); break;
      case 8: TPMLP_LN_FWD_REG(8); break;
      case 12: TPMLP_LN_FWD_REG(12); break;
      default:
        if (vpl > LN_VMAX) goto generic;
        TPMLP_LN_FWD_REG(0);
        break;
    }
#undef TPMLP_LN_FWD_REG
    return cudaGetLastError();
  }
generic:
  if (bf16) {
    ln_fwd_kernel<__nv_bfloat16><<<grid, LN_WARPS * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(X), gamma, beta,
        static_cast<__nv_bfloat16*>(Xn), mean, rstd, rows, h, eps);
  } else {
    ln_fwd_kernel<float><<<grid, LN_WARPS * 32, 0, stream>>>(
        static_cast<const float*>(X), gamma, beta, static_cast<float*>(Xn),
        mean, rstd, rows, h, eps);
  }
  return cudaGetLastError();
}

cudaError_t launch_ln_bwd(bool bf16, const float* dXn, const void* X,
                          const float* mean, const float* rstd,
                          const float* gamma, const void* dres, void* dX,
                          int rows, int h, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int grid = (rows + LN_WARPS - 1) / LN_WARPS;
  const int nv = h / (bf16 ? 8 : 4);
  const int vpl = nv % 32 == 0 ? nv / 32 : 0;
#define TPMLP_LN_BWD_REG(TY, N)                                              \
  ln_bwd_reg_kernel<TY, N><<<grid, LN_WARPS * 32, 0, stream>>>(             \
      dXn, static_cast<const TY*>(X), mean, rstd, gamma,                    \
      static_cast<const TY*>(dres), static_cast<TY*>(dX), rows, h)
  if (bf16 && (vpl == 4 || vpl == 8 || vpl == 12)) {
    if (vpl == 4) TPMLP_LN_BWD_REG(__nv_bfloat16, 4);
    else if (vpl == 8) TPMLP_LN_BWD_REG(__nv_bfloat16, 8);
    else TPMLP_LN_BWD_REG(__nv_bfloat16, 12);
  } else if (!bf16 && (vpl == 4 || vpl == 8 || vpl == 12)) {
    if (vpl == 4) TPMLP_LN_BWD_REG(float, 4);
    else if (vpl == 8) TPMLP_LN_BWD_REG(float, 8);
    else TPMLP_LN_BWD_REG(float, 12);
  } else if (bf16) {
#undef TPMLP_LN_BWD_REG
    ln_bwd_kernel<__nv_bfloat16><<<grid, LN_WARPS * 32, 0, stream>>>(
        dXn, static_cast<const __nv_bfloat16*>(X), mean, rstd, gamma,
        static_cast<const __nv_bfloat16*>(dres),
        static_cast<__nv_bfloat16*>(dX), rows, h);
  } else {
    ln_bwd_kernel<float><<<grid, LN_WARPS * 32, 0, stream>>>(
        dXn, static_cast<const float*>(X), mean, rstd, gamma,
        static_cast<const float*>(dres), static_cast<float*>(dX), rows, h);
  }
  return cudaGetLastError();
}

cudaError_t launch_colsum_partial(bool bf16, const void* src, float* part,
                                  int rows, int cols, cudaStream_t stream,
                                  unsigned int* amax) {
  const dim3 grid((cols + CS_COLS - 1) / CS_COLS, colsum_chunks(rows));
  if (bf16 && cols % 8 == 0 &&
      (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
    const dim3 grid8((cols + CS8_COLS - 1) / CS8_COLS, colsum_chunks(rows));
    colsum_partial_bf16x8_kernel<<<grid8, CS_WARPS * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(src), part, rows, cols, amax);
  } else if (bf16) {
    colsum_partial_kernel<__nv_bfloat16, 0><<<grid, CS_WARPS * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(src), nullptr, nullptr, nullptr,
        part, nullptr, rows, cols, amax);
  } else {
    colsum_partial_kernel<float, 0><<<grid, CS_WARPS * 32, 0, stream>>>(
        static_cast<const float*>(src), nullptr, nullptr, nullptr, part,
        nullptr, rows, cols, amax);
  }
  return cudaGetLastError();
}

cudaError_t launch_ln_param_partial(bool bf16, const float* dXn, const void* X,
                                    const float* mean, const float* rstd,
                                    float* part_g, float* part_b, int rows,
                                    int h, cudaStream_t stream) {
  const dim3 grid((h + CS_COLS - 1) / CS_COLS, colsum_chunks(rows));
  if (bf16 && h % 8 == 0 &&
      (reinterpret_cast<uintptr_t>(X) & 15u) == 0 &&
      (reinterpret_cast<uintptr_t>(dXn) & 15u) == 0) {
    const dim3 grid8((h + CS8_COLS - 1) / CS8_COLS, colsum_chunks(rows));
    ln_param_partial_bf16x8_kernel<<<grid8, CS_WARPS * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(X), dXn, mean, rstd, part_g, part_b,
        rows, h);
  } else if (bf16) {
    colsum_partial_kernel<__nv_bfloat16, 1><<<grid, CS_WARPS * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(X), dXn, mean, rstd, part_g, part_b,
        rows, h, nullptr);
  } else {
    colsum_partial_kernel<float, 1><<<grid, CS_WARPS * 32, 0, stream>>>(
        static_cast<const float*>(X), dXn, mean, rstd, part_g, part_b, rows,
        h, nullptr);
  }
  return cudaGetLastError();
}

cudaError_t launch_colsum_finalize(const float* part, float* out, int chunks,
                                   int cols, cudaStream_t stream) {
  if (cols <= 0) return cudaSuccess;
  colsum_finalize_kernel<<<(cols + 31) / 32, dim3(32, 8), 0, stream>>>(
      part, out, chunks, cols);
  return cudaGetLastError();
}

}  // namespace tpmlp
