// Per-tensor E4M3 scaling for the FP8 forward of the MLP block: the current
// maximum magnitude of a bf16 tensor, and quantization with the scale it
// gives (s = amax / 448 in fp32, q = e4m3(x / s), nearest-even rounding with
// saturation to +-448), in the plain layout, transposed, or both at once.  A maximum does not depend on the order its inputs
// are combined in, so the fp32-bit atomicMax keeps the result deterministic.
// All three kernels are HBM-bound streaming passes with 16-byte loads.
#include <cuda_fp8.h>

#include "internal.h"

namespace tpmlp {
namespace {

constexpr int QT = 256;          // threads per block
constexpr float E4M3_MAX = 448.f;

__device__ __forceinline__ float scale_from_amax(unsigned int bits) {
  const float amax = __uint_as_float(bits);
  return amax > 0.f ? __fdiv_rn(amax, E4M3_MAX) : 1.f;
}

__device__ __forceinline__ uint8_t to_e4m3(float x, float s) {
  return static_cast<uint8_t>(
      __nv_cvt_float_to_fp8(__fdiv_rn(x, s), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float absmax8(const uint4 u, float mx) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float a, b;
    unpack_bf16x2(w[k], a, b);
    mx = fmaxf(mx, fmaxf(fabsf(a), fabsf(b)));
  }
  return mx;
}

// 8 bf16 values per 16-byte load, four independent loads in flight per
// thread; one atomic per block after a block-wide maximum.
__global__ void __launch_bounds__(QT)
    amax_bf16_kernel(const uint4* __restrict__ x, size_t n8,
                     const __nv_bfloat16* __restrict__ tail, int ntail,
                     unsigned int* amax) {
  __shared__ unsigned int wmax[QT / 32];
  float mx = 0.f;
  const size_t stride = size_t(gridDim.x) * QT;
  size_t i = blockIdx.x * size_t(QT) + threadIdx.x;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    const uint4 u0 = x[i], u1 = x[i + stride], u2 = x[i + 2 * stride],
                u3 = x[i + 3 * stride];
    mx = absmax8(u0, mx);
    mx = absmax8(u1, mx);
    mx = absmax8(u2, mx);
    mx = absmax8(u3, mx);
  }
  for (; i < n8; i += stride) mx = absmax8(x[i], mx);
  if (blockIdx.x == 0 && threadIdx.x < ntail)
    mx = fmaxf(mx, fabsf(__bfloat162float(tail[threadIdx.x])));
  const unsigned int wm = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = wm;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned int m = 0;
#pragma unroll
    for (int k = 0; k < QT / 32; ++k) m = m > wmax[k] ? m : wmax[k];
    atomicMax(amax, m);
  }
}

// Eight bf16 values (one 16-byte load) to eight E4M3 codes (8 bytes).
__device__ __forceinline__ uint2 e4m3x8(const uint4 u, float s) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t o[2] = {0u, 0u};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float a, b;
    unpack_bf16x2(w[k], a, b);
    const uint32_t pair = uint32_t(to_e4m3(a, s)) | (uint32_t(to_e4m3(b, s)) << 8);
    o[k >> 1] |= pair << (16 * (k & 1));
  }
  return make_uint2(o[0], o[1]);
}

__global__ void quantize_kernel(const uint4* __restrict__ x, size_t n8,
                                const __nv_bfloat16* __restrict__ tail,
                                int ntail, const unsigned int* __restrict__ amax,
                                uint2* __restrict__ q, uint8_t* __restrict__ qtail,
                                float* scale_out) {
  const float s = scale_from_amax(*amax);
  if (blockIdx.x == 0 && threadIdx.x == 0 && scale_out != nullptr)
    *scale_out = s;
  const size_t stride = size_t(gridDim.x) * QT;
  size_t i = blockIdx.x * size_t(QT) + threadIdx.x;
  // two independent 16-byte loads in flight per thread
  for (; i + stride < n8; i += 2 * stride) {
    const uint4 u0 = x[i], u1 = x[i + stride];
    q[i] = e4m3x8(u0, s);
    q[i + stride] = e4m3x8(u1, s);
  }
  for (; i < n8; i += stride) q[i] = e4m3x8(x[i], s);
  if (blockIdx.x == 0 && threadIdx.x < ntail)
    qtail[threadIdx.x] = to_e4m3(__bfloat162float(tail[threadIdx.x]), s);
}

// x [rows, cols] bf16 -> qt [cols, ld_t] E4M3 (element (r, c) at
// qt[c * ld_t + r]) and, when q_row is not null, also q_row [rows, cols]
// (the plain layout), from one read of x: 64 x 64 tiles through shared
// memory (coalesced 16-byte reads, 8-byte writes).
__global__ void __launch_bounds__(QT)
    quantize_t_kernel(const __nv_bfloat16* __restrict__ x, int rows, int cols,
                      const unsigned int* __restrict__ amax,
                      uint8_t* __restrict__ qt, long long ld_t,
                      uint8_t* __restrict__ q_row, float* scale_out) {
  __shared__ uint8_t tile[64][64 + 8];
  const float s = scale_from_amax(*amax);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 &&
      scale_out != nullptr)
    *scale_out = s;
  const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
  const bool vec_in = (cols & 7) == 0;
  // load: 64 rows x 8 chunks of 8 columns; 256 threads, 2 chunks each
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int t = threadIdx.x + it * QT;
    const int r = t >> 3, ch = t & 7;
    const int gr = r0 + r, gc = c0 + ch * 8;
    uint8_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (gr < rows) {
      const size_t base = static_cast<size_t>(gr) * cols + gc;
      if (gc + 8 <= cols && vec_in) {
        const uint4 u = *reinterpret_cast<const uint4*>(x + base);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float a, b;
          unpack_bf16x2(w[k], a, b);
          v[2 * k] = to_e4m3(a, s);
          v[2 * k + 1] = to_e4m3(b, s);
        }
        if (q_row != nullptr) {
          uint2 o;
          o.x = uint32_t(v[0]) | (uint32_t(v[1]) << 8) | (uint32_t(v[2]) << 16) |
                (uint32_t(v[3]) << 24);
          o.y = uint32_t(v[4]) | (uint32_t(v[5]) << 8) | (uint32_t(v[6]) << 16) |
                (uint32_t(v[7]) << 24);
          *reinterpret_cast<uint2*>(q_row + base) = o;
        }
      } else {
        for (int k = 0; k < 8 && gc + k < cols; ++k) {
          v[k] = to_e4m3(__bfloat162float(x[base + k]), s);
          if (q_row != nullptr) q_row[base + k] = v[k];
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) tile[ch * 8 + k][r] = v[k];
  }
  __syncthreads();
  // store: 64 output rows (input columns) x 8 chunks of 8 bytes
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int t = threadIdx.x + it * QT;
    const int oc = t >> 3, ch = t & 7;
    const int grow = c0 + oc, gcol = r0 + ch * 8;
    if (grow >= cols) continue;
    uint8_t* dst = qt + static_cast<size_t>(grow) * ld_t + gcol;
    if (gcol + 8 <= rows && (reinterpret_cast<uintptr_t>(dst) & 7u) == 0) {
      *reinterpret_cast<uint2*>(dst) =
          *reinterpret_cast<const uint2*>(&tile[oc][ch * 8]);
    } else {
      for (int k = 0; k < 8 && gcol + k < rows; ++k) dst[k] = tile[oc][ch * 8 + k];
    }
  }
}

int stream_blocks(size_t n8) {
  const size_t b = (n8 + QT - 1) / QT;
  return static_cast<int>(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

}  // namespace

cudaError_t launch_amax_bf16(const void* x, size_t n, unsigned int* amax,
                             cudaStream_t s) {
  const size_t n8 = n / 8;
  const int ntail = static_cast<int>(n - n8 * 8);
  // about eight resident blocks per SM, each thread four loads deep
  const size_t want = (n8 + 4 * QT - 1) / (4 * QT);
  const int blocks = static_cast<int>(want < 1216 ? (want > 0 ? want : 1) : 1216);
  amax_bf16_kernel<<<blocks, QT, 0, s>>>(
      static_cast<const uint4*>(x), n8,
      static_cast<const __nv_bfloat16*>(x) + n8 * 8, ntail, amax);
  return cudaGetLastError();
}

cudaError_t launch_quantize_e4m3(const void* x, size_t n,
                                 const unsigned int* amax, uint8_t* q,
                                 float* scale_out, cudaStream_t s) {
  const size_t n8 = n / 8;
  const int ntail = static_cast<int>(n - n8 * 8);
  quantize_kernel<<<stream_blocks(n8), QT, 0, s>>>(
      static_cast<const uint4*>(x), n8,
      static_cast<const __nv_bfloat16*>(x) + n8 * 8, ntail, amax,
      reinterpret_cast<uint2*>(q), q + n8 * 8, scale_out);
  return cudaGetLastError();
}

cudaError_t launch_quantize_e4m3_rt(const void* x, int rows, int cols,
                                    const unsigned int* amax, uint8_t* q_row,
                                    uint8_t* qt, long long ld_t,
                                    float* scale_out, cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  if (ld_t < rows) return cudaErrorInvalidValue;
  const dim3 grid((cols + 63) / 64, (rows + 63) / 64);
  quantize_t_kernel<<<grid, QT, 0, s>>>(static_cast<const __nv_bfloat16*>(x),
                                        rows, cols, amax, qt, ld_t, q_row,
                                        scale_out);
  return cudaGetLastError();
}

}  // namespace tpmlp
