// Per-tensor E4M3 scaling for the FP8 variant of the MLP block: the
// current maximum magnitude of a bf16 tensor, and quantization with the
// scale it gives (s = amax / 448 in fp32, q = e4m3(x / s) with x / s the
// correctly rounded fp32 quotient, then nearest-even rounding with
// saturation to +-448), in the plain layout, transposed, or both at once.
// A maximum does not depend on the order its inputs are combined in, so the
// fp32-bit atomicMax keeps the result deterministic.  All kernels are
// HBM-bound streaming passes with 16-byte loads.
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

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

// Quantization by table.  The code of x is e4m3(fp32(x / s)): a function of
// x's bf16 bit pattern alone, odd in the sign (E4M3 is sign-magnitude and
// its rounding and saturation are symmetric).  Every magnitude that can
// give a nonzero code lies within QTAB_E binades below amax: |x| under
// 2^(1 - QTAB_E) amax gives |x / s| < 448 * 2^-21 < 2^-10, half the smallest
// E4M3 subnormal, hence code 0.  So each block computes the codes of those
// QTAB_E * 128 magnitudes once (the same IEEE division as above) into a
// shared-memory table, and then quantizes with one clamp and one byte
// load per value.  When that range would reach the bf16 subnormals (amax
// below 2^-105) or amax is 0, every value takes the division instead.
constexpr int QTAB_E = 22;
// entries 0 .. QTAB_E * 128 - 1: the magnitudes from 2^(e_amax - 21) up;
// the last entry, code 0, takes every magnitude outside that range
constexpr int QTAB_N = QTAB_E * 128 + 1;

struct Quantizer {
  uint32_t tab;         // shared-memory address of the QTAB_N codes
  uint32_t base;        // index = (bits & 0x7fff) - base, unsigned, clamped
  float s;
  bool use_tab;
};

// Called by every thread of the block; ends with a block barrier.
__device__ __forceinline__ Quantizer make_quantizer(uint8_t* tab,
                                                    unsigned int amax_bits) {
  const float s = scale_from_amax(amax_bits);
  const int e_lo = static_cast<int>((amax_bits >> 23) & 0xFFu) - (QTAB_E - 1);
  const Quantizer z{ptx::smem_u32(tab), static_cast<uint32_t>(e_lo) << 7, s,
                    amax_bits != 0u && e_lo >= 1};
  if (z.use_tab) {
    for (int i = threadIdx.x; i < QTAB_N; i += blockDim.x) {
      uint8_t code = 0;
      if (i < QTAB_N - 1)
        code = to_e4m3(__uint_as_float((z.base + static_cast<uint32_t>(i)) << 16), s);
      tab[i] = code;
    }
  }
  __syncthreads();
  return z;
}

__device__ __forceinline__ uint32_t ld_shared_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Two bf16 values (one word) to two codes in the low 16 bits, the first
// value lowest.  A magnitude below the table's range wraps around in the
// unsigned subtraction and lands, like one above it, on the last entry.
__device__ __forceinline__ uint32_t q_pair(const Quantizer& z, uint32_t w) {
  if (z.use_tab) {
    const uint32_t tlo = min((w & 0x7FFFu) - z.base, uint32_t(QTAB_N - 1));
    const uint32_t thi = min(((w >> 16) & 0x7FFFu) - z.base, uint32_t(QTAB_N - 1));
    // the two sign bits, moved to bits 7 and 15
    const uint32_t signs = __byte_perm(w, 0u, 0x4431u) & 0x8080u;
    return ld_shared_u8(z.tab + tlo) | (ld_shared_u8(z.tab + thi) << 8) | signs;
  }
  float a, b;
  unpack_bf16x2(w, a, b);
  return __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(a, z.s), __fdiv_rn(b, z.s)),
                                  __NV_SATFINITE, __NV_E4M3);
}

// Eight bf16 values (one 16-byte load) to eight E4M3 codes (8 bytes, the
// first value lowest).
__device__ __forceinline__ uint2 e4m3x8(const uint4 u, const Quantizer& z) {
  return make_uint2(q_pair(z, u.x) | (q_pair(z, u.y) << 16),
                    q_pair(z, u.z) | (q_pair(z, u.w) << 16));
}

__global__ void __launch_bounds__(QT)
    quantize_kernel(const uint4* __restrict__ x, size_t n8,
                    const __nv_bfloat16* __restrict__ tail, int ntail,
                    const unsigned int* __restrict__ amax,
                    uint2* __restrict__ q, uint8_t* __restrict__ qtail,
                    float* scale_out) {
  __shared__ uint8_t tab[QTAB_N];
  const Quantizer z = make_quantizer(tab, *amax);
  if (blockIdx.x == 0 && threadIdx.x == 0 && scale_out != nullptr)
    *scale_out = z.s;
  const size_t stride = size_t(gridDim.x) * QT;
  size_t i = blockIdx.x * size_t(QT) + threadIdx.x;
  // two independent 16-byte loads in flight per thread
  for (; i + stride < n8; i += 2 * stride) {
    const uint4 u0 = x[i], u1 = x[i + stride];
    q[i] = e4m3x8(u0, z);
    q[i + stride] = e4m3x8(u1, z);
  }
  for (; i < n8; i += stride) q[i] = e4m3x8(x[i], z);
  if (blockIdx.x == 0 && threadIdx.x < ntail)
    qtail[threadIdx.x] = to_e4m3(__bfloat162float(tail[threadIdx.x]), z.s);
}

// 4 x 4 byte transpose: t[b] = (a0.b, a1.b, a2.b, a3.b).
__device__ __forceinline__ void transpose4x4(uint32_t a0, uint32_t a1,
                                             uint32_t a2, uint32_t a3,
                                             uint32_t t[4]) {
  const uint32_t x0 = __byte_perm(a0, a1, 0x5140), x1 = __byte_perm(a0, a1, 0x7362);
  const uint32_t y0 = __byte_perm(a2, a3, 0x5140), y1 = __byte_perm(a2, a3, 0x7362);
  t[0] = __byte_perm(x0, y0, 0x5410);
  t[1] = __byte_perm(x0, y0, 0x7632);
  t[2] = __byte_perm(x1, y1, 0x5410);
  t[3] = __byte_perm(x1, y1, 0x7632);
}

// x [rows, cols] bf16 -> qt [cols, ld_t] E4M3 (element (r, c) at
// qt[c * ld_t + r]) and, when q_row is not null, also q_row [rows, cols]
// (the plain layout), from one read of x.  Persistent blocks walk 128 x 128
// tiles: sixteen lanes read a row's 256 bytes (16 a lane) and write its
// codes to q_row and to a shared-memory tile of codes; then each lane
// gathers an 8-row x 4-column block of codes (eight words), transposes it
// with byte permutes and writes four 8-byte column pieces, sixteen lanes
// covering a column's 128 contiguous bytes (one full line).  A thread's
// loads for the next tile are in flight during this tile's transposed
// phase.  The tile's
// words are XOR-swizzled by row group so that the gathers are free of bank
// conflicts: word w of row r sits at w ^ (2 * ((r / 8) % 16)).
constexpr int QTR_ROWS = 128, QTR_COLS = 128;
constexpr int QTR_WORDS = QTR_COLS / 4;        // words per tile row
constexpr int QTR_LPR = QTR_COLS / 8;          // lanes per row in the load
constexpr int QTR_GROUPS = QTR_ROWS / 8;       // 8-row groups
__device__ __forceinline__ int qtr_swz(int r, int w) {
  return r * QTR_WORDS + (w ^ (((r >> 3) & (QTR_GROUPS - 1)) << 1));
}

__global__ void __launch_bounds__(QT, 4)
    quantize_t_kernel(const __nv_bfloat16* __restrict__ x, int rows, int cols,
                      const unsigned int* __restrict__ amax,
                      uint8_t* __restrict__ qt, long long ld_t,
                      uint8_t* __restrict__ q_row, float* scale_out) {
  __shared__ __align__(16) uint32_t tile[QTR_ROWS * QTR_WORDS];   // 16 KB
  __shared__ uint8_t tab[QTAB_N];
  const Quantizer z = make_quantizer(tab, *amax);
  if (blockIdx.x == 0 && threadIdx.x == 0 && scale_out != nullptr)
    *scale_out = z.s;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool vec = (cols & 7) == 0;
  const int ntx = (cols + QTR_COLS - 1) / QTR_COLS;
  const int ntiles = ntx * ((rows + QTR_ROWS - 1) / QTR_ROWS);
  // load phase: lane = column chunk lc + QTR_LPR * rsub; a warp takes two
  // rows per load, the block sixteen; transposed phase: lane = row group g
  // + QTR_GROUPS * wsub
  const int lc = lane % QTR_LPR, rsub = lane / QTR_LPR;
  const int g = lane % QTR_GROUPS, wsub = lane / QTR_GROUPS;
  // The next tile's eight 16-byte loads per thread are issued before this
  // tile's transposed phase, so they stay in flight across it.
  uint4 u[8];
  auto load_tile = [&](int ti) {
    const int r0 = (ti / ntx) * QTR_ROWS, c = (ti % ntx) * QTR_COLS + lc * 8;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int r = r0 + 16 * k + 2 * warp + rsub;
      u[k] = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows && vec && c + 8 <= cols)
        u[k] = *reinterpret_cast<const uint4*>(x + static_cast<size_t>(r) * cols + c);
    }
  };
  if (static_cast<int>(blockIdx.x) < ntiles) load_tile(blockIdx.x);
  for (int tile_i = blockIdx.x; tile_i < ntiles; tile_i += gridDim.x) {
    const int r0 = (tile_i / ntx) * QTR_ROWS, c0 = (tile_i % ntx) * QTR_COLS;
    const int c = c0 + lc * 8;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int rl = 16 * k + 2 * warp + rsub, r = r0 + rl;
      uint2 o;
      if (vec || r >= rows) {
        o = e4m3x8(u[k], z);
      } else {  // columns not a multiple of 8: element by element
        uint32_t w2[2] = {0u, 0u};
        for (int j = 0; j < 8 && c + j < cols; ++j)
          w2[j >> 2] |= uint32_t(to_e4m3(
                            __bfloat162float(x[static_cast<size_t>(r) * cols + c + j]),
                            z.s))
                        << (8 * (j & 3));
        o = make_uint2(w2[0], w2[1]);
      }
      *reinterpret_cast<uint2*>(&tile[qtr_swz(rl, 2 * lc)]) = o;
      if (q_row != nullptr && r < rows) {
        uint8_t* dst = q_row + static_cast<size_t>(r) * cols + c;
        if (vec && c + 8 <= cols) {
          *reinterpret_cast<uint2*>(dst) = o;
        } else {
          for (int j = 0; j < 8 && c + j < cols; ++j)
            dst[j] = static_cast<uint8_t>((j < 4 ? o.x : o.y) >> (8 * (j & 3)));
        }
      }
    }
    if (tile_i + static_cast<int>(gridDim.x) < ntiles)
      load_tile(tile_i + gridDim.x);
    __syncthreads();
    // ---- transposed: each warp covers 2 words (8 columns) x 128 rows per
    // pass, 2 passes
    const int rl = 8 * g, r = r0 + rl;
    const bool full_rows = r + 8 <= rows && (ld_t & 7) == 0;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const int w = 2 * (pass * 8 + warp) + wsub;   // word: columns 4w..4w+3
      if (r >= rows || c0 + 4 * w >= cols) continue;
      uint32_t lo[4], hi[4];
      transpose4x4(tile[qtr_swz(rl + 0, w)], tile[qtr_swz(rl + 1, w)],
                   tile[qtr_swz(rl + 2, w)], tile[qtr_swz(rl + 3, w)], lo);
      transpose4x4(tile[qtr_swz(rl + 4, w)], tile[qtr_swz(rl + 5, w)],
                   tile[qtr_swz(rl + 6, w)], tile[qtr_swz(rl + 7, w)], hi);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int cc = c0 + 4 * w + b;
        if (cc >= cols) break;
        uint8_t* dst = qt + static_cast<size_t>(cc) * ld_t + r;
        if (full_rows) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(lo[b], hi[b]);
        } else {
          for (int i = 0; i < 8 && r + i < rows; ++i)
            dst[i] = static_cast<uint8_t>((i < 4 ? lo[b] : hi[b]) >> (8 * (i & 3)));
        }
      }
    }
    __syncthreads();   // the tile is rewritten by the next iteration
  }
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
          cudaSuccess || n <= 0)
    return 152;
  return n;
}

// Persistent grids: every block builds its code table once.
int stream_blocks(size_t n8) {
  const size_t cap = static_cast<size_t>(num_sms()) * 8;
  const size_t b = (n8 + 2 * QT - 1) / (2 * QT);
  return static_cast<int>(b < cap ? (b > 0 ? b : 1) : cap);
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
  const long long tiles = static_cast<long long>((cols + QTR_COLS - 1) / QTR_COLS) *
                          ((rows + QTR_ROWS - 1) / QTR_ROWS);
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  const long long cap = static_cast<long long>(num_sms()) * 4;
  const int grid = static_cast<int>(tiles < cap ? tiles : cap);
  quantize_t_kernel<<<grid, QT, 0, s>>>(static_cast<const __nv_bfloat16*>(x),
                                        rows, cols, amax, qt, ld_t, q_row,
                                        scale_out);
  return cudaGetLastError();
}

}  // namespace tpmlp
