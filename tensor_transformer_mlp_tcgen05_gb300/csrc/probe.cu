// Tensor-core issue-rate calibration: one thread per CTA issues back-to-back
// tcgen05.mma (M = 128, N, K = 16, bf16 operands from shared memory with
// precomputed descriptors, fp32 accumulator in TMEM) and the CTA records the
// SM clock cycles from the first issue to the completion of the last.  With
// one CTA per SM this measures the per-SM dense bf16 rate (flops per cycle)
// that a clock-based peak (SMs x rate x clock) assumes.  The operands are a
// fixed pseudo-random bf16 pattern; the accumulator is never read.
#include "internal.h"
#include "ptx.cuh"

namespace tpmlp {
namespace {

constexpr int PROBE_THREADS = 128;
// 120 KB keeps one CTA (one issuing thread) per SM.
constexpr uint32_t PROBE_SMEM = 120 * 1024;

template <int N>
__global__ void __launch_bounds__(PROBE_THREADS, 1)
    mma_rate_kernel(int n_mma, unsigned long long* cycles, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar;
  __shared__ uint32_t slot;
  // A: 128 rows x 128 B, B: N rows x 128 B (one 64-element k-block each)
  for (int i = threadIdx.x; i < 65536 / 16; i += PROBE_THREADS) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t x = static_cast<uint32_t>(i * 4 + j) * 2654435761u + 12345u;
      x ^= x >> 13;
      x *= 0x5bd1e995u;
      x ^= x >> 15;
      // two bf16 in [-2, 2): sign, exponent 127, random 7-bit mantissa
      const uint32_t lo = 0x3F80u | (x & 0x7Fu) | ((x & 0x100u) << 7);
      const uint32_t hi = 0x3F80u | ((x >> 16) & 0x7Fu) | (((x >> 24) & 1u) << 15);
      w[j] = lo | (hi << 16);
    }
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  const uint32_t b = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    ptx::fence_barrier_init();
  }
  if (threadIdx.x < 32) {
    ptx::tmem_alloc(ptx::smem_u32(&slot), 256);
    ptx::tmem_relinquish();
  }
  ptx::fence_proxy_async_shared();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = slot;
  if (threadIdx.x == 0) {
    const uint32_t sa = ptx::smem_u32(smem), sb = sa + 16384;
    constexpr uint32_t ID = idesc_bf16_f32(128, N, false, false);
    const uint64_t da = ptx::sdesc_sw128(sa, 16, 1024);
    const uint64_t db = ptx::sdesc_sw128(sb, 16, 1024);
    const long long t0 = clock64();
    for (int i = 0; i < n_mma; i += 4) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        ptx::mma_bf16(tmem, da + ((32 * k) >> 4), db + ((32 * k) >> 4), ID,
                      (i > 0 || k > 0) ? 1u : 0u);
    }
    ptx::mma_commit(b);
    const uint64_t g0 = ptx::globaltimer_ns();
    bool ok = true;
    while (!ptx::mbar_try_wait(b, 0)) {
      if (ptx::globaltimer_ns() - g0 > 1000000000ull) {
        ok = false;
        break;
      }
    }
    cycles[blockIdx.x] = static_cast<unsigned long long>(clock64() - t0);
    if (!ok) atomicExch(status, TPMLP_ERR_TIMEOUT);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 256);
  }
}

template <int N>
cudaError_t launch_probe(int ctas, int n_mma, unsigned long long* cycles,
                         int* status, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(mma_rate_kernel<N>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(PROBE_SMEM));
  if (e != cudaSuccess) return e;
  mma_rate_kernel<N><<<ctas, PROBE_THREADS, PROBE_SMEM, s>>>(n_mma, cycles,
                                                             status);
  return cudaGetLastError();
}

__global__ void gelu_probe_kernel(const float* __restrict__ x,
                                  float* __restrict__ y,
                                  float* __restrict__ dy, int n, int mode) {
  // pairs, as the GEMM epilogues evaluate them
  for (int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x); i < n;
       i += 2 * gridDim.x * blockDim.x) {
    const bool two = i + 1 < n;
    float a = x[i], b = two ? x[i + 1] : 0.f;
    float ga, gb;
    gelu_grad2_f32(a, b, ga, gb, mode);
    gelu2_f32(a, b, mode);
    y[i] = a;
    dy[i] = ga;
    if (two) {
      y[i + 1] = b;
      dy[i + 1] = gb;
    }
  }
}

}  // namespace
}  // namespace tpmlp

extern "C" int tp_mlp_probe_gelu(const float* x, float* y, float* dy, int n,
                                 int mode, void* stream) {
  using namespace tpmlp;
  if (n < 0 || (n > 0 && (x == nullptr || y == nullptr || dy == nullptr)) ||
      (mode != TPMLP_GELU_ERF && mode != TPMLP_GELU_TANH))
    return TPMLP_ERR_ARG;
  if (n == 0) return TPMLP_OK;
  const int blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
  gelu_probe_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      x, y, dy, n, mode);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_detail(cudaGetErrorString(e));
    return TPMLP_ERR_CUDA;
  }
  return TPMLP_OK;
}

extern "C" int tp_mlp_probe_mma_cycles(int n, int ctas, int n_mma,
                                       unsigned long long* cycles,
                                       int* status, void* stream) {
  using namespace tpmlp;
  if (cycles == nullptr || status == nullptr || ctas <= 0 || n_mma <= 0 ||
      n_mma % 4 != 0 || n_mma > (1 << 24))
    return TPMLP_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (n == 64)
    e = launch_probe<64>(ctas, n_mma, cycles, status, s);
  else if (n == 128)
    e = launch_probe<128>(ctas, n_mma, cycles, status, s);
  else if (n == 256)
    e = launch_probe<256>(ctas, n_mma, cycles, status, s);
  else
    return TPMLP_ERR_SHAPE;
  if (e != cudaSuccess) {
    set_last_detail(cudaGetErrorString(e));
    return TPMLP_ERR_CUDA;
  }
  return TPMLP_OK;
}
