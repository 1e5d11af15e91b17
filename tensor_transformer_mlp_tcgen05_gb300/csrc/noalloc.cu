// Bias gradient (column sums over tokens) for callers that cannot allocate
// device memory.  The regular tp_mlp_backward takes its partial-sum scratch
// from the caller's workspace; this entry point keeps it in a fixed,
// file-scope device array instead, so the caller passes only the input and
// the output.  It reuses the same two fixed-order kernels (per-chunk partial
// sums, then the chunk partials added in chunk order), so its result is
// bit-identical to the db2 that tp_mlp_backward produces (and to its db1 in
// the fp32 configuration; the bf16 db1 there comes from the dH GEMM's
// 32-row partials instead).
#include <cstdio>
#include <mutex>

#include "internal.h"

// Partial-sum scratch shared by every call in the process.  It lives on every
// GPU that loads the library until the process exits.
static __device__ __align__(256) float g_colsum_scratch[TPMLP_NOALLOC_SCRATCH_FLOATS];

namespace {

constexpr int kMaxDevices = 64;

// Device address of g_colsum_scratch on the current device, looked up once
// per device (with that device current) and cached.  In host code the
// array's name is only a host-side stand-in, never a device address.
int scratch_for_current_device(float** out) {
  static std::mutex mu;
  static float* addr[kMaxDevices] = {nullptr};
  static int state[kMaxDevices] = {0};  // 0 unknown, 1 ready, -1 not sm_103
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    tpmlp::set_last_detail("tp_mlp_bias_grad_noalloc: cudaGetDevice failed");
    return TPMLP_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return TPMLP_ERR_ARCH;
  std::lock_guard<std::mutex> lock(mu);
  if (state[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor,
                               dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor,
                               dev) != cudaSuccess) {
      tpmlp::set_last_detail(
          "tp_mlp_bias_grad_noalloc: cudaDeviceGetAttribute failed");
      return TPMLP_ERR_CUDA;
    }
    if (major != 10 || minor != 3) {
      state[dev] = -1;
    } else {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_colsum_scratch);
      if (e != cudaSuccess || p == nullptr) {
        char msg[256];
        std::snprintf(msg, sizeof(msg),
                      "tp_mlp_bias_grad_noalloc: cudaGetSymbolAddress of the "
                      "static scratch failed: %s",
                      cudaGetErrorString(e));
        tpmlp::set_last_detail(msg);
        return TPMLP_ERR_CUDA;
      }
      addr[dev] = static_cast<float*>(p);
      state[dev] = 1;
    }
  }
  if (state[dev] < 0) {
    tpmlp::set_last_detail(
        "tp_mlp_bias_grad_noalloc: the current device is not sm_103");
    return TPMLP_ERR_ARCH;
  }
  *out = addr[dev];
  return TPMLP_OK;
}

}  // namespace

extern "C" int tp_mlp_bias_grad_noalloc(int tokens, int cols, int dtype,
                                        const void* grad, float* dbias,
                                        void* stream) {
  if (dtype != TPMLP_BF16 && dtype != TPMLP_FP32) return TPMLP_ERR_ARG;
  if (dbias == nullptr || (tokens > 0 && grad == nullptr)) return TPMLP_ERR_ARG;
  if (tokens < 0 || cols <= 0 || cols % 64 != 0) return TPMLP_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(grad) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(dbias) & 15u) != 0)
    return TPMLP_ERR_ALIGN;
  const int chunks = tpmlp::colsum_chunks(tokens);
  if (static_cast<long long>(chunks) * cols > TPMLP_NOALLOC_SCRATCH_FLOATS) {
    char msg[256];
    std::snprintf(msg, sizeof(msg),
                  "tp_mlp_bias_grad_noalloc: %d tokens x %d columns need %lld "
                  "partial sums; the static scratch holds %d "
                  "(ceil(tokens / %d) * cols must not exceed it)",
                  tokens, cols, static_cast<long long>(chunks) * cols,
                  TPMLP_NOALLOC_SCRATCH_FLOATS, tpmlp::COLSUM_CHUNK_ROWS);
    tpmlp::set_last_detail(msg);
    return TPMLP_ERR_SHAPE;
  }
  float* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != TPMLP_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (tokens == 0) {  // the sum over no tokens
    e = cudaMemsetAsync(dbias, 0, static_cast<size_t>(cols) * sizeof(float), s);
  } else {
    // Stage 1 writes every partial that stage 2 reads, so nothing in the
    // scratch has to start at zero.
    const bool bf16 = dtype == TPMLP_BF16;
    e = tpmlp::launch_colsum_partial(bf16, grad, scratch, tokens, cols, s);
    if (e == cudaSuccess)
      e = tpmlp::launch_colsum_finalize(scratch, dbias, chunks, cols, s);
  }
  if (e != cudaSuccess) {
    char msg[256];
    std::snprintf(msg, sizeof(msg), "tp_mlp_bias_grad_noalloc: %s",
                  cudaGetErrorString(e));
    tpmlp::set_last_detail(msg);
    return TPMLP_ERR_CUDA;
  }
  return TPMLP_OK;
}
