// Host-side helpers shared by the C-ABI files of libtpmlp: error details,
// device checks, TMA tensor-map encoding, per-launch timing and the GEMM /
// column-sum launch wrappers.  Header-only (inline), one copy per program.
#pragma once
#include <nvtx3/nvToolsExt.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "internal.h"

namespace tpmlp {
namespace host {

// Launch bookkeeping every handle carries: wait budget, launch count and the
// optional per-kernel timing events.
struct HandleCore {
  unsigned long long budget_ns = 2000000000ull;
  long long launches = 0;
  bool timing = false;
  bool nvtx = false;  // an NVTX range, named for the kernel, around each launch
  struct Pending {
    int stat;
    cudaEvent_t a, b;
  };
  struct Stat {
    const char* name;
    long long n;
    double ms;
  };
  std::vector<Pending> pending;
  std::vector<cudaEvent_t> spare;
  std::vector<Stat> stats;

  ~HandleCore() {
    for (auto& p : pending) {
      cudaEventDestroy(p.a);
      cudaEventDestroy(p.b);
    }
    for (auto e : spare) cudaEventDestroy(e);
  }
};

inline thread_local char g_detail[512] = "";

inline void set_detail(const char* what, cudaError_t e) {
  std::snprintf(g_detail, sizeof(g_detail), "%s: %s (%d)", what,
                cudaGetErrorString(e), static_cast<int>(e));
}

inline void set_detail_msg(const char* msg) {
  std::snprintf(g_detail, sizeof(g_detail), "%s", msg);
}

// ---------------------------------------------------- workspace layout --

inline int check_device(int* num_sms) {
  static std::mutex mu;
  static int sms[64] = {0};
  static int ok[64] = {0};  // 0 unknown, 1 good, -1 bad
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_detail("cudaGetDevice", e);
    return TPMLP_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return TPMLP_ERR_ARCH;
  std::lock_guard<std::mutex> lock(mu);
  if (ok[dev] == 0) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor,
                               dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor,
                               dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess) {
      set_detail_msg("cudaDeviceGetAttribute failed");
      return TPMLP_ERR_CUDA;
    }
    ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    sms[dev] = n;
    if (ok[dev] < 0) {
      std::snprintf(g_detail, sizeof(g_detail),
                    "device %d is compute capability %d.%d; libtpmlp is built "
                    "for sm_103a only",
                    dev, major, minor);
    }
  }
  if (ok[dev] < 0) return TPMLP_ERR_ARCH;
  *num_sms = sms[dev];
  return TPMLP_OK;
}

// ----------------------------------------------------------- tensor maps --

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                  void*, const cuuint64_t*, const cuuint64_t*,
                                  const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
    }
  });
  return fn;
}

// Row-major matrix [outer, inner] (inner contiguous, pitch in elements) of
// bf16 or fp32, 128-byte swizzle, box = {box_inner, box_outer} elements.
inline int encode_map_t(CUtensorMap* m, const void* base, bool f32, uint64_t inner,
                 uint64_t outer, uint64_t pitch, uint32_t box_inner,
                 uint32_t box_outer) {
  EncodeTiledFn enc = get_encoder();
  if (enc == nullptr) {
    set_detail_msg("cuTensorMapEncodeTiled entry point not available");
    return TPMLP_ERR_CUDA;
  }
  const uint64_t es = f32 ? 4 : 2;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {pitch * es};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
          2, const_cast<void*>(base), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_detail, sizeof(g_detail),
                  "cuTensorMapEncodeTiled failed (%d): inner=%llu outer=%llu "
                  "pitch=%llu box=%ux%u",
                  static_cast<int>(r), (unsigned long long)inner,
                  (unsigned long long)outer, (unsigned long long)pitch,
                  box_inner, box_outer);
    return TPMLP_ERR_CUDA;
  }
  return TPMLP_OK;
}

// 8-bit operand [outer, inner] (pitch in bytes), 128-byte swizzle, box =
// {128 inner bytes (one swizzle row), box_outer}.
inline int encode_map_u8(CUtensorMap* m, const void* base, uint64_t inner,
                         uint64_t outer, uint64_t pitch, uint32_t box_outer) {
  EncodeTiledFn enc = get_encoder();
  if (enc == nullptr) {
    set_detail_msg("cuTensorMapEncodeTiled entry point not available");
    return TPMLP_ERR_CUDA;
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {128, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                         const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_detail, sizeof(g_detail),
                  "cuTensorMapEncodeTiled (u8) failed (%d): inner=%llu "
                  "outer=%llu pitch=%llu",
                  static_cast<int>(r), (unsigned long long)inner,
                  (unsigned long long)outer, (unsigned long long)pitch);
    return TPMLP_ERR_CUDA;
  }
  return TPMLP_OK;
}

// bf16 operand: box = {64 inner elements (one 128-byte swizzle row), box_outer}.
inline int encode_map(CUtensorMap* m, const void* base, uint64_t inner,
               uint64_t outer, uint64_t pitch, uint32_t box_outer) {
  return encode_map_t(m, base, false, inner, outer, pitch, 64, box_outer);
}

// GEMM output [rows, cols] with leading dimension ld: 32-row boxes of 128
// bytes (64 bf16 or 32 fp32 columns), the pair kernel's store chunk.
inline int out_map(CUtensorMap* m, const void* p, bool f32, int rows, int cols,
            long long ld) {
  return encode_map_t(m, p, f32, cols, rows, ld, f32 ? 32 : 64, 32);
}

// K-major operand [rows, K] with box rows = the tile's M or N extent.
inline int kmajor_map(CUtensorMap* m, const void* p, int rows, int K, int box_rows) {
  return encode_map(m, p, K, rows, K, box_rows);
}
// M/N-major operand stored [K, MN]: box = 64 (M/N) x 64 (K).
inline int mnmajor_map(CUtensorMap* m, const void* p, int K, int MN) {
  return encode_map(m, p, MN, K, MN, TC_BK);
}

inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline cudaEvent_t take_event(HandleCore* H) {
  if (!H->spare.empty()) {
    cudaEvent_t e = H->spare.back();
    H->spare.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

inline int stat_index(HandleCore* H, const char* name) {
  for (size_t i = 0; i < H->stats.size(); ++i)
    if (std::strcmp(H->stats[i].name, name) == 0) return static_cast<int>(i);
  H->stats.push_back({name, 0, 0.0});
  return static_cast<int>(H->stats.size() - 1);
}

// Run one launch, bracketing it with timing events when enabled.
template <class F>
inline int run(HandleCore* H, const char* name, cudaStream_t s, F&& launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  if (H->timing) {
    a = take_event(H);
    b = take_event(H);
    if (a && b) cudaEventRecord(a, s);
  }
  // NVTX ranges mark the host-side enqueue of each kernel; a profiler that
  // records them (ncu --nvtx, Nsight Systems) attributes the launch to the
  // range.  Without a tool attached the calls return at once.
  if (H->nvtx) nvtxRangePushA(name);
  const cudaError_t e = launch();
  if (H->nvtx) nvtxRangePop();
  H->launches++;
  if (H->timing && a && b) {
    cudaEventRecord(b, s);
    H->pending.push_back({stat_index(H, name), a, b});
  }
  if (e != cudaSuccess) {
    set_detail(name, e);
    return TPMLP_ERR_CUDA;
  }
  return TPMLP_OK;
}

#define TRY(x)                       \
  do {                               \
    const int rc_ = (x);             \
    if (rc_ != TPMLP_OK) return rc_; \
  } while (0)

// One GEMM launch on the pair kernel (K-major B maps use TC2_BN_HALF-row
// boxes).  The kernel writes through output tensor maps,
// encoded here from args.out / args.out2 (row-major, leading dimension
// args.ldo, element type fp32 for the fp32-output epilogues); EPI_GELU_BWD
// reads H through the second map (args.aux, leading dimension args.ldaux).
inline int tc_gemm(HandleCore* H, const char* name, cudaStream_t s, int sms,
            int epi, bool a_mn, bool b_mn, const CUtensorMap& ta,
            const CUtensorMap& tb, const GemmArgs& args) {
  const bool f32 = epi == EPI_STORE_F32 || (epi == EPI_SHARDSUM && args.out_f32);
  CUtensorMap to, to2;
  TRY(out_map(&to, args.out, f32, args.M, args.N, args.ldo));
  if (epi == EPI_GELU_BWD) {
    TRY(out_map(&to2, args.aux, false, args.M, args.N, args.ldaux));
  } else if (args.out2 != nullptr) {
    TRY(out_map(&to2, args.out2, false, args.M, args.N, args.ldo));
  } else {
    to2 = to;  // unused by the kernel
  }
  TailPlan plan;
  TRY(run(H, name, s, [&] {
    return launch_gemm_tc2(epi, a_mn, b_mn, ta, tb, to, to2, args, sms / 2,
                           s, args.part != nullptr ? &plan : nullptr);
  }));
  if (plan.tail == 0) return TPMLP_OK;
  return run(H, "gemm_tail_combine", s, [&] {
    return launch_gemm_tc2_tail(epi, args, plan, s);
  });
}

// LayerNorm backward (dX from dXn, plus dres when not null) and, when asked
// for, its parameter gradients (partial sums over 256-row chunks, then the
// fixed-order finalizes).  pg and pb hold colsum_chunks(T) x h floats each.
inline int ln_backward(HandleCore* H, cudaStream_t s, bool bf16,
                       const float* dXn, const void* X, const float* mean,
                       const float* rstd, const float* gamma, const void* dres,
                       void* dX, float* pg, float* pb, float* dgamma,
                       float* dbeta, int T, int h) {
  TRY(run(H, "layernorm_bwd", s, [&] {
    return launch_ln_bwd(bf16, dXn, X, mean, rstd, gamma, dres, dX, T, h, s);
  }));
  if (dgamma == nullptr && dbeta == nullptr) return TPMLP_OK;
  TRY(run(H, "layernorm_param_partial", s, [&] {
    return launch_ln_param_partial(bf16, dXn, X, mean, rstd, pg, pb, T, h, s);
  }));
  const int chunks = colsum_chunks(T);
  if (dgamma)
    TRY(run(H, "colsum_finalize", s, [&] {
      return launch_colsum_finalize(pg, dgamma, chunks, h, s);
    }));
  if (dbeta)
    TRY(run(H, "colsum_finalize", s, [&] {
      return launch_colsum_finalize(pb, dbeta, chunks, h, s);
    }));
  return TPMLP_OK;
}

inline int colsum(HandleCore* H, const char* name, cudaStream_t s, bool bf16,
           const void* src, float* part, float* out, int rows, int cols) {
  const int chunks = colsum_chunks(rows);
  TRY(run(H, name, s, [&] {
    return launch_colsum_partial(bf16, src, part, rows, cols, s);
  }));
  return run(H, "colsum_finalize", s, [&] {
    return launch_colsum_finalize(part, out, chunks, cols, s);
  });
}


// Fold finished timing events into the per-kernel totals and report entry
// `index` (TPMLP_ERR_ARG past the last one).
inline int timing_get(HandleCore* H, int index, const char** name,
                      long long* launches, double* total_ms) {
  for (auto& p : H->pending) {
    if (cudaEventSynchronize(p.b) != cudaSuccess) return TPMLP_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess)
      return TPMLP_ERR_CUDA;
    H->stats[p.stat].n += 1;
    H->stats[p.stat].ms += ms;
    H->spare.push_back(p.a);
    H->spare.push_back(p.b);
  }
  H->pending.clear();
  if (index < 0 || index >= static_cast<int>(H->stats.size()))
    return TPMLP_ERR_ARG;
  if (name) *name = H->stats[index].name;
  if (launches) *launches = H->stats[index].n;
  if (total_ms) *total_ms = H->stats[index].ms;
  return TPMLP_OK;
}

// Wait for the stream, then read and clear the status word at `status`.
inline int check_status(void* status, cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    set_detail("cudaStreamSynchronize", e);
    return TPMLP_ERR_CUDA;
  }
  int st[4] = {0, 0, 0, 0};
  e = cudaMemcpy(st, status, sizeof(st), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    set_detail("cudaMemcpy(status)", e);
    return TPMLP_ERR_CUDA;
  }
  if (st[0] != 0) {
    if (st[0] == TPMLP_ERR_CHECK) {
      std::snprintf(g_detail, sizeof(g_detail),
                    "device check failed at site %d (block %d)", st[3], st[2]);
    } else {
      std::snprintf(g_detail, sizeof(g_detail),
                    "device status %d (role %d, block %d)", st[0], st[1], st[2]);
    }
    e = cudaMemsetAsync(status, 0, 16, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
      set_detail("clearing the status word", e);
      return TPMLP_ERR_CUDA;
    }
    return (st[0] == TPMLP_ERR_TIMEOUT || st[0] == TPMLP_ERR_CHECK)
               ? st[0]
               : TPMLP_ERR_CUDA;
  }
  return TPMLP_OK;
}

}  // namespace host
}  // namespace tpmlp
