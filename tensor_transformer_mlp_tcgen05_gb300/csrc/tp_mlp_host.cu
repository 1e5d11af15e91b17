// Host side of libtpmlp: argument validation, workspace layout, TMA tensor
// maps, launch sequencing, status codes and per-kernel timing.
//
// Forward (Megatron-LM explainer, "The core idea: slicing the feed-forward
// network across units"; "The f and g operators: two lines of code"):
//   [LayerNorm] -> GEMM1 (H = Xn A + b1, Y = GeLU(H), one column block per
//   shard, no sync before GeLU) -> GEMM2 (Z = sum_i Y_i B_i + b2, the shard
//   sum replacing g's all-reduce).
// Backward: GEMM dY (dH = dZ B^T * GeLU'(H); g's backward is the identity)
//   -> column sums db2, db1 -> weight GEMMs dB = Y^T dZ, dA = Xn^T dH ->
//   GEMM dX (dXn = sum_i dH_i A_i^T, the shard sum replacing f's backward
//   all-reduce) -> [LayerNorm backward, dgamma, dbeta].
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

using namespace tpmlp;

namespace {

thread_local char g_detail[512] = "";

void set_detail(const char* what, cudaError_t e) {
  std::snprintf(g_detail, sizeof(g_detail), "%s: %s (%d)", what,
                cudaGetErrorString(e), static_cast<int>(e));
}

void set_detail_msg(const char* msg) {
  std::snprintf(g_detail, sizeof(g_detail), "%s", msg);
}

// ---------------------------------------------------- workspace layout --

struct Layout {
  size_t status = 0, xn = 0, mean = 0, rstd = 0, y = 0, h = 0, dh = 0,
         dxn = 0, dze = 0, part = 0, total = 0;
  int chunks = 0;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace sections, each 256-byte aligned: status word; [Xn, mean, rstd]
// with LayerNorm; Y; and for training H, dH, [dXn fp32 with LayerNorm],
// [the dropout-masked dZ with dropout], column-sum partials.
Layout make_layout(const tp_mlp_config& c, int tokens, int training) {
  Layout L;
  const size_t es = c.dtype == TPMLP_BF16 ? 2 : 4;
  const size_t T = static_cast<size_t>(tokens);
  const size_t h = static_cast<size_t>(c.hidden);
  const size_t f = static_cast<size_t>(c.ffn);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.status = take(256);
  if (c.use_layernorm) {
    L.xn = take(T * h * es);
    L.mean = take(T * 4);
    L.rstd = take(T * 4);
  }
  L.y = take(T * f * es);
  if (training) {
    L.h = take(T * f * es);
    L.dh = take(T * f * es);
    if (c.use_layernorm) L.dxn = take(T * h * 4);
    if (c.dropout_p > 0.f) L.dze = take(T * h * es);
    L.chunks = colsum_chunks(tokens);
    L.part = take(static_cast<size_t>(L.chunks) * (f + 3 * h) * 4);
  }
  L.total = off;
  return L;
}

// ------------------------------------------------------ device checks --

int check_device(int* num_sms) {
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

EncodeTiledFn get_encoder() {
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
int encode_map_t(CUtensorMap* m, const void* base, bool f32, uint64_t inner,
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

// bf16 operand: box = {64 inner elements (one 128-byte swizzle row), box_outer}.
int encode_map(CUtensorMap* m, const void* base, uint64_t inner,
               uint64_t outer, uint64_t pitch, uint32_t box_outer) {
  return encode_map_t(m, base, false, inner, outer, pitch, 64, box_outer);
}

// GEMM output [rows, cols] with leading dimension ld: 32-row boxes of 128
// bytes (64 bf16 or 32 fp32 columns), the pair kernel's store chunk.
int out_map(CUtensorMap* m, const void* p, bool f32, int rows, int cols,
            long long ld) {
  return encode_map_t(m, p, f32, cols, rows, ld, f32 ? 32 : 64, 32);
}

// K-major operand [rows, K] with box rows = the tile's M or N extent.
int kmajor_map(CUtensorMap* m, const void* p, int rows, int K, int box_rows) {
  return encode_map(m, p, K, rows, K, box_rows);
}
// M/N-major operand stored [K, MN]: box = 64 (M/N) x 64 (K).
int mnmajor_map(CUtensorMap* m, const void* p, int K, int MN) {
  return encode_map(m, p, MN, K, MN, TC_BK);
}

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace

void tpmlp::set_last_detail(const char* msg) { set_detail_msg(msg); }

// ------------------------------------------------------------- handle --

struct tp_mlp_handle {
  tp_mlp_config cfg;
  unsigned long long budget_ns = 2000000000ull;
  unsigned long long drop_seed = 0, drop_offset = 0;
  long long launches = 0;
  bool timing = false;
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
};

namespace {

cudaEvent_t take_event(tp_mlp_handle* H) {
  if (!H->spare.empty()) {
    cudaEvent_t e = H->spare.back();
    H->spare.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

int stat_index(tp_mlp_handle* H, const char* name) {
  for (size_t i = 0; i < H->stats.size(); ++i)
    if (std::strcmp(H->stats[i].name, name) == 0) return static_cast<int>(i);
  H->stats.push_back({name, 0, 0.0});
  return static_cast<int>(H->stats.size() - 1);
}

// Run one launch, bracketing it with timing events when enabled.
template <class F>
int run(tp_mlp_handle* H, const char* name, cudaStream_t s, F&& launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  if (H->timing) {
    a = take_event(H);
    b = take_event(H);
    if (a && b) cudaEventRecord(a, s);
  }
  const cudaError_t e = launch();
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

int grid_for(int M, int N, int sms) {
  const long long tiles = static_cast<long long>((M + TC_BM - 1) / TC_BM) *
                          ((N + TC_BN - 1) / TC_BN);
  return static_cast<int>(tiles < sms ? tiles : sms);
}

GemmArgs base_args(const tp_mlp_handle* H, void* ws, const Layout& L) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.group_m = 16;
  a.gelu_mode = H->cfg.gelu_mode;
  a.status = reinterpret_cast<int*>(static_cast<char*>(ws) + L.status);
  a.budget_ns = H->budget_ns;
  a.num_seg = 1;
  return a;
}

// Dropout parameters of the output dropout (keep when the 32-bit Philox
// draw is >= floor(p 2^32), scale kept values by 1 / (1 - p)).
void set_dropout(const tp_mlp_handle* H, GemmArgs& a) {
  const double p = H->cfg.dropout_p;
  double thr = p * 4294967296.0;
  if (thr > 4294967295.0) thr = 4294967295.0;
  a.dropout = 1;
  a.drop_threshold = static_cast<uint32_t>(thr);
  a.drop_scale = 1.0f / (1.0f - H->cfg.dropout_p);
  a.drop_seed = H->drop_seed;
  a.drop_offset = H->drop_offset;
}

#define TRY(x)                       \
  do {                               \
    const int rc_ = (x);             \
    if (rc_ != TPMLP_OK) return rc_; \
  } while (0)

// GEMM kernel selection: CTA pairs (256 x 256 tiles) by default; setting
// TPMLP_GEMM_VARIANT=single in the environment selects the one-CTA kernel.
bool use_pairs() {
  static const bool pairs = [] {
    const char* v = std::getenv("TPMLP_GEMM_VARIANT");
    return !(v != nullptr && std::strcmp(v, "single") == 0);
  }();
  return pairs;
}

// Box height of a K-major B operand for the selected kernel.
int b_box_rows() { return use_pairs() ? TC2_BN_HALF : TC_BN; }

// One GEMM launch.  The pair kernel writes through output tensor maps,
// encoded here from args.out / args.out2 (row-major, leading dimension
// args.ldo, element type fp32 for the fp32-output epilogues).
int tc_gemm(tp_mlp_handle* H, const char* name, cudaStream_t s, int sms,
            int epi, bool a_mn, bool b_mn, const CUtensorMap& ta,
            const CUtensorMap& tb, const GemmArgs& args) {
  if (use_pairs()) {
    const bool f32 = epi == EPI_STORE_F32 || (epi == EPI_SHARDSUM && args.out_f32);
    CUtensorMap to, to2;
    TRY(out_map(&to, args.out, f32, args.M, args.N, args.ldo));
    if (args.out2 != nullptr) {
      TRY(out_map(&to2, args.out2, false, args.M, args.N, args.ldo));
    } else {
      to2 = to;  // unused by the kernel
    }
    return run(H, name, s, [&] {
      return launch_gemm_tc2(epi, a_mn, b_mn, ta, tb, to, to2, args, sms / 2,
                             s);
    });
  }
  const int grid = grid_for(args.M, args.N, sms);
  return run(H, name, s, [&] {
    return launch_gemm_tc(epi, a_mn, b_mn, ta, tb, args, grid, s);
  });
}

int colsum(tp_mlp_handle* H, const char* name, cudaStream_t s, bool bf16,
           const void* src, float* part, float* out, int rows, int cols) {
  const int chunks = colsum_chunks(rows);
  TRY(run(H, name, s, [&] {
    return launch_colsum_partial(bf16, src, part, rows, cols, s);
  }));
  return run(H, "colsum_finalize", s, [&] {
    return launch_colsum_finalize(part, out, chunks, cols, s);
  });
}

}  // namespace

// ================================================================= ABI ==

extern "C" {

int tp_mlp_create(const tp_mlp_config* cfg, tp_mlp_handle** out) {
  if (cfg == nullptr || out == nullptr) return TPMLP_ERR_ARG;
  if (cfg->dtype != TPMLP_BF16 && cfg->dtype != TPMLP_FP32) return TPMLP_ERR_ARG;
  if (cfg->gelu_mode != TPMLP_GELU_ERF && cfg->gelu_mode != TPMLP_GELU_TANH)
    return TPMLP_ERR_ARG;
  if (cfg->use_layernorm != 0 && cfg->use_layernorm != 1) return TPMLP_ERR_ARG;
  if (cfg->use_residual != 0 && cfg->use_residual != 1) return TPMLP_ERR_ARG;
  if (!(cfg->dropout_p >= 0.f && cfg->dropout_p < 1.f)) return TPMLP_ERR_ARG;
  if (cfg->use_layernorm &&
      !(cfg->ln_eps >= 0.f && std::isfinite(cfg->ln_eps)))
    return TPMLP_ERR_ARG;
  if (cfg->hidden <= 0 || cfg->ffn <= 0 || cfg->shards <= 0 ||
      cfg->max_tokens < 0)
    return TPMLP_ERR_SHAPE;
  if (cfg->hidden % 64 != 0) return TPMLP_ERR_SHAPE;
  if (cfg->ffn % cfg->shards != 0) return TPMLP_ERR_SHAPE;
  if ((cfg->ffn / cfg->shards) % 64 != 0) return TPMLP_ERR_SHAPE;
  // Element coordinates and tile indices stay within int32.
  if (static_cast<long long>(cfg->max_tokens) > (1LL << 30) ||
      cfg->ffn > (1 << 24) || cfg->hidden > (1 << 24))
    return TPMLP_ERR_SHAPE;
  tp_mlp_handle* h = new (std::nothrow) tp_mlp_handle();
  if (h == nullptr) return TPMLP_ERR_ARG;
  h->cfg = *cfg;
  *out = h;
  return TPMLP_OK;
}

int tp_mlp_destroy(tp_mlp_handle* handle) {
  if (handle == nullptr) return TPMLP_OK;
  for (auto& p : handle->pending) {
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  for (auto e : handle->spare) cudaEventDestroy(e);
  delete handle;
  return TPMLP_OK;
}

size_t tp_mlp_workspace_bytes(const tp_mlp_handle* handle, int tokens,
                              int training) {
  if (handle == nullptr || tokens < 0) return 0;
  return make_layout(handle->cfg, tokens, training ? 1 : 0).total;
}

int tp_mlp_forward(tp_mlp_handle* H, int tokens, const void* X, const void* A,
                   const void* B, const float* bias1, const float* bias2,
                   const float* ln_gamma, const float* ln_beta, void* Z,
                   void* workspace, size_t workspace_bytes, int training,
                   void* stream) {
  if (H == nullptr) return TPMLP_ERR_ARG;
  const tp_mlp_config& c = H->cfg;
  if (tokens < 0 || tokens > c.max_tokens) return TPMLP_ERR_SHAPE;
  // Token-sized arrays may be NULL when there are no tokens.
  if (!A || !B || !workspace || (tokens > 0 && (!X || !Z))) return TPMLP_ERR_ARG;
  if (c.use_layernorm && (!ln_gamma || !ln_beta)) return TPMLP_ERR_ARG;
  const void* ptrs[] = {X, A, B, Z, workspace, bias1, bias2, ln_gamma, ln_beta};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return TPMLP_ERR_ALIGN;
  const Layout L = make_layout(c, tokens, training ? 1 : 0);
  if (workspace_bytes < L.total) return TPMLP_ERR_WORKSPACE;
  int sms = 0;
  TRY(check_device(&sms));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  cudaError_t e = cudaMemsetAsync(ws + L.status, 0, 16, s);
  if (e != cudaSuccess) {
    set_detail("cudaMemsetAsync(status)", e);
    return TPMLP_ERR_CUDA;
  }
  if (tokens == 0) return TPMLP_OK;

  const bool bf16 = c.dtype == TPMLP_BF16;
  const int T = tokens, h = c.hidden, f = c.ffn, t = c.shards, ft = f / t;
  void* Y = ws + L.y;
  void* Hbuf = training ? ws + L.h : nullptr;
  const void* Xop = X;
  if (c.use_layernorm) {
    void* Xn = ws + L.xn;
    TRY(run(H, "layernorm_fwd", s, [&] {
      return launch_ln_fwd(bf16, X, ln_gamma, ln_beta, Xn,
                           reinterpret_cast<float*>(ws + L.mean),
                           reinterpret_cast<float*>(ws + L.rstd), T, h,
                           c.ln_eps, s);
    }));
    Xop = Xn;
  }

  GemmArgs g1 = base_args(H, ws, L);
  g1.M = T; g1.N = f; g1.K = h;
  g1.out = Y; g1.ldo = f; g1.out2 = Hbuf; g1.bias = bias1;
  GemmArgs g2 = base_args(H, ws, L);
  g2.M = T; g2.N = h; g2.K = f; g2.num_seg = t;
  g2.out = Z; g2.ldo = h; g2.bias = bias2;
  if (c.use_residual) {  // Z += X (the raw input), before the one rounding
    g2.aux = X;
    g2.ldaux = h;
  }
  if (training && c.dropout_p > 0.f) set_dropout(H, g2);  // training only

  if (bf16) {
    CUtensorMap ta, tb;
    g1.kb_per_seg = h / TC_BK;
    TRY(kmajor_map(&ta, Xop, T, h, TC_BM));
    TRY(mnmajor_map(&tb, A, h, f));
    TRY(tc_gemm(H, "gemm1_gelu", s, sms, EPI_GELU_FWD, false, true, ta, tb,
                g1));
    g2.kb_per_seg = ft / TC_BK;
    TRY(kmajor_map(&ta, Y, T, f, TC_BM));
    TRY(mnmajor_map(&tb, B, f, h));
    TRY(tc_gemm(H, "gemm2_shardsum", s, sms, EPI_SHARDSUM, false, true, ta, tb,
                g2));
  } else {
    g1.kb_per_seg = h;
    const SimtOperands o1{static_cast<const float*>(Xop), h, 1,
                          static_cast<const float*>(A), f, 1};
    TRY(run(H, "simt_gemm1_gelu", s,
            [&] { return launch_gemm_simt(EPI_GELU_FWD, o1, g1, s); }));
    g2.kb_per_seg = ft;
    g2.out_f32 = 1;
    const SimtOperands o2{static_cast<const float*>(Y), f, 1,
                          static_cast<const float*>(B), h, 1};
    TRY(run(H, "simt_gemm2_shardsum", s,
            [&] { return launch_gemm_simt(EPI_SHARDSUM, o2, g2, s); }));
  }
  return TPMLP_OK;
}

int tp_mlp_backward(tp_mlp_handle* H, int tokens, const void* dZ,
                    const void* X, const void* A, const void* B,
                    const float* ln_gamma, void* workspace,
                    size_t workspace_bytes, void* dX, float* dA, float* dB,
                    float* dbias1, float* dbias2, float* dgamma, float* dbeta,
                    void* stream) {
  if (H == nullptr) return TPMLP_ERR_ARG;
  const tp_mlp_config& c = H->cfg;
  if (tokens < 0 || tokens > c.max_tokens) return TPMLP_ERR_SHAPE;
  if (!A || !B || !workspace || !dA || !dB ||
      (tokens > 0 && (!dZ || !X || !dX)))
    return TPMLP_ERR_ARG;
  if (c.use_layernorm && !ln_gamma) return TPMLP_ERR_ARG;
  const void* ptrs[] = {dZ, X, A, B, ln_gamma, workspace, dX, dA, dB,
                        dbias1, dbias2, dgamma, dbeta};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return TPMLP_ERR_ALIGN;
  const Layout L = make_layout(c, tokens, 1);
  if (workspace_bytes < L.total) return TPMLP_ERR_WORKSPACE;
  int sms = 0;
  TRY(check_device(&sms));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const bool bf16 = c.dtype == TPMLP_BF16;
  const int T = tokens, h = c.hidden, f = c.ffn, t = c.shards, ft = f / t;
  const bool ln = c.use_layernorm != 0;

  if (T == 0) {  // sums over an empty token set
    struct Zero {
      void* p;
      size_t n;
    } zs[] = {{dA, size_t(h) * f * 4},
              {dB, size_t(f) * h * 4},
              {dbias1, size_t(f) * 4},
              {dbias2, size_t(h) * 4},
              {ln ? dgamma : nullptr, size_t(h) * 4},
              {ln ? dbeta : nullptr, size_t(h) * 4}};
    for (auto& z : zs) {
      if (!z.p) continue;
      const cudaError_t e = cudaMemsetAsync(z.p, 0, z.n, s);
      if (e != cudaSuccess) {
        set_detail("cudaMemsetAsync(zero gradients)", e);
        return TPMLP_ERR_CUDA;
      }
    }
    return TPMLP_OK;
  }

  const void* Y = ws + L.y;
  const void* Hb = ws + L.h;
  void* dH = ws + L.dh;
  // The block's own gradients see the dropout-masked dZ; the residual path
  // (below) keeps the raw dZ.
  const void* dZg = dZ;
  if (c.dropout_p > 0.f) {
    GemmArgs dp;
    std::memset(&dp, 0, sizeof(dp));
    set_dropout(H, dp);
    void* dze = ws + L.dze;
    TRY(run(H, "dropout_bwd", s, [&] {
      return launch_dropout_grad(bf16, dZ, dze, T, h, dp.drop_threshold,
                                 dp.drop_scale, dp.drop_seed, dp.drop_offset,
                                 s);
    }));
    dZg = dze;
  }
  const void* Xop = ln ? static_cast<const void*>(ws + L.xn) : X;
  float* part = reinterpret_cast<float*>(ws + L.part);
  void* dXdst = ln ? static_cast<void*>(ws + L.dxn) : dX;

  GemmArgs gy = base_args(H, ws, L);  // dH = (dZ B^T) * GeLU'(H)
  gy.M = T; gy.N = f; gy.K = h;
  gy.out = dH; gy.ldo = f; gy.aux = Hb; gy.ldaux = f;
  GemmArgs gb = base_args(H, ws, L);  // dB = Y^T dZ
  gb.M = f; gb.N = h; gb.K = T;
  gb.out = dB; gb.ldo = h;
  GemmArgs ga = base_args(H, ws, L);  // dA = Xn^T dH
  ga.M = h; ga.N = f; ga.K = T;
  ga.out = dA; ga.ldo = f;
  GemmArgs gx = base_args(H, ws, L);  // dXn = sum_i dH_i A_i^T
  gx.M = T; gx.N = h; gx.K = f; gx.num_seg = t;
  gx.out = dXdst; gx.ldo = h; gx.out_f32 = (ln || !bf16) ? 1 : 0;
  if (c.use_residual && !ln) {  // dX = dXn + dZ in the GEMM epilogue
    gx.aux = dZ;
    gx.ldaux = h;
  }
  // With LayerNorm the residual gradient is added by the LN backward kernel.
  const void* dres = (c.use_residual && ln) ? dZ : nullptr;

  if (bf16) {
    CUtensorMap ta, tb;
    gy.kb_per_seg = h / TC_BK;
    TRY(kmajor_map(&ta, dZg, T, h, TC_BM));
    TRY(kmajor_map(&tb, B, f, h, b_box_rows()));
    TRY(tc_gemm(H, "gemm_dh_gelu_bwd", s, sms, EPI_GELU_BWD, false, false, ta,
                tb, gy));
    if (dbias2) TRY(colsum(H, "colsum_db2", s, true, dZg, part, dbias2, T, h));
    if (dbias1)
      TRY(colsum(H, "colsum_db1", s, true, dH, part + size_t(L.chunks) * h,
                 dbias1, T, f));
    const int kbT = (T + TC_BK - 1) / TC_BK;
    gb.kb_per_seg = kbT;
    TRY(mnmajor_map(&ta, Y, T, f));
    TRY(mnmajor_map(&tb, dZg, T, h));
    TRY(tc_gemm(H, "gemm_wgrad_dB", s, sms, EPI_STORE_F32, true, true, ta, tb,
                gb));
    ga.kb_per_seg = kbT;
    TRY(mnmajor_map(&ta, Xop, T, h));
    TRY(mnmajor_map(&tb, dH, T, f));
    TRY(tc_gemm(H, "gemm_wgrad_dA", s, sms, EPI_STORE_F32, true, true, ta, tb,
                ga));
    gx.kb_per_seg = ft / TC_BK;
    TRY(kmajor_map(&ta, dH, T, f, TC_BM));
    TRY(kmajor_map(&tb, A, h, f, b_box_rows()));
    TRY(tc_gemm(H, "gemm_dx_shardsum", s, sms, EPI_SHARDSUM, false, false, ta,
                tb, gx));
  } else {
    const float* fY = static_cast<const float*>(Y);
    const float* fdZ = static_cast<const float*>(dZg);
    const float* fdH = static_cast<const float*>(dH);
    gy.kb_per_seg = h;
    const SimtOperands oy{fdZ, h, 1, static_cast<const float*>(B), 1, h};
    TRY(run(H, "simt_gemm_dh_gelu_bwd", s,
            [&] { return launch_gemm_simt(EPI_GELU_BWD, oy, gy, s); }));
    if (dbias2) TRY(colsum(H, "colsum_db2", s, false, dZg, part, dbias2, T, h));
    if (dbias1)
      TRY(colsum(H, "colsum_db1", s, false, dH, part + size_t(L.chunks) * h,
                 dbias1, T, f));
    gb.kb_per_seg = T;
    const SimtOperands ob{fY, 1, f, fdZ, h, 1};
    TRY(run(H, "simt_gemm_wgrad_dB", s,
            [&] { return launch_gemm_simt(EPI_STORE_F32, ob, gb, s); }));
    ga.kb_per_seg = T;
    const SimtOperands oa{static_cast<const float*>(Xop), 1, h, fdH, f, 1};
    TRY(run(H, "simt_gemm_wgrad_dA", s,
            [&] { return launch_gemm_simt(EPI_STORE_F32, oa, ga, s); }));
    gx.kb_per_seg = ft;
    const SimtOperands ox{fdH, f, 1, static_cast<const float*>(A), 1, f};
    TRY(run(H, "simt_gemm_dx_shardsum", s,
            [&] { return launch_gemm_simt(EPI_SHARDSUM, ox, gx, s); }));
  }

  if (ln) {
    const float* dXn = reinterpret_cast<const float*>(ws + L.dxn);
    const float* mean = reinterpret_cast<const float*>(ws + L.mean);
    const float* rstd = reinterpret_cast<const float*>(ws + L.rstd);
    TRY(run(H, "layernorm_bwd", s, [&] {
      return launch_ln_bwd(bf16, dXn, X, mean, rstd, ln_gamma, dres, dX, T, h,
                           s);
    }));
    if (dgamma || dbeta) {
      float* pg = part + size_t(L.chunks) * (h + f);
      float* pb = pg + size_t(L.chunks) * h;
      TRY(run(H, "layernorm_param_partial", s, [&] {
        return launch_ln_param_partial(bf16, dXn, X, mean, rstd, pg, pb, T, h,
                                       s);
      }));
      if (dgamma)
        TRY(run(H, "colsum_finalize", s, [&] {
          return launch_colsum_finalize(pg, dgamma, L.chunks, h, s);
        }));
      if (dbeta)
        TRY(run(H, "colsum_finalize", s, [&] {
          return launch_colsum_finalize(pb, dbeta, L.chunks, h, s);
        }));
    }
  }
  return TPMLP_OK;
}

int tp_mlp_check(tp_mlp_handle* H, void* workspace, void* stream) {
  if (H == nullptr || workspace == nullptr) return TPMLP_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    set_detail("cudaStreamSynchronize", e);
    return TPMLP_ERR_CUDA;
  }
  int st[4] = {0, 0, 0, 0};
  e = cudaMemcpy(st, workspace, sizeof(st), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    set_detail("cudaMemcpy(status)", e);
    return TPMLP_ERR_CUDA;
  }
  if (st[0] != 0) {
    std::snprintf(g_detail, sizeof(g_detail),
                  "device status %d (role %d, block %d)", st[0], st[1], st[2]);
    e = cudaMemsetAsync(workspace, 0, 16, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
      set_detail("clearing the status word", e);
      return TPMLP_ERR_CUDA;
    }
    return st[0] == TPMLP_ERR_TIMEOUT ? TPMLP_ERR_TIMEOUT : TPMLP_ERR_CUDA;
  }
  return TPMLP_OK;
}

const char* tp_mlp_status_string(int status) {
  switch (status) {
    case TPMLP_OK: return "ok";
    case TPMLP_ERR_ARG: return "invalid argument";
    case TPMLP_ERR_SHAPE: return "unsupported shape";
    case TPMLP_ERR_ALIGN: return "pointer not 16-byte aligned";
    case TPMLP_ERR_ARCH: return "device is not sm_103 (GB300)";
    case TPMLP_ERR_CUDA: return "CUDA error";
    case TPMLP_ERR_TIMEOUT: return "bounded device wait timed out";
    case TPMLP_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

const char* tp_mlp_last_detail(void) { return g_detail; }

long long tp_mlp_launch_count(const tp_mlp_handle* handle) {
  return handle ? handle->launches : -1;
}

int tp_mlp_set_timing(tp_mlp_handle* handle, int enable) {
  if (handle == nullptr) return TPMLP_ERR_ARG;
  handle->timing = enable != 0;
  return TPMLP_OK;
}

int tp_mlp_timing_get(tp_mlp_handle* H, int index, const char** name,
                      long long* launches, double* total_ms) {
  if (H == nullptr) return TPMLP_ERR_ARG;
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

int tp_mlp_timing_reset(tp_mlp_handle* H) {
  if (H == nullptr) return TPMLP_ERR_ARG;
  tp_mlp_timing_get(H, -1, nullptr, nullptr, nullptr);  // drain pending
  H->stats.clear();
  return TPMLP_OK;
}

int tp_mlp_set_dropout_seed(tp_mlp_handle* handle, unsigned long long seed,
                            unsigned long long offset) {
  if (handle == nullptr) return TPMLP_ERR_ARG;
  handle->drop_seed = seed;
  handle->drop_offset = offset;
  return TPMLP_OK;
}

int tp_mlp_set_wait_budget(tp_mlp_handle* handle, unsigned long long ns) {
  if (handle == nullptr) return TPMLP_ERR_ARG;
  handle->budget_ns = ns;
  return TPMLP_OK;
}

}  // extern "C"
