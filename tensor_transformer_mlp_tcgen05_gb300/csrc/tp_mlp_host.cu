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

#include "host_common.cuh"

using namespace tpmlp;

using namespace tpmlp::host;

namespace {

struct Layout {
  size_t status = 0, xn = 0, mean = 0, rstd = 0, y = 0, h = 0, dh = 0,
         dxn = 0, dze = 0, part = 0, tailp = 0, total = 0;
  // the fused LayerNorm prologue's counters (GemmArgs::ln_sync), right
  // after the 16-byte status word so one memset clears both
  size_t lnsync = 0, lnsync_words = 0;
  size_t lnp = 0;   // rows of each LayerNorm-parameter partial section
  int chunks = 0;   // 256-row column-sum chunks
  int groups = 0;   // 32-row groups of the dH GEMM's fused db1 partials
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace sections, each 256-byte aligned: status word [+ with bf16
// LayerNorm, the prologue's row counters: 1 + ceil(T / 128) words];
// [Xn, mean, rstd] with LayerNorm; Y; [bf16: the GEMM tail-split partials, TAIL_PART_BYTES];
// and for training H, dH, [dXn fp32 with LayerNorm], [the dropout-masked dZ
// with dropout], column-sum partials: db2 (chunks x h), db1 (max(groups,
// chunks) x f), dgamma and dbeta (lnp = chunks x h each).
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
  if (c.use_layernorm && c.dtype == TPMLP_BF16) {
    L.lnsync_words = 1 + (T + 127) / 128;
    L.lnsync = 16;
    L.status = take(16 + 4 * L.lnsync_words);
  } else {
    L.status = take(256);
  }
  if (c.use_layernorm) {
    L.xn = take(T * h * es);
    L.mean = take(T * 4);
    L.rstd = take(T * 4);
  }
  L.y = take(T * f * es);
  if (c.dtype == TPMLP_BF16) L.tailp = take(static_cast<size_t>(TAIL_PART_BYTES));
  if (training) {
    L.h = take(T * f * es);
    L.dh = take(T * f * es);
    if (c.use_layernorm) L.dxn = take(T * h * 4);
    if (c.dropout_p > 0.f) L.dze = take(T * h * es);
    L.chunks = colsum_chunks(tokens);
    L.groups = (tokens + 31) / 32;
    const size_t rows1 = static_cast<size_t>(L.groups > L.chunks ? L.groups : L.chunks);
    // db2 (chunks x h), db1 (rows1 x f), then the LayerNorm parameter
    // partials (2 x chunks x h)
    L.lnp = static_cast<size_t>(L.chunks);
    L.part = take((static_cast<size_t>(L.chunks) * h + rows1 * f + 2 * L.lnp * h) * 4);
  }
  L.total = off;
  return L;
}

// FP8: packed weights and workspace.
struct Fp8Pack {
  size_t scales = 0, aqt = 0, bqt = 0, aq = 0, bq = 0, total = 0;
};
// [amax_a, amax_b (u32), s_a, s_b (f32)] | A^T codes [f, h] | B^T codes
// [h, f] | A codes [h, f] | B codes [f, h]
Fp8Pack fp8_pack_layout(const tp_mlp_config& c) {
  Fp8Pack P;
  const size_t h = static_cast<size_t>(c.hidden), f = static_cast<size_t>(c.ffn);
  P.scales = 0;
  P.aqt = 256;
  P.bqt = align_up(P.aqt + f * h, 256);
  P.aq = align_up(P.bqt + h * f, 256);
  P.bq = align_up(P.aq + h * f, 256);
  P.total = align_up(P.bq + f * h, 256);
  return P;
}

struct Fp8Layout {
  size_t status = 0, xn = 0, mean = 0, rstd = 0, scales = 0, xq = 0, y = 0,
         yq = 0, tailp = 0, total = 0;
  // training sections
  size_t tpitch = 0;  // row pitch (bytes) of the transposed code sections
  size_t hb = 0, xqt = 0, yqt = 0, bscales = 0, dzq = 0, dzqt = 0, dh = 0,
         dhq = 0, dhqt = 0, dxn = 0, part = 0, train_total = 0;
  size_t lnp = 0;
  int chunks = 0, groups = 0;
};
// status | [Xn, mean, rstd] | [amax_x, amax_y (u32), s_x, s_y (f32)] |
// Xq [T, h] | Y [T, f] bf16 | Yq [T, f] | GEMM tail-split partials
// (TAIL_PART_BYTES) -- the forward's workspace; the
// training workspace goes on with H [T, f] bf16 | Xq^T [h, Tp] | Yq^T
// [f, Tp] | [amax_dz, amax_dh (u32), s_dz, s_dh (f32)] | dZq [T, h] |
// dZq^T [h, Tp] | dH [T, f] bf16 | dHq [T, f] | dHq^T [f, Tp] | [dXn fp32
// [T, h] with LayerNorm] | column-sum partials (as the bf16 backward's),
// Tp = T rounded up to 16 (the tensor-map row pitch rule).
Fp8Layout fp8_layout(const tp_mlp_config& c, int tokens) {
  Fp8Layout L;
  const size_t T = static_cast<size_t>(tokens);
  const size_t h = static_cast<size_t>(c.hidden), f = static_cast<size_t>(c.ffn);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.status = take(256);
  if (c.use_layernorm) {
    L.xn = take(T * h * 2);
    L.mean = take(T * 4);
    L.rstd = take(T * 4);
  }
  L.scales = take(16);
  L.xq = take(T * h);
  L.y = take(T * f * 2);
  L.yq = take(T * f);
  L.tailp = take(static_cast<size_t>(TAIL_PART_BYTES));
  L.total = off;
  L.tpitch = align_up(T, 16);
  L.hb = take(T * f * 2);
  L.xqt = take(h * L.tpitch);
  L.yqt = take(f * L.tpitch);
  L.bscales = take(16);
  L.dzq = take(T * h);
  L.dzqt = take(h * L.tpitch);
  L.dh = take(T * f * 2);
  L.dhq = take(T * f);
  L.dhqt = take(f * L.tpitch);
  if (c.use_layernorm) L.dxn = take(T * h * 4);
  L.chunks = colsum_chunks(tokens);
  L.groups = (tokens + 31) / 32;
  const size_t rows1 = static_cast<size_t>(L.groups > L.chunks ? L.groups : L.chunks);
  L.lnp = static_cast<size_t>(L.chunks);
  L.part = take((static_cast<size_t>(L.chunks) * h + rows1 * f + 2 * L.lnp * h) * 4);
  L.train_total = off;
  return L;
}

// ------------------------------------------------------ device checks --

}  // namespace

void tpmlp::set_last_detail(const char* msg) { set_detail_msg(msg); }

// ------------------------------------------------------------- handle --

struct tp_mlp_handle {
  tpmlp::host::HandleCore core;
  tp_mlp_config cfg;
  unsigned long long drop_seed = 0, drop_offset = 0;
  bool ln_prologue = true;   // tp_mlp_set_ln_prologue
};

namespace {

GemmArgs base_args(const tp_mlp_handle* H, void* ws, size_t status_off) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.group_m = 16;
  a.gelu_mode = H->cfg.gelu_mode;
  a.status = reinterpret_cast<int*>(static_cast<char*>(ws) + status_off);
  a.budget_ns = H->core.budget_ns;
  a.num_seg = 1;
  return a;
}

GemmArgs base_args(const tp_mlp_handle* H, void* ws, const Layout& L) {
  GemmArgs a = base_args(H, ws, L.status);
  if (L.tailp != 0) {
    a.part = reinterpret_cast<float*>(static_cast<char*>(ws) + L.tailp);
    a.part_bytes = TAIL_PART_BYTES;
  }
  return a;
}

// An E4M3 pair GEMM, with the tail split when args.part is given.
int f8_gemm(HandleCore* H, const char* name, cudaStream_t s, int sms, int epi,
            const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to,
            const CUtensorMap& to2, const GemmArgs& g) {
  TailPlan plan;
  TRY(run(H, name, s, [&] {
    return launch_gemm_tc2_e4m3(epi, ta, tb, to, to2, g, sms / 2, s,
                                g.part != nullptr ? &plan : nullptr);
  }));
  if (plan.tail == 0) return TPMLP_OK;
  return run(H, "gemm_tail_combine", s,
             [&] { return launch_gemm_tc2_tail(epi, g, plan, s); });
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
  const bool bf16 = c.dtype == TPMLP_BF16;
  const int T = tokens, h = c.hidden, f = c.ffn, t = c.shards, ft = f / t;
  // LayerNorm inside GEMM1's launch (GemmArgs::ln_x)
  const bool ln_fused = c.use_layernorm && bf16 && H->ln_prologue &&
                        h % 256 == 0 && h / 256 <= LN_VMAX;
  // the status word, and with the fused LayerNorm its counters, cleared
  const size_t clear = ln_fused ? 16 + 4 * L.lnsync_words : 16;
  cudaError_t e = cudaMemsetAsync(ws + L.status, 0, clear, s);
  if (e != cudaSuccess) {
    set_detail("cudaMemsetAsync(status)", e);
    return TPMLP_ERR_CUDA;
  }
  if (tokens == 0) return TPMLP_OK;

  void* Y = ws + L.y;
  void* Hbuf = training ? ws + L.h : nullptr;
  const void* Xop = X;
  if (ln_fused) {
    Xop = ws + L.xn;
  } else if (c.use_layernorm) {
    void* Xn = ws + L.xn;
    TRY(run(&H->core, "layernorm_fwd", s, [&] {
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
  if (ln_fused) {
    g1.ln_x = static_cast<const __nv_bfloat16*>(X);
    g1.ln_gamma = ln_gamma;
    g1.ln_beta = ln_beta;
    g1.ln_xn = reinterpret_cast<__nv_bfloat16*>(ws + L.xn);
    g1.ln_mean = reinterpret_cast<float*>(ws + L.mean);
    g1.ln_rstd = reinterpret_cast<float*>(ws + L.rstd);
    g1.ln_eps = c.ln_eps;
    g1.ln_sync = reinterpret_cast<unsigned int*>(ws + L.status + L.lnsync);
  }
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
    TRY(tc_gemm(&H->core, ln_fused ? "gemm1_ln_gelu" : "gemm1_gelu", s, sms,
                EPI_GELU_FWD, false, true, ta, tb, g1));
    g2.kb_per_seg = ft / TC_BK;
    TRY(kmajor_map(&ta, Y, T, f, TC_BM));
    TRY(mnmajor_map(&tb, B, f, h));
    TRY(tc_gemm(&H->core, "gemm2_shardsum", s, sms, EPI_SHARDSUM, false, true, ta, tb,
                g2));
  } else {
    g1.kb_per_seg = h;
    const SimtOperands o1{static_cast<const float*>(Xop), h, 1,
                          static_cast<const float*>(A), f, 1};
    TRY(run(&H->core, "simt_gemm1_gelu", s,
            [&] { return launch_gemm_simt(EPI_GELU_FWD, o1, g1, s); }));
    g2.kb_per_seg = ft;
    g2.out_f32 = 1;
    const SimtOperands o2{static_cast<const float*>(Y), f, 1,
                          static_cast<const float*>(B), h, 1};
    TRY(run(&H->core, "simt_gemm2_shardsum", s,
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
    TRY(run(&H->core, "dropout_bwd", s, [&] {
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
  float* part1 = part + size_t(L.chunks) * h;   // db1 partials
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
    TRY(kmajor_map(&tb, B, f, h, TC2_BN_HALF));
    // db1 = sum_T dH: 32-row partials from the GEMM's epilogue, then one
    // fixed-order pass over them
    if (dbias1 != nullptr) {
      gy.colsum = part1;
      gy.ld_colsum = f;
    }
    TRY(tc_gemm(&H->core, "gemm_dh_gelu_bwd", s, sms, EPI_GELU_BWD, false, false, ta,
                tb, gy));
    if (dbias2) TRY(colsum(&H->core, "colsum_db2", s, true, dZg, part, dbias2, T, h));
    if (dbias1 != nullptr) {
      TRY(run(&H->core, "colsum_finalize", s, [&] {
        return launch_colsum_finalize(part1, dbias1, L.groups, f, s);
      }));
    }
    const int kbT = (T + TC_BK - 1) / TC_BK;
    gb.kb_per_seg = kbT;
    TRY(mnmajor_map(&ta, Y, T, f));
    TRY(mnmajor_map(&tb, dZg, T, h));
    TRY(tc_gemm(&H->core, "gemm_wgrad_dB", s, sms, EPI_STORE_F32, true, true, ta, tb,
                gb));
    ga.kb_per_seg = kbT;
    TRY(mnmajor_map(&ta, Xop, T, h));
    TRY(mnmajor_map(&tb, dH, T, f));
    TRY(tc_gemm(&H->core, "gemm_wgrad_dA", s, sms, EPI_STORE_F32, true, true, ta, tb,
                ga));
    gx.kb_per_seg = ft / TC_BK;
    TRY(kmajor_map(&ta, dH, T, f, TC_BM));
    TRY(kmajor_map(&tb, A, h, f, TC2_BN_HALF));
    TRY(tc_gemm(&H->core, "gemm_dx_shardsum", s, sms, EPI_SHARDSUM, false, false, ta,
                tb, gx));
  } else {
    const float* fY = static_cast<const float*>(Y);
    const float* fdZ = static_cast<const float*>(dZg);
    const float* fdH = static_cast<const float*>(dH);
    gy.kb_per_seg = h;
    const SimtOperands oy{fdZ, h, 1, static_cast<const float*>(B), 1, h};
    TRY(run(&H->core, "simt_gemm_dh_gelu_bwd", s,
            [&] { return launch_gemm_simt(EPI_GELU_BWD, oy, gy, s); }));
    if (dbias2) TRY(colsum(&H->core, "colsum_db2", s, false, dZg, part, dbias2, T, h));
    if (dbias1)
      TRY(colsum(&H->core, "colsum_db1", s, false, dH, part1, dbias1, T, f));
    gb.kb_per_seg = T;
    const SimtOperands ob{fY, 1, f, fdZ, h, 1};
    TRY(run(&H->core, "simt_gemm_wgrad_dB", s,
            [&] { return launch_gemm_simt(EPI_STORE_F32, ob, gb, s); }));
    ga.kb_per_seg = T;
    const SimtOperands oa{static_cast<const float*>(Xop), 1, h, fdH, f, 1};
    TRY(run(&H->core, "simt_gemm_wgrad_dA", s,
            [&] { return launch_gemm_simt(EPI_STORE_F32, oa, ga, s); }));
    gx.kb_per_seg = ft;
    const SimtOperands ox{fdH, f, 1, static_cast<const float*>(A), 1, f};
    TRY(run(&H->core, "simt_gemm_dx_shardsum", s,
            [&] { return launch_gemm_simt(EPI_SHARDSUM, ox, gx, s); }));
  }

  if (ln) {
    const float* dXn = reinterpret_cast<const float*>(ws + L.dxn);
    const float* mean = reinterpret_cast<const float*>(ws + L.mean);
    const float* rstd = reinterpret_cast<const float*>(ws + L.rstd);
    float* pg = part1 + size_t(L.groups > L.chunks ? L.groups : L.chunks) * f;
    float* pb = pg + L.lnp * h;
    TRY(ln_backward(&H->core, s, bf16, dXn, X, mean, rstd, ln_gamma, dres, dX,
                    pg, pb, dgamma, dbeta, T, h));
  }
  return TPMLP_OK;
}

// ============================================================ FP8 ====

static int fp8_config_ok(const tp_mlp_config& c) {
  if (c.dtype != TPMLP_BF16) return TPMLP_ERR_ARG;
  if (c.dropout_p > 0.f) return TPMLP_ERR_ARG;
  // A k-block of 128 E4M3 elements must not straddle two shards.
  if ((c.ffn / c.shards) % 128 != 0) return TPMLP_ERR_SHAPE;
  return TPMLP_OK;
}

size_t tp_mlp_fp8_weights_bytes(const tp_mlp_handle* H) {
  if (H == nullptr || fp8_config_ok(H->cfg) != TPMLP_OK) return 0;
  return fp8_pack_layout(H->cfg).total;
}

size_t tp_mlp_fp8_workspace_bytes(const tp_mlp_handle* H, int tokens) {
  if (H == nullptr || tokens < 0 || fp8_config_ok(H->cfg) != TPMLP_OK)
    return 0;
  return fp8_layout(H->cfg, tokens).total;
}

size_t tp_mlp_fp8_train_workspace_bytes(const tp_mlp_handle* H, int tokens) {
  if (H == nullptr || tokens < 0 || fp8_config_ok(H->cfg) != TPMLP_OK)
    return 0;
  return fp8_layout(H->cfg, tokens).train_total;
}

long long tp_mlp_fp8_offset(const tp_mlp_handle* H, int tokens, int which) {
  if (H == nullptr || tokens < 0) return -1;
  const Fp8Pack P = fp8_pack_layout(H->cfg);
  const Fp8Layout L = fp8_layout(H->cfg, tokens);
  switch (which) {
    case TPMLP_FP8_PACK_SCALES: return static_cast<long long>(P.scales);
    case TPMLP_FP8_PACK_AQT: return static_cast<long long>(P.aqt);
    case TPMLP_FP8_PACK_BQT: return static_cast<long long>(P.bqt);
    case TPMLP_FP8_PACK_AQ: return static_cast<long long>(P.aq);
    case TPMLP_FP8_PACK_BQ: return static_cast<long long>(P.bq);
    case TPMLP_FP8_WS_SCALES: return static_cast<long long>(L.scales);
    case TPMLP_FP8_WS_XQ: return static_cast<long long>(L.xq);
    case TPMLP_FP8_WS_Y: return static_cast<long long>(L.y);
    case TPMLP_FP8_WS_YQ: return static_cast<long long>(L.yq);
    case TPMLP_FP8_WS_H: return static_cast<long long>(L.hb);
    case TPMLP_FP8_WS_XQT: return static_cast<long long>(L.xqt);
    case TPMLP_FP8_WS_YQT: return static_cast<long long>(L.yqt);
    case TPMLP_FP8_WS_BSCALES: return static_cast<long long>(L.bscales);
    case TPMLP_FP8_WS_DZQ: return static_cast<long long>(L.dzq);
    case TPMLP_FP8_WS_DZQT: return static_cast<long long>(L.dzqt);
    case TPMLP_FP8_WS_DH: return static_cast<long long>(L.dh);
    case TPMLP_FP8_WS_DHQ: return static_cast<long long>(L.dhq);
    case TPMLP_FP8_WS_DHQT: return static_cast<long long>(L.dhqt);
    default: return -1;
  }
}

int tp_mlp_fp8_pack_weights(tp_mlp_handle* H, const void* A, const void* B,
                            void* packed, size_t packed_bytes, void* stream) {
  if (H == nullptr || !A || !B || !packed) return TPMLP_ERR_ARG;
  TRY(fp8_config_ok(H->cfg));
  const void* ptrs[] = {A, B, packed};
  for (const void* p : ptrs)
    if (!aligned16(p)) return TPMLP_ERR_ALIGN;
  const Fp8Pack P = fp8_pack_layout(H->cfg);
  if (packed_bytes < P.total) return TPMLP_ERR_WORKSPACE;
  int sms = 0;
  TRY(check_device(&sms));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* pk = static_cast<char*>(packed);
  const int h = H->cfg.hidden, f = H->cfg.ffn;
  unsigned int* amax = reinterpret_cast<unsigned int*>(pk + P.scales);
  float* scl = reinterpret_cast<float*>(pk + P.scales) + 2;
  cudaError_t e = cudaMemsetAsync(amax, 0, 8, s);
  if (e != cudaSuccess) {
    set_detail("cudaMemsetAsync(amax)", e);
    return TPMLP_ERR_CUDA;
  }
  TRY(run(&H->core, "fp8_amax_weights", s, [&] {
    return launch_amax_bf16(A, size_t(h) * f, amax, s);
  }));
  TRY(run(&H->core, "fp8_amax_weights", s, [&] {
    return launch_amax_bf16(B, size_t(f) * h, amax + 1, s);
  }));
  // both layouts of each weight from one read
  TRY(run(&H->core, "fp8_quantize_weights", s, [&] {
    return launch_quantize_e4m3_rt(A, h, f, amax,
                                   reinterpret_cast<uint8_t*>(pk + P.aq),
                                   reinterpret_cast<uint8_t*>(pk + P.aqt), h,
                                   scl, s);
  }));
  return run(&H->core, "fp8_quantize_weights", s, [&] {
    return launch_quantize_e4m3_rt(B, f, h, amax + 1,
                                   reinterpret_cast<uint8_t*>(pk + P.bq),
                                   reinterpret_cast<uint8_t*>(pk + P.bqt), f,
                                   scl + 1, s);
  });
}

static int forward_fp8_impl(tp_mlp_handle* H, int tokens, const void* X,
                            const void* packed, const float* bias1,
                            const float* bias2, const float* ln_gamma,
                            const float* ln_beta, void* Z, void* workspace,
                            size_t workspace_bytes, cudaStream_t s,
                            bool train) {
  if (H == nullptr) return TPMLP_ERR_ARG;
  const tp_mlp_config& c = H->cfg;
  TRY(fp8_config_ok(c));
  if (tokens < 0 || tokens > c.max_tokens) return TPMLP_ERR_SHAPE;
  if (!packed || !workspace || (tokens > 0 && (!X || !Z))) return TPMLP_ERR_ARG;
  if (c.use_layernorm && (!ln_gamma || !ln_beta)) return TPMLP_ERR_ARG;
  const void* ptrs[] = {X, packed, Z, workspace, bias1, bias2, ln_gamma, ln_beta};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return TPMLP_ERR_ALIGN;
  const Fp8Layout L = fp8_layout(c, tokens);
  if (workspace_bytes < (train ? L.train_total : L.total))
    return TPMLP_ERR_WORKSPACE;
  int sms = 0;
  TRY(check_device(&sms));
  char* ws = static_cast<char*>(workspace);
  const char* pk = static_cast<const char*>(packed);
  const Fp8Pack P = fp8_pack_layout(c);
  cudaError_t e = cudaMemsetAsync(ws + L.status, 0, 16, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws + L.scales, 0, 8, s);
  if (e != cudaSuccess) {
    set_detail("cudaMemsetAsync(status, amax)", e);
    return TPMLP_ERR_CUDA;
  }
  if (tokens == 0) return TPMLP_OK;
  const int T = tokens, h = c.hidden, f = c.ffn, t = c.shards, ft = f / t;
  const void* Xop = X;
  if (c.use_layernorm) {
    void* Xn = ws + L.xn;
    TRY(run(&H->core, "layernorm_fwd", s, [&] {
      return launch_ln_fwd(true, X, ln_gamma, ln_beta, Xn,
                           reinterpret_cast<float*>(ws + L.mean),
                           reinterpret_cast<float*>(ws + L.rstd), T, h,
                           c.ln_eps, s);
    }));
    Xop = Xn;
  }
  unsigned int* amax = reinterpret_cast<unsigned int*>(ws + L.scales);
  float* scl = reinterpret_cast<float*>(ws + L.scales) + 2;
  const float* wscl = reinterpret_cast<const float*>(pk + P.scales) + 2;
  uint8_t* Xq = reinterpret_cast<uint8_t*>(ws + L.xq);
  void* Y = ws + L.y;
  uint8_t* Yq = reinterpret_cast<uint8_t*>(ws + L.yq);
  TRY(run(&H->core, "fp8_amax_x", s,
          [&] { return launch_amax_bf16(Xop, size_t(T) * h, amax, s); }));
  TRY(run(&H->core, "fp8_quantize_x", s, [&] {
    if (train)  // Xq and, for dA, Xq^T
      return launch_quantize_e4m3_rt(Xop, T, h, amax, Xq,
                                     reinterpret_cast<uint8_t*>(ws + L.xqt),
                                     static_cast<long long>(L.tpitch), scl, s);
    return launch_quantize_e4m3(Xop, size_t(T) * h, amax, Xq, scl, s);
  }));
  CUtensorMap ta, tb, to, to2;
  GemmArgs g1 = base_args(H, ws, L.status);
  g1.M = T; g1.N = f; g1.K = h; g1.kb_per_seg = (h + 127) / 128;
  g1.out = Y; g1.ldo = f; g1.bias = bias1;
  g1.scale_a = scl; g1.scale_b = wscl; g1.amax_out = amax + 1;
  TRY(encode_map_u8(&ta, Xq, h, T, h, TC_BM));
  TRY(encode_map_u8(&tb, pk + P.aqt, h, f, h, TC2_BN_HALF));
  TRY(out_map(&to, Y, false, T, f, f));
  to2 = to;
  if (train) {  // H for GeLU's derivative in the backward
    g1.out2 = ws + L.hb;
    TRY(out_map(&to2, g1.out2, false, T, f, f));
  }
  TRY(run(&H->core, "gemm1_gelu_fp8", s, [&] {
    return launch_gemm_tc2_e4m3(EPI_GELU_FWD, ta, tb, to, to2, g1, sms / 2, s);
  }));
  TRY(run(&H->core, "fp8_quantize_y", s, [&] {
    if (train)  // Yq and, for dB, Yq^T
      return launch_quantize_e4m3_rt(Y, T, f, amax + 1, Yq,
                                     reinterpret_cast<uint8_t*>(ws + L.yqt),
                                     static_cast<long long>(L.tpitch), scl + 1,
                                     s);
    return launch_quantize_e4m3(Y, size_t(T) * f, amax + 1, Yq, scl + 1, s);
  }));
  GemmArgs g2 = base_args(H, ws, L.status);
  g2.M = T; g2.N = h; g2.K = f; g2.num_seg = t; g2.kb_per_seg = ft / 128;
  g2.out = Z; g2.ldo = h; g2.bias = bias2;
  g2.scale_a = scl + 1; g2.scale_b = wscl + 1;
  g2.part = reinterpret_cast<float*>(ws + L.tailp);
  g2.part_bytes = TAIL_PART_BYTES;
  if (c.use_residual) {
    g2.aux = X;
    g2.ldaux = h;
  }
  TRY(encode_map_u8(&ta, Yq, f, T, f, TC_BM));
  TRY(encode_map_u8(&tb, pk + P.bqt, f, h, f, TC2_BN_HALF));
  TRY(out_map(&to2, Z, false, T, h, h));
  return f8_gemm(&H->core, "gemm2_shardsum_fp8", s, sms, EPI_SHARDSUM, ta, tb,
                 to2, to2, g2);
}

int tp_mlp_forward_fp8(tp_mlp_handle* H, int tokens, const void* X,
                       const void* packed, const float* bias1,
                       const float* bias2, const float* ln_gamma,
                       const float* ln_beta, void* Z, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return forward_fp8_impl(H, tokens, X, packed, bias1, bias2, ln_gamma,
                          ln_beta, Z, workspace, workspace_bytes,
                          static_cast<cudaStream_t>(stream), false);
}

int tp_mlp_forward_fp8_train(tp_mlp_handle* H, int tokens, const void* X,
                             const void* packed, const float* bias1,
                             const float* bias2, const float* ln_gamma,
                             const float* ln_beta, void* Z, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return forward_fp8_impl(H, tokens, X, packed, bias1, bias2, ln_gamma,
                          ln_beta, Z, workspace, workspace_bytes,
                          static_cast<cudaStream_t>(stream), true);
}

int tp_mlp_backward_fp8(tp_mlp_handle* H, int tokens, const void* dZ,
                        const void* X, const void* packed,
                        const float* ln_gamma, void* workspace,
                        size_t workspace_bytes, void* dX, float* dA, float* dB,
                        float* dbias1, float* dbias2, float* dgamma,
                        float* dbeta, void* stream) {
  if (H == nullptr) return TPMLP_ERR_ARG;
  const tp_mlp_config& c = H->cfg;
  TRY(fp8_config_ok(c));
  if (tokens < 0 || tokens > c.max_tokens) return TPMLP_ERR_SHAPE;
  if (!packed || !workspace || !dA || !dB ||
      (tokens > 0 && (!dZ || !X || !dX)))
    return TPMLP_ERR_ARG;
  if (c.use_layernorm && !ln_gamma) return TPMLP_ERR_ARG;
  const void* ptrs[] = {dZ, X, packed, ln_gamma, workspace, dX, dA, dB,
                        dbias1, dbias2, dgamma, dbeta};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return TPMLP_ERR_ALIGN;
  const Fp8Layout L = fp8_layout(c, tokens);
  if (workspace_bytes < L.train_total) return TPMLP_ERR_WORKSPACE;
  int sms = 0;
  TRY(check_device(&sms));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const char* pk = static_cast<const char*>(packed);
  const Fp8Pack P = fp8_pack_layout(c);
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

  unsigned int* bamax = reinterpret_cast<unsigned int*>(ws + L.bscales);
  float* bscl = reinterpret_cast<float*>(ws + L.bscales) + 2;  // s_dz, s_dh
  const float* fscl = reinterpret_cast<const float*>(ws + L.scales) + 2;  // s_x, s_y
  const float* wscl = reinterpret_cast<const float*>(pk + P.scales) + 2;  // s_a, s_b
  const cudaError_t e = cudaMemsetAsync(bamax, 0, 8, s);
  if (e != cudaSuccess) {
    set_detail("cudaMemsetAsync(amax)", e);
    return TPMLP_ERR_CUDA;
  }
  const long long tp = static_cast<long long>(L.tpitch);
  uint8_t* dZq = reinterpret_cast<uint8_t*>(ws + L.dzq);
  uint8_t* dZqT = reinterpret_cast<uint8_t*>(ws + L.dzqt);
  void* dH = ws + L.dh;
  uint8_t* dHq = reinterpret_cast<uint8_t*>(ws + L.dhq);
  uint8_t* dHqT = reinterpret_cast<uint8_t*>(ws + L.dhqt);
  float* part = reinterpret_cast<float*>(ws + L.part);
  float* part1 = part + size_t(L.chunks) * h;  // db1 partials

  // dZ: current amax (from the db2 column-sum pass when db2 is wanted, which
  // reads dZ anyway), then codes in both layouts from one read
  if (dbias2) {
    TRY(run(&H->core, "colsum_db2_amax_dz", s, [&] {
      return launch_colsum_partial(true, dZ, part, T, h, s, bamax);
    }));
  } else {
    TRY(run(&H->core, "fp8_amax_dz", s,
            [&] { return launch_amax_bf16(dZ, size_t(T) * h, bamax, s); }));
  }
  TRY(run(&H->core, "fp8_quantize_dz", s, [&] {
    return launch_quantize_e4m3_rt(dZ, T, h, bamax, dZq, dZqT, tp, bscl, s);
  }));
  // dH = (s_dz s_b) (dZq Bq^T) * GeLU'(H), raising amax_dh, with the db1
  // partials of 32-row groups
  CUtensorMap ta, tb, to;
  GemmArgs gy = base_args(H, ws, L.status);
  gy.M = T; gy.N = f; gy.K = h; gy.kb_per_seg = (h + 127) / 128;
  gy.out = dH; gy.ldo = f; gy.aux = ws + L.hb; gy.ldaux = f;
  gy.scale_a = bscl; gy.scale_b = wscl + 1; gy.amax_out = bamax + 1;
  if (dbias1) {
    gy.colsum = part1;
    gy.ld_colsum = f;
  }
  TRY(encode_map_u8(&ta, dZq, h, T, h, TC_BM));
  TRY(encode_map_u8(&tb, pk + P.bq, h, f, h, TC2_BN_HALF));
  CUtensorMap th;  // H, read by the epilogue through a tensor map
  TRY(out_map(&to, dH, false, T, f, f));
  TRY(out_map(&th, ws + L.hb, false, T, f, f));
  TRY(run(&H->core, "gemm_dh_gelu_bwd_fp8", s, [&] {
    return launch_gemm_tc2_e4m3(EPI_GELU_BWD, ta, tb, to, th, gy, sms / 2, s);
  }));
  TRY(run(&H->core, "fp8_quantize_dh", s, [&] {
    return launch_quantize_e4m3_rt(dH, T, f, bamax + 1, dHq, dHqT, tp,
                                   bscl + 1, s);
  }));
  if (dbias2)
    TRY(run(&H->core, "colsum_finalize", s, [&] {
      return launch_colsum_finalize(part, dbias2, L.chunks, h, s);
    }));
  if (dbias1)
    TRY(run(&H->core, "colsum_finalize", s, [&] {
      return launch_colsum_finalize(part1, dbias1, L.groups, f, s);
    }));
  // dB = (s_y s_dz) (Yq^T dZq): K = T over the transposed codes
  const int kbT = (T + 127) / 128;
  GemmArgs gb = base_args(H, ws, L.status);
  gb.M = f; gb.N = h; gb.K = T; gb.kb_per_seg = kbT;
  gb.out = dB; gb.ldo = h;
  gb.scale_a = fscl + 1; gb.scale_b = bscl;
  gb.part = reinterpret_cast<float*>(ws + L.tailp);
  gb.part_bytes = TAIL_PART_BYTES;
  TRY(encode_map_u8(&ta, ws + L.yqt, T, f, tp, TC_BM));
  TRY(encode_map_u8(&tb, dZqT, T, h, tp, TC2_BN_HALF));
  TRY(out_map(&to, dB, true, f, h, h));
  TRY(f8_gemm(&H->core, "gemm_wgrad_dB_fp8", s, sms, EPI_STORE_F32, ta, tb, to,
              to, gb));
  // dA = (s_x s_dh) (Xq^T dHq)
  GemmArgs ga = base_args(H, ws, L.status);
  ga.M = h; ga.N = f; ga.K = T; ga.kb_per_seg = kbT;
  ga.out = dA; ga.ldo = f;
  ga.scale_a = fscl; ga.scale_b = bscl + 1;
  ga.part = reinterpret_cast<float*>(ws + L.tailp);
  ga.part_bytes = TAIL_PART_BYTES;
  TRY(encode_map_u8(&ta, ws + L.xqt, T, h, tp, TC_BM));
  TRY(encode_map_u8(&tb, dHqT, T, f, tp, TC2_BN_HALF));
  TRY(out_map(&to, dA, true, h, f, f));
  TRY(f8_gemm(&H->core, "gemm_wgrad_dA_fp8", s, sms, EPI_STORE_F32, ta, tb, to,
              to, ga));
  // dXn = sum_i (s_dh s_a) (dHq_i Aq_i^T) in shard order: fp32 for the
  // LayerNorm backward, else dX itself (+ dZ with the residual)
  void* dXdst = ln ? static_cast<void*>(ws + L.dxn) : dX;
  GemmArgs gx = base_args(H, ws, L.status);
  gx.M = T; gx.N = h; gx.K = f; gx.num_seg = t; gx.kb_per_seg = ft / 128;
  gx.out = dXdst; gx.ldo = h; gx.out_f32 = ln ? 1 : 0;
  gx.scale_a = bscl + 1; gx.scale_b = wscl;
  gx.part = reinterpret_cast<float*>(ws + L.tailp);
  gx.part_bytes = TAIL_PART_BYTES;
  if (c.use_residual && !ln) {
    gx.aux = dZ;
    gx.ldaux = h;
  }
  TRY(encode_map_u8(&ta, dHq, f, T, f, TC_BM));
  TRY(encode_map_u8(&tb, pk + P.aq, f, h, f, TC2_BN_HALF));
  TRY(out_map(&to, dXdst, ln, T, h, h));
  TRY(f8_gemm(&H->core, "gemm_dx_shardsum_fp8", s, sms, EPI_SHARDSUM, ta, tb,
              to, to, gx));
  if (ln) {
    const float* dXn = reinterpret_cast<const float*>(ws + L.dxn);
    const float* mean = reinterpret_cast<const float*>(ws + L.mean);
    const float* rstd = reinterpret_cast<const float*>(ws + L.rstd);
    const void* dres = c.use_residual ? dZ : nullptr;
    float* pg = part1 + size_t(L.groups > L.chunks ? L.groups : L.chunks) * f;
    float* pb = pg + L.lnp * h;
    TRY(ln_backward(&H->core, s, true, dXn, X, mean, rstd, ln_gamma, dres, dX,
                    pg, pb, dgamma, dbeta, T, h));
  }
  return TPMLP_OK;
}

int tp_mlp_check(tp_mlp_handle* H, void* workspace, void* stream) {
  if (H == nullptr || workspace == nullptr) return TPMLP_ERR_ARG;
  return check_status(workspace, static_cast<cudaStream_t>(stream));
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
    case TPMLP_ERR_CHECK: return "device-side check failed (debug build)";
    default: return "unknown status";
  }
}

const char* tp_mlp_last_detail(void) { return g_detail; }

long long tp_mlp_launch_count(const tp_mlp_handle* handle) {
  return handle ? handle->core.launches : -1;
}

int tp_mlp_set_timing(tp_mlp_handle* handle, int enable) {
  if (handle == nullptr) return TPMLP_ERR_ARG;
  handle->core.timing = enable != 0;
  return TPMLP_OK;
}

int tp_mlp_timing_get(tp_mlp_handle* H, int index, const char** name,
                      long long* launches, double* total_ms) {
  if (H == nullptr) return TPMLP_ERR_ARG;
  return timing_get(&H->core, index, name, launches, total_ms);
}

int tp_mlp_timing_reset(tp_mlp_handle* H) {
  if (H == nullptr) return TPMLP_ERR_ARG;
  timing_get(&H->core, -1, nullptr, nullptr, nullptr);  // drain pending
  H->core.stats.clear();
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
  handle->core.budget_ns = ns;
  return TPMLP_OK;
}

int tp_mlp_set_nvtx(tp_mlp_handle* handle, int enable) {
  if (handle == nullptr || (enable != 0 && enable != 1)) return TPMLP_ERR_ARG;
  handle->core.nvtx = enable != 0;
  return TPMLP_OK;
}

int tp_mlp_set_ln_prologue(tp_mlp_handle* handle, int enable) {
  if (handle == nullptr || (enable != 0 && enable != 1)) return TPMLP_ERR_ARG;
  handle->ln_prologue = enable != 0;
  return TPMLP_OK;
}

}  // extern "C"
