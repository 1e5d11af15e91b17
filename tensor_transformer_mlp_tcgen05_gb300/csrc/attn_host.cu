// Host side of the head-parallel self-attention block: validation,
// workspace layout, tensor maps and launch sequencing.
//
// Forward (Megatron-LM explainer, "Attention: a design that parallelises
// naturally"; Megatron-LM notes, "Self-attention block split"):
//   [LayerNorm] -> QKV = Xn W_qkv + b_qkv (pair GEMM, one column group per
//   shard) -> attention core per (sequence, head, query block) -> Z =
//   sum_i Ctx_i W_o,i + b_o (pair GEMM, fixed-order shard sum = g) [+ X].
// Backward: db_o, dW_o = Ctx^T dZ, dCtx = dZ W_o^T -> dQ and delta =
//   rowsum(dCtx * Ctx) per head (one CTA per query block) -> dK, dV (one CTA
//   per key block) -> db_qkv, dW_qkv = Xn^T dQKV, dXn = sum_i dQKV_i W_qkv,i^T
//   (fixed-order shard sum = f's backward) -> [LayerNorm backward] [+ dZ].
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>

#include "host_common.cuh"
#include "tp_attn.h"

using namespace tpmlp;
using namespace tpmlp::host;

namespace {

struct AttnLayout {
  size_t status = 0, xn = 0, mean = 0, rstd = 0, qkv = 0, ctx = 0, lse = 0,
         dctx = 0, delta = 0, dqkv = 0, dxn = 0, part = 0, tailp = 0,
         total = 0, lnp = 0;
  size_t lnsync_words = 0;   // the LayerNorm prologue's counters
  int chunks = 0;   // 256-row column-sum chunks
  int groups = 0;   // 32-row groups of the core kernels' fused db_qkv partials
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

AttnLayout attn_layout(const tp_attn_config& c, int tokens, int training) {
  AttnLayout L;
  const size_t T = static_cast<size_t>(tokens);
  const size_t h = static_cast<size_t>(c.hidden);
  const size_t H = static_cast<size_t>(c.heads);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  if (c.use_layernorm) {
    // the status word, then the LayerNorm prologue's row counters
    // (GemmArgs::ln_sync: 1 + ceil(T / 128) words)
    L.lnsync_words = 1 + (T + 127) / 128;
    L.status = take(16 + 4 * L.lnsync_words);
  } else {
    L.status = take(256);
  }
  if (c.use_layernorm) {
    L.xn = take(T * h * 2);
    L.mean = take(T * 4);
    L.rstd = take(T * 4);
  }
  L.qkv = take(T * 3 * h * 2);
  L.ctx = take(T * h * 2);
  L.lse = take(H * T * 4);
  L.tailp = take(static_cast<size_t>(TAIL_PART_BYTES));  // GEMM tail split
  if (training) {
    L.dctx = take(T * h * 2);
    L.delta = take(2 * H * T * 4);   // -lse2 and -delta' (AttnArgs::delta)
    L.dqkv = take(T * 3 * h * 2);
    if (c.use_layernorm) L.dxn = take(T * h * 4);
    L.chunks = colsum_chunks(tokens);
    L.groups = (tokens + 31) / 32;
    // db_o (chunks x h), db_qkv (max(groups, chunks) x 3h), dgamma and
    // dbeta (lnp x h each)
    const size_t rows3 = static_cast<size_t>(L.groups > L.chunks ? L.groups : L.chunks);
    L.lnp = static_cast<size_t>(L.chunks);
    L.part = take((static_cast<size_t>(L.chunks) * h + rows3 * 3 * h +
                   2 * L.lnp * h) * 4);
  }
  L.total = off;
  return L;
}

}  // namespace

struct tp_attn_handle {
  HandleCore core;
  tp_attn_config cfg;
  bool ln_prologue = true;   // tp_attn_set_ln_prologue
};

namespace {

GemmArgs gemm_args(const tp_attn_handle* H, char* ws, const AttnLayout& L) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.group_m = 16;
  a.status = reinterpret_cast<int*>(ws + L.status);
  a.budget_ns = H->core.budget_ns;
  a.num_seg = 1;
  a.part = reinterpret_cast<float*>(ws + L.tailp);
  a.part_bytes = TAIL_PART_BYTES;
  return a;
}

AttnArgs core_args(const tp_attn_handle* H, char* ws, const AttnLayout& L,
                   int tokens) {
  const tp_attn_config& c = H->cfg;
  AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.heads = c.heads;
  a.heads_per_shard = c.heads / c.shards;
  a.head_dim = c.hidden / c.heads;
  a.shard_width = c.hidden / c.shards;
  a.seq_len = c.seq_len;
  a.nq = c.seq_len / 128;
  a.causal = c.causal;
  a.scale_log2 = static_cast<float>(1.4426950408889634 /
                                    std::sqrt(static_cast<double>(a.head_dim)));
  a.ctx = reinterpret_cast<__nv_bfloat16*>(ws + L.ctx);
  a.ld_ctx = c.hidden;
  a.lse = reinterpret_cast<float*>(ws + L.lse);
  a.ld_stat = tokens;
  a.ld_qkv = 3LL * c.hidden;
  a.status = reinterpret_cast<int*>(ws + L.status);
  a.budget_ns = H->core.budget_ns;
  return a;
}

int check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return TPMLP_ERR_ALIGN;
  return TPMLP_OK;
}

}  // namespace

extern "C" {

int tp_attn_create(const tp_attn_config* cfg, tp_attn_handle** out) {
  if (cfg == nullptr || out == nullptr) return TPMLP_ERR_ARG;
  if ((cfg->causal != 0 && cfg->causal != 1) ||
      (cfg->use_layernorm != 0 && cfg->use_layernorm != 1) ||
      (cfg->use_residual != 0 && cfg->use_residual != 1))
    return TPMLP_ERR_ARG;
  if (cfg->use_layernorm && !(cfg->ln_eps >= 0.f && std::isfinite(cfg->ln_eps)))
    return TPMLP_ERR_ARG;
  if (cfg->hidden <= 0 || cfg->heads <= 0 || cfg->shards <= 0 ||
      cfg->seq_len <= 0 || cfg->max_tokens < 0)
    return TPMLP_ERR_SHAPE;
  if (cfg->hidden % cfg->heads != 0 || cfg->heads % cfg->shards != 0)
    return TPMLP_ERR_SHAPE;
  const int d = cfg->hidden / cfg->heads;
  if (d != 64 && d != 96 && d != 128) return TPMLP_ERR_SHAPE;
  if ((cfg->hidden / cfg->shards) % 64 != 0) return TPMLP_ERR_SHAPE;
  if (cfg->seq_len % 128 != 0) return TPMLP_ERR_SHAPE;
  if (static_cast<long long>(cfg->max_tokens) > (1LL << 28) ||
      cfg->hidden > (1 << 20))
    return TPMLP_ERR_SHAPE;
  tp_attn_handle* h = new (std::nothrow) tp_attn_handle();
  if (h == nullptr) return TPMLP_ERR_ARG;
  h->cfg = *cfg;
  *out = h;
  return TPMLP_OK;
}

int tp_attn_destroy(tp_attn_handle* handle) {
  delete handle;
  return TPMLP_OK;
}

size_t tp_attn_workspace_bytes(const tp_attn_handle* handle, int tokens,
                               int training) {
  if (handle == nullptr || tokens < 0) return 0;
  return attn_layout(handle->cfg, tokens, training ? 1 : 0).total;
}

long long tp_attn_workspace_offset(const tp_attn_handle* handle, int tokens,
                                   int training, int which) {
  if (handle == nullptr || tokens < 0) return -1;
  const AttnLayout L = attn_layout(handle->cfg, tokens, training ? 1 : 0);
  switch (which) {
    case TPATTN_WS_QKV: return static_cast<long long>(L.qkv);
    case TPATTN_WS_CTX: return static_cast<long long>(L.ctx);
    case TPATTN_WS_LSE: return static_cast<long long>(L.lse);
    case TPATTN_WS_DQKV:
      return training ? static_cast<long long>(L.dqkv) : -1;
    default: return -1;
  }
}

int tp_attn_forward(tp_attn_handle* H, int tokens, const void* X,
                    const void* Wqkv, const void* Wo, const float* bqkv,
                    const float* bo, const float* ln_gamma,
                    const float* ln_beta, void* Z, void* workspace,
                    size_t workspace_bytes, int training, void* stream) {
  if (H == nullptr) return TPMLP_ERR_ARG;
  const tp_attn_config& c = H->cfg;
  if (tokens < 0 || tokens > c.max_tokens || tokens % c.seq_len != 0)
    return TPMLP_ERR_SHAPE;
  if (!Wqkv || !Wo || !workspace || (tokens > 0 && (!X || !Z)))
    return TPMLP_ERR_ARG;
  if (c.use_layernorm && (!ln_gamma || !ln_beta)) return TPMLP_ERR_ARG;
  TRY(check_ptrs({X, Wqkv, Wo, bqkv, bo, ln_gamma, ln_beta, Z, workspace}));
  const AttnLayout L = attn_layout(c, tokens, training ? 1 : 0);
  if (workspace_bytes < L.total) return TPMLP_ERR_WORKSPACE;
  int sms = 0;
  TRY(check_device(&sms));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  // LayerNorm inside the QKV projection's launch (GemmArgs::ln_x)
  const bool ln_fused = c.use_layernorm && H->ln_prologue &&
                        c.hidden % 256 == 0 && c.hidden / 256 <= LN_VMAX;
  // the status word, and with the fused LayerNorm its counters, cleared
  const size_t clear = ln_fused ? 16 + 4 * L.lnsync_words : 16;
  cudaError_t e = cudaMemsetAsync(ws + L.status, 0, clear, s);
  if (e != cudaSuccess) {
    set_detail("cudaMemsetAsync(status)", e);
    return TPMLP_ERR_CUDA;
  }
  if (tokens == 0) return TPMLP_OK;

  const int T = tokens, h = c.hidden, ht = h / c.shards;
  const void* Xop = X;
  if (ln_fused) {
    Xop = ws + L.xn;
  } else if (c.use_layernorm) {
    void* Xn = ws + L.xn;
    TRY(run(&H->core, "layernorm_fwd", s, [&] {
      return launch_ln_fwd(true, X, ln_gamma, ln_beta, Xn,
                           reinterpret_cast<float*>(ws + L.mean),
                           reinterpret_cast<float*>(ws + L.rstd), T, h,
                           c.ln_eps, s);
    }));
    Xop = Xn;
  }
  CUtensorMap ta, tb;
  // QKV = Xn W_qkv + b_qkv
  GemmArgs gq = gemm_args(H, ws, L);
  gq.M = T; gq.N = 3 * h; gq.K = h; gq.kb_per_seg = h / TC_BK;
  gq.out = ws + L.qkv; gq.ldo = 3LL * h; gq.bias = bqkv;
  if (ln_fused) {
    gq.ln_x = static_cast<const __nv_bfloat16*>(X);
    gq.ln_gamma = ln_gamma;
    gq.ln_beta = ln_beta;
    gq.ln_xn = reinterpret_cast<__nv_bfloat16*>(ws + L.xn);
    gq.ln_mean = reinterpret_cast<float*>(ws + L.mean);
    gq.ln_rstd = reinterpret_cast<float*>(ws + L.rstd);
    gq.ln_eps = c.ln_eps;
    gq.ln_sync = reinterpret_cast<unsigned int*>(ws + L.status + 16);
  }
  TRY(kmajor_map(&ta, Xop, T, h, TC_BM));
  TRY(mnmajor_map(&tb, Wqkv, h, 3 * h));
  TRY(tc_gemm(&H->core, ln_fused ? "gemm_ln_qkv" : "gemm_qkv", s, sms,
              EPI_BIAS_BF16, false, true, ta, tb, gq));
  // attention core
  AttnArgs aa = core_args(H, ws, L, T);
  CUtensorMap tqk, tv;
  TRY(encode_map(&tqk, ws + L.qkv, 3ULL * h, T, 3ULL * h, 128));
  TRY(encode_map(&tv, ws + L.qkv, 3ULL * h, T, 3ULL * h, 64));
  // persistent forward: two CTAs per SM walk the items, one group of
  // (sequence, head) pairs per round
  const int items = (T / c.seq_len) * c.heads * aa.nq;
  const int grid = std::min(items, 2 * sms);
  aa.hs_group = std::max(1, grid / aa.nq);
  TRY(run(&H->core, "attn_fwd", s,
          [&] { return launch_attn_fwd(tqk, tv, aa, grid, s); }));
  // Z = sum_i Ctx_i W_o,i + b_o [+ X]
  GemmArgs go = gemm_args(H, ws, L);
  go.M = T; go.N = h; go.K = h; go.num_seg = c.shards;
  go.kb_per_seg = ht / TC_BK;
  go.out = Z; go.ldo = h; go.bias = bo;
  if (c.use_residual) {
    go.aux = X;
    go.ldaux = h;
  }
  TRY(kmajor_map(&ta, ws + L.ctx, T, h, TC_BM));
  TRY(mnmajor_map(&tb, Wo, h, h));
  return tc_gemm(&H->core, "gemm_out_shardsum", s, sms, EPI_SHARDSUM, false,
                 true, ta, tb, go);
}

int tp_attn_backward(tp_attn_handle* H, int tokens, const void* dZ,
                     const void* X, const void* Wqkv, const void* Wo,
                     const float* ln_gamma, void* workspace,
                     size_t workspace_bytes, void* dX, float* dWqkv,
                     float* dWo, float* dbqkv, float* dbo, float* dgamma,
                     float* dbeta, void* stream) {
  if (H == nullptr) return TPMLP_ERR_ARG;
  const tp_attn_config& c = H->cfg;
  if (tokens < 0 || tokens > c.max_tokens || tokens % c.seq_len != 0)
    return TPMLP_ERR_SHAPE;
  if (!Wqkv || !Wo || !workspace || !dWqkv || !dWo ||
      (tokens > 0 && (!dZ || !X || !dX)))
    return TPMLP_ERR_ARG;
  if (c.use_layernorm && !ln_gamma) return TPMLP_ERR_ARG;
  TRY(check_ptrs({dZ, X, Wqkv, Wo, ln_gamma, workspace, dX, dWqkv, dWo, dbqkv,
                  dbo, dgamma, dbeta}));
  const AttnLayout L = attn_layout(c, tokens, 1);
  if (workspace_bytes < L.total) return TPMLP_ERR_WORKSPACE;
  int sms = 0;
  TRY(check_device(&sms));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const int T = tokens, h = c.hidden, ht = h / c.shards;
  const bool ln = c.use_layernorm != 0;

  if (T == 0) {
    struct Zero {
      void* p;
      size_t n;
    } zs[] = {{dWqkv, size_t(h) * 3 * h * 4}, {dWo, size_t(h) * h * 4},
              {dbqkv, size_t(3) * h * 4},      {dbo, size_t(h) * 4},
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

  float* part = reinterpret_cast<float*>(ws + L.part);
  const void* Xop = ln ? static_cast<const void*>(ws + L.xn) : X;
  void* ctx = ws + L.ctx;
  void* dctx = ws + L.dctx;
  void* dqkv = ws + L.dqkv;
  CUtensorMap ta, tb;
  const int kbT = (T + TC_BK - 1) / TC_BK;

  if (dbo) TRY(colsum(&H->core, "colsum_dbo", s, true, dZ, part, dbo, T, h));
  // dW_o = Ctx^T dZ
  GemmArgs gw = gemm_args(H, ws, L);
  gw.M = h; gw.N = h; gw.K = T; gw.kb_per_seg = kbT;
  gw.out = dWo; gw.ldo = h;
  TRY(mnmajor_map(&ta, ctx, T, h));
  TRY(mnmajor_map(&tb, dZ, T, h));
  TRY(tc_gemm(&H->core, "gemm_wgrad_dWo", s, sms, EPI_STORE_F32, true, true, ta,
              tb, gw));
  // dCtx = dZ W_o^T
  GemmArgs gc = gemm_args(H, ws, L);
  gc.M = T; gc.N = h; gc.K = h; gc.kb_per_seg = h / TC_BK;
  gc.out = dctx; gc.ldo = h;
  TRY(kmajor_map(&ta, dZ, T, h, TC_BM));
  TRY(kmajor_map(&tb, Wo, h, h, TC2_BN_HALF));
  TRY(tc_gemm(&H->core, "gemm_dctx", s, sms, EPI_BIAS_BF16, false, false, ta,
              tb, gc));
  // attention core backward
  AttnArgs aa = core_args(H, ws, L, T);
  aa.dctx = static_cast<const __nv_bfloat16*>(dctx);
  aa.delta = reinterpret_cast<float*>(ws + L.delta);
  aa.dqkv = static_cast<__nv_bfloat16*>(dqkv);
  CUtensorMap tq128, tq64, tdo128, tdo64, tctx128, tdqkv_out;
  TRY(encode_map(&tq128, ws + L.qkv, 3ULL * h, T, 3ULL * h, 128));
  TRY(encode_map(&tq64, ws + L.qkv, 3ULL * h, T, 3ULL * h, 64));
  TRY(encode_map(&tdo128, dctx, h, T, h, 128));
  TRY(encode_map(&tdo64, dctx, h, T, h, 64));
  TRY(encode_map(&tctx128, ctx, h, T, h, 128));
  TRY(out_map(&tdqkv_out, dqkv, false, T, 3 * h, 3LL * h));
  const int grid = (T / c.seq_len) * c.heads * aa.nq;
  aa.hs_group = std::max(1, sms / aa.nq);   // one backward CTA per SM
  // db_qkv = sum_T dQKV: both kernels write 32-row partials of what they
  // store (the chunks they stage for their TMA stores, and at d = 96 the
  // 32-column tails); one fixed-order pass sums them
  float* part3 = part + size_t(L.chunks) * h;
  const bool fused_dbqkv = dbqkv != nullptr;
  if (fused_dbqkv) {
    aa.colsum = part3;
    aa.ld_colsum = 3LL * h;
  }
  // the query kernel also writes delta = rowsum(dCtx * Ctx), which the
  // key/value kernel reads
  TRY(run(&H->core, "attn_bwd_dq", s, [&] {
    return launch_attn_dq(tq128, tq64, tdo128, tctx128, tdqkv_out, aa, grid, s);
  }));
  TRY(run(&H->core, "attn_bwd_dkdv", s, [&] {
    return launch_attn_dkdv(tq128, tq64, tdo64, tdqkv_out, aa, grid, s);
  }));
  if (fused_dbqkv) {
    TRY(run(&H->core, "colsum_finalize", s, [&] {
      return launch_colsum_finalize(part3, dbqkv, L.groups, 3 * h, s);
    }));
  }
  // dW_qkv = Xn^T dQKV
  GemmArgs gwq = gemm_args(H, ws, L);
  gwq.M = h; gwq.N = 3 * h; gwq.K = T; gwq.kb_per_seg = kbT;
  gwq.out = dWqkv; gwq.ldo = 3LL * h;
  TRY(mnmajor_map(&ta, Xop, T, h));
  TRY(mnmajor_map(&tb, dqkv, T, 3 * h));
  TRY(tc_gemm(&H->core, "gemm_wgrad_dWqkv", s, sms, EPI_STORE_F32, true, true,
              ta, tb, gwq));
  // dXn = sum_i dQKV_i W_qkv,i^T (segment i = shard i's 3 h_t columns)
  GemmArgs gx = gemm_args(H, ws, L);
  gx.M = T; gx.N = h; gx.K = 3 * h; gx.num_seg = c.shards;
  gx.kb_per_seg = 3 * ht / TC_BK;
  gx.out = ln ? static_cast<void*>(ws + L.dxn) : dX;
  gx.ldo = h;
  gx.out_f32 = ln ? 1 : 0;
  if (c.use_residual && !ln) {
    gx.aux = dZ;
    gx.ldaux = h;
  }
  TRY(kmajor_map(&ta, dqkv, T, 3 * h, TC_BM));
  TRY(kmajor_map(&tb, Wqkv, h, 3 * h, TC2_BN_HALF));
  TRY(tc_gemm(&H->core, "gemm_dx_shardsum", s, sms, EPI_SHARDSUM, false, false,
              ta, tb, gx));
  if (ln) {
    const float* dXn = reinterpret_cast<const float*>(ws + L.dxn);
    const float* mean = reinterpret_cast<const float*>(ws + L.mean);
    const float* rstd = reinterpret_cast<const float*>(ws + L.rstd);
    const void* dres = c.use_residual ? dZ : nullptr;
    float* pg = part3 + size_t(L.groups > L.chunks ? L.groups : L.chunks) * 3 * h;
    float* pb = pg + L.lnp * h;
    TRY(ln_backward(&H->core, s, true, dXn, X, mean, rstd, ln_gamma, dres, dX,
                    pg, pb, dgamma, dbeta, T, h));
  }
  return TPMLP_OK;
}

int tp_attn_check(tp_attn_handle* H, void* workspace, void* stream) {
  if (H == nullptr || workspace == nullptr) return TPMLP_ERR_ARG;
  return check_status(workspace, static_cast<cudaStream_t>(stream));
}

long long tp_attn_launch_count(const tp_attn_handle* handle) {
  return handle ? handle->core.launches : -1;
}

int tp_attn_set_timing(tp_attn_handle* handle, int enable) {
  if (handle == nullptr) return TPMLP_ERR_ARG;
  handle->core.timing = enable != 0;
  return TPMLP_OK;
}

int tp_attn_timing_get(tp_attn_handle* H, int index, const char** name,
                       long long* launches, double* total_ms) {
  if (H == nullptr) return TPMLP_ERR_ARG;
  return timing_get(&H->core, index, name, launches, total_ms);
}

int tp_attn_timing_reset(tp_attn_handle* H) {
  if (H == nullptr) return TPMLP_ERR_ARG;
  timing_get(&H->core, -1, nullptr, nullptr, nullptr);
  H->core.stats.clear();
  return TPMLP_OK;
}

int tp_attn_set_nvtx(tp_attn_handle* handle, int enable) {
  if (handle == nullptr || (enable != 0 && enable != 1)) return TPMLP_ERR_ARG;
  handle->core.nvtx = enable != 0;
  return TPMLP_OK;
}

int tp_attn_set_ln_prologue(tp_attn_handle* handle, int enable) {
  if (handle == nullptr || (enable != 0 && enable != 1)) return TPMLP_ERR_ARG;
  handle->ln_prologue = enable != 0;
  return TPMLP_OK;
}

int tp_attn_set_wait_budget(tp_attn_handle* handle, unsigned long long ns) {
  if (handle == nullptr) return TPMLP_ERR_ARG;
  handle->core.budget_ns = ns;
  return TPMLP_OK;
}

}  // extern "C"
