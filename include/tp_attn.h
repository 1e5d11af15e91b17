/*
 * tp_attn.h - C ABI of libtpmlp's head-parallel self-attention block on one
 * GB300 (sm_103a).  Status codes, tp_mlp_status_string() and
 * tp_mlp_last_detail() are shared with tp_mlp.h.
 *
 * What the block computes (Megatron-LM explainer, azimuth.plus, section
 * "Attention: a design that parallelises naturally"; Megatron-LM notes,
 * notes.yuuk.io, section "Self-attention block split"): the heads are
 * independent, so the Q, K and V projections are split by columns head
 * group by head group, each shard runs the attention of its own heads with
 * no communication, and the output projection W_o is split by rows, with one
 * all-reduce (operator g) after it - the pattern of the MLP block:
 *
 *     Xn     = LayerNorm(X)                optional pre-LN
 *     QKV    = Xn W_qkv + b_qkv            W_qkv [h, 3h], shard-grouped
 *     Ctx_j  = softmax(Q_j K_j^T / sqrt(d) [causal mask]) V_j   per head j
 *     Z      = sum_{i=0}^{t-1} Ctx_i W_o,i + b_o     W_o split by rows
 *     [Z    += X]                          optional residual
 *
 * The t shards are logical; g becomes a fixed-order sum of fresh fp32
 * partials in the output GEMM's epilogue (and f's backward the same sum in
 * the dX GEMM), so repeated calls are bit-identical.  The attention backward
 * gives every output element one writer (the key/value gradients from one
 * kernel, the query gradients from another that recomputes the scores), so
 * it needs no atomics either.
 *
 * Conventions
 * -----------
 * - Shapes: T = tokens = batches * seq_len (sequence-major rows), h = hidden,
 *   H = heads, d = h / H, t = shards, h_t = h / t, H_t = H / t.
 * - W_qkv [h, 3h] columns are grouped by shard: shard i owns columns
 *   [3 i h_t, 3 (i+1) h_t) = [Q_i | K_i | V_i], each h_t wide, holding heads
 *   i H_t .. (i+1) H_t - 1 in order (head j of shard i at offset
 *   (j - i H_t) d inside each group).  b_qkv [3h] likewise.  The context
 *   Ctx [T, h] holds head j in columns [j d, (j+1) d), so row block i of
 *   W_o [h, h] belongs to shard i.  b_o [h] is added once, after the sum.
 * - Element types: X, W_qkv, W_o, Z, dZ, dX are bf16; biases, LayerNorm
 *   parameters and all weight, bias and LayerNorm gradients are fp32.
 *   Accumulation is fp32 throughout.
 * - Pointers are DEVICE pointers the caller owns, 16-byte aligned; the
 *   library never allocates device memory.  Calls only enqueue work on
 *   `stream` (a cudaStream_t as void*); tp_attn_check() waits and reports
 *   device-side errors.  Every function returns a status code and touches
 *   no output when argument validation fails.
 */
#ifndef TP_ATTN_H_
#define TP_ATTN_H_

#include <stddef.h>

#include "tp_mlp.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tp_attn_config {
  int   hidden;          /* h; multiple of 64                                */
  int   heads;           /* H; d = h / H must be 64, 96 or 128; H % t == 0   */
  int   shards;          /* t; h_t = h / t multiple of 64                    */
  int   max_tokens;      /* largest T any call will pass                     */
  int   seq_len;         /* tokens per sequence; multiple of 128             */
  int   causal;          /* 1: query i sees keys j <= i of its sequence      */
  int   use_layernorm;   /* 1: pre-LayerNorm on X                            */
  float ln_eps;          /* LayerNorm epsilon (e.g. 1e-5)                    */
  int   use_residual;    /* 1: Z = X + block(X)                              */
} tp_attn_config;

typedef struct tp_attn_handle tp_attn_handle;

/* Validates the configuration (TPMLP_ERR_ARG / TPMLP_ERR_SHAPE) and creates
 * a host-side handle.  No device work. */
int tp_attn_create(const tp_attn_config* config, tp_attn_handle** handle);
int tp_attn_destroy(tp_attn_handle* handle);

/* Workspace bytes for `tokens` tokens; training = 1 sizes it for
 * tp_attn_forward(training = 1) followed by tp_attn_backward on the same
 * workspace.  It holds the status word, [Xn, mean, rstd], QKV [T, 3h] bf16,
 * Ctx [T, h] bf16, the softmax log-sum-exp [H, T] fp32 and, for training,
 * the backward's intermediates.  Returns 0 for a NULL handle or T < 0. */
size_t tp_attn_workspace_bytes(const tp_attn_handle* handle, int tokens,
                               int training);

/* Forward pass.
 *   tokens     T, a multiple of seq_len, 0 <= T <= max_tokens (T = 0
 *              enqueues nothing; X and Z may then be NULL)
 *   X [T,h]    input (bf16);  Wqkv [h,3h], Wo [h,h] bf16 weights
 *   bqkv [3h], bo [h]   fp32 biases, each may be NULL (zero)
 *   ln_gamma, ln_beta [h] fp32, required iff use_layernorm
 *   Z [T,h]    output (bf16), overwritten
 *   workspace  >= tp_attn_workspace_bytes(handle, T, training) bytes; with
 *              training = 1 it must reach tp_attn_backward unchanged. */
int tp_attn_forward(tp_attn_handle* handle, int tokens, const void* X,
                    const void* Wqkv, const void* Wo, const float* bqkv,
                    const float* bo, const float* ln_gamma,
                    const float* ln_beta, void* Z, void* workspace,
                    size_t workspace_bytes, int training, void* stream);

/* Backward pass given dZ:
 *   dbo = sum_T dZ;  dWo = Ctx^T dZ;  dCtx = dZ Wo^T;
 *   per sequence and head: dV = P^T dO, dP = dO V^T,
 *   dS = P * (dP - rowsum(dO * O)), dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d);
 *   dbqkv = sum_T dQKV;  dWqkv = Xn^T dQKV;
 *   dXn = sum_{i=0}^{t-1} dQKV_i Wqkv_i^T (fixed shard order);
 *   dX = LayerNorm-backward(dXn) (or dXn) [+ dZ with the residual].
 *   dZ [T,h] bf16; X, Wqkv, Wo, ln_gamma as passed to the forward call;
 *   workspace  the forward call's (training = 1), unchanged;
 *   dX [T,h] bf16; dWqkv [h,3h], dWo [h,h] fp32: overwritten;
 *   dbqkv [3h], dbo [h], dgamma, dbeta [h] fp32: overwritten, each may be
 *   NULL to skip it.  With T = 0 the weight and bias gradients are zeroed. */
int tp_attn_backward(tp_attn_handle* handle, int tokens, const void* dZ,
                     const void* X, const void* Wqkv, const void* Wo,
                     const float* ln_gamma, void* workspace,
                     size_t workspace_bytes, void* dX, float* dWqkv,
                     float* dWo, float* dbqkv, float* dbo, float* dgamma,
                     float* dbeta, void* stream);

/* Waits for `stream`, then reads and clears the workspace's status word:
 * TPMLP_OK, TPMLP_ERR_TIMEOUT (a bounded device wait gave up; outputs of
 * that call are undefined) or TPMLP_ERR_CUDA. */
int tp_attn_check(tp_attn_handle* handle, void* workspace, void* stream);

/* Kernel launches issued through this handle so far; -1 for NULL. */
long long tp_attn_launch_count(const tp_attn_handle* handle);

/* Per-kernel CUDA-event timing, as tp_mlp_set_timing / tp_mlp_timing_get /
 * tp_mlp_timing_reset; bounded-wait budget as tp_mlp_set_wait_budget. */
int tp_attn_set_timing(tp_attn_handle* handle, int enable);
int tp_attn_timing_get(tp_attn_handle* handle, int index, const char** name,
                       long long* launches, double* total_ms);
int tp_attn_timing_reset(tp_attn_handle* handle);
int tp_attn_set_wait_budget(tp_attn_handle* handle, unsigned long long ns);
/* NVTX ranges around each launch, as tp_mlp_set_nvtx. */
int tp_attn_set_nvtx(tp_attn_handle* handle, int enable);

/* Enable (1, the default) or disable (0) the fused pre-LayerNorm prologue
 * of the forward (pre-LN placement: Megatron-LM explainer, "Fixing BERT:
 * reordering layer normalisation for scaling"), as tp_mlp_set_ln_prologue
 * for the MLP block: with use_layernorm and hidden = 256 v for v <= 24, the
 * QKV projection's launch normalises the token rows itself (its epilogue
 * warps, before their first tile) and loads each 128-row block of its A
 * operand once written; otherwise a stand-alone LayerNorm kernel runs
 * first.  Both compute the same bits.  TPMLP_ERR_ARG for a NULL handle or
 * another value. */
int tp_attn_set_ln_prologue(tp_attn_handle* handle, int enable);

/* Offsets in bytes, inside a workspace laid out for (tokens, training), of
 * the saved QKV [T,3h] bf16, Ctx [T,h] bf16, log-sum-exp [H,T] fp32 and
 * (training layouts only) dQKV [T,3h] bf16, for inspection by tests; -1 for
 * a NULL handle or an unknown `which`.  The log-sum-exp is kept in base 2 of
 * the scores scaled by log2(e)/sqrt(d): lse2 = log2 sum_j 2^(s_j log2(e) /
 * sqrt(d)), i.e. the natural-log value times log2(e). */
long long tp_attn_workspace_offset(const tp_attn_handle* handle, int tokens,
                                   int training, int which);
#define TPATTN_WS_QKV 0
#define TPATTN_WS_CTX 1
#define TPATTN_WS_LSE 2
#define TPATTN_WS_DQKV 3

#ifdef __cplusplus
}
#endif

#endif /* TP_ATTN_H_ */
