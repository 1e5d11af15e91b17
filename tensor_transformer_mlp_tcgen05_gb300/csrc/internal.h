// Launchers shared between the translation units of libtpmlp (host side).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace tpmlp {

// Tensor-core GEMM k-blocks are 64 deep (one 128-byte swizzle row of
// bf16); each CTA stages 128 rows of the A operand (the box height of
// K-major A maps).
constexpr int TC_BM = 128;
constexpr int TC_BK = 64;

// D = Aop * Bop on CTA pairs (tcgen05 cta_group::2, 256 x 256 tile per
// pair).  a_mn / b_mn select M/N-major operands (the tensor map's innermost
// dimension runs along M or N) instead of K-major ones.  Supported
// combinations: (K, MN, GELU_FWD), (K, MN, SHARDSUM), (K, K, GELU_BWD),
// (K, K, SHARDSUM), (MN, MN, STORE_F32), (K, MN or K, BIAS_BF16).
// K-major B operands must be encoded with 128-row boxes (each CTA stages half
// of the tile's N).  Outputs are written through tensor maps: `to` for
// args.out and `to2` for args.out2 (EPI_GELU_FWD's H), 128-byte-swizzled
// boxes of 32 rows x 128 bytes (64 bf16 or 32 fp32 columns); EPI_GELU_BWD
// reads H (args.aux) through `to2`, encoded the same way.  At most
// `max_pairs` clusters are launched.
constexpr int TC2_BN_HALF = 128;
// The tail split a pair-GEMM launch used (see GemmArgs::part); tail = 0
// when it used none.  launch_gemm_tc2_tail then combines the partials.
struct TailPlan {
  int tail = 0, pieces = 0, nslots = 0;
  int num_full = 0, num_msup = 0, num_n = 0, group_sup = 0;
};
// Partial-sum capacity the library's workspaces reserve for the tail split.
constexpr long long TAIL_PART_BYTES = 64ll << 20;
cudaError_t launch_gemm_tc2(int epi, bool a_mn, bool b_mn,
                            const CUtensorMap& ta, const CUtensorMap& tb,
                            const CUtensorMap& to, const CUtensorMap& to2,
                            const GemmArgs& args, int max_pairs,
                            cudaStream_t stream, TailPlan* plan = nullptr);
// Combine a tail split's partials (fixed order) and apply the launch's
// epilogue to the tail super-tiles: EPI_SHARDSUM (bias, dropout, residual,
// bf16 or fp32 output, bitwise equal to the unsplit epilogue) or
// EPI_STORE_F32.  `args` as given to the GEMM launch.
cudaError_t launch_gemm_tc2_tail(int epi, const GemmArgs& args,
                                 const TailPlan& plan, cudaStream_t stream);

// The pair GEMM on E4M3 operands (both K-major, 8-bit tensor maps with
// 128 x 128-byte boxes; args.kb_per_seg counts 128-element k-blocks;
// args.scale_a and args.scale_b required).  Epilogues EPI_GELU_FWD and
// EPI_GELU_BWD (each optionally raising args.amax_out to the largest |out|
// stored; EPI_GELU_BWD also with the args.colsum partials), EPI_SHARDSUM and
// EPI_STORE_F32.
cudaError_t launch_gemm_tc2_e4m3(int epi, const CUtensorMap& ta,
                                 const CUtensorMap& tb, const CUtensorMap& to,
                                 const CUtensorMap& to2, const GemmArgs& args,
                                 int max_pairs, cudaStream_t stream,
                                 TailPlan* plan = nullptr);

// FP8 helpers (csrc/fp8.cu).  amax: *amax = max(*amax, max |x|) as fp32
// bits (the caller zeroes it first).  Quantization: s = amax / 448 in fp32
// (1 when amax = 0), q = e4m3(x / s) rounded to nearest even with
// saturation; scale_out (nullable) receives s.
cudaError_t launch_amax_bf16(const void* x, size_t n, unsigned int* amax,
                             cudaStream_t stream);
cudaError_t launch_quantize_e4m3(const void* x, size_t n,
                                 const unsigned int* amax, uint8_t* q,
                                 float* scale_out, cudaStream_t stream);
// Quantization of a bf16 [rows, cols] matrix into both layouts from one
// read: q_row [rows, cols] (nullable) and qt [cols,
// ld_t] (element (r, c) at qt[c * ld_t + r], ld_t >= rows; columns past
// `rows` are left untouched).
cudaError_t launch_quantize_e4m3_rt(const void* x, int rows, int cols,
                                    const unsigned int* amax, uint8_t* q_row,
                                    uint8_t* qt, long long ld_t,
                                    float* scale_out, cudaStream_t stream);

// fp32 CUDA-core GEMM with the same epilogues.  Element (m, k) of the first
// operand is a[m * a_sm + k * a_sk]; element (k, n) of the second is
// b[k * b_sk + n * b_sn].  args.kb_per_seg is the shard segment length in K.
struct SimtOperands {
  const float* a;
  long long a_sm, a_sk;
  const float* b;
  long long b_sk, b_sn;
};
cudaError_t launch_gemm_simt(int epi, const SimtOperands& ops,
                             const GemmArgs& args, cudaStream_t stream);

// LayerNorm forward: Xn = (X - mean) * rstd * gamma + beta per row of h.
cudaError_t launch_ln_fwd(bool bf16, const void* X, const float* gamma,
                          const float* beta, void* Xn, float* mean,
                          float* rstd, int rows, int h, float eps,
                          cudaStream_t stream);

// LayerNorm backward for dX given dXn (fp32); dres (nullable, element type
// of X) is added to dX (the residual connection's gradient).
cudaError_t launch_ln_bwd(bool bf16, const float* dXn, const void* X,
                          const float* mean, const float* rstd,
                          const float* gamma, const void* dres, void* dX,
                          int rows, int h, cudaStream_t stream);

// Rows per chunk of the two-stage fixed-order column sums.
constexpr int COLSUM_CHUNK_ROWS = 256;
inline int colsum_chunks(int rows) {
  return (rows + COLSUM_CHUNK_ROWS - 1) / COLSUM_CHUNK_ROWS;
}

// part[chunk][c] = sum over the chunk's rows of src[r][c] (src bf16/fp32).
// amax (nullable): raised to the largest |src| (fp32 bits), as
// launch_amax_bf16 does, from the same read.
cudaError_t launch_colsum_partial(bool bf16, const void* src, float* part,
                                  int rows, int cols, cudaStream_t stream,
                                  unsigned int* amax = nullptr);

// LayerNorm parameter gradients, stage 1: part_g[chunk][c] = sum dXn * xhat,
// part_b[chunk][c] = sum dXn over the chunk's rows (colsum_chunks(rows)
// chunks; the chunks are visited last first, so that the rows the LayerNorm
// backward read last are still in L2).
cudaError_t launch_ln_param_partial(bool bf16, const float* dXn, const void* X,
                                    const float* mean, const float* rstd,
                                    float* part_g, float* part_b, int rows,
                                    int h, cudaStream_t stream);

// out[c] = sum over chunks (in chunk order) of part[chunk][c].
cudaError_t launch_colsum_finalize(const float* part, float* out, int chunks,
                                   int cols, cudaStream_t stream);

// Backward of the output dropout: out = mask * scale * dZ ([rows, cols]).
cudaError_t launch_dropout_grad(bool bf16, const void* dZ, void* out, int rows,
                                int cols, uint32_t threshold, float scale,
                                unsigned long long seed,
                                unsigned long long offset,
                                cudaStream_t stream);

// ---------------------------------------------------------------- attention
// Head-parallel attention core over the fused projection QKV [T, 3h]
// (columns grouped by shard: [Q_i | K_i | V_i], each h/t wide; head j of
// shard i = j / (H/t) sits at offset (j mod H/t) d inside each group).
// Tokens are sequence-major: T = batches * seq_len, seq_len % 128 == 0.
struct AttnArgs {
  int heads;            // H
  int heads_per_shard;  // H / t
  int head_dim;         // d (64 or 128)
  int shard_width;      // h / t
  int seq_len;
  int nq;               // seq_len / 128
  int causal;
  float scale_log2;     // log2(e) / sqrt(d)
  __nv_bfloat16* ctx;   // forward output [T, h], head j in columns j d..
  long long ld_ctx;
  float* lse;           // [H, T] base-2 log-sum-exp of the scores scaled by
                        // log2(e) / sqrt(d)
  long long ld_stat;    // row pitch of lse / delta (= T)
  const __nv_bfloat16* dctx;  // backward: dCtx [T, h]
  float* delta;               // backward, [2][H][T]: written by the query
                              // kernel, read by the key/value kernel:
                              // [0] -lse2 of each query row, [1] -delta'
                              // (delta' = sum_j P dP with the query
                              // kernel's own P and dP), negated so that the
                              // key/value kernel adds them
  __nv_bfloat16* dqkv;        // backward output [T, 3h] (same layout as QKV)
  long long ld_qkv;
  float* colsum;              // backward (nullable, d = 128): per 32-row group
  long long ld_colsum;        // g and dQKV column c, the fp32 sum of the
                              // stored values, at colsum[g * ld_colsum + c]
  int* status;
  unsigned long long budget_ns;
  int hs_group;               // (sequence, head) pairs per scheduling group
                              // of the core kernels (attn::core_item)
};

// Forward: tqk maps QKV with 64 x 128 boxes (Q and K tiles), tv with
// 64 x 64 boxes (V tiles, M/N-major operand).  Persistent: any grid of at
// least one CTA walks the batches * H * nq items (the host launches two CTAs
// per SM, at most one per item).
cudaError_t launch_attn_fwd(const CUtensorMap& tqk, const CUtensorMap& tv,
                            const AttnArgs& a, int grid, cudaStream_t stream);

// Backward, key/value gradients (one CTA per 128 keys of a sequence and
// head) and query gradients (one CTA per 128 queries).  tq128 / tq64 map
// QKV with 64 x 128 / 64 x 64 boxes, tdo128 / tdo64 map dCtx [T, h] alike,
// tctx128 maps the forward's Ctx [T, h] with 64 x 128 boxes, tdqkv_out maps
// dQKV [T, 3h] with 64 x 32 store boxes (both kernels' output).
// Both write their columns of a.dqkv; grid = batches * H * nq.  The query
// kernel also writes delta = rowsum(dCtx * Ctx) for every (head, token), which
// the key/value kernel reads: launch the query kernel first.
cudaError_t launch_attn_dkdv(const CUtensorMap& tq128, const CUtensorMap& tq64,
                             const CUtensorMap& tdo64,
                             const CUtensorMap& tdqkv_out, const AttnArgs& a,
                             int grid, cudaStream_t stream);
cudaError_t launch_attn_dq(const CUtensorMap& tq128, const CUtensorMap& tq64,
                           const CUtensorMap& tdo128, const CUtensorMap& tctx128,
                           const CUtensorMap& tdqkv_out, const AttnArgs& a,
                           int grid, cudaStream_t stream);

// Record a message for tp_mlp_last_detail() on the calling thread.
void set_last_detail(const char* msg);

}  // namespace tpmlp
