/*
 * tp_mlp.h - C ABI of libtpmlp: the Megatron-LM intra-layer tensor-parallel
 * transformer MLP block on one GB300 (sm_103a).
 *
 * What the block computes (Megatron-LM explainer, azimuth.plus, section "The
 * core idea: slicing the feed-forward network across units"; Megatron-LM
 * notes, notes.yuuk.io, section "MLP block split"):
 *
 *     Xn  = LayerNorm(X)            (optional pre-LN, explainer section
 *                                    "Fixing BERT: reordering layer
 *                                    normalisation for scaling")
 *     Y_i = GeLU(Xn A_i + b1_i)     A = [A_1 .. A_t] split by columns
 *     Z   = sum_{i=0}^{t-1} Y_i B_i + b2    B split by rows into B_i
 *     Z   = Dropout(Z)              optional, training calls only (the pages'
 *                                   Z = Dropout(YB)), before the residual
 *     [Z += X]                      optional residual connection: the whole
 *                                   pre-LN sub-block X + MLP(LN(X)) (same
 *                                   explainer section on pre-LN: the residual
 *                                   path carries the raw input)
 *
 * The t shards are logical: they run as independent tiles on one GPU.  The
 * operator g (explainer section "The f and g operators: two lines of code"),
 * an all-reduce of the partial outputs Y_i B_i on the pages, becomes a sum of
 * fp32 partials in the fixed order i = 0 .. t-1 inside the second GEMM's
 * epilogue, each partial with a fresh accumulator.  Its conjugate f (identity
 * forward, all-reduce of input gradients backward) becomes the same fixed-
 * order sum in the dX GEMM.  There are no atomics and no split-K with
 * atomic adds: every output element has exactly one writer and every
 * reduction runs in a fixed order, so two calls with the same inputs give
 * bit-identical outputs (the determinism rule of the Megatron Core article,
 * news.hamidun.com, "bitwise determinism at 2432 GPUs": fixed-order
 * reductions and private output space per writer).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Shapes: T = tokens (batch * sequence), h = hidden, f = ffn, t = shards,
 *   f_t = f / t.  Shard i owns ffn columns [i f_t, (i+1) f_t).
 * - Layouts: every matrix is row-major and contiguous: X, Z, dZ, dX [T, h];
 *   A and dA [h, f]; B and dB [f, h].  Vectors b1, db1 [f]; b2, db2, gamma,
 *   beta, dgamma, dbeta [h].
 * - Element types: X, A, B, Z, dZ, dX are bf16 (TPMLP_BF16) or fp32
 *   (TPMLP_FP32) as the configuration says.  Biases, LayerNorm parameters
 *   and every weight/bias/LayerNorm gradient are fp32.  Accumulation is fp32.
 * - Pointers: every data pointer is a DEVICE pointer to memory the caller
 *   owns, 16-byte aligned.  The library never allocates, frees or retains
 *   device memory; it owns only the host-side handle.
 * - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *   default stream).  Calls only enqueue work and return without waiting;
 *   tp_mlp_check() waits and reports device-side errors.
 * - Errors: every function returns a status code (TPMLP_OK = 0, negative on
 *   error); nothing is thrown across the ABI and no output is touched when
 *   argument validation fails.
 */
#ifndef TP_MLP_H_
#define TP_MLP_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define TPMLP_OK              0
#define TPMLP_ERR_ARG        -1  /* null handle/pointer, bad enum value      */
#define TPMLP_ERR_SHAPE      -2  /* h % 64, f % (64 t), tokens > max_tokens  */
#define TPMLP_ERR_ALIGN      -3  /* a pointer is not 16-byte aligned         */
#define TPMLP_ERR_ARCH       -4  /* current device is not compute cap. 10.3  */
#define TPMLP_ERR_CUDA       -5  /* a CUDA runtime/driver call failed        */
#define TPMLP_ERR_TIMEOUT    -6  /* a bounded on-device wait gave up         */
#define TPMLP_ERR_WORKSPACE  -7  /* workspace too small for this call        */
#define TPMLP_ERR_CHECK      -8  /* a device-side check of a debug build
                                    (TPMLP_CHECKS) failed; see
                                    tp_mlp_last_detail for the site        */

/* ---- configuration values --------------------------------------------- */
#define TPMLP_BF16        0      /* bf16 storage, fp32 accumulate (tcgen05) */
#define TPMLP_FP32        1      /* fp32 storage and arithmetic (CUDA cores) */
#define TPMLP_GELU_ERF    0      /* GeLU(x) = x Phi(x) (default)             */
#define TPMLP_GELU_TANH   1      /* tanh approximation of GeLU               */

typedef struct tp_mlp_config {
  int   hidden;          /* h; multiple of 64                                */
  int   ffn;             /* f; f / shards must be a multiple of 64           */
  int   shards;          /* t >= 1, the number of column/row shards          */
  int   max_tokens;      /* largest T any call will pass                     */
  int   dtype;           /* TPMLP_BF16 or TPMLP_FP32                         */
  int   use_layernorm;   /* 1: pre-LayerNorm on X before the first GEMM      */
  float ln_eps;          /* LayerNorm epsilon (added to the biased variance) */
  int   gelu_mode;       /* TPMLP_GELU_ERF or TPMLP_GELU_TANH                */
  int   use_residual;    /* 1: Z = X + MLP(...), added before the rounding  */
  float dropout_p;       /* output dropout probability in [0, 1); training
                            calls only; 0 = off (see tp_mlp_set_dropout_seed) */
} tp_mlp_config;

typedef struct tp_mlp_handle tp_mlp_handle;

/* Validate `cfg` and create a host-side handle (no device work, no device
 * memory).  Returns TPMLP_ERR_ARG / TPMLP_ERR_SHAPE for invalid
 * configurations; *out is set only on success. */
int tp_mlp_create(const tp_mlp_config* cfg, tp_mlp_handle** out);

/* Release the handle.  Passing NULL is allowed and returns TPMLP_OK. */
int tp_mlp_destroy(tp_mlp_handle* handle);

/* Bytes of device workspace a call with `tokens` tokens needs.  training = 1
 * sizes it for tp_mlp_forward(training = 1) followed by tp_mlp_backward on
 * the same workspace; training = 0 for inference-only forward calls.  Besides
 * the saved activations and gradient partial sums, a bf16 handle's
 * workspace (and the FP8 and attention workspaces) holds 64 MiB of fp32
 * partial results for the GEMMs' last round of tiles, which the library
 * splits along K when that round would leave SMs idle (summed again in a
 * fixed order).  Returns 0 for a NULL handle or a negative token count. */
size_t tp_mlp_workspace_bytes(const tp_mlp_handle* handle, int tokens,
                              int training);

/* Forward pass (pages: f forward = identity; Y_i = GeLU(X A_i); Z_i = Y_i
 * B_i; g forward = sum of the Z_i).
 *   tokens      T, 0 <= T <= max_tokens (T = 0 enqueues nothing; X and Z
 *               may then be NULL)
 *   X  [T,h]    input activations (dtype)
 *   A  [h,f], B [f,h]  weights (dtype)
 *   bias1 [f], bias2 [h]  fp32, each may be NULL (treated as zero)
 *   ln_gamma, ln_beta [h] fp32, required iff use_layernorm
 *   Z  [T,h]    output (dtype), overwritten
 *   workspace   device scratch of at least
 *               tp_mlp_workspace_bytes(handle, T, training) bytes; with
 *               training = 1 it keeps what tp_mlp_backward needs (LayerNorm
 *               output and statistics, H = Xn A + b1, Y) and must be passed
 *               to tp_mlp_backward unchanged.
 *   training    1 to save activations for backward, 0 for inference
 *   stream      cudaStream_t the work is enqueued on */
int tp_mlp_forward(tp_mlp_handle* handle, int tokens, const void* X,
                   const void* A, const void* B, const float* bias1,
                   const float* bias2, const float* ln_gamma,
                   const float* ln_beta, void* Z, void* workspace,
                   size_t workspace_bytes, int training, void* stream);

/* Backward pass given dZ = dL/dZ (pages: g backward = identity; f backward =
 * sum of the per-shard input gradients, here in fixed shard order):
 *   dB_i = Y_i^T dZ;  db2 = sum_T dZ;  dH_i = (dZ B_i^T) * GeLU'(H_i);
 *   db1_i = sum_T dH_i;  dA_i = Xn^T dH_i;  dXn = sum_{i=0}^{t-1} dH_i A_i^T;
 *   dX = LayerNorm-backward(dXn) (or dXn) [+ dZ with the residual],
 *   dgamma, dbeta.
 *   dZ [T,h] (dtype); X, A, B, ln_gamma as passed to the forward call.
 *   workspace   the forward call's workspace (training = 1), unchanged.
 *   dX [T,h] (dtype); dA [h,f], dB [f,h] fp32; all overwritten.
 *   dbias1 [f], dbias2 [h], dgamma, dbeta [h] fp32: overwritten; each may be
 *   NULL to skip it (dgamma/dbeta are ignored without LayerNorm).
 * With T = 0 the weight and bias gradients are set to zero (dZ, X and dX
 * may then be NULL). */
int tp_mlp_backward(tp_mlp_handle* handle, int tokens, const void* dZ,
                    const void* X, const void* A, const void* B,
                    const float* ln_gamma, void* workspace,
                    size_t workspace_bytes, void* dX, float* dA, float* dB,
                    float* dbias1, float* dbias2, float* dgamma, float* dbeta,
                    void* stream);

/* ---- FP8 (E4M3) variant: forward and backward --------------------------
 * The block's forward with both GEMMs on 8-bit E4M3 operands (the
 * low-precision runs of the Megatron Core determinism article, read as
 * plain per-tensor FP8): every operand tensor T (Xn, A, B and Y) is scaled
 * by s_T = amax(T) / 448 (fp32; 1 for an all-zero tensor) and stored as
 * codes q = e4m3(x / s_T) (x / s_T an fp32 division, nearest-even rounding,
 * saturation to +-448).  H = (s_x s_a) (Xq Aq) + b1 with fp32 accumulation,
 * Y = GeLU(H) stored bf16 and quantized with its own current amax, Z =
 * sum_i (s_y s_b) (Yq_i Bq_i) + b2 [+ X] in fixed shard order, one bf16
 * rounding.  The handle must be TPMLP_BF16 without dropout, and f / t must
 * be a multiple of 128 (TPMLP_ERR_ARG / TPMLP_ERR_SHAPE otherwise).  The
 * weights are quantized once by tp_mlp_fp8_pack_weights into a
 * caller-owned buffer of tp_mlp_fp8_weights_bytes bytes (layout: amax_a,
 * amax_b as fp32 bits and s_a, s_b as fp32, then A^T codes [f, h], B^T
 * codes [h, f], A codes [h, f] and B codes [f, h], each section 256-byte
 * aligned: the forward reads the transposed codes, the backward the plain
 * ones); the forward quantizes Xn and Y itself. */
size_t tp_mlp_fp8_weights_bytes(const tp_mlp_handle* handle);
int tp_mlp_fp8_pack_weights(tp_mlp_handle* handle, const void* A,
                            const void* B, void* packed, size_t packed_bytes,
                            void* stream);
/* Workspace of tp_mlp_forward_fp8 for `tokens` tokens (0 on a bad handle). */
size_t tp_mlp_fp8_workspace_bytes(const tp_mlp_handle* handle, int tokens);
/* X [T,h] bf16, packed weights from tp_mlp_fp8_pack_weights, bias1 [f],
 * bias2 [h], ln_gamma/ln_beta as tp_mlp_forward; Z [T,h] bf16. */
int tp_mlp_forward_fp8(tp_mlp_handle* handle, int tokens, const void* X,
                       const void* packed, const float* bias1,
                       const float* bias2, const float* ln_gamma,
                       const float* ln_beta, void* Z, void* workspace,
                       size_t workspace_bytes, void* stream);
/* Training step in FP8.  The backward uses E4M3 for the gradients too,
 * with the same per-tensor current scaling (the determinism article names
 * no gradient format; this is the plain reading):
 *   dZq = e4m3(dZ / s_dz);  db2 = sum_T dZ;
 *   dH = bf16((s_dz s_b) (dZq Bq^T) * GeLU'(H)) with H as the training
 *     forward stored it (bf16);  db1 = sum_T dH;  dHq = e4m3(dH / s_dh);
 *   dXn = sum_i (s_dh s_a) (dHq_i Aq_i^T) in fixed shard order (fp32),
 *     then LayerNorm's backward with the forward's statistics, or dXn
 *     itself; + dZ with the residual; dX rounded to bf16 once;
 *   dA = (s_x s_dh) (Xq^T dHq), dB = (s_y s_dz) (Yq^T dZq), fp32.
 * Every scale product is rounded to fp32.  Bias and LayerNorm-parameter
 * sums run in fixed order (bitwise reproducible), as in tp_mlp_backward.
 *
 * tp_mlp_forward_fp8_train is tp_mlp_forward_fp8 that also keeps what the
 * backward needs in its workspace (H bf16, Xq^T and Yq^T codes); its
 * workspace has tp_mlp_fp8_train_workspace_bytes bytes (the sections of
 * the plain forward at the same offsets, then the training sections) and
 * must be passed, unchanged, to tp_mlp_backward_fp8 with the same tokens,
 * X and packed weights.  tp_mlp_backward_fp8 arguments as tp_mlp_backward
 * (dZ, X, dX bf16 [T,h]; dA [h,f], dB [f,h] and the nullable bias and
 * LayerNorm-parameter gradients fp32, all overwritten); with T = 0 the
 * weight and bias gradients are set to zero.  Errors as the forward. */
size_t tp_mlp_fp8_train_workspace_bytes(const tp_mlp_handle* handle,
                                        int tokens);
int tp_mlp_forward_fp8_train(tp_mlp_handle* handle, int tokens,
                             const void* X, const void* packed,
                             const float* bias1, const float* bias2,
                             const float* ln_gamma, const float* ln_beta,
                             void* Z, void* workspace, size_t workspace_bytes,
                             void* stream);
int tp_mlp_backward_fp8(tp_mlp_handle* handle, int tokens, const void* dZ,
                        const void* X, const void* packed,
                        const float* ln_gamma, void* workspace,
                        size_t workspace_bytes, void* dX, float* dA, float* dB,
                        float* dbias1, float* dbias2, float* dgamma,
                        float* dbeta, void* stream);
/* Byte offsets of the packed-weight sections and of the forward's and the
 * training step's workspace sections (for inspection by tests); -1 if
 * unknown.  Transposed code sections of T columns have a row pitch of
 * T rounded up to a multiple of 16 bytes. */
long long tp_mlp_fp8_offset(const tp_mlp_handle* handle, int tokens,
                            int which);
#define TPMLP_FP8_PACK_SCALES 0   /* amax_a, amax_b (u32), s_a, s_b (f32) */
#define TPMLP_FP8_PACK_AQT    1   /* A^T codes [f, h]                     */
#define TPMLP_FP8_PACK_BQT    2   /* B^T codes [h, f]                     */
#define TPMLP_FP8_WS_SCALES   3   /* amax_x, amax_y (u32), s_x, s_y (f32) */
#define TPMLP_FP8_WS_XQ       4   /* Xn codes [T, h]                      */
#define TPMLP_FP8_WS_Y        5   /* Y [T, f] bf16                        */
#define TPMLP_FP8_WS_YQ       6   /* Y codes [T, f]                       */
#define TPMLP_FP8_PACK_AQ     7   /* A codes [h, f]                       */
#define TPMLP_FP8_PACK_BQ     8   /* B codes [f, h]                       */
#define TPMLP_FP8_WS_H        9   /* H [T, f] bf16 (training)             */
#define TPMLP_FP8_WS_XQT     10   /* Xn codes transposed [h, T]           */
#define TPMLP_FP8_WS_YQT     11   /* Y codes transposed [f, T]            */
#define TPMLP_FP8_WS_BSCALES 12   /* amax_dz, amax_dh (u32), s_dz, s_dh   */
#define TPMLP_FP8_WS_DZQ     13   /* dZ codes [T, h]                      */
#define TPMLP_FP8_WS_DZQT    14   /* dZ codes transposed [h, T]           */
#define TPMLP_FP8_WS_DH      15   /* dH [T, f] bf16                       */
#define TPMLP_FP8_WS_DHQ     16   /* dH codes [T, f]                      */
#define TPMLP_FP8_WS_DHQT    17   /* dH codes transposed [f, T]           */

/* Tensor-core rate calibration (instrumentation, not part of the block):
 * launches `ctas` CTAs (one per SM when ctas <= the SM count), each with one
 * thread issuing `n_mma` (a multiple of 4, <= 2^24) back-to-back
 * tcgen05.mma of shape M = 128, N = n (64, 128 or 256), K = 16, bf16
 * operands from shared memory, fp32 accumulator in tensor memory, and writes
 * the SM clock cycles from first issue to last completion of CTA i to
 * cycles[i] (device memory, >= ctas entries).  status (device int, zeroed
 * by the caller) becomes TPMLP_ERR_TIMEOUT if a completion wait gave up.
 * 2 * 128 * n * 16 * n_mma / cycles is the per-SM dense bf16 rate in flops
 * per cycle.  Asynchronous on `stream`. */
int tp_mlp_probe_mma_cycles(int n, int ctas, int n_mma,
                            unsigned long long* cycles, int* status,
                            void* stream);

/* The library's device GeLU (instrumentation, not part of the block):
 * y[i] = GeLU(x[i]) and dy[i] = GeLU'(x[i]) for n fp32 values in device
 * memory, exactly as the GEMM epilogues evaluate them (mode
 * TPMLP_GELU_ERF or TPMLP_GELU_TANH).  Lets tests check the epilogues' GeLU
 * against CUDA's erf and the oracle.  TPMLP_ERR_ARG for a bad mode, n < 0 or
 * null pointers with n > 0.  Asynchronous on `stream`. */
int tp_mlp_probe_gelu(const float* x, float* y, float* dy, int n, int mode,
                      void* stream);

/* Bias gradient without any device allocation: dbias[c] = sum over the
 * `tokens` rows of grad[r][c], for a row-major [tokens, cols] gradient
 * (e.g. dZ, giving db2).  The pages have no counterpart for this entry
 * point; it exists for callers that cannot allocate device memory, such as
 * a host engine that reserves the whole device memory pool for itself at
 * start-up, or a tool that must not change the process's device-memory
 * footprint while it runs, and so cannot provide the workspace that
 * tp_mlp_backward takes its scratch from.
 *   tokens  T >= 0 (T = 0 writes zeros); cols > 0, a multiple of 64
 *   dtype   TPMLP_BF16 or TPMLP_FP32: the element type of `grad`
 *   grad    device pointer, [T, cols]; may be NULL when T = 0
 *   dbias   device pointer, [cols] fp32, overwritten
 * The partial sums go to one static device array of
 * TPMLP_NOALLOC_SCRATCH_FLOATS floats (4 MiB), which every GPU that loads
 * the library holds until the process exits; calls need
 * ceil(T / 256) * cols <= TPMLP_NOALLOC_SCRATCH_FLOATS and return
 * TPMLP_ERR_SHAPE (with tp_mlp_last_detail() saying why) otherwise.  The
 * first call on a device looks the array's device address up with that
 * device current; make that first call before any stream capture.  Every
 * call shares the array and it keeps the last call's contents (each call
 * overwrites all it reads, so nothing needs clearing); calls that overlap on
 * the GPU, on different streams, race on it.  The result is bit-identical to
 * the db2 of tp_mlp_backward for the same dZ (the same two fixed-order
 * kernels), and to its db1 in the fp32 configuration; the bf16 path sums
 * db1 from 32-row partials written by the dH GEMM's epilogue instead, which
 * agrees within fp32 rounding, not bitwise.  No cudaMalloc, cudaFree or
 * allocating library routine is called. */
#define TPMLP_NOALLOC_SCRATCH_FLOATS (1 << 20)
int tp_mlp_bias_grad_noalloc(int tokens, int cols, int dtype, const void* grad,
                             float* dbias, void* stream);

/* Wait for `stream`, then read and clear the device status word kept in
 * `workspace`.  Returns TPMLP_OK, TPMLP_ERR_TIMEOUT (a bounded wait inside a
 * GEMM kernel gave up; the outputs of that call are undefined) or
 * TPMLP_ERR_CUDA. */
int tp_mlp_check(tp_mlp_handle* handle, void* workspace, void* stream);

/* Human-readable text for a status code (static storage). */
const char* tp_mlp_status_string(int status);

/* Detail of the most recent failure on the calling thread (which CUDA call
 * failed and why, or the device status word's role/block); thread-local
 * storage, overwritten by the next failure. */
const char* tp_mlp_last_detail(void);

/* ---- instrumentation --------------------------------------------------- */

/* Number of kernels this handle has launched since creation (memsets not
 * counted). */
long long tp_mlp_launch_count(const tp_mlp_handle* handle);

/* Enable (1) or disable (0) per-kernel timing: when enabled every launch is
 * bracketed by CUDA events on its stream.  Costs one event pair per launch. */
int tp_mlp_set_timing(tp_mlp_handle* handle, int enable);

/* Wait for the recorded events and fold them into per-kernel totals, then
 * report kernel `index` (0-based): its name (static storage), launches and
 * total milliseconds.  Returns TPMLP_ERR_ARG once `index` is past the last
 * kernel.  tp_mlp_timing_reset() clears the totals. */
int tp_mlp_timing_get(tp_mlp_handle* handle, int index, const char** name,
                      long long* launches, double* total_ms);
int tp_mlp_timing_reset(tp_mlp_handle* handle);

/* Seed and counter offset of the output dropout (default 0, 0).  The mask
 * is a pure function of (seed, offset, token row, column), so it does not
 * depend on the shard count or on the launch configuration: element (r, c)
 * is kept when 32-bit word c % 4 of Philox4x32-10 (Salmon et al., SC 2011)
 * of counter (c / 4, r, offset low, offset high) under key (seed low, seed
 * high) is >= floor(dropout_p 2^32); kept values are scaled by
 * 1 / (1 - dropout_p).  tp_mlp_backward regenerates the same mask from the
 * handle's current seed and offset, so they must not change between a
 * forward call and its backward call. */
int tp_mlp_set_dropout_seed(tp_mlp_handle* handle, unsigned long long seed,
                            unsigned long long offset);

/* Budget, in nanoseconds, for each bounded wait inside the GEMM kernels
 * (default 2e9).  A wait that exceeds it makes the kernel record
 * TPMLP_ERR_TIMEOUT in the status word and return early. */
int tp_mlp_set_wait_budget(tp_mlp_handle* handle, unsigned long long ns);

/* Enable (1) or disable (0, the default) an NVTX range around the enqueue
 * of every kernel this handle launches, named for the kernel (the names
 * tp_mlp_timing_get reports), so that a profiler recording NVTX (ncu
 * --nvtx, Nsight Systems) can attribute each launch to its step of the
 * block.  Without a tool attached the ranges cost a function call each.
 * Tracing only: the pages describe no profiling hooks.
 * TPMLP_ERR_ARG for a NULL handle or another value. */
int tp_mlp_set_nvtx(tp_mlp_handle* handle, int enable);

/* Enable (1, the default) or disable (0) the fused pre-LayerNorm prologue
 * of the bf16 forward (pre-LN placement: Megatron-LM explainer, "Fixing
 * BERT: reordering layer normalisation for scaling").  Enabled, with
 * use_layernorm, dtype TPMLP_BF16 and hidden = 256 v for v <= 24 (hidden
 * <= 6144), the LayerNorm runs inside the first GEMM's launch: that
 * kernel's epilogue warps normalise the token rows (one row per warp at a
 * time, the row held in registers: coalesced 16-byte loads, warp-shuffle
 * reductions) before their first tile, and each 128-row block of the GEMM's
 * A operand is loaded as soon as its rows are written, so the LayerNorm
 * overlaps the GEMM instead of running as its own launch.  Disabled, or for
 * other shapes, a stand-alone LayerNorm kernel runs first.  Both compute
 * the same bits (one device function normalises a row on either path):
 * Xn, mean, rstd and every output are identical.  Takes effect from the
 * next tp_mlp_forward call.  TPMLP_ERR_ARG for a NULL handle or another
 * value. */
int tp_mlp_set_ln_prologue(tp_mlp_handle* handle, int enable);

#ifdef __cplusplus
}
#endif
#endif /* TP_MLP_H_ */
