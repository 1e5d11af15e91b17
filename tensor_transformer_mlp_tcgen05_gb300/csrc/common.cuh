// Definitions shared by the kernels of libtpmlp.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tp_mlp.h"

namespace tpmlp {

// Epilogues of the GEMM kernels.
enum Epilogue : int {
  // H = acc + b1; Y = GeLU(H); writes Y (out) and, if out2 != null, H.
  EPI_GELU_FWD = 0,
  // fixed-order sum over shard segments of fresh fp32 partials, + bias,
  // one rounding to the output type (bf16 or fp32).
  EPI_SHARDSUM = 1,
  // dH = acc * GeLU'(H) with H read from `aux`; writes dH (out).
  EPI_GELU_BWD = 2,
  // plain fp32 store (weight gradients).
  EPI_STORE_F32 = 3,
  // acc (+ bias) rounded to bf16 (projections without an activation).
  EPI_BIAS_BF16 = 4,
};

// Rows of LayerNorm held in registers by one warp (ln_row.cuh): h = 256 vpl
// with vpl <= LN_VMAX, i.e. h <= 6144 (96 registers of raw row per lane).
constexpr int LN_VMAX = 24;

// Arguments of one GEMM launch: D[M,N] = sum over K of Aop[m,k] * Bop[k,n],
// K split into `num_seg` equal segments of `kb_per_seg` k-blocks; each
// segment accumulates into a fresh accumulator (used for the shard sum).
// (The fp32 CUDA-core GEMM reads kb_per_seg as the segment length in K.)
struct GemmArgs {
  int M, N, K;
  int kb_per_seg;
  int num_seg;
  int group_m;            // tile rasterisation: m-tiles per group
  int gelu_mode;
  int out_f32;            // EPI_SHARDSUM output type: 1 fp32, 0 bf16
  void* out;              // [M, N] row-major, leading dimension ldo
  long long ldo;
  void* out2;             // EPI_GELU_FWD: H (nullable)
  const void* aux;        // EPI_GELU_BWD: H; EPI_SHARDSUM: residual added
                          // before the rounding (nullable); leading dim ldaux
  long long ldaux;
  const float* bias;      // [N] fp32 (nullable)
  int* status;            // device status word: [0] code, [1] role, [2] block
  unsigned long long budget_ns;
  // EPI_SHARDSUM dropout (applied after the bias, before the residual).
  int dropout;            // 0 = off
  uint32_t drop_threshold;  // keep when the 32-bit draw >= threshold
  float drop_scale;       // 1 / (1 - p)
  unsigned long long drop_seed, drop_offset;
  // E4M3 operand GEMMs: the accumulator is multiplied by *scale_a *
  // *scale_b (the two operands' per-tensor scales, device memory, product
  // rounded to fp32) before the bias.  amax_out (nullable): EPI_GELU_FWD
  // and EPI_GELU_BWD raise it to the largest |Y| or |dH| written (fp32 bits
  // of a bf16 value).
  const float* scale_a;
  const float* scale_b;
  unsigned int* amax_out;
  // EPI_GELU_BWD (nullable): for every 32-row group g of the output and
  // column c, the fp32 sum of the stored (bf16) values over the group's rows
  // (in row order), written to colsum[g * ld_colsum + c] — the first stage of
  // the bias gradient sum over the tokens.
  float* colsum;
  long long ld_colsum;
  // Tail split (EPI_SHARDSUM with num_seg >= 2, EPI_STORE_F32; pair kernel).
  // part / part_bytes (nullable / 0 = off): a caller-owned fp32 buffer.  The
  // launcher sets tail, pieces and nslots when the last round of super-tiles
  // would leave groups idle: the last `tail` super-tiles are then computed
  // as `pieces` items each, over consecutive k-ranges (whole shard segments
  // for EPI_SHARDSUM, k-blocks for EPI_STORE_F32), whose raw fp32
  // accumulators go to `part` (nslots 512 x 256 slots per tail super-tile)
  // and are combined in a fixed order by launch_gemm_tc2_tail.
  float* part;
  long long part_bytes;
  int tail, pieces, nslots;
  // Fused LayerNorm prologue (EPI_GELU_FWD or EPI_BIAS_BF16 with K-major
  // bf16 A and M/N-major B; ln_x null = off).  The A tensor map points at ln_xn.  The epilogue warps of every
  // CTA first normalise rows of ln_x [M, K] (K = 256 vpl, vpl <= LN_VMAX)
  // into ln_xn and write ln_mean / ln_rstd, claiming one or two rows at a
  // time from ln_sync[0]; after a claim's rows are written they add their
  // count to ln_sync[1 + r / 128].  The producer loads a 128-row A block only
  // once its count is complete.  ln_sync (1 + ceil(M / 128) words) must be
  // zero at launch.
  const __nv_bfloat16* ln_x;
  const float* ln_gamma;
  const float* ln_beta;
  __nv_bfloat16* ln_xn;
  float* ln_mean;
  float* ln_rstd;
  float ln_eps;
  unsigned int* ln_sync;
};

// Roles recorded in status[1] when a bounded wait gives up (ROLE_CHECK: a
// debug-build device check failed; status[3] then names the site).
enum WaitRole : int {
  ROLE_PRODUCER = 1, ROLE_MMA = 2, ROLE_EPILOGUE = 3, ROLE_CHECK = 4,
  ROLE_LN_READY = 5   // the producer waiting for fused-LayerNorm rows
};

// Debug builds (-DTPMLP_CHECKS) verify, before each TMA copy and each
// computed store, the conditions the hardware does not check itself (the
// innermost tile coordinate of a tensor copy on a 16-byte boundary, index
// ranges of plain stores).  A failed check records TPMLP_ERR_CHECK and its
// site in the status word, raises the kernel's abort flag (the other roles
// stop at their next bounded wait) and the access is skipped.  Release
// builds compile the checks out.
enum CheckSite : int {
  SITE_GEMM_LOAD_A = 1, SITE_GEMM_LOAD_B = 2, SITE_GEMM_STORE = 3,
  SITE_GEMM_COLSUM = 4, SITE_ATTN_FWD_LOAD = 5, SITE_ATTN_FWD_STORE = 6,
  SITE_ATTN_BWD_LOAD = 7, SITE_ATTN_BWD_VEC = 8, SITE_ATTN_BWD_STORE = 9,
  SITE_GEMM_LN = 10
};
#ifdef TPMLP_CHECKS
__device__ __forceinline__ bool device_check(bool ok, int* status,
                                             int* abort_flag, int site) {
  if (ok) return true;
  if (atomicCAS(status, 0, TPMLP_ERR_CHECK) == 0) {
    status[1] = ROLE_CHECK;
    status[2] = static_cast<int>(blockIdx.x);
    status[3] = site;
  }
  *reinterpret_cast<volatile int*>(abort_flag) = 1;
  __threadfence();
  return false;
}
#define TPMLP_CHECK(ok, status, abort_flag, site) \
  device_check((ok), (status), (abort_flag), (site))
#else
#define TPMLP_CHECK(ok, status, abort_flag, site) ((void)sizeof(ok), true)
#endif

// GeLU and its derivative in fp32.  Exact form: GeLU(x) = x Phi(x) with
// Phi the standard normal CDF, GeLU'(x) = Phi(x) + x phi(x).  Tanh form
// (Hendrycks & Gimpel): 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
//
// Phi comes from the upper tail Q(|x|) = erfc(|x| / sqrt 2) / 2 with erfc
// from the rational approximation of Abramowitz & Stegun, formula 7.1.26
// (Hastings): erfc(z) = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2),
// t = 1 / (1 + p z), z >= 0, |error| <= 1.5e-7 on erf (so <= 7.5e-8 on
// Phi), and Phi(x) = 1 - Q(x) for x >= 0, Q(-x) otherwise.  exp(-z^2) =
// exp(-x^2 / 2) is also phi(x) sqrt(2 pi), so GeLU' takes one exponential.
// The reciprocal and the exponential are the SFU's approximate
// instructions (rcp.approx, ex2.approx: relative errors near 2^-23 and
// 2^-22), far below the bf16 rounding every GeLU output goes through.
// The GEMM epilogues use the paired forms below (gelu2_f32, gelu_grad2_f32,
// identical results); tp_mlp_probe_gelu evaluates those on a device array
// for the tests.
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float ex2_approx_f32(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Phi(x) and exp(-x^2 / 2).
__device__ __forceinline__ void normal_cdf_exp(float x, float& cdf, float& e) {
  const float z = fabsf(x) * 0.70710678118654752f;          // |x| / sqrt 2
  const float t = rcp_approx(fmaf(0.3275911f, z, 1.0f));
  e = ex2_approx_f32(-(z * z) * 1.44269504088896341f);      // exp(-z^2)
  float poly = fmaf(1.061405429f, t, -1.453152027f);
  poly = fmaf(poly, t, 1.421413741f);
  poly = fmaf(poly, t, -0.284496736f);
  poly = fmaf(poly, t, 0.254829592f);
  const float q = 0.5f * (poly * t) * e;                    // Q(|x|)
  cdf = x >= 0.f ? 1.0f - q : q;
}

__device__ __forceinline__ float gelu_f32(float x, int mode) {
  if (mode == TPMLP_GELU_ERF) {
    float cdf, e;
    normal_cdf_exp(x, cdf, e);
    return x * cdf;
  }
  const float u = 0.79788456080286536f * (x + 0.044715f * x * x * x);
  return 0.5f * x * (1.0f + tanhf(u));
}

__device__ __forceinline__ float gelu_grad_f32(float x, int mode) {
  if (mode == TPMLP_GELU_ERF) {
    float cdf, e;
    normal_cdf_exp(x, cdf, e);
    return fmaf(x * 0.39894228040143268f, e, cdf);          // Phi + x phi
  }
  const float u = 0.79788456080286536f * (x + 0.044715f * x * x * x);
  const float th = tanhf(u);
  const float du = 0.79788456080286536f * (1.0f + 3.0f * 0.044715f * x * x);
  return 0.5f * (1.0f + th) + 0.5f * x * (1.0f - th * th) * du;
}

// The same for two values at once, with packed fp32x2 arithmetic
// (fma/mul.rn.f32x2: two IEEE fp32 operations per instruction, results
// identical to the scalar ones).  The factor 1/2 of Q is folded into the
// polynomial's coefficients (an exact scaling).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// (Phi(x0), Phi(x1)) and (exp(-x0^2/2), exp(-x1^2/2)).
__device__ __forceinline__ void normal_cdf_exp2(float x0, float x1, float& c0,
                                                float& c1, float& e0,
                                                float& e1) {
  const uint64_t z = f2_mul(f2_pack(fabsf(x0), fabsf(x1)),
                            f2_pack(0.70710678118654752f, 0.70710678118654752f));
  float d0, d1;
  f2_unpack(f2_fma(z, f2_pack(0.3275911f, 0.3275911f), f2_pack(1.0f, 1.0f)),
            d0, d1);
  const uint64_t t = f2_pack(rcp_approx(d0), rcp_approx(d1));
  float a0, a1;
  f2_unpack(f2_mul(f2_mul(z, z),
                   f2_pack(-1.44269504088896341f, -1.44269504088896341f)),
            a0, a1);
  e0 = ex2_approx_f32(a0);
  e1 = ex2_approx_f32(a1);
  // 0.5 * (a1 + t (a2 + t (a3 + t (a4 + t a5))))
  uint64_t p = f2_fma(f2_pack(0.5307027145f, 0.5307027145f), t,
                      f2_pack(-0.7265760135f, -0.7265760135f));
  p = f2_fma(p, t, f2_pack(0.7107068705f, 0.7107068705f));
  p = f2_fma(p, t, f2_pack(-0.142248368f, -0.142248368f));
  p = f2_fma(p, t, f2_pack(0.127414796f, 0.127414796f));
  float q0, q1;
  f2_unpack(f2_mul(f2_mul(p, t), f2_pack(e0, e1)), q0, q1);
  c0 = x0 >= 0.f ? 1.0f - q0 : q0;
  c1 = x1 >= 0.f ? 1.0f - q1 : q1;
}

__device__ __forceinline__ void gelu2_f32(float& x0, float& x1, int mode) {
  if (mode == TPMLP_GELU_ERF) {
    float c0, c1, e0, e1;
    normal_cdf_exp2(x0, x1, c0, c1, e0, e1);
    f2_unpack(f2_mul(f2_pack(x0, x1), f2_pack(c0, c1)), x0, x1);
    return;
  }
  x0 = gelu_f32(x0, mode);
  x1 = gelu_f32(x1, mode);
}

// (GeLU'(x0), GeLU'(x1)).
__device__ __forceinline__ void gelu_grad2_f32(float x0, float x1, float& g0,
                                               float& g1, int mode) {
  if (mode == TPMLP_GELU_ERF) {
    float c0, c1, e0, e1;
    normal_cdf_exp2(x0, x1, c0, c1, e0, e1);
    const uint64_t xp = f2_mul(f2_pack(x0, x1),
                               f2_pack(0.39894228040143268f, 0.39894228040143268f));
    f2_unpack(f2_fma(xp, f2_pack(e0, e1), f2_pack(c0, c1)), g0, g1);
    return;
  }
  g0 = gelu_grad_f32(x0, mode);
  g1 = gelu_grad_f32(x1, mode);
}

// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, SC 2011): 10 rounds; a round
// multiplies counter words 0 and 2 by 0xD2511F53 and 0xCD9E8D57 and maps
// (c0, c1, c2, c3) to (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1,
// lo(M0 c0)); the key advances by (0x9E3779B9, 0xBB67AE85) between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0,
                                               uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Dropout of the block's output: element (row, col) is kept when word
// col % 4 of Philox4x32-10(counter (col / 4, row, offset), key = seed) is
// >= threshold; kept values are scaled.  Applies to n consecutive columns
// from c0 (c0 % 4 == 0, n % 4 == 0).
__device__ __forceinline__ void apply_dropout(uint32_t threshold, float scale,
                                              unsigned long long seed,
                                              unsigned long long offset,
                                              int row, int c0, float* v,
                                              int n) {
#pragma unroll
  for (int i = 0; i < n / 4; ++i) {
    const uint4 w = philox4x32_10(
        make_uint4(static_cast<uint32_t>(c0 / 4 + i), static_cast<uint32_t>(row),
                   static_cast<uint32_t>(offset),
                   static_cast<uint32_t>(offset >> 32)),
        static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
    v[4 * i + 0] = w.x >= threshold ? v[4 * i + 0] * scale : 0.f;
    v[4 * i + 1] = w.y >= threshold ? v[4 * i + 1] * scale : 0.f;
    v[4 * i + 2] = w.z >= threshold ? v[4 * i + 2] * scale : 0.f;
    v[4 * i + 3] = w.w >= threshold ? v[4 * i + 3] * scale : 0.f;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void unpack_bf16x2(uint32_t u, float& lo,
                                              float& hi) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  lo = __low2float(v);
  hi = __high2float(v);
}

}  // namespace tpmlp
