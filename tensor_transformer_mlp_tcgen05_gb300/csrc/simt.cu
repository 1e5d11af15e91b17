// fp32 CUDA-core GEMM with the tensor-core kernel's epilogues, for the fp32
// configuration (TPMLP_FP32), whose tolerance tf32 tensor cores would not
// meet.  16 x 16 output tile per block, operand tiles staged in shared
// memory, one output element per thread.  The shard sum follows the same
// rule as the tensor-core path: every shard segment accumulates into a fresh
// fp32 partial, partials are added in shard order, the bias is added last.
#include "internal.h"

namespace tpmlp {
namespace {

constexpr int TS = 16;

__global__ void __launch_bounds__(TS* TS)
    simt_gemm_kernel(SimtOperands ops, GemmArgs a, int epi, int seg_len) {
  __shared__ float sa[TS][TS + 1];
  __shared__ float sb[TS][TS + 1];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int n = blockIdx.x * TS + tx;
  const int m = blockIdx.y * TS + ty;
  float total = 0.f;
  for (int seg = 0; seg < a.num_seg; ++seg) {
    const int k_begin = seg * seg_len;
    const int k_end = min(a.K, k_begin + seg_len);
    float part = 0.f;
    for (int k0 = k_begin; k0 < k_end; k0 += TS) {
      // sa[ty][tx] = Aop(m_tile + ty, k0 + tx); sb[ty][tx] = Bop(k0 + ty, n)
      const int am = blockIdx.y * TS + ty, ak = k0 + tx;
      sa[ty][tx] =
          (am < a.M && ak < k_end)
              ? ops.a[am * ops.a_sm + static_cast<long long>(ak) * ops.a_sk]
              : 0.f;
      const int bk = k0 + ty;
      sb[ty][tx] =
          (n < a.N && bk < k_end)
              ? ops.b[static_cast<long long>(bk) * ops.b_sk + n * ops.b_sn]
              : 0.f;
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < TS; ++kk) part = fmaf(sa[ty][kk], sb[kk][tx], part);
      __syncthreads();
    }
    total = (seg == 0) ? part : total + part;
  }
  if (m >= a.M || n >= a.N) return;
  const size_t off = static_cast<size_t>(m) * a.ldo + n;
  float* out = static_cast<float*>(a.out);
  switch (epi) {
    case EPI_GELU_FWD: {
      const float h = total + (a.bias ? a.bias[n] : 0.f);
      if (a.out2) static_cast<float*>(a.out2)[off] = h;
      out[off] = gelu_f32(h, a.gelu_mode);
      break;
    }
    case EPI_SHARDSUM: {
      float v = total + (a.bias ? a.bias[n] : 0.f);
      if (a.dropout) {
        float q[4] = {0.f, 0.f, 0.f, 0.f};
        q[n & 3] = v;
        apply_dropout(a.drop_threshold, a.drop_scale, a.drop_seed,
                      a.drop_offset, m, n & ~3, q, 4);
        v = q[n & 3];
      }
      if (a.aux) {
        v += static_cast<const float*>(a.aux)[static_cast<size_t>(m) * a.ldaux + n];
      }
      out[off] = v;
      break;
    }
    case EPI_GELU_BWD: {
      const float h = static_cast<const float*>(
          a.aux)[static_cast<size_t>(m) * a.ldaux + n];
      out[off] = total * gelu_grad_f32(h, a.gelu_mode);
      break;
    }
    default:
      out[off] = total;
  }
}

}  // namespace

cudaError_t launch_gemm_simt(int epi, const SimtOperands& ops,
                             const GemmArgs& args, cudaStream_t stream) {
  const dim3 block(TS, TS);
  const dim3 grid((args.N + TS - 1) / TS, (args.M + TS - 1) / TS);
  simt_gemm_kernel<<<grid, block, 0, stream>>>(ops, args, epi,
                                               args.kb_per_seg);
  return cudaGetLastError();
}

}  // namespace tpmlp
