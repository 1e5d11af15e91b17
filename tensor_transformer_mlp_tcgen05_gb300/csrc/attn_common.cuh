// Device helpers shared by the attention kernels (forward and backward).
#pragma once
#include "gemm_common.cuh"

namespace tpmlp {
namespace attn {

using gemm::Ctl;
using gemm::wait_bounded;

// 12 warps: 0 TMA producer, 1 TMEM allocator + MMA issuer, 2-3 idle,
// 4-11 softmax / elementwise.  Softmax warp w reads TMEM lane quarter
// w mod 4 (its rows) and handles column half (w - 4) / 4 of each tile, so
// every SM sub-partition runs two softmax warps.
constexpr int ATT_THREADS = 384;
constexpr int SOFTMAX_WARP0 = 4;
constexpr int SOFTMAX_WARPS = 8;
constexpr uint32_t KBLOCK_BYTES = 128 * 128;  // 128 rows x 64 bf16
constexpr uint32_t ATOM_BYTES = 64 * 128;     // 64 K-rows x 64 bf16 (MN-major)
constexpr unsigned long long ABORT_SETTLE_NS = 2000000ull;

__device__ __forceinline__ void cta_barrier_att() {
  asm volatile("bar.sync 1, %0;" ::"n"(ATT_THREADS) : "memory");
}

// Named barrier among the softmax warps only.
__device__ __forceinline__ void softmax_barrier() {
  asm volatile("bar.sync 2, %0;" ::"n"(SOFTMAX_WARPS * 32) : "memory");
}

// Warp-uniform bounded wait (every lane polls; the result is agreed).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity,
                                          const Ctl& c, int role) {
  bool ok = wait_bounded(bar, parity, c, role);
  return __all_sync(0xffffffffu, ok);
}

// Store 16-byte units u0 .. u0 + N/4 - 1 (N 32-bit words, 2 bf16 each) of
// row `r` of a 128-row K-major, 128-byte-swizzled operand k-block (64 bf16
// per row; unit u of row r sits at unit u ^ (r mod 8)).
template <int N>
__device__ __forceinline__ void stage_units(uint32_t kblock, int r, int u0,
                                            const uint32_t (&w)[N]) {
  const uint32_t row = kblock + static_cast<uint32_t>(r) * 128u;
#pragma unroll
  for (int u = 0; u < N / 4; ++u) {
    const uint32_t pu = static_cast<uint32_t>((u0 + u) ^ (r & 7));
    ptx::st_shared_v4(row + pu * 16u, w[4 * u], w[4 * u + 1], w[4 * u + 2],
                      w[4 * u + 3]);
  }
}

// A whole 64-value row.
__device__ __forceinline__ void stage_row64(uint32_t kblock, int r,
                                            const uint32_t (&w)[32]) {
  stage_units<32>(kblock, r, 0, w);
}

__device__ __forceinline__ void tmem_ld_128(uint32_t taddr, uint32_t (&r)[128]) {
  uint32_t (&r0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[0]);
  uint32_t (&r1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[32]);
  uint32_t (&r2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[64]);
  uint32_t (&r3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[96]);
  ptx::tmem_ld_32x32b_x32(taddr, r0);
  ptx::tmem_ld_32x32b_x32(taddr + 32, r1);
  ptx::tmem_ld_32x32b_x32(taddr + 64, r2);
  ptx::tmem_ld_32x32b_x32(taddr + 96, r3);
  ptx::tmem_ld_wait();
}

// Column offsets of head j's Q, K and V inside the shard-grouped QKV rows.
struct HeadCols {
  int q, k, v;
};
__device__ __forceinline__ HeadCols head_cols(const AttnArgs& a, int head) {
  const int shard = head / a.heads_per_shard;
  const int jj = head - shard * a.heads_per_shard;
  const int q = 3 * a.shard_width * shard + jj * a.head_dim;
  return {q, q + a.shard_width, q + 2 * a.shard_width};
}

}  // namespace attn
}  // namespace tpmlp
