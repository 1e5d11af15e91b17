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

// A shared-memory descriptor moved by `bytes` (a multiple of 16): the start
// address field holds addr >> 4 in 14 bits and shared-memory addresses are
// below 2^18, so the addition never carries out of the field.  Lets the MMA
// issuer build each operand's descriptor once and step it with constants,
// keeping the single issuing thread ahead of 64-cycle MMAs.
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) {
  return desc + (bytes >> 4);
}

// The (sequence, head, block rank) of work item b of a core kernel (items =
// hs_total (sequence, head) pairs x nq blocks).  Items come in groups of
// hs_group (sequence, head) pairs, about one wave of CTAs, so that a group's
// K and V stay in L2 while it runs; inside a group the items with the most
// blocks to walk come first (rank 0 = the longest: the last query block of a
// causal forward or query kernel, the first key block of the key/value
// kernel), so the short ones fill the end.  A bijection of the item index:
// each item's work, and so every result, does not depend on the grouping.
struct CoreItem {
  int rank, head, seq;
};
__device__ __forceinline__ CoreItem core_item(int b, int hs_total, int nq,
                                              int heads, int hs_group) {
  const int G = hs_group > 0 ? hs_group : 1;
  const int g = b / (G * nq);
  const int within = b - g * G * nq;
  const int count = min(G, hs_total - g * G);
  CoreItem it;
  it.rank = within / count;
  const int hs = g * G + within % count;
  it.head = hs % heads;
  it.seq = hs / heads;
  return it;
}

// The fp32 column sums over a warp's 32 rows (in row order) of 32 bf16
// columns that the warp stores itself (the last 32 columns of a d = 96 head,
// which a 64-column chunk store would overrun): each lane's row is written,
// as the first half of a 128-byte-swizzled chunk row, into the stager's next
// buffer once earlier stores have read it, and summed like a staged chunk.
// Lanes 0-15 get columns 2l and 2l + 1; the buffer is free again on return.
__device__ __forceinline__ float2 tail_colsum_bf16(const gemm::ChunkStager& st,
                                                   const float (&v)[32],
                                                   int lane) {
  const uint32_t buf = st.buffer(0);   // the buffer put two chunks ago
  if (lane == 0) ptx::bulk_wait_read<1>();
  __syncwarp();
  const uint32_t row = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t u = static_cast<uint32_t>(c ^ (lane & 7));
    ptx::st_shared_v4(row + u * 16u, pack_bf16x2(v[8 * c], v[8 * c + 1]),
                      pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                      pack_bf16x2(v[8 * c + 4], v[8 * c + 5]),
                      pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
  }
  __syncwarp();
  const float2 cs = gemm::chunk_colsum_bf16(buf, lane);
  __syncwarp();
  return cs;
}

// Named barrier between the two softmax warps of row quarter q (ids 3-6).
__device__ __forceinline__ void pair_barrier(int q) {
  asm volatile("bar.sync %0, 64;" ::"r"(3 + q) : "memory");
}

// 32 TMEM lanes x 32 consecutive 32-bit columns from registers (the store
// counterpart of ptx::tmem_ld_32x32b_x32), and the wait for such stores.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr,
                                                   const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
      "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]),
      "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),
      "r"(r[30]), "r"(r[31])
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: bf16 A read from tensor memory (row m in
// lane m, K packed two bf16 per 32-bit column, lower K index in the low
// half), B from a shared-memory descriptor, fp32 accumulator.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem,
                                            uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2^x by the SFU's approximate base-2 exponential (ex2.approx.ftz.f32: the
// hardware instruction, relative error far below bf16's half ulp; inputs here
// are at most 8 and results that would be subnormal flush to zero, which the
// bf16 P and the fp32 row sums never resolve anyway).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (three-input max.f32).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// One lane of a fully active warp (elect.sync).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// The MMA role runs on all 32 lanes of warp 1, so that its descriptors and
// addresses stay warp-uniform, and one elected lane issues each tcgen05
// instruction.  (A loop run by lane 0 alone lost issue slots to the softmax
// warps sharing its SM sub-partition: its MMAs then ran at 40-50 % rate.)
__device__ __forceinline__ void mma_ss_el(uint32_t d_tmem, uint64_t adesc,
                                          uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  if (elect_one()) ptx::mma_bf16(d_tmem, adesc, bdesc, idesc, accumulate);
}
__device__ __forceinline__ void mma_ts_el(uint32_t d_tmem, uint32_t a_tmem,
                                          uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  if (elect_one()) mma_bf16_ts(d_tmem, a_tmem, bdesc, idesc, accumulate);
}
__device__ __forceinline__ void commit_el(uint32_t bar) {
  if (elect_one()) ptx::mma_commit(bar);
}

// 32 TMEM lanes x 16 consecutive 32-bit columns from registers.
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr,
                                                   const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
      "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]),
      "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Named barrier among the softmax warps only.
__device__ __forceinline__ void softmax_barrier() {
  asm volatile("bar.sync 2, %0;" ::"n"(SOFTMAX_WARPS * 32) : "memory");
}

// The same barrier, ANDing a predicate over the softmax warps: every warp
// leaves with the same answer (a persistent kernel's warps agree on whether
// to go on to the next item, so none waits at a named barrier alone).
__device__ __forceinline__ bool softmax_barrier_and(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, 2, %2, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(p ? 1u : 0u), "n"(SOFTMAX_WARPS * 32)
      : "memory");
  return r != 0;
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
