// Backward of the attention core (per sequence and head; scaled dot-product
// attention, Megatron-LM explainer section on attention and notes section
// "Self-attention block split": the heads stay independent in the backward
// too, so no shard exchanges anything here).
//
// With P = exp2(S log2(e)/sqrt(d) - lse2) (the forward's saved base-2
// log-sum-exp), dO = dCtx and delta = rowsum(dO * O) = sum_j P dP (the query
// kernel starts from the first form, from its dO tile and the forward's
// context rows, and writes the second, from its own P and dP, for the
// key/value kernel, which therefore runs second; it writes -lse2 and
// -delta', so that the key/value kernel's per-column terms enter its packed
// fused multiply-adds and additions without a negation):
//   dV = P^T dO,   dP = dO V^T,   dS = P * (dP - delta) / sqrt(d),
//   dK = dS^T Q,   dQ = dS K.
// Every output element has exactly one writer and no atomics are used:
//   * the KV kernel owns 128 keys of one (sequence, head) and walks the
//     64-query blocks that may see them, accumulating dK and dV in TMEM;
//   * the Q kernel owns 128 queries and walks the 64-key blocks they see,
//     recomputing S and dP, accumulating dQ in TMEM.
// Both are one template: a fixed 128-row pair of operand tiles (A1, A2) and a
// stream of 64-row tile pairs (B1, B2):
//           rows   A1  A2   B1  B2   S1 = A1 B1^T  S2 = A2 B2^T    outputs
//   KV      keys   K   V    Q   dO   S^T           dP^T            dK += dS^T Q, dV += P^T dO
//   Q       query  Q   dO   K   V    S             dP              dQ += dS K, PK += P K
// The Q kernel also forms delta for its 128 queries from its dO tile and the
// forward's context rows (loaded into the last ring stage before the ring
// first reaches it), and at its end writes sum_j P dP for the KV kernel.
// The elementwise step writes P and dS as bf16 into a tensor-memory buffer of
// their own, where the output MMAs take them as A operands (their B operands
// are the streamed tiles read M/N-major, the same bytes); S and dP have one
// buffer, which the next step's score MMAs overwrite as soon as the
// elementwise warps have loaded it, so the tensor pipe goes from one step's
// gradient MMAs to the next step's score MMAs without waiting for the former
// to finish.  A1 (K for KV, Q for Q) is copied once into tensor memory by
// the elementwise warps, so the S1 MMAs read only the streamed tile from
// shared memory (a 128 x 64 x 16 MMA with both operands in shared memory
// needs 6 KB per instruction and runs at the shared-memory operand rate,
// 48 cycles; with A in tensor memory, 2 KB and 32 cycles).
// Outputs leave as 32-row x 64-column bf16 chunks staged in the idle B ring
// and stored by TMA (at d = 96 the last 32 columns of dK, dV and dQ with
// plain 16-byte stores); each chunk, and each such 32-column tail, is also
// summed over its 32 rows into the partials of the QKV bias gradient.
//
// Warp roles: warp 0 TMA producer, warp 1 TMEM allocator and issuer of the
// score MMAs, warp 2 issuer of the gradient MMAs (each the whole warp, one
// elected lane issuing), warps 4-11 elementwise (thread = row = TMEM lane,
// two warps per row quarter, one per half of the columns).  With one issuer
// per kind, the next step's score MMAs are queued while this step's
// gradient MMAs are still being issued, so the tensor pipe does not idle
// between them.  All waits are bounded.
#include "attn_common.cuh"

namespace tpmlp {
namespace {

using namespace gemm;
using namespace attn;

template <int D, bool KV>
__global__ void __launch_bounds__(ATT_THREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmA2,
                    const __grid_constant__ CUtensorMap tmB1,
                    const __grid_constant__ CUtensorMap tmB2,
                    const __grid_constant__ CUtensorMap tmCtx,
                    const __grid_constant__ CUtensorMap tmOut,
                    const AttnArgs a) {
  // 64-wide blocks of d (d = 96: the second block's upper 32 columns are
  // loaded but never used; the MMAs stop at K = d and N = d)
  constexpr int KB = (D + 63) / 64;
  constexpr uint32_t A_TILE = KB * KBLOCK_BYTES;   // 128 rows x D
  constexpr uint32_t B_TILE = KB * ATOM_BYTES;     // 64 rows x D
  // Stages of the streamed tile pair: the load for step n + NB can only
  // start once step n's gradient MMAs have read its stage, so the ring must
  // cover the TMA latency (4 fit for KV next to its lse / delta vectors, 5
  // for Q).
  constexpr int NB = KV ? 4 : 5;
  constexpr uint32_t VEC_BYTES = 512;              // 64 -lse2 + 64 -delta
  // KV: lse2 / delta of the streamed queries per stage; Q: the two column
  // halves' partial row sums of dS, exchanged at the end
  constexpr uint32_t VEC_TOTAL = KV ? NB * VEC_BYTES : 1024;
  constexpr int NBARS = 12 + 2 * NB;
  constexpr uint32_t B_TX = 2 * B_TILE + (KV ? VEC_BYTES : 0);
  constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 64, false, false);
  constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, false, true);
  // TMEM columns: S1 (S or S^T) and S2 (dP or dP^T) of the current step,
  // 64 each; the bf16 P and dS operands (P then dS, 32 packed columns
  // apiece); A1 as a bf16 MMA operand (row m in lane m, two elements per
  // column, D / 2 columns); the two fp32 accumulators.
  constexpr uint32_t TMEM_S1 = 0, TMEM_S2 = 64, TMEM_PDS = 128;
  constexpr uint32_t TMEM_A1 = 192;
  constexpr uint32_t TMEM_OUT2 = 256;              // dK (KV) or dQ
  constexpr uint32_t TMEM_OUT1 = 256 + 64 * KB;    // dV (KV) or P K (Q)
  constexpr float INV_SQRT_D = D == 64   ? 0.125f
                               : D == 96 ? 0.10206207261596575f
                                         : 0.08838834764831845f;
  static_assert(D == 64 || D == 96 || D == 128, "head dim");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA1 = ptx::smem_u32(smem);
  const uint32_t sA2 = sA1 + A_TILE;
  const uint32_t sB = sA2 + A_TILE;                // [stage][B1 | B2]
  uint8_t* vec_gen = smem + 2 * A_TILE + NB * 2 * B_TILE;
  const uint32_t sVec = ptx::smem_u32(vec_gen);    // [stage][-lse2 | -delta]
  uint64_t* bars = reinterpret_cast<uint64_t*>(vec_gen + VEC_TOTAL);
  const uint32_t b0 = ptx::smem_u32(bars);
  // s_full: S and dP of the step are in TMEM (one buffer); s_read: the
  // elementwise warps have loaded them, so the next step's MMAs may
  // overwrite them; a1_full: A1 is in tensor memory; e_full / e_empty: P
  // and dS of the step are in their
  // TMEM buffer (two, by step parity) / its gradient MMAs have read them.
  const uint32_t a_full = b0, b_full = b0 + 8, b_empty = b_full + 8 * NB,
                 s_full = b_empty + 8 * NB, s_read = s_full + 8,
                 e_full = s_full + 16, a1_full = e_full + 8,
                 e_empty = e_full + 16,
                 o_full = e_empty + 16,
                 done_bar = o_full + 8, ctx_full = done_bar + 8,
                 ctx_free = ctx_full + 8, done2 = ctx_free + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = a.nq;
  const CoreItem item =
      core_item(static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x) / nq,
                nq, a.heads, a.hs_group);
  const int rb = KV ? item.rank : nq - 1 - item.rank;
  const int head = item.head;
  const int seq = item.seq;
  const int row0 = seq * a.seq_len + rb * 128;
  // 64-wide column blocks: queries >= the first key (KV), keys <= the last
  // query (Q) when causal.
  const int cb_begin = (KV && a.causal) ? 2 * rb : 0;
  const int cb_end = (!KV && a.causal) ? 2 * rb + 2 : 2 * nq;
  const int nsteps = cb_end - cb_begin;
  const HeadCols hc = head_cols(a, head);
  const int cA1 = KV ? hc.k : hc.q;
  const int cA2 = KV ? hc.v : head * D;
  const int cB1 = KV ? hc.q : hc.k;
  const int cB2 = KV ? head * D : hc.v;

  if (threadIdx.x == 0) {
    ptx::mbar_init(a_full, 1);
    for (int i = 0; i < NB; ++i) {
      ptx::mbar_init(b_full + 8 * i, 1);
      ptx::mbar_init(b_empty + 8 * i, 1);
    }
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(s_read, SOFTMAX_WARPS);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(e_full + 8 * i, SOFTMAX_WARPS);   // [1]: a1_full
      ptx::mbar_init(e_empty + 8 * i, 1);
    }
    ptx::mbar_init(o_full, 1);
    ptx::mbar_init(done_bar, 1);
    ptx::mbar_init(ctx_full, 1);
    ptx::mbar_init(ctx_free, SOFTMAX_WARPS);
    ptx::mbar_init(done2, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const Ctl ctl{abort_flag, a.status, a.budget_ns};

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------- producer --
      // (debug builds: the copies' innermost coordinates on a 16-byte
      // boundary, the 1-D copies of lse2 / delta on 16-byte addresses)
      if (TPMLP_CHECK(cA1 % 8 == 0 && cA2 % 8 == 0 && cB1 % 8 == 0 &&
                          cB2 % 8 == 0 && (head * D) % 8 == 0 &&
                          (static_cast<long long>(head) * a.ld_stat +
                           seq * a.seq_len) % 4 == 0,
                      a.status, abort_flag, SITE_ATTN_BWD_LOAD))
      {
      ptx::mbar_arrive_expect_tx(a_full, 2 * A_TILE);
#pragma unroll
      for (int kk = 0; kk < KB; ++kk) {
        ptx::tma_load_2d(sA1 + kk * KBLOCK_BYTES, &tmA1, a_full, cA1 + 64 * kk,
                         row0);
        ptx::tma_load_2d(sA2 + kk * KBLOCK_BYTES, &tmA2, a_full, cA2 + 64 * kk,
                         row0);
      }
      if constexpr (!KV) {
        // Q: the forward's context rows of this block, for delta, borrow the
        // last stage of the ring until the elementwise warps have read them
        ptx::mbar_arrive_expect_tx(ctx_full, KB * KBLOCK_BYTES);
#pragma unroll
        for (int kk = 0; kk < KB; ++kk)
          ptx::tma_load_2d(sB + (NB - 1) * 2 * B_TILE + kk * KBLOCK_BYTES,
                           &tmCtx, ctx_full, head * D + 64 * kk, row0);
      }
      for (int n = 0; n < nsteps; ++n) {
        const uint32_t bs = n % NB, bph = (n / NB) & 1;
        if (!KV && n == NB - 1 &&
            !wait_bounded(ctx_free, 0, ctl, ROLE_PRODUCER))
          break;
        if (!wait_bounded(b_empty + 8 * bs, bph ^ 1, ctl, ROLE_PRODUCER)) break;
        const int col0 = seq * a.seq_len + (cb_begin + n) * 64;
        const uint32_t bf = b_full + 8 * bs;
        const uint32_t dB1 = sB + bs * 2 * B_TILE, dB2 = dB1 + B_TILE;
        ptx::mbar_arrive_expect_tx(bf, B_TX);
#pragma unroll
        for (int kk = 0; kk < KB; ++kk) {
          ptx::tma_load_2d(dB1 + kk * ATOM_BYTES, &tmB1, bf, cB1 + 64 * kk, col0);
          ptx::tma_load_2d(dB2 + kk * ATOM_BYTES, &tmB2, bf, cB2 + 64 * kk, col0);
        }
        if constexpr (KV) {
          const size_t off = static_cast<size_t>(head) * a.ld_stat + col0;
          const size_t plane = static_cast<size_t>(a.heads) * a.ld_stat;
          ptx::bulk_load_1d(sVec + bs * VEC_BYTES, a.delta + off, 256, bf);
          ptx::bulk_load_1d(sVec + bs * VEC_BYTES + 256, a.delta + plane + off,
                            256, bf);
        }
      }
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    {
      // ------------------------ MMA issuers (whole warp, elected lane) --
      // warp 1: S1, S2 of every step; warp 2: the step's gradient MMAs.
      // Each tcgen05.commit tracks its own thread's MMAs only: s_full the
      // score MMAs; b_empty, e_empty and o_full the gradient MMAs, which
      // start after the same step's score MMAs have completed (e_full is
      // arrived after s_full), so a ring stage is released only when both
      // kinds have read it.
      bool alive = warp == 2 || warp_wait(a_full, 0, ctl, ROLE_MMA);
      const uint64_t dA2 = ptx::sdesc_sw128(sA2, 16, 1024);
      const uint64_t dBk = ptx::sdesc_sw128(sB, 16, 1024);          // K-major
      const uint64_t dBm = ptx::sdesc_sw128(sB, ATOM_BYTES, 1024);  // MN-major
      auto issue_s = [&](int n) -> bool {
        const uint32_t bs = n % NB, bph = (n / NB) & 1;
        if (!warp_wait(b_full + 8 * bs, bph, ctl, ROLE_MMA)) return false;
        // the score buffer still holds step n - 1's S and dP until the
        // elementwise warps have loaded them
        if (n >= 1 && !warp_wait(s_read, static_cast<uint32_t>(n - 1) & 1u,
                                 ctl, ROLE_MMA))
          return false;
        if (n == 0 && !warp_wait(a1_full, 0, ctl, ROLE_MMA)) return false;
        ptx::tc_fence_after();
        const uint64_t b1 = desc_add(dBk, bs * 2 * B_TILE);
        const uint64_t b2 = desc_add(b1, B_TILE);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t bo = (k / 4) * ATOM_BYTES + (k % 4) * 32;
          mma_ts_el(tmem + TMEM_S1, tmem + TMEM_A1 + 8 * k, desc_add(b1, bo),
                    IDESC_S, k > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ao = (k / 4) * KBLOCK_BYTES + (k % 4) * 32;
          const uint32_t bo = (k / 4) * ATOM_BYTES + (k % 4) * 32;
          mma_ss_el(tmem + TMEM_S2, desc_add(dA2, ao),
                    desc_add(b2, bo), IDESC_S, k > 0 ? 1u : 0u);
        }
        commit_el(s_full);
        return true;
      };
      auto issue_o = [&](int n) -> bool {
        const uint32_t bs = n % NB, bph = (n / NB) & 1;
        // (the stage's b_full phase is still step n's: its refill for step
        // n + NB waits for this step's commit to b_empty)
        if (!warp_wait(e_full, static_cast<uint32_t>(n) & 1u, ctl, ROLE_MMA) ||
            !warp_wait(b_full + 8 * bs, bph, ctl, ROLE_MMA))
          return false;
        ptx::tc_fence_after();
        const uint64_t b1 = desc_add(dBm, bs * 2 * B_TILE);
        const uint64_t b2 = desc_add(b1, B_TILE);
        // A operands in TMEM: P and dS, 32 packed columns each (the column
        // half hf of the elementwise warps wrote its 32 queries or keys at
        // +16 hf): k-step k (16 of the step's 64) at +8 k
        const uint32_t e1 = tmem + TMEM_PDS, e2 = e1 + 32;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts_el(tmem + TMEM_OUT2, e2 + 8 * k, desc_add(b1, 2048 * k),
                    IDESC_O, (n > 0 || k > 0) ? 1u : 0u);
        // KV: dV += P^T dO.  Q: sum_j P_ij k_j += P K (same B as dQ), for
        // the row-sum correction of dQ below.
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts_el(tmem + TMEM_OUT1, e1 + 8 * k,
                    desc_add(KV ? b2 : b1, 2048 * k), IDESC_O,
                    (n > 0 || k > 0) ? 1u : 0u);
        commit_el(b_empty + 8 * bs);
        commit_el(e_empty);
        return true;
      };
      if (warp == 1) {
        for (int n = 0; alive && n < nsteps; ++n) alive = issue_s(n);
      } else {
        for (int n = 0; alive && n < nsteps; ++n) alive = issue_o(n);
        if (alive) commit_el(o_full);
      }
      if (*reinterpret_cast<volatile int*>(abort_flag)) {
        // every MMA this warp issued has completed before TMEM is freed
        const uint32_t db = warp == 1 ? done_bar : done2;
        commit_el(db);
        wait_teardown(db, 0);
      }
    }
    __syncwarp();
  } else if (warp >= SOFTMAX_WARP0) {
    // -------------------------------------------------- elementwise --
    // Two warps per row quarter, each on 32 of the step's 64 columns (and
    // on half of the output columns at the end).
    const int q = warp & 3;
    const int hf = (warp - SOFTMAX_WARP0) >> 2;
    const int r = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const float sl2 = a.scale_log2;
    float lse_r = 0.f, delta_r = 0.f;
    bool alive = warp_wait(a_full, 0, ctl, ROLE_EPILOGUE);
    if (alive) {
      // A1 into tensor memory for the S1 MMAs: this warp's 32 rows of
      // k-block hf (64 elements, or D - 64 of them; none for hf = 1 when
      // D = 64), column 32 hf + j holding elements 2j and 2j + 1 of the
      // k-block (16-byte unit u of row r sits at u ^ (r mod 8))
      constexpr int U1 = D > 64 ? (D - 64) / 8 : 0;
      const int units = hf == 0 ? 8 : U1;
      if (units > 0) {
        const uint32_t rowa = sA1 + static_cast<uint32_t>(hf) * KBLOCK_BYTES +
                              static_cast<uint32_t>(r) * 128u;
        uint32_t w[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint32_t v[4] = {0u, 0u, 0u, 0u};
          if (u < units)
            ptx::ld_shared_v4(rowa + 16u * static_cast<uint32_t>(u ^ (r & 7)), v);
#pragma unroll
          for (int t = 0; t < 4; ++t) w[4 * u + t] = v[t];
        }
        const uint32_t dst = tmem + lane_base + TMEM_A1 + 32u * hf;
        if (units == 8) {
          tmem_st_32x32b_x32(dst, w);
        } else {
          uint32_t w16[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) w16[t] = w[t];
          tmem_st_32x32b_x16(dst, w16);
        }
        tmem_st_wait();
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(a1_full);
    }
    if constexpr (!KV) {
      // delta of this query row = sum_e dO[r][e] O[r][e], both tiles in shared
      // memory (128-byte-swizzled rows; O, the forward's context, in the last
      // ring stage until ctx_free), summed in fp32 in column order by both
      // warps of the row (so both hold the same value without an exchange).
      const size_t off = static_cast<size_t>(head) * a.ld_stat + row0 + r;
      lse_r = a.lse[off];
      alive = alive && warp_wait(ctx_full, 0, ctl, ROLE_EPILOGUE);
      if (alive) {
#pragma unroll
        for (int u = 0; u < D / 8; ++u) {
          const uint32_t at = (u / 8) * KBLOCK_BYTES + r * 128 +
                              16 * ((u % 8) ^ (r & 7));
          const uint4 dv = *reinterpret_cast<const uint4*>(smem + A_TILE + at);
          const uint4 ov = *reinterpret_cast<const uint4*>(
              smem + 2 * A_TILE + (NB - 1) * 2 * B_TILE + at);
          const uint32_t dw4[4] = {dv.x, dv.y, dv.z, dv.w};
          const uint32_t ow4[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float d0, d1, o0, o1;
            unpack_bf16x2(dw4[k], d0, d1);
            unpack_bf16x2(ow4[k], o0, o1);
            delta_r = fmaf(d0, o0, delta_r);
            delta_r = fmaf(d1, o1, delta_r);
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ctx_free);
      }
    }
    float rsum = 0.f;              // Q: this half's sum of dS over its keys
    for (int n = 0; alive && n < nsteps; ++n) {
      const uint32_t bs = n % NB, bph = (n / NB) & 1;
      if (!warp_wait(s_full, static_cast<uint32_t>(n) & 1u, ctl,
                     ROLE_EPILOGUE) ||
          (KV && !warp_wait(b_full + 8 * bs, bph, ctl, ROLE_EPILOGUE))) {
        alive = false;
        break;
      }
      ptx::tc_fence_after();
      const int cb = cb_begin + n;
      // Causal validity of column c: KV (row = key): c >= lo; Q (row =
      // query): c <= hi.  Without the mask every column is valid.
      const int diff = rb * 128 + r - cb * 64 - 32 * hf;
      const int lo = (KV && a.causal) ? diff : -1;
      const int hi = (!KV && a.causal) ? diff : 64;
      uint32_t s1[32], s2[32];
      ptx::tmem_ld_32x32b_x32(tmem + lane_base + TMEM_S1 + 32 * hf, s1);
      ptx::tmem_ld_32x32b_x32(tmem + lane_base + TMEM_S2 + 32 * hf, s2);
      ptx::tmem_ld_wait();
      // S and dP are in registers: the next step's score MMAs may overwrite
      // them while this step's P and dS are formed
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(s_read);
      uint32_t pw[16], dw[16];
      // column pairs with packed fp32x2 arithmetic:
      // P = 2^(S sl2 - L), dS = P (dP - delta) / sqrt(d), from nL = -L and
      // nD = -delta
      const uint64_t scale = f2_pack(sl2, sl2);
      const uint64_t inv_sqrt_d = f2_pack(INV_SQRT_D, INV_SQRT_D);
      // the causal mask touches no column of this warp's rows: no selects
      const bool unmasked = __all_sync(0xffffffffu, lo <= 0 && hi >= 31);
      auto pair = [&](int i, float nL0, float nL1, float nD0, float nD1,
                      bool masked) {
        float a0, a1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(s1[i]), __uint_as_float(s1[i + 1])),
                         scale, f2_pack(nL0, nL1)),
                  a0, a1);
        float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
        if (masked) {
          p0 = (i >= lo && i <= hi) ? p0 : 0.f;
          p1 = (i + 1 >= lo && i + 1 <= hi) ? p1 : 0.f;
        }
        const uint64_t dp = f2_add(
            f2_pack(__uint_as_float(s2[i]), __uint_as_float(s2[i + 1])),
            f2_pack(nD0, nD1));
        float ds0, ds1;
        f2_unpack(f2_mul(f2_mul(f2_pack(p0, p1), dp), inv_sqrt_d), ds0, ds1);
        pw[i / 2] = pack_bf16x2(p0, p1);
        dw[i / 2] = pack_bf16x2(ds0, ds1);
        rsum += ds0 + ds1;
      };
      auto columns = [&](bool masked) {
        if constexpr (KV) {
          // the streamed queries' -lse2 and -delta', four columns a load,
          // each loaded two groups ahead of its use (the loads' latency
          // otherwise lies on the chain)
          const uint32_t va = sVec + bs * VEC_BYTES + 128u * hf;
          uint32_t l4[3][4], d4[3][4];
          ptx::ld_shared_v4(va, l4[0]);
          ptx::ld_shared_v4(va + 256u, d4[0]);
          ptx::ld_shared_v4(va + 16u, l4[1]);
          ptx::ld_shared_v4(va + 256u + 16u, d4[1]);
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const int g = i / 4;
            if (i + 8 < 32) {
              ptx::ld_shared_v4(va + 4u * (i + 8), l4[(g + 2) % 3]);
              ptx::ld_shared_v4(va + 256u + 4u * (i + 8), d4[(g + 2) % 3]);
            }
            const uint32_t(&l)[4] = l4[g % 3];
            const uint32_t(&d)[4] = d4[g % 3];
            pair(i, __uint_as_float(l[0]), __uint_as_float(l[1]),
                 __uint_as_float(d[0]), __uint_as_float(d[1]), masked);
            pair(i + 2, __uint_as_float(l[2]), __uint_as_float(l[3]),
                 __uint_as_float(d[2]), __uint_as_float(d[3]), masked);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            pair(i, -lse_r, -lse_r, -delta_r, -delta_r, masked);
            pair(i + 2, -lse_r, -lse_r, -delta_r, -delta_r, masked);
          }
        }
      };
      if (unmasked) {
        columns(false);
      } else {
        columns(true);
      }
      // P and dS into their buffer, this half's 32 columns packed two per
      // column, once step n - 1's gradient MMAs have read it
      if (n >= 1 &&
          !warp_wait(e_empty, static_cast<uint32_t>(n - 1) & 1u, ctl,
                     ROLE_EPILOGUE)) {
        alive = false;
        break;
      }
      ptx::tc_fence_after();
      tmem_st_32x32b_x16(tmem + lane_base + TMEM_PDS + 16 * hf, pw);
      tmem_st_32x32b_x16(tmem + lane_base + TMEM_PDS + 32 + 16 * hf, dw);
      tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(e_full);
    }
    float rrow = 0.f;
    if constexpr (!KV) {
      // Row sums of dS: zero for exact arithmetic, but delta comes from the
      // forward's rounded context while P and dP are this kernel's own, so
      // r = (sum_j P dP - delta) / sqrt(d) is not.  Every dS in the row
      // carries that offset, and the component shared by all keys, which
      // cancels in the exact dQ, would be amplified; subtracting r sum_j P k
      // gives dQ = sum_j P (dP - sum_j P dP) k / sqrt(d) with this kernel's
      // own P and dP.  The halves meet once (every path passes the barrier).
      float* red = reinterpret_cast<float*>(vec_gen);
      red[hf * 128 + r] = rsum;
      pair_barrier(q);
      rrow = red[r] + red[128 + r];
      // For the key/value kernel: delta' = sum_j P dP with this kernel's own
      // P and dP (= delta + r sqrt(d), the P of a row summing to 1), so that
      // its dS rows, formed from its own recomputed P and dP, carry no
      // offset either.  With delta from the rounded context instead, every
      // dS of a query row would be off by P times that rounding error,
      // which dK = dS^T Q does not cancel.
      if (alive && hf == 0) {
        const size_t off = static_cast<size_t>(head) * a.ld_stat + row0 + r;
        a.delta[off] = -lse_r;
        a.delta[static_cast<size_t>(a.heads) * a.ld_stat + off] =
            -(delta_r + rrow / INV_SQRT_D);
      }
    }
    if (alive && warp_wait(o_full, 0, ctl, ROLE_EPILOGUE)) {
      ptx::tc_fence_after();
      if constexpr (KV) {
        // Each warp writes its 32 rows of one output (half 0: dK, half 1:
        // dV), all D columns, as 32-row x 64-column bf16 chunks staged in
        // the (now idle) B ring and stored by TMA: full-line writes instead
        // of one row per thread.
        ChunkStager st{sB + static_cast<uint32_t>(warp - SOFTMAX_WARP0) * 2u *
                                STAGE_CHUNK_BYTES,
                       0u};
        const uint32_t src =
            tmem + lane_base + (hf == 0 ? TMEM_OUT2 : TMEM_OUT1);
        const int col = hf == 0 ? hc.k : hc.v;
#pragma unroll 1
        for (int j = 0; j < D / 64; ++j) {
          uint32_t r0[32], r1[32];
          ptx::tmem_ld_32x32b_x32(src + 64 * j, r0);
          ptx::tmem_ld_32x32b_x32(src + 64 * j + 32, r1);
          ptx::tmem_ld_wait();
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w[i] = pack_bf16x2(__uint_as_float(r0[2 * i]),
                               __uint_as_float(r0[2 * i + 1]));
            w[16 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]),
                                    __uint_as_float(r1[2 * i + 1]));
          }
          const uint32_t buf = st.put(&tmOut, col + 64 * j, row0 + q * 32, w, lane);
          if (a.colsum != nullptr) {     // bias-gradient partials, 32 rows
            const float2 cs = chunk_colsum_bf16(buf, lane);
            *reinterpret_cast<float2*>(
                a.colsum + static_cast<size_t>((row0 + q * 32) / 32) * a.ld_colsum +
                col + 64 * j + 2 * lane) = cs;
          }
        }
        if constexpr (D % 64 != 0) {
          // the last 32 columns (a 64-column chunk would reach into the next
          // head's columns): each thread its own row, 64 bytes
          const bool st_ok = TPMLP_CHECK(
              __all_sync(0xffffffffu,
                         (reinterpret_cast<uintptr_t>(
                              a.dqkv + static_cast<size_t>(row0 + r) * a.ld_qkv +
                              col + 64 * (D / 64)) & 15u) == 0),
              a.status, abort_flag, SITE_ATTN_BWD_STORE);
          uint32_t rr[32];
          ptx::tmem_ld_32x32b_x32(src + 64 * (D / 64), rr);
          ptx::tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(rr[i]);
          if (st_ok)
            store_bf16x32(a.dqkv + static_cast<size_t>(row0 + r) * a.ld_qkv +
                              col + 64 * (D / 64),
                          v);
          if (a.colsum != nullptr) {     // their bias-gradient partials
            const float2 cs = tail_colsum_bf16(st, v, lane);
            if (lane < 16)
              *reinterpret_cast<float2*>(
                  a.colsum +
                  static_cast<size_t>((row0 + q * 32) / 32) * a.ld_colsum +
                  col + 64 * (D / 64) + 2 * lane) = cs;
          }
        }
        st.drain(lane);
      } else if constexpr (D == 96) {
        // dQ: the first column half's warps 64 columns as one chunk (staged,
        // stored by TMA, summed for the bias-gradient partials), the second
        // half's warps the last 32 columns with 16-byte stores of their rows
        ChunkStager st{sB + static_cast<uint32_t>(warp - SOFTMAX_WARP0) * 2u *
                                STAGE_CHUNK_BYTES,
                       0u};
        const uint32_t src2 = tmem + lane_base + TMEM_OUT2 + hf * 64;
        const uint32_t src1 = tmem + lane_base + TMEM_OUT1 + hf * 64;
        if (hf == 0) {
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            uint32_t ov[32], kv[32];
            ptx::tmem_ld_32x32b_x32(src2 + 32 * j, ov);
            ptx::tmem_ld_32x32b_x32(src1 + 32 * j, kv);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[16 * j + i] = pack_bf16x2(
                  fmaf(-rrow, __uint_as_float(kv[2 * i]),
                       __uint_as_float(ov[2 * i])),
                  fmaf(-rrow, __uint_as_float(kv[2 * i + 1]),
                       __uint_as_float(ov[2 * i + 1])));
          }
          const uint32_t buf = st.put(&tmOut, hc.q, row0 + q * 32, w, lane);
          if (a.colsum != nullptr) {
            const float2 cs = chunk_colsum_bf16(buf, lane);
            *reinterpret_cast<float2*>(
                a.colsum +
                static_cast<size_t>((row0 + q * 32) / 32) * a.ld_colsum +
                hc.q + 2 * lane) = cs;
          }
        } else {
          uint32_t ov[32], kv[32];
          ptx::tmem_ld_32x32b_x32(src2, ov);
          ptx::tmem_ld_32x32b_x32(src1, kv);
          ptx::tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i)
            v[i] = fmaf(-rrow, __uint_as_float(kv[i]), __uint_as_float(ov[i]));
          __nv_bfloat16* out2 =
              a.dqkv + static_cast<size_t>(row0 + r) * a.ld_qkv + hc.q + 64;
          if (TPMLP_CHECK(__all_sync(0xffffffffu,
                                     (reinterpret_cast<uintptr_t>(out2) & 15u) == 0),
                          a.status, abort_flag, SITE_ATTN_BWD_STORE))
            store_bf16x32(out2, v);
          if (a.colsum != nullptr) {
            const float2 cs = tail_colsum_bf16(st, v, lane);
            if (lane < 16)
              *reinterpret_cast<float2*>(
                  a.colsum +
                  static_cast<size_t>((row0 + q * 32) / 32) * a.ld_colsum +
                  hc.q + 64 + 2 * lane) = cs;
          }
        }
        st.drain(lane);
      } else if constexpr (D == 128 || D == 64) {
        // dQ: each warp its 32 rows x 64 columns (one chunk; at d = 64 the
        // first column half's warps hold all of them), staged and stored by
        // TMA like the key/value outputs
        if (hf * 64 < D) {
          ChunkStager st{sB + static_cast<uint32_t>(warp - SOFTMAX_WARP0) * 2u *
                                  STAGE_CHUNK_BYTES,
                         0u};
          const uint32_t src2 = tmem + lane_base + TMEM_OUT2 + hf * 64;
          const uint32_t src1 = tmem + lane_base + TMEM_OUT1 + hf * 64;
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            uint32_t ov[32], kv[32];
            ptx::tmem_ld_32x32b_x32(src2 + 32 * j, ov);
            ptx::tmem_ld_32x32b_x32(src1 + 32 * j, kv);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[16 * j + i] = pack_bf16x2(
                  fmaf(-rrow, __uint_as_float(kv[2 * i]), __uint_as_float(ov[2 * i])),
                  fmaf(-rrow, __uint_as_float(kv[2 * i + 1]),
                       __uint_as_float(ov[2 * i + 1])));
          }
          const uint32_t buf = st.put(&tmOut, hc.q + 64 * hf, row0 + q * 32, w, lane);
          if (a.colsum != nullptr) {
            const float2 cs = chunk_colsum_bf16(buf, lane);
            *reinterpret_cast<float2*>(
                a.colsum + static_cast<size_t>((row0 + q * 32) / 32) * a.ld_colsum +
                hc.q + 64 * hf + 2 * lane) = cs;
          }
          st.drain(lane);
        }
      } else {
        // dQ: this warp's D / 2 columns of its row, 16 at a time
        __nv_bfloat16* out2 = a.dqkv + static_cast<size_t>(row0 + r) * a.ld_qkv +
                              hc.q + hf * (D / 2);
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {
          uint32_t ov[16], kv[16];
          ptx::tmem_ld_32x32b_x16(
              tmem + lane_base + TMEM_OUT2 + hf * (D / 2) + 16 * j, ov);
          ptx::tmem_ld_32x32b_x16(
              tmem + lane_base + TMEM_OUT1 + hf * (D / 2) + 16 * j, kv);
          ptx::tmem_ld_wait();
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            v[i] = fmaf(-rrow, __uint_as_float(kv[i]), __uint_as_float(ov[i]));
          store_bf16x16(out2 + 16 * j, v);
        }
      }
    }
    __syncwarp();
  }

  // --------------------------------------------------------- teardown --
  ptx::tc_fence_before();
  cta_barrier_att();
  if (*reinterpret_cast<volatile int*>(abort_flag) && threadIdx.x == 0) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < ABORT_SETTLE_NS) {
    }
  }
  cta_barrier_att();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// Dynamic shared memory; at least 116 KB so that a second CTA (and its 512
// TMEM columns) never shares the SM.
template <int D, bool KV>
size_t attn_bwd_smem() {
  constexpr int KB = (D + 63) / 64;
  constexpr int NB = KV ? 4 : 5;
  const size_t need = 1024 + 2 * KB * KBLOCK_BYTES + NB * 2 * KB * ATOM_BYTES +
                      (KV ? NB * 512 : 1024) + (12 + 2 * NB) * 8 + 16;
  return need > 116 * 1024 ? need : 116 * 1024;
}

template <int D, bool KV>
cudaError_t launch_bwd(const CUtensorMap& a1, const CUtensorMap& a2,
                       const CUtensorMap& b1, const CUtensorMap& b2,
                       const CUtensorMap& tctx, const CUtensorMap& tout,
                       const AttnArgs& a, int grid, cudaStream_t s) {
  auto kern = attn_bwd_kernel<D, KV>;
  const size_t smem = attn_bwd_smem<D, KV>();
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, ATT_THREADS, smem, s>>>(a1, a2, b1, b2, tctx, tout, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_dkdv(const CUtensorMap& tq128, const CUtensorMap& tq64,
                             const CUtensorMap& tdo64,
                             const CUtensorMap& tdqkv_out, const AttnArgs& a,
                             int grid, cudaStream_t s) {
  if (a.head_dim == 128)
    return launch_bwd<128, true>(tq128, tq128, tq64, tdo64, tq128, tdqkv_out, a,
                                 grid, s);
  if (a.head_dim == 96)
    return launch_bwd<96, true>(tq128, tq128, tq64, tdo64, tq128, tdqkv_out, a,
                                grid, s);
  if (a.head_dim == 64)
    return launch_bwd<64, true>(tq128, tq128, tq64, tdo64, tq128, tdqkv_out, a,
                                grid, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_dq(const CUtensorMap& tq128, const CUtensorMap& tq64,
                           const CUtensorMap& tdo128, const CUtensorMap& tctx128,
                           const CUtensorMap& tdqkv_out, const AttnArgs& a,
                           int grid, cudaStream_t s) {
  if (a.head_dim == 128)
    return launch_bwd<128, false>(tq128, tdo128, tq64, tq64, tctx128, tdqkv_out,
                                  a, grid, s);
  if (a.head_dim == 96)
    return launch_bwd<96, false>(tq128, tdo128, tq64, tq64, tctx128, tdqkv_out,
                                 a, grid, s);
  if (a.head_dim == 64)
    return launch_bwd<64, false>(tq128, tdo128, tq64, tq64, tctx128, tdqkv_out,
                                 a, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace tpmlp
