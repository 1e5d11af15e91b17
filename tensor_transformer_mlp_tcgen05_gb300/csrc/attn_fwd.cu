// Attention core of the head-parallel self-attention block on sm_103a.
//
// The heads are independent (Megatron-LM explainer, section on attention;
// notes, "Self-attention block split"), so each (sequence, head, 128-query
// block) item is computed on its own and no CTA communicates with another.
// Q, K and V are read in
// place from the fused projection output QKV [T, 3h] (columns grouped by
// shard: [Q_i | K_i | V_i], head j of shard i at offset (j mod H/t) d inside
// each group) through TMA tensor maps; scores, probabilities and the output
// accumulator live in TMEM.
//
// Forward, one pass over the key blocks the query block may see (all of
// them, or blocks 0..qb when causal): S = Q K^T (tcgen05, M = N = 128,
// K = d) into TMEM -> P = exp2(S log2e / sqrt d - m_ref) with a lazily
// raised reference max -> bf16 P stored by the softmax threads over the
// scores (one row per lane) -> O += P V with A read from TMEM (only V comes
// from shared memory, which keeps the MMA's operand reads under the SM's
// shared-memory bandwidth); O / l at the end.
// Outputs: the context rows (bf16) and, for the backward, every (head,
// token) row's log-sum-exp in base 2 of the scores scaled by log2(e)/sqrt(d),
// lse2 = m + log2(l), so that P = exp2(S log2(e)/sqrt(d) - lse2).
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 TMEM allocator and
// MMA issuer (the whole warp; one elected lane issues), warps 2-9 softmax
// (thread = query row = TMEM lane, two warps per row quarter, one per half
// of the columns).  Each CTA walks its key blocks strictly in turn (S, then
// the softmax, then P V, then the next S over the same TMEM columns) and
// holds 256 TMEM columns and ~100 KB of shared memory, so two CTAs share an
// SM and the tensor core works for one while the other is in its softmax.
// The CTAs are persistent (two per SM), each walking a list of (sequence,
// head, query block) items: the next item's Q and first K and V load, and
// its first S runs, while the softmax warps finish the previous item's
// output, which frees O for the next item's first P V.  All waits are
// bounded as in the GEMM kernels.
#include "attn_common.cuh"

namespace tpmlp {
namespace {

using namespace gemm;
using namespace attn;

constexpr int FWD_THREADS = 320;
constexpr int FWD_SOFTMAX_WARP0 = 2;
constexpr uint32_t FWD_TMEM_COLS = 256;

__device__ __forceinline__ void fwd_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(FWD_THREADS) : "memory");
}

// TMEM column of the packed P values for keys 16k .. 16k + 15: each column
// half of the softmax writes its 64 keys' P over the first 32 of its own 64
// score columns.
__device__ __forceinline__ constexpr uint32_t p_col(int k) {
  return 64u * static_cast<uint32_t>(k / 4) + 8u * static_cast<uint32_t>(k % 4);
}

template <int D>
__global__ void __launch_bounds__(FWD_THREADS, 2)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQK,
                    const __grid_constant__ CUtensorMap tmV,
                    const AttnArgs a) {
  // 64-wide blocks of d (d = 96: the second block's upper 32 columns belong
  // to the next head or lie past the tensor; they are loaded, never used:
  // the MMAs below stop at K = d and N = d)
  constexpr int KB = (D + 63) / 64;
  constexpr uint32_t QK_TILE = KB * KBLOCK_BYTES;      // 128 x D
  constexpr uint32_t V_TILE = 2 * KB * ATOM_BYTES;     // 128 keys x D
  constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, false, true);
  constexpr uint32_t TMEM_O = 128;   // S in columns 0-127, P over S

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = ptx::smem_u32(smem);
  const uint32_t sK = sQ + QK_TILE;
  const uint32_t sV = sK + QK_TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * QK_TILE + V_TILE);
  const uint32_t b0 = ptx::smem_u32(bars);
  const uint32_t q_full = b0, k_full = b0 + 8, k_empty = b0 + 16,
                 v_full = b0 + 24, v_empty = b0 + 32, s_full = b0 + 40,
                 p_full = b0 + 48, pv_done = b0 + 56, done_bar = b0 + 64,
                 q_empty = b0 + 72, o_free = b0 + 80;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 11);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  // Row max (per block, two parities) and row sum exchange between the two
  // column halves: [3][2][128].
  float* red = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 128);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = a.nq;
  // Persistent: the (sequence, head, query block) items in core_item order,
  // dealt to the CTAs in rounds, forwards in even rounds and backwards in odd
  // ones, so that with the longest items first in each round every CTA gets
  // about the same total; every role walks the same list.
  const int hs_total = (static_cast<int>(a.ld_stat) / a.seq_len) * a.heads;
  const int n_items = hs_total * nq;
  const int C = static_cast<int>(gridDim.x);
  auto item_at = [&](int ic) -> int {
    const int base = ic * C;
    return base + ((ic & 1) ? C - 1 - static_cast<int>(blockIdx.x)
                            : static_cast<int>(blockIdx.x));
  };
  struct Work {
    int qb, head, seq, row0, nk;
    HeadCols hc;
  };
  auto decode = [&](int idx) -> Work {
    const CoreItem it = core_item(idx, hs_total, nq, a.heads, a.hs_group);
    Work w;
    w.qb = nq - 1 - it.rank;
    w.head = it.head;
    w.seq = it.seq;
    w.row0 = it.seq * a.seq_len + w.qb * 128;
    w.nk = a.causal ? w.qb + 1 : nq;
    w.hc = head_cols(a, it.head);
    return w;
  };

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1);
    ptx::mbar_init(k_full, 1);
    ptx::mbar_init(k_empty, 1);
    ptx::mbar_init(v_full, 1);
    ptx::mbar_init(v_empty, 1);
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(p_full, SOFTMAX_WARPS);
    ptx::mbar_init(pv_done, 1);
    ptx::mbar_init(o_free, SOFTMAX_WARPS);
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), FWD_TMEM_COLS);
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
      // One stage each for Q, K and V: Q of the next item once the MMAs
      // have read this item's Q for the last time, K(j) once S(j - 1) is
      // done, V(j) once P V(j - 1) is done (j counts key blocks over all of
      // this CTA's items).  (Debug builds: the head's column offsets, the
      // copies' innermost coordinates, on a 16-byte boundary.)
      uint32_t kc = 0;
      bool alive = true;
      for (int ic = 0; alive; ++ic) {
        const int idx = item_at(ic);
        if (idx >= n_items) break;
        const Work w = decode(idx);
        if (!TPMLP_CHECK(w.hc.q % 8 == 0 && w.hc.k % 8 == 0 && w.hc.v % 8 == 0,
                         a.status, abort_flag, SITE_ATTN_FWD_LOAD))
          break;
        if (ic > 0 && !wait_bounded(q_empty, static_cast<uint32_t>(ic - 1) & 1u,
                                    ctl, ROLE_PRODUCER))
          break;
        ptx::mbar_arrive_expect_tx(q_full, QK_TILE);
#pragma unroll
        for (int kk = 0; kk < KB; ++kk)
          ptx::tma_load_2d(sQ + kk * KBLOCK_BYTES, &tmQK, q_full,
                           w.hc.q + 64 * kk, w.row0);
        for (int kb = 0; kb < w.nk; ++kb, ++kc) {
          const int key0 = w.seq * a.seq_len + kb * 128;
          const uint32_t prev = (kc - 1u) & 1u;
          if (kc > 0 && !wait_bounded(k_empty, prev, ctl, ROLE_PRODUCER)) {
            alive = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(k_full, QK_TILE);
#pragma unroll
          for (int kk = 0; kk < KB; ++kk)
            ptx::tma_load_2d(sK + kk * KBLOCK_BYTES, &tmQK, k_full,
                             w.hc.k + 64 * kk, key0);
          if (kc > 0 && !wait_bounded(v_empty, prev, ctl, ROLE_PRODUCER)) {
            alive = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(v_full, V_TILE);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
            for (int at = 0; at < KB; ++at)
              ptx::tma_load_2d(sV + (h2 * KB + at) * ATOM_BYTES, &tmV, v_full,
                               w.hc.v + 64 * at, key0 + 64 * h2);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    {
      // ------------------------ MMA issuer (whole warp, elected lane) --
      const uint64_t dQ = ptx::sdesc_sw128(sQ, 16, 1024);
      const uint64_t dK = ptx::sdesc_sw128(sK, 16, 1024);
      const uint64_t dV = ptx::sdesc_sw128(sV, ATOM_BYTES, 1024);
      uint32_t kc = 0;
      bool alive = true;
      for (int ic = 0; alive; ++ic) {
        const int idx = item_at(ic);
        if (idx >= n_items) break;
        const Work w = decode(idx);
        if (!warp_wait(q_full, static_cast<uint32_t>(ic) & 1u, ctl, ROLE_MMA))
          break;
        for (int kb = 0; kb < w.nk; ++kb, ++kc) {
          const uint32_t ph = kc & 1u;
          // S = Q K^T into the score columns, once P V of the previous key
          // block (of this item or the last one) has read its P from them
          if (!warp_wait(k_full, ph, ctl, ROLE_MMA) ||
              (kc > 0 && !warp_wait(pv_done, ph ^ 1u, ctl, ROLE_MMA))) {
            alive = false;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k / 4) * KBLOCK_BYTES + (k % 4) * 32;
            mma_ss_el(tmem, desc_add(dQ, off), desc_add(dK, off), IDESC_S,
                      k > 0 ? 1u : 0u);
          }
          commit_el(k_empty);
          commit_el(s_full);
          if (kb == w.nk - 1) commit_el(q_empty);
          // O += P V once the softmax has written P over the scores (the
          // first block of an item also once the previous item's output has
          // been read out of O)
          if (!warp_wait(p_full, ph, ctl, ROLE_MMA) ||
              !warp_wait(v_full, ph, ctl, ROLE_MMA) ||
              (kb == 0 && ic > 0 &&
               !warp_wait(o_free, static_cast<uint32_t>(ic - 1) & 1u, ctl,
                          ROLE_MMA))) {
            alive = false;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts_el(tmem + TMEM_O, tmem + p_col(k),
                      desc_add(dV, (k / 4) * KB * ATOM_BYTES + (k % 4) * 2048),
                      IDESC_O, (kb > 0 || k > 0) ? 1u : 0u);
          commit_el(v_empty);
          commit_el(pv_done);
        }
      }
      if (*reinterpret_cast<volatile int*>(abort_flag)) {
        commit_el(done_bar);
        wait_teardown(done_bar, 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ softmax --
    // One pass over each item's key blocks with a lazily updated reference
    // max (log2 units of the scaled scores).  Two warps share each row
    // quarter, one per column half; per block they exchange their halves'
    // maxima through shared memory.  P = exp2(x - m_ref) is written as bf16
    // over the half's own score columns, 32 columns at a time (the scores
    // are read twice, for the max and for P, to keep register use low enough
    // for two CTAs per SM).  Only when the block max exceeds m_ref by more
    // than RESCALE_LOG2 does m_ref move up, with O (each warp its half of
    // the D columns) and the partial row sums scaled by exp2(m_old - m_new);
    // the previous P V is complete by then, since S(kb) was issued after it.
    // The decision depends only on the scores, so it is deterministic, and
    // P stays below 2^RESCALE_LOG2.  Output O / (l0 + l1); saved lse2 =
    // m_ref + log2 l; then O is released for the next item.  Every softmax
    // warp passes the same barriers on every path.
    constexpr float RESCALE_LOG2 = 8.f;
    const int q = warp & 3;
    const int hf = (warp - FWD_SOFTMAX_WARP0) >> 2;
    const int r = q * 32 + lane;          // query row inside the block
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t scol = tmem + lane_base + 64 * hf;
    const float sl2 = a.scale_log2;
    uint32_t kc = 0;
    bool alive = true;
    for (int ic = 0; alive; ++ic) {
      const int idx = item_at(ic);
      if (idx >= n_items) break;
      const Work w = decode(idx);
      float m_ref = -INFINITY, l = 0.f;
      for (int kb = 0; kb < w.nk; ++kb, ++kc) {
        bool ok = alive && warp_wait(s_full, kc & 1u, ctl, ROLE_EPILOGUE);
        // only the diagonal block of a causal row masks anything
        const bool diag = a.causal && kb == w.qb;
        const int lim = diag ? r - 64 * hf : 63;
        float mb = -INFINITY;
        if (ok) {
          ptx::tc_fence_after();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t sv[32];
            ptx::tmem_ld_32x32b_x32(scol + 32 * c, sv);
            ptx::tmem_ld_wait();
            if (diag) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (32 * c + j <= lim) mb = fmaxf(mb, __uint_as_float(sv[j]));
            } else {
              // two chains of three-input maxima
              float m0 = mb, m1 = mb;
#pragma unroll
              for (int j = 0; j < 32; j += 4) {
                m0 = max3(m0, __uint_as_float(sv[j]), __uint_as_float(sv[j + 1]));
                m1 = max3(m1, __uint_as_float(sv[j + 2]),
                          __uint_as_float(sv[j + 3]));
              }
              mb = fmaxf(m0, m1);
            }
          }
        }
        // exchange the halves' maxima (double-buffered by block parity)
        red[(kc & 1u) * 256 + hf * 128 + r] = mb * sl2;
        pair_barrier(q);
        mb = fmaxf(red[(kc & 1u) * 256 + r], red[(kc & 1u) * 256 + 128 + r]);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          alive = false;
          continue;              // keep meeting the sibling's barriers
        }
        float alpha = 1.f;
        const bool move = mb > m_ref + RESCALE_LOG2;
        if (move) {
          alpha = exp2f(m_ref - mb);       // 0 on the first block
          m_ref = mb;
        }
        if (__any_sync(0xffffffffu, move) && kb > 0) {
          // this warp's D / 2 output columns, 16 at a time
#pragma unroll 1
          for (int j = 0; j < D / 32; ++j) {
            const uint32_t oc =
                tmem + lane_base + TMEM_O + hf * (D / 2) + 16 * j;
            uint32_t ov[16];
            ptx::tmem_ld_32x32b_x16(oc, ov);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st_32x32b_x16(oc, ov);
          }
        }
        // P: 32 scores at a time, packed two per column over columns that
        // this warp has already read
        float lb0 = 0.f, lb1 = 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t sv[32];
          ptx::tmem_ld_32x32b_x32(scol + 32 * c, sv);
          ptx::tmem_ld_wait();
          uint32_t pw[16];
          if (!diag) {
            // pairs of columns with packed fp32x2 arithmetic (same results
            // as the scalar form below; lb0 / lb1 are the pair's two lanes)
            const uint64_t scale = f2_pack(sl2, sl2);
            const uint64_t shift = f2_pack(-m_ref, -m_ref);
            uint64_t lb = f2_pack(lb0, lb1);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              float a0, a1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[j]),
                                       __uint_as_float(sv[j + 1])),
                               scale, shift),
                        a0, a1);
              const float p0 = ex2_approx(a0);
              const float p1 = ex2_approx(a1);
              lb = f2_add(lb, f2_pack(p0, p1));
              pw[j / 2] = pack_bf16x2(p0, p1);
            }
            f2_unpack(lb, lb0, lb1);
          } else {
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              float p0 =
                  ex2_approx(fmaf(__uint_as_float(sv[j]), sl2, -m_ref));
              float p1 =
                  ex2_approx(fmaf(__uint_as_float(sv[j + 1]), sl2, -m_ref));
              p0 = 32 * c + j <= lim ? p0 : 0.f;
              p1 = 32 * c + j + 1 <= lim ? p1 : 0.f;
              lb0 += p0;
              lb1 += p1;
              pw[j / 2] = pack_bf16x2(p0, p1);
            }
          }
          tmem_st_32x32b_x16(scol + 16 * c, pw);
        }
        l = l * alpha + (lb0 + lb1);
        tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(p_full);
      }
      red[512 + hf * 128 + r] = l;
      alive = softmax_barrier_and(alive);
      l = red[512 + r] + red[512 + 128 + r];
      const bool done =
          alive && warp_wait(pv_done, (kc - 1u) & 1u, ctl, ROLE_EPILOGUE);
      if (done) {
        ptx::tc_fence_after();
        const float inv_l = 1.0f / l;
        // this warp's D / 2 context columns, 16 at a time (32 bytes a row)
        __nv_bfloat16* out = a.ctx +
                             static_cast<size_t>(w.row0 + r) * a.ld_ctx +
                             w.head * D + hf * (D / 2);
        // (warp-uniform: the loop's TMEM loads are warp-collective)
        if (TPMLP_CHECK(__all_sync(0xffffffffu,
                                   (reinterpret_cast<uintptr_t>(out) & 15u) == 0 &&
                                       w.row0 + r < a.ld_stat),
                        a.status, abort_flag, SITE_ATTN_FWD_STORE))
#pragma unroll 1
        for (int j = 0; j < D / 32; ++j) {
          uint32_t ov[16];
          ptx::tmem_ld_32x32b_x16(
              tmem + lane_base + TMEM_O + hf * (D / 2) + 16 * j, ov);
          ptx::tmem_ld_wait();
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(ov[i]) * inv_l;
          store_bf16x16(out + 16 * j, v);
        }
        if (hf == 0)
          a.lse[static_cast<size_t>(w.head) * a.ld_stat + w.row0 + r] =
              m_ref + log2f(l);
        // O has been read: the next item's first P V may overwrite it
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(o_free);
      }
      // every softmax warp goes on to the next item, or none does
      alive = softmax_barrier_and(done);
    }
    __syncwarp();
  }

  // --------------------------------------------------------- teardown --
  ptx::tc_fence_before();
  fwd_barrier();
  if (*reinterpret_cast<volatile int*>(abort_flag) && threadIdx.x == 0) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < ABORT_SETTLE_NS) {
    }
  }
  fwd_barrier();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, FWD_TMEM_COLS);
  }
}

// Dynamic shared memory: Q, one K and one V stage, barriers and the
// exchange buffers (~100 KB at d = 128), and at least 80 KB so that never
// more than two CTAs (2 x 256 TMEM columns) share an SM.
template <int D>
size_t attn_fwd_smem() {
  constexpr int KB = (D + 63) / 64;
  const size_t need = 1024 + 2 * KB * KBLOCK_BYTES + 2 * KB * ATOM_BYTES +
                      128 + 6 * 128 * 4;
  return need > 80 * 1024 ? need : 80 * 1024;
}

template <int D>
cudaError_t launch_fwd(const CUtensorMap& tqk, const CUtensorMap& tv,
                       const AttnArgs& a, int grid, cudaStream_t s) {
  auto kern = attn_fwd_kernel<D>;
  const size_t smem = attn_fwd_smem<D>();
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, FWD_THREADS, smem, s>>>(tqk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const CUtensorMap& tqk, const CUtensorMap& tv,
                            const AttnArgs& a, int grid, cudaStream_t s) {
  if (a.head_dim == 128) return launch_fwd<128>(tqk, tv, a, grid, s);
  if (a.head_dim == 96) return launch_fwd<96>(tqk, tv, a, grid, s);
  if (a.head_dim == 64) return launch_fwd<64>(tqk, tv, a, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace tpmlp
