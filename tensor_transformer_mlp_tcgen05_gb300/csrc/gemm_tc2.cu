// Persistent, warp-specialised CTA-pair tcgen05 GEMM for sm_103a
// (cta_group::2) with fused epilogues, 256 x 256 output tile per pair.
//
// Clusters of 2 CTAs; the pair (CTA ranks 0 and 1) owns one 256 x 256 tile
// at a time, persistent over the tile list.  Per k-block each CTA loads only
// its half of the operands into its own shared memory: rank r loads A rows
// [m0 + 128 r, +128) and B columns [n0 + 128 r, +128), 32 KB per stage.  The
// even CTA issues tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16): the
// tensor cores of both SMs read A from their own CTA and B from both, and
// each CTA receives its 128 rows of D (all 256 columns) in its own TMEM.  The
// ring has 5 stages (160 KB) next to 64 KB of epilogue staging.
//
// 12 warps in 3 warpgroups per CTA:
//   warp 0      TMA producer (one lane).
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators,
//               so the epilogue of one tile runs while the MMAs of the next
//               proceed); on the even CTA one lane issues the MMAs and
//               commits.
//   warps 2-3   idle.
//   warps 4-11  epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 (its
//               sub-partition) and one 128-column half of the tile.  With
//               the fused LayerNorm prologue (GemmArgs::ln_x) they first
//               normalise rows of the raw input into the A operand, one row
//               per warp at a time, claimed from a counter shared by the
//               whole grid, while the producers of tiles whose 128-row A
//               blocks are complete already load and the MMAs run.
// Registers: the CTA is launched with 168 per thread (384 x 168 = 64512); the
// first warpgroup gives registers back (down to REGS_CONTROL) and the two
// epilogue warpgroups take them (up to REGS_EPILOGUE), enough to hold a
// 128-column fp32 shard-sum row per thread.
//
// Shard sum (the on-device form of the pages' g forward and f backward
// all-reduces): the K range is cut into `num_seg` segments, one per shard.
// Each segment starts a fresh accumulator (the MMA's accumulate flag is off
// on its first k-step); the epilogue adds the segment partials into fp32
// registers in segment order 0..t-1, adds the bias and rounds once.  Every
// output element has one writer and a fixed summation order, so results are
// bitwise reproducible.
//
// Every pair loads its own operands: the launch uses clusters of exactly two
// CTAs, and no copy writes into another pair's shared memory.
//
// Synchronisation:
//   full[s]   (pair leader only) counts the TMA bytes landing in both CTAs of
//             the pair: the leader arms it with the pair's 64 KB, both CTAs'
//             copies complete on it.
//   empty[s]  (each CTA) arrived by the MMA issuer's commit (signalled to
//             both CTAs of the pair) when the MMAs have read stage s,
//             releasing the producers.
//   tfull[b]  (each CTA) arrived by a commit signalled to both CTAs when
//             accumulator b is ready in both TMEMs.
//   tempty[b] (rank 0 only) 16 arrivals: 8 epilogue warps of each CTA, the
//             peer's arriving remotely.
// Epilogue: each warp turns its 32 TMEM lanes into 32-row x 128-byte chunks
// (64 bf16 or 32 fp32 columns), stages them in shared memory and writes them
// with asynchronous TMA stores (coalesced full-line writes; rows or columns
// past the tensor's edge are clipped by the TMA unit), double-buffered per
// warp, so the epilogue never issues row-strided global stores.
// Every mbarrier wait is bounded by a time budget; on expiry the CTA records
// TPMLP_ERR_TIMEOUT in the status word, the other roles see a shared abort
// flag and stop, outstanding copies and MMAs are waited for (bounded), TMEM
// is freed and the kernel returns.  Both CTAs meet at cluster barriers
// before the first copy and before TMEM is freed, so no CTA leaves while its
// peer may still touch its shared memory or barriers.
//
// With F8 the operands are E4M3 bytes (both K-major): a k-block is 128
// elements, still one 128-byte swizzle row, each MMA (kind::f8f6f4, K = 32)
// consumes the same 32 bytes as a bf16 K = 16 step, so the ring, the
// descriptors and the tile shapes are unchanged; the epilogue multiplies the
// fp32 accumulator by the product of the operands' per-tensor scales.
#include <cstdlib>
#include <cstring>

#include "gemm_common.cuh"
#include "host_common.cuh"

namespace tpmlp {
namespace {

using namespace gemm;

constexpr int PM = 256;  // tile rows per pair
constexpr int PN = 256;  // tile columns per pair
constexpr int HM = 128;  // rows per CTA
constexpr int HN = 128;  // B columns staged per CTA
constexpr int BK = TC_BK;
constexpr int STAGES = 5;
constexpr int NUM_THREADS = 384;
constexpr int NUM_EPI_WARPS = 8;
constexpr int FIRST_EPI_WARP = 4;
constexpr int REGS_LAUNCH = 168;
constexpr int REGS_CONTROL = 56;
constexpr int REGS_EPILOGUE = 224;
static_assert(REGS_CONTROL * 128 + REGS_EPILOGUE * 256 <=
                  REGS_LAUNCH * NUM_THREADS,
              "register split exceeds the launch allocation");
constexpr uint32_t A_STAGE_BYTES = HM * BK * 2;  // 16 KiB
constexpr uint32_t B_STAGE_BYTES = HN * BK * 2;  // 16 KiB
constexpr uint32_t STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr uint32_t PAIR_STAGE_BYTES = 2 * STAGE_BYTES;
constexpr uint32_t TMEM_COLS = 2 * PN;
// full, empty (per stage), tfull, tempty (per accumulator), done, and one
// per epilogue warp for EPI_GELU_BWD's H chunks
constexpr int NUM_BARRIERS = 2 * STAGES + 5 + NUM_EPI_WARPS;
constexpr uint32_t EPI_STAGING_BYTES = NUM_EPI_WARPS * 2 * STAGE_CHUNK_BYTES;
constexpr size_t SMEM_BYTES = 1024 + size_t(STAGES) * STAGE_BYTES +
                              EPI_STAGING_BYTES + NUM_BARRIERS * 8 + 16;
// On an abort, copies this CTA issued may still be landing in its shared
// memory (their completions are counted on the peer's barrier), so the CTA
// waits this long before freeing its resources.
constexpr unsigned long long ABORT_SETTLE_NS = 2000000ull;

static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ void cta_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(NUM_THREADS) : "memory");
}

// The epilogue warps only.
__device__ __forceinline__ void epilogue_barrier() {
  asm volatile("bar.sync 2, %0;" ::"n"(NUM_EPI_WARPS * 32) : "memory");
}

// The fused LayerNorm prologue stages gamma and beta (fp32, up to 256
// LN_VMAX values each) in the epilogue staging buffers before their first use.
static_assert(2 * 256 * LN_VMAX * 4 <= EPI_STAGING_BYTES,
              "LayerNorm parameters exceed the staging buffers");

// Bounded wait with cluster-scope acquire (tempty: arrivals from both CTAs).
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar,
                                                     uint32_t parity,
                                                     const Ctl& c, int role) {
  if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    if (*c.abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > c.budget) {
      *c.abort_flag = 1;
      if (atomicCAS(c.status, 0, TPMLP_ERR_TIMEOUT) == 0) {
        c.status[1] = role;
        c.status[2] = static_cast<int>(blockIdx.x);
      }
      __threadfence();
      return false;
    }
  }
}

// One unit of a group's work: a whole super-tile, or one piece of a tail
// super-tile (see GemmArgs::part): segments [seg_lo, seg_hi) and k-blocks
// [kb_lo, kb_hi), kbs k-blocks per accumulator.
struct Item {
  int sup, piece;  // piece -1: the whole super-tile
  int seg_lo, seg_hi, kb_lo, kb_hi, kbs;
};

__device__ __forceinline__ Item decode_item(int item, int num_full,
                                            const GemmArgs& a) {
  Item it;
  const int kb_total = a.kb_per_seg * a.num_seg;
  if (item < num_full) {
    it.sup = item;
    it.piece = -1;
    it.seg_lo = 0;
    it.seg_hi = a.num_seg;
    it.kb_lo = 0;
    it.kb_hi = kb_total;
    it.kbs = a.kb_per_seg;
    return it;
  }
  const int j = item - num_full;
  it.sup = num_full + j / a.pieces;
  it.piece = j % a.pieces;
  if (a.num_seg > 1) {  // whole shard segments
    it.seg_lo = a.num_seg * it.piece / a.pieces;
    it.seg_hi = a.num_seg * (it.piece + 1) / a.pieces;
    it.kb_lo = it.seg_lo * a.kb_per_seg;
    it.kb_hi = it.seg_hi * a.kb_per_seg;
    it.kbs = a.kb_per_seg;
  } else {              // k-blocks of the single accumulation
    it.seg_lo = 0;
    it.seg_hi = 1;
    it.kb_lo = kb_total * it.piece / a.pieces;
    it.kb_hi = kb_total * (it.piece + 1) / a.pieces;
    it.kbs = it.kb_hi - it.kb_lo;
  }
  return it;
}

template <bool A_MN, bool B_MN, int EPI, bool F8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmO,
                    const __grid_constant__ CUtensorMap tmO2,
                    const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_a = ptx::smem_u32(smem);
  const uint32_t s_b = s_a + STAGES * A_STAGE_BYTES;
  const uint32_t s_epi = s_a + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      smem + size_t(STAGES) * STAGE_BYTES + EPI_STAGING_BYTES);
  const uint32_t bar0 = ptx::smem_u32(bars);
  const uint32_t full0 = bar0;
  const uint32_t empty0 = bar0 + 8u * STAGES;
  const uint32_t tfull0 = bar0 + 16u * STAGES;
  const uint32_t tempty0 = tfull0 + 16u;
  const uint32_t done_bar = tempty0 + 16u;
  const uint32_t hbar0 = done_bar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARRIERS);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The fused LayerNorm prologue is compiled only into the GEMMs that take
  // it: the first GEMM of the MLP block and the attention block's QKV
  // projection (K-major bf16 A, B M/N-major).
  constexpr bool LN_PROLOGUE = (EPI == EPI_GELU_FWD || EPI == EPI_BIAS_BF16) &&
                               !A_MN && B_MN && !F8;
  // Work is dealt to groups of four CTAs (two pairs, two clusters) in
  // blockIdx order: a group owns a 512 x 256 "super-tile", its pairs the
  // upper and lower 256 x 256 tiles, which read the same B columns at about
  // the same time (one trip from DRAM to L2 for both).
  const uint32_t prank = ptx::cluster_ctarank();  // rank inside the pair
  const bool leader = prank == 0;
  const int pg = static_cast<int>(blockIdx.x >> 1) & 1;  // pair in its group
  const int group = static_cast<int>(blockIdx.x >> 2);
  const int num_groups = static_cast<int>(gridDim.x >> 2);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full0 + 8u * s, 1);
      ptx::mbar_init(empty0 + 8u * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull0 + 8u * b, 1);
      ptx::mbar_init(tempty0 + 8u * b, 2 * NUM_EPI_WARPS);
    }
    ptx::mbar_init(done_bar, 1);
    for (int w = 0; w < NUM_EPI_WARPS; ++w) ptx::mbar_init(hbar0 + 8u * w, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmO);
    if constexpr (EPI == EPI_GELU_BWD) ptx::prefetch_tmap(&tmO2);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  const Ctl ctl{abort_flag, args.status, args.budget_ns};
  const int num_m = (args.M + PM - 1) / PM;
  const int num_n = (args.N + PN - 1) / PN;
  const int num_msup = (num_m + 1) / 2;   // super-tile rows
  const int num_super = num_msup * num_n;
  const int group_sup = args.group_m > 1 ? args.group_m / 2 : 1;
  // tail split: the first num_full super-tiles whole, then the pieces
  const int num_full = num_super - args.tail;
  const int num_items = num_full + args.tail * args.pieces;
  // The even CTA's full and tempty barriers, as cluster addresses.
  const uint32_t lead_full0 = ptx::mapa_shared(full0, 0u);
  const uint32_t lead_tempty0 = ptx::mapa_shared(tempty0, 0u);

  if (warp < FIRST_EPI_WARP) {
    ptx::setmaxnreg_dec<REGS_CONTROL>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------- producer --
      uint32_t stage = 0, phase = 0;
      bool alive = true;
      for (int item = group; alive && item < num_items; item += num_groups) {
        const Item it = decode_item(item, num_full, args);
        int msup, nb;
        tile_coords(it.sup, num_msup, num_n, group_sup, msup, nb);
        const int mb = 2 * msup + pg;   // may lie past M: zero-filled, unused
        const int m0 = mb * PM + static_cast<int>(prank) * HM;
        const int n0 = nb * PN + static_cast<int>(prank) * HN;
        if constexpr (LN_PROLOGUE) {
          // fused LayerNorm: this CTA's 128 A rows must all be written
          if (args.ln_x != nullptr && m0 < args.M &&
              !wait_count(args.ln_sync + 1 + m0 / HM,
                          static_cast<uint32_t>(min(HM, args.M - m0)), ctl,
                          ROLE_LN_READY)) {
            alive = false;
            break;
          }
        }
        for (int kb = it.kb_lo; kb < it.kb_hi; ++kb) {
          if (!wait_bounded(empty0 + 8u * stage, phase ^ 1u, ctl,
                            ROLE_PRODUCER)) {
            alive = false;
            break;
          }
          const int k0 = kb * (F8 ? 2 * BK : BK);  // 128 bytes of K either way
          // the innermost coordinate of each copy on a 16-byte boundary
          constexpr int XAL = F8 ? 16 : 8;
          if (!TPMLP_CHECK((A_MN ? m0 : k0) % XAL == 0, ctl.status, abort_flag,
                           SITE_GEMM_LOAD_A) ||
              !TPMLP_CHECK((B_MN ? n0 : k0) % XAL == 0, ctl.status, abort_flag,
                           SITE_GEMM_LOAD_B)) {
            alive = false;
            break;
          }
          if (leader) ptx::mbar_arrive_expect_tx(full0 + 8u * stage,
                                                 PAIR_STAGE_BYTES);
          const uint32_t fb = lead_full0 + 8u * stage;
          const uint32_t da = s_a + stage * A_STAGE_BYTES;
          const uint32_t db = s_b + stage * B_STAGE_BYTES;
          if constexpr (!A_MN) {
            ptx::tma_load_2d_pair(da, &tmA, fb, k0, m0);
          } else {
#pragma unroll
            for (int j = 0; j < HM / 64; ++j)
              ptx::tma_load_2d_pair(da + j * (BK * 128), &tmA, fb, m0 + 64 * j,
                                    k0);
          }
          if constexpr (!B_MN) {
            ptx::tma_load_2d_pair(db, &tmB, fb, k0, n0);
          } else {
#pragma unroll
            for (int j = 0; j < HN / 64; ++j)
              ptx::tma_load_2d_pair(db + j * (BK * 128), &tmB, fb, n0 + 64 * j,
                                    k0);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    } else if (warp == 1 && lane == 0 && leader) {
      // -------------------------------------------------- MMA issuer --
      constexpr uint32_t IDESC =
          F8 ? idesc_e4m3_f32(PM, PN) : idesc_bf16_f32(PM, PN, A_MN, B_MN);
      constexpr uint32_t A_KSTEP = A_MN ? 16 * 128 : 32;
      constexpr uint32_t B_KSTEP = B_MN ? 16 * 128 : 32;
      constexpr uint32_t A_LBO = A_MN ? BK * 128 : 16;
      constexpr uint32_t B_LBO = B_MN ? BK * 128 : 16;
      // commits signal the barrier of both CTAs of the pair
      constexpr uint16_t pair_mask = 0x3;
      uint32_t stage = 0, phase = 0, acc = 0;
      bool alive = true;
      for (int item = group; alive && item < num_items; item += num_groups) {
        const Item it = decode_item(item, num_full, args);
        for (int seg = it.seg_lo; alive && seg < it.seg_hi; ++seg, ++acc) {
          const uint32_t b = acc & 1u;
          const uint32_t aph = (acc >> 1) & 1u;
          if (!wait_bounded_cluster(tempty0 + 8u * b, aph ^ 1u, ctl,
                                    ROLE_MMA)) {
            alive = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem_base + b * PN;
          for (int kb = 0; kb < it.kbs; ++kb) {
            if (!wait_bounded(full0 + 8u * stage, phase, ctl, ROLE_MMA)) {
              alive = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t a_addr = s_a + stage * A_STAGE_BYTES;
            const uint32_t b_addr = s_b + stage * B_STAGE_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint64_t adesc =
                  ptx::sdesc_sw128(a_addr + k * A_KSTEP, A_LBO, 1024);
              const uint64_t bdesc =
                  ptx::sdesc_sw128(b_addr + k * B_KSTEP, B_LBO, 1024);
              if constexpr (F8) {
                ptx::mma_f8_pair(d_tmem, adesc, bdesc, IDESC,
                                 (kb > 0 || k > 0) ? 1u : 0u);
              } else {
                ptx::mma_bf16_pair(d_tmem, adesc, bdesc, IDESC,
                                   (kb > 0 || k > 0) ? 1u : 0u);
              }
            }
            ptx::mma_commit_pair(empty0 + 8u * stage, pair_mask);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (alive) ptx::mma_commit_pair(tfull0 + 8u * b, pair_mask);
        }
      }
      if (*reinterpret_cast<volatile int*>(abort_flag)) {
        // Wait for every MMA this thread issued before TMEM is freed.
        ptx::mma_commit_pair(done_bar, static_cast<uint16_t>(1u << prank));
        wait_teardown(done_bar, 0);
      }
    }
    // ------------------------------------------------------ teardown --
    cta_barrier();
    if (*reinterpret_cast<volatile int*>(abort_flag) && warp == 0 &&
        lane == 0) {
      const uint64_t t0 = ptx::globaltimer_ns();
      while (ptx::globaltimer_ns() - t0 < ABORT_SETTLE_NS) {
      }
    }
    cta_barrier();
    ptx::cluster_sync();
    if (warp == 1) {
      __syncwarp();
      ptx::tc_fence_after();
      ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
  } else {
    ptx::setmaxnreg_inc<REGS_EPILOGUE>();
    if constexpr (LN_PROLOGUE) {
      // ------------------------------------ fused LayerNorm prologue --
      // gamma and beta go to the staging buffers (not yet in use: the
      // epilogue starts after the second barrier), read from there by
      // every row
      if (args.ln_x != nullptr &&
          TPMLP_CHECK(args.K % 256 == 0 && args.K / 256 <= LN_VMAX,
                      ctl.status, abort_flag, SITE_GEMM_LN)) {
        float* sg = reinterpret_cast<float*>(smem + size_t(STAGES) * STAGE_BYTES);
        float* sb = sg + args.K;
        const int et = static_cast<int>(threadIdx.x) - FIRST_EPI_WARP * 32;
        for (int i = 4 * et; i < args.K; i += 4 * NUM_EPI_WARPS * 32) {
          *reinterpret_cast<float4*>(sg + i) =
              __ldg(reinterpret_cast<const float4*>(args.ln_gamma + i));
          *reinterpret_cast<float4*>(sb + i) =
              __ldg(reinterpret_cast<const float4*>(args.ln_beta + i));
        }
        epilogue_barrier();
        ln_prologue(args, sg, sb, lane);
        epilogue_barrier();
      }
    }
    // ------------------------------------------------------ epilogue --
    const int ew = warp - FIRST_EPI_WARP;
    const int q = warp & 3;      // TMEM sub-partition this warp may read
    const int half = ew >> 2;    // which 128-column half of the tile
    ChunkStager st{s_epi + static_cast<uint32_t>(ew) * 2u * STAGE_CHUNK_BYTES,
                   0u};
    // E4M3 operands: the product of the two per-tensor scales.
    const float acc_scale = F8 ? *args.scale_a * *args.scale_b : 1.f;
    // EPI_GELU_BWD: this warp's barrier for its H chunks, and its phase
    const uint32_t hbar = hbar0 + 8u * static_cast<uint32_t>(ew);
    uint32_t hphase = 0;
    uint32_t acc = 0;
    bool alive = true;
    for (int item = group; alive && item < num_items; item += num_groups) {
      const Item it = decode_item(item, num_full, args);
      int msup, nb;
      tile_coords(it.sup, num_msup, num_n, group_sup, msup, nb);
      const int mb = 2 * msup + pg;
      const int row0 = mb * PM + static_cast<int>(prank) * HM + q * 32;
      // a tail piece's partials: slot rows of this warp in `part` (tmO2)
      const int prow0 = ((it.sup - num_full) * args.nslots) * 2 * PM +
                        (row0 - msup * 2 * PM);
      const int pcol0 = half * 128;
      // EPI_SHARDSUM: the first later segment (slots 1..) of a tail piece
      const int s1 = args.pieces > 0 ? args.num_seg / args.pieces : 0;
      const int row = row0 + lane;
      const bool live = row0 < args.M;  // warp-uniform: any row in range
      const int col_base = nb * PN + half * 128;
      float S[EPI == EPI_SHARDSUM ? 128 : 1];
      uint32_t cbuf[2] = {0u, 0u};   // EPI_GELU_BWD: the staged dH chunks
      // EPI_GELU_BWD: this warp's two 32 x 64 chunks of H are copied by TMA
      // into the two staging buffers the dH chunks will be written from
      // (once those buffers' earlier stores have read them), in flight
      // while the accumulator is computed; each lane then reads its row
      // there, writes its dH row over it and stores the chunk.  One full-line
      // copy per chunk instead of row-strided loads.
      const int hchunks = (EPI == EPI_GELU_BWD && live)
                              ? (col_base < args.N) + (col_base + 64 < args.N)
                              : 0;
      if constexpr (EPI == EPI_GELU_BWD) {
        if (hchunks > 0) {
          ptx::fence_proxy_async_shared();  // earlier reads of the buffers
          __syncwarp();
          if (lane == 0) {
            ptx::bulk_wait_read<0>();
            ptx::mbar_arrive_expect_tx(hbar, hchunks * STAGE_CHUNK_BYTES);
            for (int j = 0; j < hchunks; ++j)
              ptx::tma_load_2d(st.buffer(j), &tmO2, hbar, col_base + 64 * j,
                               row0);
          }
        }
      }
      for (int seg = it.seg_lo; seg < it.seg_hi; ++seg, ++acc) {
        const uint32_t b = acc & 1u;
        const uint32_t aph = (acc >> 1) & 1u;
        bool ok = wait_bounded(tfull0 + 8u * b, aph, ctl, ROLE_EPILOGUE);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          alive = false;
          break;
        }
        if constexpr (EPI == EPI_GELU_BWD) {
          if (hchunks > 0) {
            bool hok = wait_bounded(hbar, hphase, ctl, ROLE_EPILOGUE);
            hok = __all_sync(0xffffffffu, hok);
            hphase ^= 1u;
            if (!hok) {
              alive = false;
              break;
            }
          }
        }
        ptx::tc_fence_after();
        const uint32_t taddr =
            tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * PN +
            half * 128;
        if constexpr (EPI == EPI_SHARDSUM) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(taddr + j * 32, r);
            ptx::tmem_ld_wait();
            if (it.piece > 0) {
              // a later piece of a tail super-tile: each segment's raw
              // accumulator to its own slot
              st.put(&tmO2, pcol0 + j * 32,
                     prow0 + (1 + seg - s1) * 2 * PM, r, lane);
            } else if (seg == it.seg_lo) {
#pragma unroll
              for (int i = 0; i < 32; ++i) S[j * 32 + i] = __uint_as_float(r[i]);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) S[j * 32 + i] += __uint_as_float(r[i]);
            }
          }
        } else if constexpr (EPI == EPI_STORE_F32) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(taddr + j * 32, r);
            ptx::tmem_ld_wait();
            const int c0 = col_base + j * 32;
            if (it.piece >= 0) {
              // a piece of a tail super-tile: the raw accumulator to its slot
              st.put(&tmO2, pcol0 + j * 32, prow0 + it.piece * 2 * PM, r,
                     lane);
              continue;
            }
            if constexpr (F8) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                r[i] = __float_as_uint(__uint_as_float(r[i]) * acc_scale);
            }
            if (live && c0 < args.N) st.put(&tmO, c0, row0, r, lane);
          }
        } else {
          // GeLU forward / backward, plain bf16: two 64-column bf16 chunks.
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            uint32_t r0[32], r1[32];
            ptx::tmem_ld_32x32b_x32(taddr + j * 64, r0);
            ptx::tmem_ld_32x32b_x32(taddr + j * 64 + 32, r1);
            ptx::tmem_ld_wait();
            const int c0 = col_base + j * 64;
            if (live && c0 < args.N) {
              float v[64];
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                v[i] = __uint_as_float(r0[i]);
                v[32 + i] = __uint_as_float(r1[i]);
              }
              uint32_t w[32];
              if constexpr (F8) {
#pragma unroll
                for (int i = 0; i < 64; ++i) v[i] *= acc_scale;
              }
              if constexpr (EPI == EPI_BIAS_BF16) {
                add_bias_n(args.bias, c0, v, 64);
              } else if constexpr (EPI == EPI_GELU_FWD) {
                add_bias_n(args.bias, c0, v, 64);
                if (args.out2 != nullptr) {
                  pack_bf16x64(v, w);
                  st.put(&tmO2, c0, row0, w, lane);
                }
#pragma unroll
                for (int i = 0; i < 64; i += 2)
                  gelu2_f32(v[i], v[i + 1], args.gelu_mode);
                if (args.amax_out != nullptr) {
                  // largest |Y| of this warp's rows in range, as stored (bf16)
                  float mx = 0.f;
#pragma unroll
                  for (int i = 0; i < 64; ++i) mx = fmaxf(mx, fabsf(v[i]));
                  mx = row < args.M ? __bfloat162float(__float2bfloat16_rn(mx))
                                    : 0.f;
                  const unsigned int wm =
                      __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
                  if (lane == 0) atomicMax(args.amax_out, wm);
                }
              } else {
                // H from the staged chunk (128-byte-swizzled rows)
                const uint32_t hrow =
                    st.buffer(0) + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  uint32_t hw[4];
                  ptx::ld_shared_v4(
                      hrow + static_cast<uint32_t>(i ^ (lane & 7)) * 16u, hw);
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    float h0, h1;
                    unpack_bf16x2(hw[k], h0, h1);
                    float g0, g1;
                    gelu_grad2_f32(h0, h1, g0, g1, args.gelu_mode);
                    v[8 * i + 2 * k + 0] *= g0;
                    v[8 * i + 2 * k + 1] *= g1;
                  }
                }
                if (F8 && args.amax_out != nullptr) {
                  // largest |dH| of this warp's rows in range, as stored
                  float mx = 0.f;
#pragma unroll
                  for (int i = 0; i < 64; ++i) mx = fmaxf(mx, fabsf(v[i]));
                  mx = row < args.M ? __bfloat162float(__float2bfloat16_rn(mx))
                                    : 0.f;
                  const unsigned int wm =
                      __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
                  if (lane == 0) atomicMax(args.amax_out, wm);
                }
              }
              pack_bf16x64(v, w);
              cbuf[j] = st.put(&tmO, c0, row0, w, lane);
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) {
            ptx::mbar_arrive(tempty0 + 8u * b);
          } else {
            ptx::mbar_arrive_cluster(lead_tempty0 + 8u * b);
          }
        }
        if constexpr (EPI == EPI_GELU_BWD) {
          // bias-gradient partials of this warp's 32 rows, from the chunks
          // still staged in shared memory (after the accumulator is released)
          if (args.colsum != nullptr && live) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int c0 = col_base + j * 64;
              if (c0 < args.N &&
                  TPMLP_CHECK(c0 + 64 <= args.ld_colsum && c0 % 8 == 0,
                              ctl.status, abort_flag, SITE_GEMM_COLSUM)) {
                const float2 cs = chunk_colsum_bf16(cbuf[j], lane);
                *reinterpret_cast<float2*>(
                    args.colsum + static_cast<size_t>(row0 / 32) * args.ld_colsum +
                    c0 + 2 * lane) = cs;
              }
            }
          }
        }
      }
      if constexpr (EPI == EPI_SHARDSUM) {
        if (it.piece == 0) {
          // first piece of a tail super-tile: its running sum, raw, to slot 0
          if (alive) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t w[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(S[j * 32 + i]);
              st.put(&tmO2, pcol0 + j * 32, prow0, w, lane);
            }
          }
        } else if (it.piece < 0) {
        if constexpr (F8) {
#pragma unroll
          for (int i = 0; i < 128; ++i) S[i] *= acc_scale;
        }
        if (alive && live) {
          if (args.out_f32) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int c0 = col_base + j * 32;
              if (c0 < args.N) {
                add_bias_n(args.bias, c0, &S[j * 32], 32);
                if (args.dropout)
                  apply_dropout(args.drop_threshold, args.drop_scale,
                                args.drop_seed, args.drop_offset, row, c0,
                                &S[j * 32], 32);
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(S[j * 32 + i]);
                st.put(&tmO, c0, row0, w, lane);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int c0 = col_base + j * 64;
              if (c0 < args.N) {
                add_bias_n(args.bias, c0, &S[j * 64], 64);
                if (args.dropout)
                  apply_dropout(args.drop_threshold, args.drop_scale,
                                args.drop_seed, args.drop_offset, row, c0,
                                &S[j * 64], 64);
                add_residual_bf16(args.aux, args.ldaux, row, args.M, c0,
                                  &S[j * 64], 64);
                uint32_t w[32];
                pack_bf16x64(&S[j * 64], w);
                st.put(&tmO, c0, row0, w, lane);
              }
            }
          }
        }
        }
      }
    }
    st.drain(lane);
    cta_barrier();
    cta_barrier();
    ptx::cluster_sync();
  }
}

// Test knobs, read once: TPMLP_GEMM_MAX_PAIRS caps the pairs a launch uses
// (so that small problems run several rounds); TPMLP_TAIL_SPLIT=0 turns the
// tail split off, =2 makes it whenever it fits (no cost threshold).
int env_max_pairs() {
  static const int v = [] {
    const char* e = std::getenv("TPMLP_GEMM_MAX_PAIRS");
    const int n = e ? std::atoi(e) : 0;
    return n >= 2 ? n : 0;
  }();
  return v;
}
int env_tail_split() {
  static const int v = [] {
    const char* e = std::getenv("TPMLP_TAIL_SPLIT");
    if (e != nullptr && std::strcmp(e, "0") == 0) return 0;
    if (e != nullptr && std::strcmp(e, "2") == 0) return 2;
    return 1;
  }();
  return v;
}

// Tail split plan for `groups` groups of two pairs (see GemmArgs::part):
// the remainder of the super-tiles over the groups, each cut into as many
// pieces as there are groups for it (at most the split units: shard
// segments or k-blocks), reduced until the partials fit `part_bytes`.  Only
// worth it when the k-blocks taken off the last round, kb_total (P-1)/P,
// outweigh the pieces' own overhead and the combine pass (about 10 us);
// measured on the GPT-3-13B-shaped layer, that holds from roughly 96
// k-blocks (a k-block of MMAs is ~0.27 us at full rate), so shorter splits
// are not made.
constexpr int TAIL_MIN_SAVED_KB = 96;
template <int EPI>
TailPlan plan_tail(const GemmArgs& a, int groups) {
  TailPlan p;
  if (!(EPI == EPI_SHARDSUM || EPI == EPI_STORE_F32)) return p;
  if (a.part == nullptr || env_tail_split() == 0 || groups < 2 ||
      a.N % 32 != 0)
    return p;
  if (EPI == EPI_SHARDSUM && a.num_seg < 2) return p;
  const int num_m = (a.M + PM - 1) / PM;
  const int num_n = (a.N + PN - 1) / PN;
  const int num_msup = (num_m + 1) / 2;
  const long long num_super = static_cast<long long>(num_msup) * num_n;
  const int rem = static_cast<int>(num_super % groups);
  if (rem == 0) return p;
  const int units = EPI == EPI_SHARDSUM ? a.num_seg : a.kb_per_seg * a.num_seg;
  const long long kb_total = static_cast<long long>(a.kb_per_seg) * a.num_seg;
  for (int P = std::min(groups / rem, units); P >= 2; --P) {
    if (env_tail_split() != 2 && kb_total * (P - 1) / P < TAIL_MIN_SAVED_KB)
      break;
    const int nslots = EPI == EPI_SHARDSUM ? 1 + a.num_seg - a.num_seg / P : P;
    const long long need =
        static_cast<long long>(rem) * nslots * (2 * PM) * PN * 4;
    if (need > a.part_bytes) continue;
    p.tail = rem;
    p.pieces = P;
    p.nslots = nslots;
    p.num_full = static_cast<int>(num_super) - rem;
    p.num_msup = num_msup;
    p.num_n = num_n;
    p.group_sup = a.group_m > 1 ? a.group_m / 2 : 1;
    break;
  }
  return p;
}

template <bool A_MN, bool B_MN, int EPI, bool F8 = false>
cudaError_t launch_impl(const CUtensorMap& ta, const CUtensorMap& tb,
                        const CUtensorMap& to, const CUtensorMap& to2,
                        const GemmArgs& args, int max_pairs,
                        cudaStream_t stream, TailPlan* plan) {
  auto kern = gemm_tc2_kernel<A_MN, B_MN, EPI, F8>;
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * NUM_THREADS <
      REGS_CONTROL * 128 + REGS_EPILOGUE * NUM_EPI_WARPS * 32)
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (env_max_pairs() > 0 && max_pairs > env_max_pairs())
    max_pairs = env_max_pairs();
  cfg.gridDim = dim3(2);
  int resident = 0;
  e = cudaOccupancyMaxActiveClusters(&resident, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  // Work goes to groups of two pairs (an even number of pairs).  The pair
  // count, and with it the tail-split plan (and so the last bits of the
  // split fp32 weight gradients), is a function of `max_pairs` (half the
  // device's SM count) and the shape alone: the runtime's residency answer
  // is not used, so that two processes on the same GPU model compute the
  // same bits.  If fewer pairs fit at once (an SM limit imposed by the
  // environment), the later clusters start when earlier ones finish: the
  // work each does is fixed by its index, so results do not change.
  const long long sup = static_cast<long long>((args.M + 2 * PM - 1) / (2 * PM)) *
                        ((args.N + PN - 1) / PN);
  long long pairs = 2 * sup < max_pairs ? 2 * sup : max_pairs;
  pairs &= ~1LL;
  if (pairs < 2) pairs = 2;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  GemmArgs a = args;
  a.tail = a.pieces = a.nslots = 0;
  CUtensorMap tp = to2;
  TailPlan tpl;
  if (plan != nullptr) tpl = plan_tail<EPI>(args, static_cast<int>(pairs / 2));
  if (tpl.tail > 0) {
    // the partials: fp32 [tail x nslots x 512 rows, 256 columns]
    if (host::out_map(&tp, args.part, true, tpl.tail * tpl.nslots * 2 * PM, PN,
                      PN) != TPMLP_OK)
      return cudaErrorInvalidValue;
    a.tail = tpl.tail;
    a.pieces = tpl.pieces;
    a.nslots = tpl.nslots;
  }
  if (plan != nullptr) *plan = tpl;
  e = cudaLaunchKernelEx(&cfg, kern, ta, tb, to, tp, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Tail combine: one thread per (tail super-tile, row of 512, 8 columns):
// two 16-byte loads per slot, up to eight slots' loads in flight at once.
// Slots are added in slot order, which for EPI_SHARDSUM is the shard order
// (slot 0: the first piece's running sum; then one slot per later segment),
// then the epilogue's own steps in its order.
constexpr int TC_COLS = 8;
template <int EPI>
__global__ void __launch_bounds__(256)
    tail_combine_kernel(const GemmArgs a, const TailPlan p) {
  const long long gid = blockIdx.x * 256ll + threadIdx.x;
  const int cc = static_cast<int>(gid % (PN / TC_COLS));
  const int lr = static_cast<int>((gid / (PN / TC_COLS)) % (2 * PM));
  const int r = static_cast<int>(gid / (PN / TC_COLS) / (2 * PM));
  if (r >= p.tail) return;
  int msup, nb;
  tile_coords(p.num_full + r, p.num_msup, p.num_n, p.group_sup, msup, nb);
  const int row = msup * 2 * PM + lr;
  const int c0 = nb * PN + cc * TC_COLS;
  if (row >= a.M || c0 >= a.N) return;
  const float4* src = reinterpret_cast<const float4*>(
      a.part + (static_cast<size_t>(r) * p.nslots * 2 * PM + lr) * PN +
      cc * TC_COLS);
  const size_t stride4 = static_cast<size_t>(2 * PM) * PN / 4;
  float v[TC_COLS] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s0 = 0; s0 < p.nslots; s0 += 8) {
    float4 t[8][2];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (s0 + k < p.nslots) {
        t[k][0] = src[(s0 + k) * stride4];
        t[k][1] = src[(s0 + k) * stride4 + 1];
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (s0 + k >= p.nslots) break;
      if (s0 + k == 0) {
        v[0] = t[0][0].x; v[1] = t[0][0].y; v[2] = t[0][0].z; v[3] = t[0][0].w;
        v[4] = t[0][1].x; v[5] = t[0][1].y; v[6] = t[0][1].z; v[7] = t[0][1].w;
      } else {
        v[0] += t[k][0].x; v[1] += t[k][0].y; v[2] += t[k][0].z; v[3] += t[k][0].w;
        v[4] += t[k][1].x; v[5] += t[k][1].y; v[6] += t[k][1].z; v[7] += t[k][1].w;
      }
    }
  }
  if (a.scale_a != nullptr) {  // E4M3 operands
    const float acc_scale = *a.scale_a * *a.scale_b;
#pragma unroll
    for (int i = 0; i < TC_COLS; ++i) v[i] *= acc_scale;
  }
  if constexpr (EPI == EPI_SHARDSUM) {
    add_bias_n(a.bias, c0, v, TC_COLS);
    if (a.dropout)
      apply_dropout(a.drop_threshold, a.drop_scale, a.drop_seed, a.drop_offset,
                    row, c0, v, TC_COLS);
    if (!a.out_f32) add_residual_bf16(a.aux, a.ldaux, row, a.M, c0, v, TC_COLS);
  }
  if (EPI == EPI_STORE_F32 || a.out_f32) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(a.out) +
                                          static_cast<size_t>(row) * a.ldo + c0);
    d[0] = make_float4(v[0], v[1], v[2], v[3]);
    d[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) +
                              static_cast<size_t>(row) * a.ldo + c0) =
        make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                   pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
  }
}

}  // namespace

cudaError_t launch_gemm_tc2(int epi, bool a_mn, bool b_mn,
                            const CUtensorMap& ta, const CUtensorMap& tb,
                            const CUtensorMap& to, const CUtensorMap& to2,
                            const GemmArgs& args, int max_pairs,
                            cudaStream_t stream, TailPlan* plan) {
  if (plan != nullptr) *plan = TailPlan{};
  if (!a_mn && b_mn && epi == EPI_GELU_FWD)
    return launch_impl<false, true, EPI_GELU_FWD>(ta, tb, to, to2, args,
                                                  max_pairs, stream, plan);
  if (!a_mn && b_mn && epi == EPI_SHARDSUM)
    return launch_impl<false, true, EPI_SHARDSUM>(ta, tb, to, to2, args,
                                                  max_pairs, stream, plan);
  if (!a_mn && !b_mn && epi == EPI_GELU_BWD)
    return launch_impl<false, false, EPI_GELU_BWD>(ta, tb, to, to2, args,
                                                   max_pairs, stream, plan);
  if (!a_mn && !b_mn && epi == EPI_SHARDSUM)
    return launch_impl<false, false, EPI_SHARDSUM>(ta, tb, to, to2, args,
                                                   max_pairs, stream, plan);
  if (a_mn && b_mn && epi == EPI_STORE_F32)
    return launch_impl<true, true, EPI_STORE_F32>(ta, tb, to, to2, args,
                                                  max_pairs, stream, plan);
  if (!a_mn && b_mn && epi == EPI_BIAS_BF16)
    return launch_impl<false, true, EPI_BIAS_BF16>(ta, tb, to, to2, args,
                                                   max_pairs, stream, plan);
  if (!a_mn && !b_mn && epi == EPI_BIAS_BF16)
    return launch_impl<false, false, EPI_BIAS_BF16>(ta, tb, to, to2, args,
                                                    max_pairs, stream, plan);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc2_e4m3(int epi, const CUtensorMap& ta,
                                 const CUtensorMap& tb, const CUtensorMap& to,
                                 const CUtensorMap& to2, const GemmArgs& args,
                                 int max_pairs, cudaStream_t stream,
                                 TailPlan* plan) {
  if (plan != nullptr) *plan = TailPlan{};
  if (args.scale_a == nullptr || args.scale_b == nullptr)
    return cudaErrorInvalidValue;
  if (epi == EPI_GELU_FWD)
    return launch_impl<false, false, EPI_GELU_FWD, true>(ta, tb, to, to2, args,
                                                         max_pairs, stream, plan);
  if (epi == EPI_SHARDSUM)
    return launch_impl<false, false, EPI_SHARDSUM, true>(ta, tb, to, to2, args,
                                                         max_pairs, stream, plan);
  if (epi == EPI_GELU_BWD)
    return launch_impl<false, false, EPI_GELU_BWD, true>(ta, tb, to, to2, args,
                                                         max_pairs, stream, plan);
  if (epi == EPI_STORE_F32)
    return launch_impl<false, false, EPI_STORE_F32, true>(ta, tb, to, to2, args,
                                                          max_pairs, stream, plan);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc2_tail(int epi, const GemmArgs& args,
                                 const TailPlan& plan, cudaStream_t stream) {
  if (plan.tail <= 0) return cudaSuccess;
  const long long threads =
      static_cast<long long>(plan.tail) * 2 * PM * (PN / TC_COLS);
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  if (epi == EPI_SHARDSUM)
    tail_combine_kernel<EPI_SHARDSUM><<<blocks, 256, 0, stream>>>(args, plan);
  else if (epi == EPI_STORE_F32)
    tail_combine_kernel<EPI_STORE_F32><<<blocks, 256, 0, stream>>>(args, plan);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace tpmlp
