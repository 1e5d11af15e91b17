// Persistent, warp-specialised tcgen05 GEMM for sm_103a with fused epilogues.
//
// One CTA per SM (grid = min(tiles, SMs)), 12 warps in 3 warpgroups:
//   warp 0      TMA producer (one lane): fills a 4-stage ring of A/B k-blocks
//               in 128-byte-swizzled shared memory, tracked by mbarriers.
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32
//               accumulators); one lane issues tcgen05.mma (M=128, N=256,
//               K=16) and tcgen05.commit.
//   warps 2-3   idle.
//   warps 4-11  epilogue: tcgen05.ld of the accumulator, fused GeLU / GeLU' /
//               shard sum / bias, stores to global memory.  Warp w reads TMEM
//               lanes 32*(w%4) .. +31 (its sub-partition) and one 128-column
//               half of the tile.
// Registers: the CTA is launched with 168 per thread (384 x 168 = 64512); the
// first warpgroup gives registers back (down to REGS_CONTROL) and the two
// epilogue warpgroups take them (up to REGS_EPILOGUE), enough to hold a
// 128-column fp32 shard-sum row per thread.  Each role runs to the end of
// the kernel inside its own register budget; the roles meet only at named
// barriers.
// The two accumulators alternate, so the epilogue of one accumulation runs
// while the MMAs of the next one proceed.
//
// Shard sum (the on-device form of the pages' g forward and f backward
// all-reduces): the K range is cut into `num_seg` segments, one per shard.
// Each segment starts a fresh accumulator (the MMA's accumulate flag is off
// on its first k-step); the epilogue adds the segment partials into fp32
// registers in segment order 0..t-1, adds the bias and rounds once.  Every
// output element has one writer and a fixed summation order, so results are
// bitwise reproducible.
//
// Every mbarrier wait is bounded by a time budget; on expiry the CTA records
// TPMLP_ERR_TIMEOUT in the status word, the other roles see a shared abort
// flag and stop, outstanding TMA copies and MMAs are waited for (bounded),
// TMEM is freed and the kernel returns.
#include "gemm_common.cuh"

namespace tpmlp {
namespace {

using namespace gemm;

constexpr int BM = TC_BM;
constexpr int BN = TC_BN;
constexpr int BK = TC_BK;
constexpr int STAGES = 4;
constexpr int NUM_THREADS = 384;
constexpr int NUM_EPI_WARPS = 8;
constexpr int FIRST_EPI_WARP = 4;
constexpr int REGS_LAUNCH = 168;
constexpr int REGS_CONTROL = 40;
constexpr int REGS_EPILOGUE = 232;
static_assert(REGS_CONTROL * 128 + REGS_EPILOGUE * 256 <=
                  REGS_LAUNCH * NUM_THREADS,
              "register split exceeds the launch allocation");
constexpr uint32_t A_STAGE_BYTES = BM * BK * 2;  // 16 KiB
constexpr uint32_t B_STAGE_BYTES = BN * BK * 2;  // 32 KiB
constexpr uint32_t STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int NUM_BARRIERS = 2 * STAGES + 5;
constexpr size_t SMEM_BYTES =
    1024 + size_t(STAGES) * STAGE_BYTES + NUM_BARRIERS * 8 + 16;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// CTA-wide named barrier (id 1) for the teardown; every thread of the CTA
// arrives, from whichever role branch it is in.
__device__ __forceinline__ void cta_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(NUM_THREADS) : "memory");
}

template <bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_a = ptx::smem_u32(smem);
  const uint32_t s_b = s_a + STAGES * A_STAGE_BYTES;
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + size_t(STAGES) * STAGE_BYTES);
  const uint32_t bar0 = ptx::smem_u32(bars);
  // full[s] = bar0 + 8 s, empty[s] = full + 8 STAGES, tfull[b], tempty[b],
  // done (teardown) follow.
  const uint32_t full0 = bar0;
  const uint32_t empty0 = bar0 + 8u * STAGES;
  const uint32_t tfull0 = bar0 + 16u * STAGES;
  const uint32_t tempty0 = tfull0 + 16u;
  const uint32_t done_bar = tempty0 + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARRIERS);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full0 + 8u * s, 1);
      ptx::mbar_init(empty0 + 8u * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull0 + 8u * b, 1);
      ptx::mbar_init(tempty0 + 8u * b, NUM_EPI_WARPS);
    }
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  const Ctl ctl{abort_flag, args.status, args.budget_ns};
  const int num_m = (args.M + BM - 1) / BM;
  const int num_n = (args.N + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int kb_total = args.kb_per_seg * args.num_seg;

  if (warp < FIRST_EPI_WARP) {
    ptx::setmaxnreg_dec<REGS_CONTROL>();
    uint32_t issued = 0;  // producer: k-blocks issued (for teardown)
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------- producer --
      uint32_t stage = 0, phase = 0;
      bool alive = true;
      for (int tile = blockIdx.x; alive && tile < num_tiles;
           tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, num_m, num_n, args.group_m, mb, nb);
        const int m0 = mb * BM, n0 = nb * BN;
        for (int kb = 0; kb < kb_total; ++kb) {
          if (!wait_bounded(empty0 + 8u * stage, phase ^ 1u, ctl,
                            ROLE_PRODUCER)) {
            alive = false;
            break;
          }
          const uint32_t fb = full0 + 8u * stage;
          ptx::mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const int k0 = kb * BK;
          const uint32_t da = s_a + stage * A_STAGE_BYTES;
          const uint32_t db = s_b + stage * B_STAGE_BYTES;
          if constexpr (!A_MN) {
            ptx::tma_load_2d(da, &tmA, fb, k0, m0);
          } else {
#pragma unroll
            for (int j = 0; j < BM / 64; ++j)
              ptx::tma_load_2d(da + j * (BK * 128), &tmA, fb, m0 + 64 * j, k0);
          }
          if constexpr (!B_MN) {
            ptx::tma_load_2d(db, &tmB, fb, k0, n0);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              ptx::tma_load_2d(db + j * (BK * 128), &tmB, fb, n0 + 64 * j, k0);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    } else if (warp == 1 && lane == 0) {
      // -------------------------------------------------- MMA issuer --
      constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, A_MN, B_MN);
      // Per 16-deep k-step advance inside a stage: K-major operands move 32 B
      // along the swizzled row; M/N-major operands move 16 rows of 128 B.
      constexpr uint32_t A_KSTEP = A_MN ? 16 * 128 : 32;
      constexpr uint32_t B_KSTEP = B_MN ? 16 * 128 : 32;
      constexpr uint32_t A_LBO = A_MN ? BK * 128 : 16;
      constexpr uint32_t B_LBO = B_MN ? BK * 128 : 16;
      uint32_t stage = 0, phase = 0, acc = 0;
      bool alive = true;
      for (int tile = blockIdx.x; alive && tile < num_tiles;
           tile += gridDim.x) {
        for (int seg = 0; alive && seg < args.num_seg; ++seg, ++acc) {
          const uint32_t b = acc & 1u;
          const uint32_t aph = (acc >> 1) & 1u;
          if (!wait_bounded(tempty0 + 8u * b, aph ^ 1u, ctl, ROLE_MMA)) {
            alive = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem_base + b * BN;
          for (int kb = 0; kb < args.kb_per_seg; ++kb) {
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
              ptx::mma_bf16(d_tmem, adesc, bdesc, IDESC,
                            (kb > 0 || k > 0) ? 1u : 0u);
            }
            ptx::mma_commit(empty0 + 8u * stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (alive) ptx::mma_commit(tfull0 + 8u * b);
        }
      }
    }
    // ------------------------------------------------------ teardown --
    cta_barrier();
    if (*reinterpret_cast<volatile int*>(abort_flag)) {
      if (warp == 0 && lane == 0) {
        // Wait for every TMA copy still in flight into this CTA's ring.
        for (uint32_t s = 0; s < STAGES; ++s) {
          if (issued > s) {
            const uint32_t uses = (issued - 1 - s) / STAGES + 1;
            wait_teardown(full0 + 8u * s, (uses - 1) & 1u);
          }
        }
      }
      if (warp == 1 && lane == 0) {
        // Wait for every MMA this thread issued before freeing TMEM.
        ptx::mma_commit(done_bar);
        wait_teardown(done_bar, 0);
      }
    }
    cta_barrier();
    if (warp == 1) {
      __syncwarp();
      ptx::tc_fence_after();
      ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
  } else {
    ptx::setmaxnreg_inc<REGS_EPILOGUE>();
    // ------------------------------------------------------ epilogue --
    const int ew = warp - FIRST_EPI_WARP;
    const int q = warp & 3;      // TMEM sub-partition this warp may read
    const int half = ew >> 2;    // which 128-column half of the tile
    uint32_t acc = 0;
    bool alive = true;
    for (int tile = blockIdx.x; alive && tile < num_tiles;
         tile += gridDim.x) {
      int mb, nb;
      tile_coords(tile, num_m, num_n, args.group_m, mb, nb);
      const int row = mb * BM + q * 32 + lane;
      const int col_base = nb * BN + half * 128;
      const bool row_ok = row < args.M;
      float S[EPI == EPI_SHARDSUM ? 128 : 1];
      for (int seg = 0; seg < args.num_seg; ++seg, ++acc) {
        const uint32_t b = acc & 1u;
        const uint32_t aph = (acc >> 1) & 1u;
        bool ok = wait_bounded(tfull0 + 8u * b, aph, ctl, ROLE_EPILOGUE);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          alive = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t taddr =
            tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * BN +
            half * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(taddr + j * 32, r);
          ptx::tmem_ld_wait();
          if constexpr (EPI == EPI_SHARDSUM) {
            if (seg == 0) {
#pragma unroll
              for (int i = 0; i < 32; ++i) S[j * 32 + i] = __uint_as_float(r[i]);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) S[j * 32 + i] += __uint_as_float(r[i]);
            }
          } else {
            const int c0 = col_base + j * 32;
            if (row_ok && c0 < args.N) {
              float v[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
              epilogue_chunk<EPI>(args, row, c0, v);
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(tempty0 + 8u * b);
      }
      if constexpr (EPI == EPI_SHARDSUM) {
        if (alive && row_ok) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c0 = col_base + j * 32;
            if (c0 < args.N) {
              float v[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = S[j * 32 + i];
              add_bias32(args.bias, c0, v);
              if (args.dropout)
                apply_dropout(args.drop_threshold, args.drop_scale,
                              args.drop_seed, args.drop_offset, row, c0, v, 32);
              if (!args.out_f32)
                add_residual_bf16(args.aux, args.ldaux, row, args.M, c0, v, 32);
              const size_t off = static_cast<size_t>(row) * args.ldo + c0;
              if (args.out_f32) {
                store_f32x32(static_cast<float*>(args.out) + off, v);
              } else {
                store_bf16x32(static_cast<__nv_bfloat16*>(args.out) + off, v);
              }
            }
          }
        }
      }
    }
    cta_barrier();
    cta_barrier();
  }
}

template <bool A_MN, bool B_MN, int EPI>
cudaError_t launch_impl(const CUtensorMap& ta, const CUtensorMap& tb,
                        const GemmArgs& args, int grid, cudaStream_t stream) {
  auto kern = gemm_tc_kernel<A_MN, B_MN, EPI>;
  // The setmaxnreg split only adds up if the kernel was compiled with the
  // full launch allocation; refuse to launch otherwise (an increase that
  // cannot be satisfied would wait forever).
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * NUM_THREADS <
      REGS_CONTROL * 128 + REGS_EPILOGUE * NUM_EPI_WARPS * 32)
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  kern<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(ta, tb, args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_tc(int epi, bool a_mn, bool b_mn, const CUtensorMap& ta,
                           const CUtensorMap& tb, const GemmArgs& args,
                           int grid, cudaStream_t stream) {
  if (!a_mn && b_mn && epi == EPI_GELU_FWD)
    return launch_impl<false, true, EPI_GELU_FWD>(ta, tb, args, grid, stream);
  if (!a_mn && b_mn && epi == EPI_SHARDSUM)
    return launch_impl<false, true, EPI_SHARDSUM>(ta, tb, args, grid, stream);
  if (!a_mn && !b_mn && epi == EPI_GELU_BWD)
    return launch_impl<false, false, EPI_GELU_BWD>(ta, tb, args, grid, stream);
  if (!a_mn && !b_mn && epi == EPI_SHARDSUM)
    return launch_impl<false, false, EPI_SHARDSUM>(ta, tb, args, grid, stream);
  if (a_mn && b_mn && epi == EPI_STORE_F32)
    return launch_impl<true, true, EPI_STORE_F32>(ta, tb, args, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace tpmlp
