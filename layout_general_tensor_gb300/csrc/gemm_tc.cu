// Any-layout fp16 / bf16 GEMM on the sm_103a tensor cores.
//
// One persistent CTA per SM walks (tile, split) work units.  Warp roles:
//   warp 0      TMA producer: one elected lane loads the P and Q tiles of each
//               64-deep K block into a ring of shared-memory stages.
//   warp 1      MMA issuer: allocates TMEM, one lane issues tcgen05.mma into a
//               double-buffered fp32 accumulator and commits each stage back.
//   warps 2..5  epilogue: tcgen05.ld the accumulator, then either convert and
//               store C, or add the fp32 partial into the workspace and let the
//               last-arriving CTA of the tile convert and store.
//   warps 6..9  stream-K fixup: convert this CTA's share of the tail tiles
//               once their partial sums are complete (idle without a tail);
//               or, for an operand TMA cannot address (rows not 16-byte
//               multiples apart, or an unaligned base), its realigning
//               loader (realign.cuh), which fills that operand's part of each
//               stage and arrives on the stage beside the TMA bytes of the
//               other.
//
// Operand layouts.  The Triton inThreadTranspose page ("Feature description")
// fixes the problem: a dot operand that is not contiguous along K must still
// reach the matrix unit as K-ordered fragments with conflict-free shared
// memory reads; it transposes in registers.  Here the TMA box is laid along
// the contiguous dimension and written with the 128-byte swizzle, and the
// tcgen05 shared-memory descriptor is marked K-major or MN-major to match
// (the SharedEncodingAttr order swap of the same page, "PR description",
// item 1), so no operand is transposed by threads at all.
//
// Split-K: unit u covers tile u / split and K blocks
// [(u % split) * kb_per_split, ...) -- the per-split K offset of the BitBLAS
// TileLang page's T.Parallel / T.copy example.  With split > 1 each CTA takes
// a contiguous run of units, so consecutive splits of one tile accumulate in
// TMEM and only the run's total leaves the SM; the partial runs of a tile are
// reduced in fp32 through L2 (red.global.add) and an arrival counter -- the
// partials -> shared storage -> second reduction pattern of the IREE page
// ("Add support for inter-subgroup multi_reduction"), lifted from subgroups
// to CTAs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "realign.cuh"
#include "tc_common.cuh"

namespace lgt {
namespace {

constexpr int kThreads = 320;  // 6 warps + 4 stream-K fixup warps
constexpr int kFixWarp0 = 6;
constexpr uint32_t kRlWarps = 4;  // the fixup warps, as realigning loader
constexpr int kEpiWarp0 = 2;
constexpr uint32_t kP_BYTES = TILE_P * TILE_K * 2;   // 16 KiB
constexpr uint32_t kMnChunkBytes = 64 * TILE_K * 2;  // one 64-wide MN box, 64 K rows: 8 KiB

template <int BN>
struct Cfg {
  static constexpr uint32_t Q_BYTES = BN * TILE_K * 2;
  static constexpr uint32_t STAGE_BYTES = kP_BYTES + Q_BYTES;
  static constexpr int STAGES_RAW = (194 * 1024) / STAGE_BYTES;  // leaves room for the epilogue staging
  static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
  // two accumulator buffers of BN fp32 columns, rounded up to a power of two
  static constexpr uint32_t TMEM_COLS = (2 * BN) <= 32 ? 32 : (2 * BN) <= 64 ? 64 : (2 * BN) <= 128 ? 128
                                        : (2 * BN) <= 256 ? 256 : 512;
  static constexpr int CH = BN < 32 ? BN : 32;          // accumulator columns per tcgen05.ld
  static constexpr uint32_t EPI_OFF = STAGES * STAGE_BYTES;  // 1024-aligned (stages are 2 KiB multiples)
  // barriers: full[S], empty[S], acc_full[2], acc_empty[2], teardown, cluster slices received,
  // realigning loader staging slots landed[kRlMaxStg]
  static constexpr uint32_t BAR_OFF = EPI_OFF + EPI_STAGING_BYTES;
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 6 + kRlMaxStg;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr uint32_t SMEM_USED = MISC_OFF + 64;
  static constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;  // slack for 1024-byte alignment
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N must be a multiple of 16 in [16, 256]");
  static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0 && TMEM_COLS <= 512, "TMEM allocation");
  static_assert(EPI_OFF % 1024 == 0 && SMEM_ALLOC <= 227 * 1024, "shared memory layout");
  // cluster split-K (BN <= 64): the outgoing slices (up to BN x 128 fp32) and
  // a 16-bit transpose of one slice fit in the idle pipeline stages
  static_assert(BN > 64 || EPI_OFF >= TILE_P * 4 * BN + TILE_P * 2 * BN, "cluster split-K staging");
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ TcArgs a) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);

  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = base + C::BAR_OFF;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 + b); };
  const uint32_t teardown_bar = bar0 + 8u * (2 * C::STAGES + 4);
  const uint32_t cl_bar0 = bar0 + 8u * (2 * C::STAGES + 5);  // cluster split-K: slices received
  auto stg_full = [&](int i) { return bar0 + 8u * (2 * C::STAGES + 6 + i); };
  // Realigning loader (realign.cuh): its staging ring takes the last rl_take
  // pipeline stages' memory; nst stages remain.
  const bool rl = a.rl_on[0] || a.rl_on[1];
  const uint32_t rl_bytes_p = a.rl_on[0] ? rl_stage_bytes(a.p_mn, TILE_P, a.rl_cls[0]) : 0u;
  const uint32_t rl_bytes_q = a.rl_on[1] ? rl_stage_bytes(a.q_mn, BN, a.rl_cls[1]) : 0u;
  const uint32_t rl_slot = rl_bytes_p + rl_bytes_q;
  int rl_take = 0, rl_nstg = 0;
  rl_ring(C::STAGES, C::STAGE_BYTES, rl_slot, rl_take, rl_nstg);
  const int nst = C::STAGES - rl_take;
  const uint32_t stg0 = base + static_cast<uint32_t>(nst) * C::STAGE_BYTES;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  volatile int* consumed_slot = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 12);

  if (threadIdx.x == 0) {
    // (a realigned operand: the loader arrives on the stage too)
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), rl ? 2u : 1u);
      mbar_init(empty_bar(s), 1);
    }
    for (int i = 0; i < kRlMaxStg; ++i) mbar_init(stg_full(i), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), kEpiThreads / 32);
    }
    mbar_init(teardown_bar, 1);
    mbar_init(cl_bar0, 1);
    *abort_flag = 0;
    *consumed_slot = 0;
    fence_barrier_init();
    // cluster split-K: the (cl - 1) slices the peers send land on this
    // barrier (they start sending only after the cluster barrier below)
    if (a.cl_size > 1)
      mbar_arrive_expect_tx(cl_bar0, static_cast<uint32_t>(a.cl_size - 1) * TILE_P * 4u *
                                         static_cast<uint32_t>(BN / a.cl_size));
    fence_proxy_async_smem();
    tma_prefetch_desc(&a.tm_p);
    tma_prefetch_desc(&a.tm_q);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the peers' barriers are initialised before anyone arrives on them remotely
  if (a.cl_size > 1) cluster_sync_all();
  const uint32_t tmem_base = *tmem_slot;

  // A stage's boxes: P (128 rows; two 64-wide boxes when MN-major) and Q.
  auto load_p = [&](uint32_t sp, uint32_t bar, int32_t k0, int32_t prow) {
    if (!a.p_mn) {
      tma_load_2d(sp, &a.tm_p, bar, k0, prow);
    } else {
      tma_load_2d(sp, &a.tm_p, bar, prow, k0);
      tma_load_2d(sp + kMnChunkBytes, &a.tm_p, bar, prow + 64, k0);
    }
  };
  auto load_q = [&](uint32_t sq, uint32_t bar, int32_t k0, int32_t qrow) {
    if (!a.q_mn) {
      tma_load_2d(sq, &a.tm_q, bar, k0, qrow);
    } else {
#pragma unroll
      for (int j = 0; j < BN / 64; ++j) tma_load_2d(sq + j * kMnChunkBytes, &a.tm_q, bar, qrow + 64 * j, k0);
    }
  };
  // operands, C and the split-K workspace may be written by the previous kernel
  pdl_wait();

  int issued = 0;  // producer lane: K blocks whose loads were issued

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Sched sched(a);
      Group g;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      while (ok && sched.next(a, g)) {
        int32_t tp, tq, m0, m1, n0, n1;
        tile_ranges(a, g.tile, BN, tp, tq, m0, m1, n0, n1);
        const int32_t prow = tp * TILE_P, qrow = tq * BN;
        for (int kb = 0; kb < g.nkb; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, a.wait_limit_ns, abort_flag)) {
            if (!*abort_flag) record_timeout(a, abort_flag, 0 * 16 + 1);
            ok = false;
            break;
          }
          const uint32_t sp = base + stage * C::STAGE_BYTES;
          const uint32_t sq = sp + kP_BYTES;
          const int32_t k0 = (g.kb0 + kb) * TILE_K;
          if (a.withhold && blockIdx.x == 0 && issued == 0) {
            // test aid (a.withhold): this stage is never filled, so the MMA
            // issuer's bounded wait on it runs out
            ++issued;
            if (++stage == nst) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          // (realigned operands come from the loader warps)
          mbar_arrive_expect_tx(full_bar(stage), (a.rl_on[0] ? 0u : kP_BYTES) + (a.rl_on[1] ? 0u : C::Q_BYTES));
          if (!a.rl_on[0]) load_p(sp, full_bar(stage), k0, prow);
          if (!a.rl_on[1]) load_q(sq, full_bar(stage), k0, qrow);
          ++issued;
          if (++stage == nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      Sched sched(a);
      Group g;
      int stage = 0;
      uint32_t phase = 0;
      int acc_iter = 0;
      int consumed = 0;
      bool ok = true;
      // Per-MMA (K = 16) start-address advance inside a stage, and the
      // descriptor offsets: K-major rows are 128 bytes along K (advance 32 B
      // per 16 elements, LBO unused); MN-major tiles hold 128-byte rows along
      // M/N, one per k (advance 16 rows = 2 KiB), 64-wide chunks 8 KiB apart.
      const uint32_t p_step = a.p_mn ? 2048u : 32u;
      const uint32_t q_step = a.q_mn ? 2048u : 32u;
      const uint32_t p_lbo = a.p_mn ? kMnChunkBytes : 16u;
      const uint32_t q_lbo = a.q_mn ? kMnChunkBytes : 16u;
      while (ok && sched.next(a, g)) {
        if (g.nkb == 0) continue;
        const int buf = acc_iter & 1;
        const uint32_t acc_phase = (acc_iter >> 1) & 1;
        if (!mbar_wait_bounded(acce_bar(buf), acc_phase ^ 1u, a.wait_limit_ns, abort_flag)) {
          if (!*abort_flag) record_timeout(a, abort_flag, 1 * 16 + 3);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < g.nkb; ++kb) {
          if (!mbar_wait_bounded(full_bar(stage), phase, a.wait_limit_ns, abort_flag)) {
            if (!*abort_flag) record_timeout(a, abort_flag, 1 * 16 + 0);
            ok = false;
            break;
          }
          ++consumed;
          tc_fence_after();
          const uint32_t sp = base + stage * C::STAGE_BYTES;
          const uint32_t sq = sp + kP_BYTES;
#pragma unroll
          for (int k = 0; k < TILE_K / 16; ++k) {
            const uint64_t pd = sw128_desc(sp + k * p_step, p_lbo, 1024u);
            const uint64_t qd = sw128_desc(sq + k * q_step, q_lbo, 1024u);
            tc_mma_f16_ss(d_tmem, pd, qd, a.idesc, (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(empty_bar(stage));
          if (++stage == nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(accf_bar(buf));
        ++acc_iter;
      }
      *consumed_slot = consumed;
    }
  } else if (warp >= kFixWarp0) {
    if (rl) {
      // ---------------------------------------------------------- realigning loader
      // The staging ring is the loader's own: the first loader warp copies
      // the class boxes of K block it + rl_nstg into the slot that K block
      // `it` has just been realigned out of (its lanes share the boxes), and
      // all four warps realign each K block into its pipeline stage once the
      // stage is free (the planner gives such plans no fixup work).
      const int t = threadIdx.x - kFixWarp0 * 32;
      const bool issuer = warp == kFixWarp0;
      const uint32_t tx = (a.rl_on[0] ? rl_stage_tx(a.p_mn, TILE_P, a.rl_cls[0]) : 0u) +
                          (a.rl_on[1] ? rl_stage_tx(a.q_mn, BN, a.rl_cls[1]) : 0u);
      KbIter ahead(a);
      int stg_issued = 0, stg_done = 0;
      auto fill = [&](int sl) {  // the next K block's boxes into slot sl (first loader warp)
        int tile, kb;
        if (!ahead.next(a, tile, kb)) return;
        int32_t tp, tq, m0, m1, n0, n1;
        tile_ranges(a, tile, BN, tp, tq, m0, m1, n0, n1);
        const uint32_t dst = stg0 + static_cast<uint32_t>(sl) * rl_slot;
        if (lane == 0) mbar_arrive_expect_tx(stg_full(sl), tx);
        __syncwarp();
        if (a.rl_on[0]) rl_issue(a.tm_rl[0], a.rl_cls[0], a.p_mn, TILE_P, tp * TILE_P, kb * TILE_K, dst, stg_full(sl), lane, 32);
        if (a.rl_on[1])
          rl_issue(a.tm_rl[1], a.rl_cls[1], a.q_mn, BN, tq * BN, kb * TILE_K, dst + rl_bytes_p, stg_full(sl), lane, 32);
        ++stg_issued;
      };
      if (issuer)
        for (int sl = 0; sl < rl_nstg; ++sl) fill(sl);
      Sched sched(a);
      Group g;
      int stage = 0, slot = 0;
      uint32_t phase = 0, sphase = 0;
      bool ok = true;
      while (ok && sched.next(a, g)) {
        for (int kb = 0; kb < g.nkb; ++kb) {
          const bool got = mbar_wait_bounded(stg_full(slot), sphase, a.wait_limit_ns, abort_flag) &&
                           mbar_wait_bounded(empty_bar(stage), phase ^ 1u, a.wait_limit_ns, abort_flag);
          if (!got && !*abort_flag) record_timeout(a, abort_flag, 0 * 16 + 6);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          const uint32_t src = stg0 + static_cast<uint32_t>(slot) * rl_slot;
          const uint32_t sp = base + static_cast<uint32_t>(stage) * C::STAGE_BYTES;
          if (a.rl_on[0]) rl_pass(a.rl_d[0], a.rl_cls[0], a.p_mn, TILE_P, src, sp, t, kRlWarps * 32);
          if (a.rl_on[1]) rl_pass(a.rl_d[1], a.rl_cls[1], a.q_mn, BN, src + rl_bytes_p, sp + kP_BYTES, t, kRlWarps * 32);
          // the stage is read by the MMA (async proxy); the slot is refilled by TMA
          fence_proxy_async_smem();
          named_bar_sync(3, kRlWarps * 32);
          ++stg_done;
          if (t == 0) mbar_arrive(full_bar(stage));
          if (issuer) fill(slot);
          if (++stage == nst) {
            stage = 0;
            phase ^= 1u;
          }
          if (++slot == rl_nstg) {
            slot = 0;
            sphase ^= 1u;
          }
        }
      }
      if (issuer && lane == 0 && *abort_flag) {
        // copies still in flight land before the CTA exits
        volatile int no_abort = 0;
        for (int it = stg_done; it < stg_issued; ++it)
          mbar_wait_bounded(stg_full(it % rl_nstg), (it / rl_nstg) & 1, a.wait_limit_ns, &no_abort);
      }
    } else if (a.tail_tiles) {
      // ---------------------------------------------------------- stream-K fixup
      finish_tail<BN>(a, abort_flag, threadIdx.x - kFixWarp0 * 32);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;                  // TMEM lane quadrant this warp may access
    const int et = threadIdx.x - kEpiWarp0 * 32;
    Sched sched(a);
    Group g;
    int acc_iter = 0;
    int ring = 0;
    const uint32_t stage_smem = base + C::EPI_OFF + static_cast<uint32_t>(warp - kEpiWarp0) * 8192u;
    while (sched.next(a, g)) {
      if (!epilogue_group<BN, C::CH>(a, g, tmem_base, accf_bar(0), acce_bar(0), acc_iter, abort_flag, q4, lane, et,
                                     0, stage_smem, ring, NoFix(), 1u, cl_bar0, base + C::EPI_OFF, base))
        break;
    }
    if (lane == 0) bulk_wait_group<0>();  // staged stores finished before the CTA exits
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0) {
      // Let every TMA load still in flight land before the CTA exits.
      volatile int no_abort = 0;
      const int consumed = *consumed_slot;
      for (int it = consumed; it < issued; ++it) {
        if (a.withhold && blockIdx.x == 0 && it == 0) continue;  // the withheld stage has no copy in flight
        mbar_wait_bounded(full_bar(it % nst), (it / nst) & 1, a.wait_limit_ns, &no_abort);
      }

    }
  }
  if (warp == 1 && lane == 0) {
    // Wait until every MMA this CTA issued has completed.
    volatile int no_abort = 0;
    tc_commit(teardown_bar);
    mbar_wait_bounded(teardown_bar, 0, a.wait_limit_ns, &no_abort);
  }
  tc_fence_before();
  __syncthreads();
  // Split-K in a cluster: no CTA leaves while a peer may still push its slice
  // into this CTA's shared memory (a peer that gave up a wait still reaches
  // this barrier: every wait before it is bounded).
  if (a.cl_size > 1) cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

template <int BN>
cudaError_t launch_bn(const TcArgs& args, int grid, cudaStream_t stream) {
  using C = Cfg<BN>;
  cudaError_t e = set_smem_once<tc_gemm_kernel<BN>>(static_cast<int>(C::SMEM_ALLOC));
  if (e != cudaSuccess) return e;
  // CTAs that convert split tiles wait for other CTAs' partial sums; they
  // start waiting only after pdl_wait (the previous kernel has left every
  // SM), and the grid never exceeds the CTAs the device holds at once.
  if (args.cl_size > 1)
    return launch_pdl_cluster(tc_gemm_kernel<BN>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), C::SMEM_ALLOC,
                              stream, static_cast<unsigned>(args.cl_size), args);
  return launch_pdl(tc_gemm_kernel<BN>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), C::SMEM_ALLOC, stream, args);
}

template <int BN>
cudaError_t max_clusters_bn(int cluster, int* clusters) {
  using C = Cfg<BN>;
  cudaError_t e = set_smem_once<tc_gemm_kernel<BN>>(static_cast<int>(C::SMEM_ALLOC));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM_ALLOC;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, tc_gemm_kernel<BN>, &cfg);
}

}  // namespace

size_t tc_gemm_smem_bytes(int bn) {
  switch (bn) {
    case 16: return Cfg<16>::SMEM_ALLOC;
    case 32: return Cfg<32>::SMEM_ALLOC;
    case 64: return Cfg<64>::SMEM_ALLOC;
    case 128: return Cfg<128>::SMEM_ALLOC;
    case 192: return Cfg<192>::SMEM_ALLOC;
    case 256: return Cfg<256>::SMEM_ALLOC;
    default: return 0;
  }
}

bool tc_gemm_rl_fits(int bn, int p_mn, int q_mn, int p_cls, int q_cls) {
  auto fits = [&](int stages, uint32_t stage_bytes) {
    const uint32_t stg = (p_cls ? rl_stage_bytes(p_mn, TILE_P, p_cls) : 0u) + (q_cls ? rl_stage_bytes(q_mn, bn, q_cls) : 0u);
    int take, nstg;
    return rl_ring(stages, stage_bytes, stg, take, nstg) && (stg == 0 || nstg >= 2);
  };
  switch (bn) {
    case 16: return fits(Cfg<16>::STAGES, Cfg<16>::STAGE_BYTES);
    case 32: return fits(Cfg<32>::STAGES, Cfg<32>::STAGE_BYTES);
    case 64: return fits(Cfg<64>::STAGES, Cfg<64>::STAGE_BYTES);
    case 128: return fits(Cfg<128>::STAGES, Cfg<128>::STAGE_BYTES);
    case 192: return fits(Cfg<192>::STAGES, Cfg<192>::STAGE_BYTES);
    case 256: return fits(Cfg<256>::STAGES, Cfg<256>::STAGE_BYTES);
    default: return false;
  }
}

cudaError_t tc_gemm_max_clusters(int bn, int cluster, int* clusters) {
  *clusters = 0;
  switch (bn) {
    case 16: return max_clusters_bn<16>(cluster, clusters);
    case 32: return max_clusters_bn<32>(cluster, clusters);
    case 64: return max_clusters_bn<64>(cluster, clusters);
    default: return cudaSuccess;
  }
}

cudaError_t launch_tc_gemm(const TcArgs& args, int bn, int grid, cudaStream_t stream) {
  switch (bn) {
    case 16: return launch_bn<16>(args, grid, stream);
    case 32: return launch_bn<32>(args, grid, stream);
    case 64: return launch_bn<64>(args, grid, stream);
    case 128: return launch_bn<128>(args, grid, stream);
    case 192: return launch_bn<192>(args, grid, stream);
    case 256: return launch_bn<256>(args, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lgt
