// CTA-pair variant of the any-layout fp16 / bf16 GEMM (tcgen05 cta_group::2).
//
// Two CTAs of a cluster share a 256 x BN output tile (BN in 128..256).  Each
// CTA loads 128 rows of the P operand and BN/2 rows of the Q operand per
// 64-deep K block; one thread of the even CTA issues a 256 x BN x 16 MMA
// that reads both CTAs' shared memory and writes 128 accumulator rows into
// each CTA's TMEM.  Against the single-CTA 128 x 256 tile this moves a third
// fewer bytes from L2 into shared memory per FLOP and frees room for more
// pipeline stages.  The planner picks BN so that the tiles fill whole waves
// of CTA pairs.
//
// Roles (320 threads per CTA, in both CTAs):
//   warp 0      TMA producer of this CTA's halves; the copies of both CTAs
//               complete on the even CTA's stage barrier, which the even
//               CTA's producer arms with the bytes of both.
//   warp 1      TMEM allocation (both CTAs, jointly); in the even CTA one lane
//               issues the MMAs and multicasts each commit to both CTAs'
//               stage-free / accumulator-full barriers.
//   warps 2..5  epilogue of the CTA's own 128 accumulator rows (shared code
//               with the single-CTA kernel); each warp signals "buffer
//               drained" on the even CTA's barrier.
//   warps 6..9  stream-K fixup of this CTA's share of the tail tiles; or
//               the realigning loader (realign.cuh) of an operand TMA cannot
//               address: this CTA's halves of it, each stage announced on
//               the even CTA's stage barrier.
//
// Operand layouts are handled exactly as in the single-CTA kernel (TMA box
// along the contiguous dimension, 128-byte swizzle, K- or MN-major shared
// memory descriptors), following the inThreadTranspose page's "Feature
// description": no operand is transposed by threads.
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
constexpr uint32_t kRlWarps = 4;                      // the fixup warps, as realigning loader
constexpr int kEpiWarp0 = 2;
constexpr int kHalf = 128;                            // P rows per CTA
constexpr uint32_t kHalfBytes = kHalf * TILE_K * 2;   // 16 KiB: the P half, and room for the Q half
constexpr uint32_t kStageBytes = 2 * kHalfBytes;      // this CTA's P half + Q half
constexpr uint32_t kMnChunkBytes = 64 * TILE_K * 2;   // one 64-wide MN box, 64 K rows: 8 KiB
constexpr uint32_t kSmemLimit = 227 * 1024;
constexpr uint32_t kNumBarsFor = 5 + kRlMaxStg;       // accf[2], acce[2], teardown, staging slots landed (+ 2 per stage)
constexpr int kStages = static_cast<int>((kSmemLimit - EPI_STAGING_BYTES - 1024 - 64 - 8 * kNumBarsFor) /
                                         (kStageBytes + 16));
constexpr uint32_t kEpiOff = kStages * kStageBytes;
constexpr uint32_t kBarOff = kEpiOff + EPI_STAGING_BYTES;
constexpr uint32_t kNumBars = 2 * kStages + kNumBarsFor;
constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
constexpr uint32_t kSmemAlloc = kMiscOff + 64 + 1024;  // slack for 1024-byte alignment
constexpr uint32_t kTmemCols = 512;                   // two accumulator buffers of BN <= 256 columns
constexpr int kCH = 32;
static_assert(kSmemAlloc <= kSmemLimit, "shared memory budget");
static_assert(kStages >= 4, "pipeline depth");

template <int kBN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_gemm_pair_kernel(const __grid_constant__ TcArgs a) {
  pdl_launch_dependents();
  static_assert(kBN % 32 == 0 && kBN >= 128 && kBN <= 256, "pair tile width");
  constexpr int kQHalf = kBN / 2;                   // Q rows per CTA
  constexpr int kQChunks = (kQHalf + 63) / 64;      // 64-wide boxes of an MN-major Q half
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const bool leader = rank == 0;
  const uint32_t bar0 = base + kBarOff;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  const uint32_t teardown_bar = bar0 + 8u * (2 * kStages + 4);
  auto stg_full = [&](int i) { return bar0 + 8u * (2 * kStages + 5 + i); };
  // Realigning loader (realign.cuh): its staging ring takes the last rl_take
  // pipeline stages' memory of each CTA; nst stages remain.
  const bool rl = a.rl_on[0] || a.rl_on[1];
  const uint32_t rl_bytes_p = a.rl_on[0] ? rl_stage_bytes(a.p_mn, kHalf, a.rl_cls[0]) : 0u;
  const uint32_t rl_bytes_q = a.rl_on[1] ? rl_stage_bytes(a.q_mn, kQHalf, a.rl_cls[1]) : 0u;
  const uint32_t rl_slot = rl_bytes_p + rl_bytes_q;
  int rl_take = 0, rl_nstg = 0;
  rl_ring(kStages, kStageBytes, rl_slot, rl_take, rl_nstg);
  const int nst = kStages - rl_take;
  const uint32_t stg0 = base + static_cast<uint32_t>(nst) * kStageBytes;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);

  if (threadIdx.x == 0) {
    // the even CTA's producer arms it with both CTAs' bytes; a realigned
    // operand's loader warps of both CTAs arrive on it too
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), rl ? 3u : 1u);
      mbar_init(empty_bar(s), 1);  // multicast MMA commit
    }
    for (int i = 0; i < kRlMaxStg; ++i) mbar_init(stg_full(i), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);                   // multicast MMA commit
      mbar_init(acce_bar(b), 2 * kEpiThreads / 32);  // epilogue warps of both CTAs
    }
    mbar_init(teardown_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&a.tm_p);
    tma_prefetch_desc(&a.tm_q);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    tmem_relinquish_pair();
  }
  // Both CTAs' barriers are initialised and TMEM is allocated before any
  // cross-CTA traffic.
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // operands, C and the split-K workspace may be written by the previous kernel
  pdl_wait();
  // The even CTA's barriers in the cluster's shared window.
  const uint32_t full_bar_leader0 = mapa_shared(full_bar(0), 0);
  const uint32_t acce_bar_leader0 = mapa_shared(acce_bar(0), 0);

  int issued = 0;  // producer lane: K blocks whose loads were issued

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Sched sched(a);
      Group g;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // Bytes of both CTAs' copies per stage (an MN-major Q half is loaded in
      // whole 64-wide boxes); realigned operands go through staging.
      const uint32_t q_bytes = a.q_mn ? kQChunks * kMnChunkBytes : kQHalf * TILE_K * 2;
      const uint32_t pair_bytes = 2 * ((a.rl_on[0] ? 0u : kHalfBytes) + (a.rl_on[1] ? 0u : q_bytes));
      while (ok && sched.next(a, g)) {
        int32_t tp, tq, m0, m1, n0, n1;
        tile_ranges(a, g.tile, kBN, tp, tq, m0, m1, n0, n1);
        const int32_t prow = tp * (2 * kHalf) + static_cast<int32_t>(rank) * kHalf;
        const int32_t qrow = tq * kBN + static_cast<int32_t>(rank) * kQHalf;
        for (int kb = 0; kb < g.nkb; ++kb) {
          if (!mbar_wait_bounded_cluster(empty_bar(stage), phase ^ 1u, a.wait_limit_ns, abort_flag)) {
            if (!*abort_flag) record_timeout(a, abort_flag, 0 * 16 + 1);
            ok = false;
            break;
          }
          const uint32_t sp = base + stage * kStageBytes;
          const uint32_t sq = sp + kHalfBytes;
          const uint32_t fb = full_bar_leader0 + 8u * stage;
          const int32_t k0 = (g.kb0 + kb) * TILE_K;
          if (leader) mbar_arrive_expect_tx(full_bar(stage), pair_bytes);
          if (a.rl_on[0]) {
            // (realigned: the loader warps fill it)
          } else if (!a.p_mn) {
            tma_load_2d_pair(sp, &a.tm_p, fb, k0, prow);
          } else {
            tma_load_2d_pair(sp, &a.tm_p, fb, prow, k0);
            tma_load_2d_pair(sp + kMnChunkBytes, &a.tm_p, fb, prow + 64, k0);
          }
          if (a.rl_on[1]) {
            // (realigned: the loader warps fill it)
          } else if (!a.q_mn) {
            tma_load_2d_pair(sq, &a.tm_q, fb, k0, qrow);
          } else {
#pragma unroll
            for (int j = 0; j < kQChunks; ++j)
              tma_load_2d_pair(sq + j * kMnChunkBytes, &a.tm_q, fb, qrow + 64 * j, k0);
          }
          ++issued;
          if (++stage == nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Wait until the MMAs have released the last stages this CTA filled, so
      // that no multicast commit targets this CTA after it exits.
      const int first = issued > nst ? issued - nst : 0;
      for (int it = first; it < issued && !*abort_flag; ++it)
        if (!mbar_wait_bounded_cluster(empty_bar(it % nst), (it / nst) & 1, a.wait_limit_ns, abort_flag) &&
            !*abort_flag)
          record_timeout(a, abort_flag, 0 * 16 + 4);

    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      Sched sched(a);
      Group g;
      int stage = 0;
      uint32_t phase = 0;
      int acc_iter = 0;
      bool ok = true;
      // Per-MMA (K = 16) start-address advance inside a stage, as in the
      // single-CTA kernel: K-major 128-byte rows (+32 B per 16 elements),
      // MN-major 128-byte rows per k (+2 KiB per 16 k), 64-wide chunks 8 KiB apart.
      const uint32_t p_step = a.p_mn ? 2048u : 32u;
      const uint32_t q_step = a.q_mn ? 2048u : 32u;
      const uint32_t p_lbo = a.p_mn ? kMnChunkBytes : 16u;
      const uint32_t q_lbo = a.q_mn ? kMnChunkBytes : 16u;
      while (ok && sched.next(a, g)) {
        if (g.nkb == 0) continue;
        const int buf = acc_iter & 1;
        const uint32_t acc_phase = (acc_iter >> 1) & 1;
        if (!mbar_wait_bounded_cluster(acce_bar(buf), acc_phase ^ 1u, a.wait_limit_ns, abort_flag)) {
          if (!*abort_flag) record_timeout(a, abort_flag, 1 * 16 + 3);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kBN);
        for (int kb = 0; kb < g.nkb; ++kb) {
          if (!mbar_wait_bounded_cluster(full_bar(stage), phase, a.wait_limit_ns, abort_flag)) {
            if (!*abort_flag) record_timeout(a, abort_flag, 1 * 16 + 0);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sp = base + stage * kStageBytes;
          const uint32_t sq = sp + kHalfBytes;
#pragma unroll
          for (int k = 0; k < TILE_K / 16; ++k) {
            const uint64_t pd = sw128_desc(sp + k * p_step, p_lbo, 1024u);
            const uint64_t qd = sw128_desc(sq + k * q_step, q_lbo, 1024u);
            tc_mma_f16_ss_pair(d_tmem, pd, qd, a.idesc, (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit_pair_mc(empty_bar(stage), 0x3);
          if (++stage == nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(accf_bar(buf), 0x3);
        ++acc_iter;
      }
    }
  } else if (warp >= kFixWarp0) {
    if (rl) {
      // ---------------------------------------------------------- realigning loader
      // As in the single-CTA kernel: the loader's own staging ring, refilled
      // by the first loader warp as each slot is realigned out; this CTA's
      // halves of each stage, then one arrive on the even CTA's stage barrier
      // (the planner gives such plans no fixup work).
      const int t = threadIdx.x - kFixWarp0 * 32;
      const bool issuer = warp == kFixWarp0;
      const uint32_t tx = (a.rl_on[0] ? rl_stage_tx(a.p_mn, kHalf, a.rl_cls[0]) : 0u) +
                          (a.rl_on[1] ? rl_stage_tx(a.q_mn, kQHalf, a.rl_cls[1]) : 0u);
      KbIter ahead(a);
      int stg_issued = 0, stg_done = 0;
      auto fill = [&](int sl) {
        int tile, kb;
        if (!ahead.next(a, tile, kb)) return;
        int32_t tp, tq, m0, m1, n0, n1;
        tile_ranges(a, tile, kBN, tp, tq, m0, m1, n0, n1);
        const int32_t prow = tp * (2 * kHalf) + static_cast<int32_t>(rank) * kHalf;
        const int32_t qrow = tq * kBN + static_cast<int32_t>(rank) * kQHalf;
        const uint32_t dst = stg0 + static_cast<uint32_t>(sl) * rl_slot;
        if (lane == 0) mbar_arrive_expect_tx(stg_full(sl), tx);
        __syncwarp();
        if (a.rl_on[0]) rl_issue(a.tm_rl[0], a.rl_cls[0], a.p_mn, kHalf, prow, kb * TILE_K, dst, stg_full(sl), lane, 32);
        if (a.rl_on[1])
          rl_issue(a.tm_rl[1], a.rl_cls[1], a.q_mn, kQHalf, qrow, kb * TILE_K, dst + rl_bytes_p, stg_full(sl), lane, 32);
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
                           mbar_wait_bounded_cluster(empty_bar(stage), phase ^ 1u, a.wait_limit_ns, abort_flag);
          if (!got && !*abort_flag) record_timeout(a, abort_flag, 0 * 16 + 6);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          const uint32_t src = stg0 + static_cast<uint32_t>(slot) * rl_slot;
          const uint32_t sp = base + static_cast<uint32_t>(stage) * kStageBytes;
          if (a.rl_on[0]) rl_pass(a.rl_d[0], a.rl_cls[0], a.p_mn, kHalf, src, sp, t, kRlWarps * 32);
          if (a.rl_on[1]) rl_pass(a.rl_d[1], a.rl_cls[1], a.q_mn, kQHalf, src + rl_bytes_p, sp + kHalfBytes, t, kRlWarps * 32);
          // the stage is read by this SM's tensor core (async proxy) for the
          // pair's MMA, which the even CTA issues after the arrive below; the
          // slot is refilled by TMA
          fence_proxy_async_smem();
          named_bar_sync(3, kRlWarps * 32);
          ++stg_done;
          if (t == 0) mbar_arrive_cluster(full_bar_leader0 + 8u * stage);
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
      finish_tail<kBN>(a, abort_flag, threadIdx.x - kFixWarp0 * 32);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;
    const int et = threadIdx.x - kEpiWarp0 * 32;
    Sched sched(a);
    Group g;
    int acc_iter = 0;
    int ring = 0;
    const uint32_t stage_smem = base + kEpiOff + static_cast<uint32_t>(warp - kEpiWarp0) * 8192u;
    while (sched.next(a, g)) {
      if (!epilogue_group<kBN, kCH, true>(a, g, tmem_base, accf_bar(0), acce_bar_leader0, acc_iter, abort_flag, q4,
                                          lane, et, static_cast<int>(rank), stage_smem, ring))
        break;
    }
    if (lane == 0) bulk_wait_group<0>();  // staged stores finished before the CTA exits
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_flag) {
    // Copies this CTA issued may still be landing (their stage barrier lives
    // in the even CTA and may never complete): give them time to arrive.
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
  }
  if (leader && warp == 1 && lane == 0) {
    // Wait until every MMA of the pair has completed.
    volatile int no_abort = 0;
    tc_commit_pair_mc(teardown_bar, 0x1);
    mbar_wait_bounded(teardown_bar, 0, a.wait_limit_ns, &no_abort);
  }
  tc_fence_before();
  __syncthreads();
  // Neither CTA leaves while the other may still touch its shared memory.
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

template <int BN>
cudaError_t launch_bn(const TcArgs& args, int grid, cudaStream_t stream) {
  cudaError_t e = set_smem_once<tc_gemm_pair_kernel<BN>>(static_cast<int>(kSmemAlloc));
  if (e != cudaSuccess) return e;
  // (the grid is at most the resident clusters; see the single-CTA launcher)
  return launch_pdl(tc_gemm_pair_kernel<BN>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmemAlloc, stream,
                    args);
}

}  // namespace

bool tc_gemm_pair_supports(int bn) { return bn == 128 || bn == 160 || bn == 192 || bn == 224 || bn == 256; }

bool tc_gemm_pair_rl_fits(int bn, int p_mn, int q_mn, int p_cls, int q_cls) {
  if (!tc_gemm_pair_supports(bn)) return false;
  const uint32_t stg = (p_cls ? rl_stage_bytes(p_mn, kHalf, p_cls) : 0u) + (q_cls ? rl_stage_bytes(q_mn, bn / 2, q_cls) : 0u);
  int take, nstg;
  return rl_ring(kStages, kStageBytes, stg, take, nstg) && (stg == 0 || nstg >= 2);
}

cudaError_t launch_tc_gemm_pair(const TcArgs& args, int bn, int grid, cudaStream_t stream) {
  if (grid < 2 || (grid & 1) || !args.pair) return cudaErrorInvalidValue;
  switch (bn) {
    case 128: return launch_bn<128>(args, grid, stream);
    case 160: return launch_bn<160>(args, grid, stream);
    case 192: return launch_bn<192>(args, grid, stream);
    case 224: return launch_bn<224>(args, grid, stream);
    case 256: return launch_bn<256>(args, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t tc_gemm_pair_max_clusters(int* clusters) {
  *clusters = 0;
  // every width has the same block size and shared memory
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_pair_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemAlloc));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemAlloc;
  return cudaOccupancyMaxActiveClusters(clusters, tc_gemm_pair_kernel<256>, &cfg);
}

}  // namespace lgt
