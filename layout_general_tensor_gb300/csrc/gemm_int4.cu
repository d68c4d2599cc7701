// int4-weight GEMM with the dequantisation inside the mainloop, fp16 form
// (activations of up to 64 rows, any activation layout, groups of 64 or more;
// the e4m3 form in gemm_int4_f8.cu takes activations of up to 16 rows).
//
//   C[m,n] = sum_k A[m,k] * w(k,n),  w(k,n) = (q(n,k) - z(n,g)) * s(n,g),
//   g = k / group_size, codes two per byte (low nibble = even k).
//
// The weight is the large operand and the activation the skinny one, so the
// MMA runs swapped: 128 weight rows (n) on the MMA's M side, the activation
// rows (m) on its N side, the accumulator holding C^T in TMEM.  The expanded
// weight tile is the MMA's A operand *in TMEM*; the activation its B operand
// in shared memory.
//
// Arithmetic.  C = sum_k A q s - sum_g z s Ag[g], with Ag[g][m] the sum of
// row m of the activation over group g.  The expanded weight is q s rounded
// to fp16 once: a code in bits 0..3 of a half ORed into 0x6400 is the fp16
// number 1024 + q, one in bits 4..7 ORed into 0x5400 is 64 + q (the
// mantissa's unit there is 1/16), and fma(1024 + q, s, -1024 s) is q s
// exactly before its one rounding (1024 s and 64 s are exact), so a pair of
// codes costs one LOP3 and one HFMA2.  The zero-point term z s Ag is formed
// in fp32 (z s is exact there) by the epilogue of the run that starts each
// tile and subtracted from that run's accumulator.
// The activation is copied once, K-contiguous, with every 8-element group of
// K reordered to that pair order (0,4,1,5,2,6,3,7) by a small pre-pass
// (int4_prep_kmajor_kernel / int4_prep_kernel), so no code is moved in the
// mainloop.  The dequantise copy of the BitBLAS TileLang page (the
// thread-level listing in "Relevant Issues") vectorises its loads of packed
// weights; here the TMA box does the addressing and every thread's shared
// loads are 128-bit.
//
// A pipeline stage is up to four 64-deep K blocks of one run: the packed
// weight as one TMA box of 128 rows x 128 bytes (128-byte swizzle; 128-byte
// row segments keep the TMA stream near the HBM rate) in the weight ring, and
// one activation box per K block in the activation ring.  The weight ring is
// freed as soon as the expanders have read a stage, so its depth is all in
// flight.  The accumulators of a run are double-buffered in TMEM, so the
// epilogue of one run overlaps the next; a run's epilogue (C, or the split-K
// partial and the arrival protocol) is the one of the dense kernels.
//
// Warp roles (512 threads):
//   warp 0       TMA producer for both rings.
//   warps 1..3   MMA issuers (NI of them active, by accumulator width).  One
//                thread issues a narrow MMA only every 150 to 200 cycles
//                whatever its width, so a stage's MMAs are spread over all
//                of them: MMA m of a stage (K block m / 4, 16-deep step
//                m % 4) goes to issuer m % NI, into that issuer's own
//                accumulator.  Every issuer waits for every stage's expanded
//                slot and activation and commits the slot and the activation
//                buffer free (NI arrivals each).  Warp 1 owns the TMEM.
//   warps 4..7   epilogue (TMEM lane quadrant warp % 4), adds the NI
//                accumulators.
//   warps 8..15  expanders: two warps per TMEM lane quadrant, each taking two
//                of every stage's four K blocks; each thread owns one weight
//                row of the tile.  A stage's codes are expanded before the
//                slot they go to is waited for.
#include <cuda_fp16.h>

#include "int4.h"
#include "kernels.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lgt {
namespace {

constexpr int kThreads4 = 512;
constexpr int kIssWarp0 = 1;                  // MMA issuer warps 1..3
constexpr int kMaxIssuers = 3;
constexpr int kEpiWarp04 = 4;                 // epilogue warps 4..7
constexpr int kExpWarp0 = 8;                  // expander warps 8..15
constexpr int kQuadK = 4;                     // K blocks per stage
constexpr uint32_t kRawBytes = TILE_P * 128;  // 128 rows x 128 bytes (256 codes)
constexpr uint32_t kWStage = kRawBytes + 1024;  // packed-weight stage (+ a pre-packed block's scale slots)
constexpr uint32_t kASlotCol0 = 128;          // A slots at [128, 512); the accumulators below

template <int BN>
struct Cfg4 {
  // MMA issuers.  One thread issues a narrow (N <= 64) MMA about every 150
  // to 200 cycles whatever N, and the tensor core takes them several times
  // faster than that, so every stage's MMAs are spread over NI issuers, each
  // with accumulators of its own (double-buffered: 2 NI BN <= 128 columns),
  // which the epilogue adds.
  static constexpr int NI = BN == 16 ? 3 : (BN == 32 ? 2 : 1);
  // TMEM A slots of 128 columns (a stage's four K blocks as fp16 pairs);
  // every issuer takes part in every stage, so it waits on every slot's and
  // activation buffer's barriers in order.
  static constexpr int TSLOTS = 3;
  static constexpr uint32_t ACT_TILE = BN * TILE_K * 2;  // one 64-deep activation box
  static constexpr uint32_t XSTAGE = kQuadK * ACT_TILE;  // a stage's activation
  // activation ring: one buffer per A slot (stage s uses both s % TSLOTS),
  // so that one barrier frees both
  static constexpr int XST = TSLOTS;
  // the tile's slice of the activation group sums, Ag[g][m0 .. m0 + BN),
  // staged in shared memory for the zero-point term (BN = 16, up to 256 groups)
  static constexpr uint32_t ZP_BYTES = BN == 16 ? 256 * BN * 4 : 0;
  static constexpr uint32_t RING_BYTES = 224 * 1024 - ZP_BYTES;
  static constexpr int WST_FIT = static_cast<int>((RING_BYTES - XST * XSTAGE) / kWStage);
  static constexpr int WST = WST_FIT > 12 ? 12 : WST_FIT;  // packed-weight ring
  static constexpr uint32_t X_OFF = WST * kWStage;
  // barriers: full_w[W], wfree[W], full_x[X], a_full[T], tfree[T], accf[2], acce[2], teardown
  static constexpr uint32_t ZP_OFF = X_OFF + XST * XSTAGE;
  static constexpr uint32_t BAR_OFF = ZP_OFF + ZP_BYTES;
  static constexpr uint32_t NUM_BARS = 2 * WST + XST + 2 * TSLOTS + 5;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr uint32_t SMEM_ALLOC = MISC_OFF + 64 + 1024;  // slack for 1024-byte alignment
  static_assert(kWStage % 1024 == 0 && ACT_TILE % 1024 == 0, "swizzled buffers stay 1024-byte aligned");
  static_assert(WST >= 4 && XST == TSLOTS, "ring depths");
  static_assert(NI <= kMaxIssuers, "issuer warps");
  static_assert(2 * NI * BN <= static_cast<int>(kASlotCol0), "accumulators fit below the A slots");
  static_assert(kASlotCol0 + TSLOTS * 128 <= 512, "A slots fit in the TMEM allocation");
};

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
  return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float half_bits_to_float(uint32_t b) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}




// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16.
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Stages of this CTA's runs, in order: up to kQuadK K blocks of one run each
// (runs without K blocks are skipped).
struct StageIter {
  Sched sched;
  Group g;
  bool have = false;
  int kb = 0;
  __device__ explicit StageIter(const TcArgs& a) : sched(a) {}
  __device__ bool next(const TcArgs& a, int& kb0, int& nk, bool& new_run) {
    new_run = false;
    while (!have || kb >= g.nkb) {
      if (!sched.next(a, g)) return false;
      have = true;
      kb = 0;
      new_run = true;
    }
    kb0 = kb;
    nk = min(kQuadK, g.nkb - kb);
    kb += nk;
    return true;
  }
};

// The zero-point term of a tile, subtracted from the run that starts at K
// block 0 (its accumulator holds sum_k A[m, k] q(n, k) s(n, g(k)) for its
// K blocks; the other runs' partials need no term): for this thread's row n,
//   corr[m] = sum over all groups g of z(n, g) s(n, g) * Ag[g][m],
// with Ag the activation's group sums.  z s is exact in fp32.  For BN = 16
// the term is formed before the accumulator is ready, else per block of
// columns when it is drained.
template <int BN>
struct ZpFix {
  static constexpr int NC = BN <= 16 ? BN : 1;
  const Int4Args* A4 = nullptr;
  const uint16_t* srow = nullptr;  // null: no term (row beyond N)
  const uint16_t* zrow = nullptr;
  uint32_t ag_smem = 0;            // staged Ag slice (fp32 [g][BN]), or 0: read from global memory
  int m0 = 0;
  bool active = false;  // the current run is one that subtracts the term
  float corr[NC];

  template <int N>
  __device__ __forceinline__ void term(int c0, float (&out)[N]) const {
#pragma unroll
    for (int j = 0; j < N; ++j) out[j] = 0.0f;
    if (!srow) return;
    const int M = A4->t.M, G = A4->groups;
    const int mc = m0 + c0;
    const bool full = mc + N <= M && (M & 3) == 0;
    // group g's Ag[g][mc .. mc + N) times zs
    auto add_group = [&](int g, float zs) {
      if (ag_smem) {
#pragma unroll
        for (int j = 0; j < N; j += 4) {
          const float4 v = ld_shared_f32x4(ag_smem + static_cast<uint32_t>((g * BN + c0 + j) * 4));
          out[j] = fmaf(zs, v.x, out[j]);
          out[j + 1] = fmaf(zs, v.y, out[j + 1]);
          out[j + 2] = fmaf(zs, v.z, out[j + 2]);
          out[j + 3] = fmaf(zs, v.w, out[j + 3]);
        }
        return;
      }
      const float* ag = A4->agsum + static_cast<int64_t>(g) * M + mc;
      if (full) {
#pragma unroll
        for (int j = 0; j < N; j += 4) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(ag + j));
          out[j] = fmaf(zs, v.x, out[j]);
          out[j + 1] = fmaf(zs, v.y, out[j + 1]);
          out[j + 2] = fmaf(zs, v.z, out[j + 2]);
          out[j + 3] = fmaf(zs, v.w, out[j + 3]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < N; ++j)
          if (mc + j < M) out[j] = fmaf(zs, __ldg(ag + j), out[j]);
      }
    };
    if (A4->vec_sz) {
      // the row's scales and zero points 16 bytes (8 groups) per load, four
      // loads of each in flight at a time
      for (int gb = 0; gb < G; gb += 32) {
        uint4 sw[4], zw[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          sw[w] = make_uint4(0u, 0u, 0u, 0u);
          zw[w] = make_uint4(0x48004800u, 0x48004800u, 0x48004800u, 0x48004800u);  // fp16 8.0
          if (gb + 8 * w < G) {
            sw[w] = __ldg(reinterpret_cast<const uint4*>(srow + gb) + w);
            if (zrow) zw[w] = __ldg(reinterpret_cast<const uint4*>(zrow + gb) + w);
          }
        }
#pragma unroll 1
        for (int w = 0; w < 4; ++w) {
          if (gb + 8 * w >= G) break;
          const uint32_t sv[4] = {sw[w].x, sw[w].y, sw[w].z, sw[w].w};
          const uint32_t zv[4] = {zw[w].x, zw[w].y, zw[w].z, zw[w].w};
#pragma unroll 2
          for (int e = 0; e < 8; ++e) {
            const uint32_t sb = (e & 1) ? (sv[e >> 1] >> 16) : (sv[e >> 1] & 0xFFFFu);
            const uint32_t zb = (e & 1) ? (zv[e >> 1] >> 16) : (zv[e >> 1] & 0xFFFFu);
            add_group(gb + 8 * w + e, half_bits_to_float(zb) * half_bits_to_float(sb));
          }
        }
      }
    } else {
      for (int g = 0; g < G; ++g)
        add_group(g, (zrow ? half_bits_to_float(__ldg(zrow + g)) : 8.0f) * half_bits_to_float(__ldg(srow + g)));
    }
  }

  // Sets up (and for BN = 16 forms) the term of a run that starts a tile.
  // All 128 epilogue threads call it together: with a staging buffer
  // (`stage` != 0, BN = 16, at most 256 groups) they first copy the tile's
  // Ag slice there, every load in flight at once.
  __device__ void prepare(const Int4Args& a4, const Group& g, int n, int n1, int m0_, uint32_t stage, int et) {
    A4 = &a4;
    m0 = m0_;
    ag_smem = 0;
    if (stage && a4.groups <= 256) {
      const int M = a4.t.M;
      named_bar_sync(1, kEpiThreads);  // the previous slice is no longer read
      for (int i = et; i < a4.groups * BN; i += kEpiThreads) {
        const int gi = i / BN, m = m0 + i % BN;
        st_shared_f32(stage + 4u * i, m < M ? __ldg(a4.agsum + static_cast<int64_t>(gi) * M + m) : 0.0f);
      }
      named_bar_sync(1, kEpiThreads);
      ag_smem = stage;
    }
    srow = n < n1 ? a4.scales + static_cast<int64_t>(n) * a4.groups : nullptr;
    zrow = (n < n1 && a4.zeros) ? a4.zeros + static_cast<int64_t>(n) * a4.groups : nullptr;
    (void)g;
    if constexpr (BN <= 16) term<NC>(0, corr);
  }

  template <int N>
  __device__ __forceinline__ void operator()(int c0, uint32_t (&v)[N]) const {
    if (!active || !srow) return;
    if constexpr (BN <= 16) {
#pragma unroll
      for (int j = 0; j < N; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) - corr[c0 + j]);
    } else {
      float t[N];
      term<N>(c0, t);
#pragma unroll
      for (int j = 0; j < N; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) - t[j]);
    }
  }
};

template <int BN>
__global__ void __launch_bounds__(kThreads4, 1) int4_gemm_kernel(const __grid_constant__ Int4Args A4) {
  pdl_launch_dependents();
  using C = Cfg4<BN>;
  constexpr int NI = C::NI;
  const TcArgs& a = A4.t;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = base + C::BAR_OFF;
  // full_w[s] / full_x[s]: a packed-weight / activation stage landed.
  // wfree[s]: the stage's eight expander warps have expanded its packed
  // weights into TMEM.
  // a_full[t]: the expanders wrote a stage's weights into TMEM A slot t.
  // tfree[t]: the MMAs reading slot t and activation buffer t completed
  // (every issuer commits), so both are free.  accf / acce: accumulator
  // buffer full (one commit per issuer at the end of each run) / drained by
  // the epilogue.
  constexpr int kB1 = 2 * C::WST + C::XST;
  auto full_w = [&](int i) { return bar0 + 8u * i; };
  auto wfree = [&](int i) { return bar0 + 8u * (C::WST + i); };
  auto full_x = [&](int i) { return bar0 + 8u * (2 * C::WST + i); };
  auto a_full = [&](int t) { return bar0 + 8u * (kB1 + t); };
  auto tfree_bar = [&](int t) { return bar0 + 8u * (kB1 + C::TSLOTS + t); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (kB1 + 2 * C::TSLOTS + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (kB1 + 2 * C::TSLOTS + 2 + b); };
  const uint32_t teardown_bar = bar0 + 8u * (kB1 + 2 * C::TSLOTS + 4);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::WST; ++i) {
      mbar_init(full_w(i), 1);
      mbar_init(wfree(i), 8);  // every expander warp, after its stores
    }
    for (int i = 0; i < C::XST; ++i) {
      mbar_init(full_x(i), 1);
    }
    for (int t = 0; t < C::TSLOTS; ++t) {
      mbar_init(a_full(t), 8);
      mbar_init(tfree_bar(t), NI);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), NI);
      mbar_init(acce_bar(b), kEpiThreads / 32);
    }
    mbar_init(teardown_bar, NI);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&A4.tm_w);
    tma_prefetch_desc(&a.tm_q);
  }
  if (warp == kIssWarp0) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the pre-pass's output, C and the split-K workspace come from earlier kernels
  pdl_wait();

  int w_issued = 0, x_issued = 0;  // producer lane: stages whose loads were issued, per ring

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Two rings fed in stage order, each as soon as its next buffer is free:
    // the packed weights (the HBM stream) never wait for an activation buffer.
    if (lane == 0) {
      StageIter itw(a), itx(a);
      int wkb0 = 0, wnk = 0, xkb0 = 0, xnk = 0;
      bool nr, whave = false, xhave = false, wdone = false, xdone = false;
      uint64_t stall_t0 = 0;
      while (true) {
        if (!whave && !wdone) {
          whave = itw.next(a, wkb0, wnk, nr);
          wdone = !whave;
        }
        if (!xhave && !xdone) {
          xhave = itx.next(a, xkb0, xnk, nr);
          xdone = !xhave;
        }
        if (wdone && xdone) break;
        bool progress = false;
        if (whave) {
          const int s = w_issued % C::WST;
          if (mbar_test_wait(wfree(s), ((w_issued / C::WST) & 1) ^ 1u)) {
            int32_t tp, tq, m0, m1, n0, n1;
            tile_ranges(a, itw.g.tile, BN, tp, tq, m0, m1, n0, n1);
            const int kb = itw.g.kb0 + wkb0;
            if (A4.wpre) {
              // pre-packed: the stage's block (codes already swizzled, then
              // its scales) in one bulk copy
              const uint8_t* src = A4.wpre + (static_cast<int64_t>(tp) * A4.pre_stages + kb / kQuadK) * A4.pre_block;
              mbar_arrive_expect_tx(full_w(s), static_cast<uint32_t>(A4.pre_block));
              bulk_load_g2s(base + s * kWStage, src, static_cast<uint32_t>(A4.pre_block), full_w(s));
            } else {
              mbar_arrive_expect_tx(full_w(s), kRawBytes);
              tma_load_2d(base + s * kWStage, &A4.tm_w, full_w(s), kb * (TILE_K / 2), n0);
            }
            ++w_issued;
            whave = false;
            progress = true;
          }
        }
        if (xhave) {
          const int s = x_issued % C::XST;
          if (mbar_test_wait(tfree_bar(s), ((x_issued / C::XST) & 1) ^ 1u)) {
            int32_t tp, tq, m0, m1, n0, n1;
            tile_ranges(a, itx.g.tile, BN, tp, tq, m0, m1, n0, n1);
            // one box: x_box_kb K blocks of bn rows (beyond the run's K blocks
            // it reads neighbours or zero fill, which no MMA uses)
            (void)xnk;
            mbar_arrive_expect_tx(full_x(s), static_cast<uint32_t>(A4.x_box_kb) * C::ACT_TILE);
            tma_load_3d(base + C::X_OFF + s * C::XSTAGE, &a.tm_q, full_x(s), 0, m0, itx.g.kb0 + xkb0);
            ++x_issued;
            xhave = false;
            progress = true;
          }
        }
        if (progress) {
          stall_t0 = 0;
          continue;
        }
        if (*abort_flag) break;
        const uint64_t now = global_timer_ns();
        if (stall_t0 == 0) {
          stall_t0 = now;
        } else if (now - stall_t0 > a.wait_limit_ns) {
          record_timeout(a, abort_flag, 0 * 16 + 1);
          break;
        }
        __nanosleep(32);
      }
    }
  } else if (warp < kEpiWarp04) {
    // ------------------------------------------------------------ MMA issuers
    // Issuer i issues MMAs m = i, i + NI, ... of every stage (m = 4 j + k:
    // K block j, 16-deep step k) into its own accumulator; its first MMA of
    // a run's first stage starts the accumulator.  One commit per stage frees
    // the stage's A slot and activation buffer.  An issuer with no MMA in
    // a run (a run of fewer than NI / 4 K blocks, rounded up) leaves its accumulator
    // untouched, and the epilogue adds only the others.  Every issuer waits
    // for every stage, so its commits on the slot and activation barriers
    // come after the stage was filled, in order; it commits the end of every
    // run.
    const int iss = warp - kIssWarp0;
    if (lane == 0 && iss < NI) {
      StageIter it(a);
      int kb0, nk, acc_iter = -1;
      bool nr;
      uint32_t d_tmem = tmem_base;
      int t = 0;            // A slot and activation buffer of this stage
      uint32_t tph = 0u;    // their phase parity
      while (it.next(a, kb0, nk, nr)) {
        if (nr) {
          ++acc_iter;
          const int buf = acc_iter & 1;
          if (!mbar_wait_bounded(acce_bar(buf), ((acc_iter >> 1) & 1) ^ 1u, a.wait_limit_ns, abort_flag)) {
            if (!*abort_flag) record_timeout(a, abort_flag, 1 * 16 + 3);
            break;
          }
          d_tmem = tmem_base + static_cast<uint32_t>((buf * NI + iss) * BN);
        }
        if (!mbar_wait_bounded(a_full(t), tph, a.wait_limit_ns, abort_flag) ||
            !mbar_wait_bounded(full_x(t), tph, a.wait_limit_ns, abort_flag)) {
          if (!*abort_flag) record_timeout(a, abort_flag, 1 * 16 + 0);
          break;
        }
        tc_fence_after();
        const uint64_t bd0 = sw128_desc(base + C::X_OFF + t * C::XSTAGE, 16u, 1024u);
        const uint32_t a0 = tmem_base + kASlotCol0 + static_cast<uint32_t>(t * 128);
        const uint32_t first = kb0 == 0;  // the run's first stage
#pragma unroll
        for (int m = iss; m < 4 * kQuadK; m += NI) {
          if (m >= 4 * nk) break;
          const int j = m >> 2, k = m & 3;
          // A: 8 TMEM columns (16 fp16 pairs) per 16-deep step; B: +32 bytes per step
          tc_mma_f16_ts(d_tmem, a0 + static_cast<uint32_t>(j * 32 + k * 8),
                        bd0 + static_cast<uint64_t>((j * C::ACT_TILE) >> 4) + static_cast<uint64_t>(2 * k), a.idesc,
                        (m == iss && first) ? 0u : 1u);
        }
        tc_commit(tfree_bar(t));
        if (kb0 + nk == it.g.nkb) tc_commit(accf_bar(acc_iter & 1));
        if (++t == C::TSLOTS) {
          t = 0;
          tph ^= 1u;
        }
      }
    }
  } else if (warp >= kExpWarp0) {
    // ------------------------------------------------------------ expanders
    const int q4 = warp & 3;
    const int h = (warp - kExpWarp0) >> 2;  // K blocks 2h, 2h + 1 of every stage
    const int r = q4 * 32 + lane;           // weight row within the tile (TMEM lane)
    // This row's scale of each of its two K blocks of a stage (raw fp16
    // bits).  Pre-packed weights carry them in the stage: K block j's in
    // slot j / (K blocks per group), at an offset fixed for this thread.
    // Otherwise they are read from the scale array two stages ahead, by a
    // look-ahead walk over the same stages, into a three-deep register
    // ring, so that each load's latency hides behind two stages' expansion.
    const bool pre = A4.wpre != nullptr;
    uint32_t pre_off[2];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
      pre_off[jj] = kRawBytes + static_cast<uint32_t>(
                                    (A4.pre_kbpg >= kQuadK ? 0 : (2 * h + jj) / max(A4.pre_kbpg, 1)) * 256 + r * 2);
    StageIter ahead(a);
    const uint16_t* arow = nullptr;  // the look-ahead stage's scale row (null: row beyond N)
    auto fetch = [&](uint32_t (&o)[2]) {
      o[0] = 0u;
      o[1] = 0u;
      int kb0a, nka;
      bool nra;
      if (!ahead.next(a, kb0a, nka, nra)) return;
      if (nra) {
        int32_t tp, tq, m0, m1, n0, n1;
        tile_ranges(a, ahead.g.tile, BN, tp, tq, m0, m1, n0, n1);
        const int n = n0 + r;
        arow = n < n1 ? A4.scales + static_cast<int64_t>(n) * A4.groups : nullptr;
      }
      if (!arow) return;
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int j = 2 * h + jj;
        if (j < nka) {
          const uint32_t g = magic_div(static_cast<uint32_t>(ahead.g.kb0 + kb0a + j), A4.div_kb_per_group);
          o[jj] = __ldg(arow + g);
        }
      }
    };
    uint32_t sc0[2] = {0u, 0u}, sc1[2] = {0u, 0u}, sc2[2] = {0u, 0u};
    if (!pre) {
      fetch(sc0);
      fetch(sc1);
    }
    // One K block (eight words of eight codes) as 32 fp16 pairs: codes
    // (p, p + 4) of a word for p = 0..3 as 1024 + q (p even) or 64 + q
    // (p odd), then (1024 + q) s - 1024 s = q s, rounded once.
    auto expand = [&](const uint4& r0, const uint4& r1, uint32_t s16, uint32_t* v) {
      const uint32_t s2 = s16 * 0x10001u;
      const uint32_t c1024 = hmul2(s2, 0xE400E400u), c64 = hmul2(s2, 0xD400D400u);
      const uint32_t words[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
      for (int w8 = 0; w8 < 8; ++w8) {
        const uint32_t lo = words[w8], hi = lo >> 8;
        v[4 * w8 + 0] = hfma2(lop3_and_or(lo, 0x000F000Fu, 0x64006400u), s2, c1024);
        v[4 * w8 + 1] = hfma2(lop3_and_or(lo, 0x00F000F0u, 0x54005400u), s2, c64);
        v[4 * w8 + 2] = hfma2(lop3_and_or(hi, 0x000F000Fu, 0x64006400u), s2, c1024);
        v[4 * w8 + 3] = hfma2(lop3_and_or(hi, 0x00F000F0u, 0x54005400u), s2, c64);
      }
    };
    StageIter it(a);
    int kb0, nk;
    bool nr;
    int sw = 0, t = 0;            // weight stage and A slot of this stage
    uint32_t wph = 0u, tph = 0u;  // their rings' phase parities
    while (it.next(a, kb0, nk, nr)) {
      if (!pre) fetch(sc2);  // two stages ahead
      const bool got = mbar_wait_bounded(full_w(sw), wph, a.wait_limit_ns, abort_flag);
      if (!got && !*abort_flag) record_timeout(a, abort_flag, 3 * 16 + 0);
      // the warp leaves together (tcgen05.st below needs every lane)
      if (!__all_sync(0xffffffffu, got)) break;
      // raw row r: eight 16-byte chunks, chunk c stored at c ^ (r mod 8)
      // (128-byte swizzle); this warp's K blocks 2h, 2h + 1 are chunks 4h..4h+3
      const uint32_t stage = base + static_cast<uint32_t>(sw) * kWStage;
      const uint8_t* rowp = smem + static_cast<uint32_t>(sw) * kWStage + r * 128;
      uint4 raw[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) raw[c] = *reinterpret_cast<const uint4*>(rowp + (((4 * h + c) ^ (r & 7)) << 4));
      uint32_t s16[2] = {sc0[0], sc0[1]};
      if (pre) {
        s16[0] = ld_shared_u16(stage + pre_off[0]);
        s16[1] = ld_shared_u16(stage + pre_off[1]);
      }
      // both K blocks are expanded before the slot is waited for (the MMAs
      // of the stage TSLOTS back may still be reading it), then stored by
      // one instruction; columns of a K block past the run's end hold values
      // no MMA reads
      uint32_t vals[64];
      expand(raw[0], raw[1], s16[0], vals);
      expand(raw[2], raw[3], s16[1], vals + 32);
      const bool freed = mbar_wait_bounded(tfree_bar(t), tph ^ 1u, a.wait_limit_ns, abort_flag);
      if (!freed && !*abort_flag) record_timeout(a, abort_flag, 3 * 16 + 1);
      if (!__all_sync(0xffffffffu, freed)) break;
      tc_fence_after();
      if (2 * h < nk) {
        const uint32_t slot = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + kASlotCol0 +
                              static_cast<uint32_t>(t * 128 + h * 64);
        tc_st_32x32b_x64_wait(slot, vals);
      }
      tc_fence_before();
      __syncwarp();
      // Both handoffs after the store: the stage's packed weights were read
      // by loads whose values the store consumed (so the next copy into the
      // stage cannot overtake them), and the A slot is written.
      if (lane == 0) {
        mbar_arrive(a_full(t));
        mbar_arrive(wfree(sw));
      }
      sc0[0] = sc1[0];
      sc0[1] = sc1[1];
      sc1[0] = sc2[0];
      sc1[1] = sc2[1];
      if (++sw == C::WST) {
        sw = 0;
        wph ^= 1u;
      }
      if (++t == C::TSLOTS) {
        t = 0;
        tph ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // (warps 4..7: TMEM lane quadrant warp % 4; tiles leave by plain stores,
    // so no staging buffer)
    const int q4 = warp & 3;
    const int et = threadIdx.x - kEpiWarp04 * 32;
    Sched sched(a);
    Group g;
    int acc_iter = 0, ring = 0;
    // The zero-point term of this CTA's first run that starts a tile is
    // formed now, while the pipeline fills; later ones when they come up.
    ZpFix<BN> fix;
    const uint32_t zp_stage = C::ZP_BYTES ? base + C::ZP_OFF : 0u;
    int first_idx = -1;
    {
      Sched look(a);
      Group gl;
      for (int idx = 0; look.next(a, gl); ++idx) {
        if (gl.s0 == 0 && gl.nkb > 0) {
          int32_t tp, tq, m0, m1, n0, n1;
          tile_ranges(a, gl.tile, BN, tp, tq, m0, m1, n0, n1);
          fix.prepare(A4, gl, n0 + q4 * 32 + lane, n1, m0, zp_stage, et);
          first_idx = idx;
          break;
        }
      }
    }
    for (int idx = 0; sched.next(a, g); ++idx) {
      fix.active = g.s0 == 0 && g.nkb > 0;
      // issuers with an MMA in the run: those of its first stage's MMAs
      // (a run with a second stage has a full first one, 16 >= NI MMAs)
      const int nmma = 4 * (g.nkb < kQuadK ? g.nkb : kQuadK);
      const uint32_t mask = nmma >= NI ? (1u << NI) - 1u : (1u << nmma) - 1u;
      if (fix.active && idx != first_idx) {
        int32_t tp, tq, m0, m1, n0, n1;
        tile_ranges(a, g.tile, BN, tp, tq, m0, m1, n0, n1);
        fix.prepare(A4, g, n0 + q4 * 32 + lane, n1, m0, zp_stage, et);
      }
      if (!epilogue_group<BN, (BN < 32 ? BN : 32), false, NI, ZpFix<BN>>(
              a, g, tmem_base, accf_bar(0), acce_bar(0), acc_iter, abort_flag, q4, lane, et, 0, 0u, ring, fix, mask))
        break;
    }
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // Let the loads still in flight land before the CTA exits: every use of a
    // buffer before its last one landed (its consumer waited for it before
    // freeing it), so only each ring's last round of uses can be pending.
    volatile int no_abort = 0;
    for (int c = w_issued > C::WST ? w_issued - C::WST : 0; c < w_issued; ++c)
      mbar_wait_bounded(full_w(c % C::WST), (c / C::WST) & 1, a.wait_limit_ns, &no_abort);
    for (int c = x_issued > C::XST ? x_issued - C::XST : 0; c < x_issued; ++c)
      mbar_wait_bounded(full_x(c % C::XST), (c / C::XST) & 1, a.wait_limit_ns, &no_abort);
  }
  // every issuer's MMAs completed before the TMEM is released
  if (warp >= kIssWarp0 && warp < kIssWarp0 + NI && lane == 0) tc_commit(teardown_bar);
  if (warp == kIssWarp0 && lane == 0) {
    volatile int no_abort = 0;
    mbar_wait_bounded(teardown_bar, 0, a.wait_limit_ns, &no_abort);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kIssWarp0) tmem_dealloc(tmem_base, 512);
}

// Activation pre-pass, K-contiguous activation: one thread per 8-element
// chunk (m, c), c fastest, so that loads and stores are coalesced 16-byte
// vectors (scalar loads when the rows are not 16-byte aligned); the chunk is
// stored K-block-major (K block c / 8 of row m at (c / 8 * M + m) * 64) with
// its elements reordered to (0,4,1,5,2,6,3,7).
__global__ void __launch_bounds__(256) int4_prep_kmajor_kernel(const uint16_t* __restrict__ A, int64_t lda, int vec,
                                                               int M, int K, int gc, uint16_t* __restrict__ Ap,
                                                               float* __restrict__ agsum) {
  pdl_launch_dependents();
  pdl_wait();
  const int chunks = K / 8;
  const int64_t total = static_cast<int64_t>(M) * chunks;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += step) {
    const int m = static_cast<int>(i / chunks);
    const int c = static_cast<int>(i - static_cast<int64_t>(m) * chunks);
    const uint16_t* src = A + static_cast<int64_t>(m) * lda + 8 * c;
    uint32_t w[4];
    if (vec) {
      const uint4 q = *reinterpret_cast<const uint4*>(src);
      w[0] = q.x;
      w[1] = q.y;
      w[2] = q.z;
      w[3] = q.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) w[e] = static_cast<uint32_t>(src[2 * e]) | (static_cast<uint32_t>(src[2 * e + 1]) << 16);
    }
    // elements e = 0..7 are the halves of w[e / 2]; the stored order is 0,4 | 1,5 | 2,6 | 3,7
    uint4 o;
    o.x = (w[0] & 0xFFFFu) | (w[2] << 16);
    o.y = (w[0] >> 16) | (w[2] & 0xFFFF0000u);
    o.z = (w[1] & 0xFFFFu) | (w[3] << 16);
    o.w = (w[1] >> 16) | (w[3] & 0xFFFF0000u);
    *reinterpret_cast<uint4*>(Ap + ((static_cast<int64_t>(c >> 3) * M + m) << 6) + 8 * (c & 7)) = o;
    if (gc) {
      // group sums: the gc (8, 16 or 32) chunks of a group are consecutive
      // lanes of this warp (chunks per row and the grid are multiples of 32,
      // so every lane is active); a butterfly gives each lane the same total
      // (element 2e of the chunk is the low half of w[e]: even k; 2e + 1 the high half: odd k)
      float se = 0.0f, so = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        se += half_bits_to_float(w[e] & 0xFFFFu);
        so += half_bits_to_float(w[e] >> 16);
      }
      for (int off = 1; off < gc; off <<= 1) {
        se += __shfl_xor_sync(0xffffffffu, se, off);
        so += __shfl_xor_sync(0xffffffffu, so, off);
      }
      if (c % gc == 0) agsum[static_cast<int64_t>(c / gc) * M + m] = se + so;
    }
  }
}

// Group sums of the prepared activation, one thread per (g, m), for the
// shapes the pre-pass does not sum itself.
__global__ void __launch_bounds__(256) int4_group_sum_kernel(const uint16_t* __restrict__ Ap, int M, int K, int group,
                                                             float* __restrict__ agsum) {
  pdl_launch_dependents();
  pdl_wait();
  const int G = K / group;
  const int64_t total = static_cast<int64_t>(G) * M;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += step) {
    const int g = static_cast<int>(i / M);
    const int m = static_cast<int>(i - static_cast<int64_t>(g) * M);
    float sum = 0.0f;
    for (int k = g * group; k < (g + 1) * group; k += 8) {
      const uint4 q = *reinterpret_cast<const uint4*>(Ap + ((static_cast<int64_t>(k >> 6) * M + m) << 6) + (k & 63));
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) sum += half_bits_to_float(w[e] & 0xFFFFu) + half_bits_to_float(w[e] >> 16);
    }
    agsum[i] = sum;
  }
}

// Same for an M-contiguous activation: one thread per (8-element K chunk, m),
// m fastest, so that each of the eight loads is coalesced across the warp.
__global__ void __launch_bounds__(256) int4_prep_mmajor_kernel(const uint16_t* __restrict__ A, int64_t lda, int M,
                                                               int K, uint16_t* __restrict__ Ap) {
  pdl_launch_dependents();
  pdl_wait();
  const int chunks = K / 8;
  const int64_t total = static_cast<int64_t>(M) * chunks;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += step) {
    const int c = static_cast<int>(i / M);
    const int m = static_cast<int>(i - static_cast<int64_t>(c) * M);
    uint16_t v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = A[static_cast<int64_t>(8 * c + e) * lda + m];
    uint4 o;
    o.x = static_cast<uint32_t>(v[0]) | (static_cast<uint32_t>(v[4]) << 16);
    o.y = static_cast<uint32_t>(v[1]) | (static_cast<uint32_t>(v[5]) << 16);
    o.z = static_cast<uint32_t>(v[2]) | (static_cast<uint32_t>(v[6]) << 16);
    o.w = static_cast<uint32_t>(v[3]) | (static_cast<uint32_t>(v[7]) << 16);
    *reinterpret_cast<uint4*>(Ap + ((static_cast<int64_t>(c >> 3) * M + m) << 6) + 8 * (c & 7)) = o;
  }
}

template <int BN>
cudaError_t launch4(const Int4Args& args, int grid, cudaStream_t stream) {
  using C = Cfg4<BN>;
  cudaError_t e = set_smem_once<int4_gemm_kernel<BN>>(static_cast<int>(C::SMEM_ALLOC));
  if (e != cudaSuccess) return e;
  return launch_pdl(int4_gemm_kernel<BN>, dim3(static_cast<unsigned>(grid)), dim3(kThreads4), C::SMEM_ALLOC,
                    stream, args);
}

// Whether the pre-pass forms the group sums in its one pass: a group's
// chunks are 8, 16 or 32 consecutive lanes of a warp.
bool int4_prep_fused(int a_mn, int K, int group) {
  const int gc = group / 8;
  return !a_mn && (gc == 8 || gc == 16 || gc == 32) && (K / 8) % 32 == 0;
}

// Offline pre-pack of the weights (layout: int4.h).  One thread per 16-byte
// chunk of codes of a block; then one per scale of a block's slots.
__global__ void __launch_bounds__(256) int4_prepack_kernel(const uint8_t* __restrict__ B, int64_t ldb,
                                                           const uint16_t* __restrict__ scales, int N, int K,
                                                           int group, int S, int block, int nslots, int64_t nblocks,
                                                           uint8_t* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t row_bytes = K / 2;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nblocks * 1024; i += step) {
    const int64_t blk = i >> 10;
    const int w = static_cast<int>(i & 1023), r = w >> 3, cout = w & 7;
    const int64_t t = blk / S, s = blk - t * S;
    const int64_t n = t * TILE_P + r;
    const int c = cout ^ (r & 7);  // the stage's chunk stored at cout
    const int64_t b0 = s * 128 + c * 16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < N && b0 < row_bytes) {
      const uint8_t* src = B + n * ldb + b0;
      if (b0 + 16 <= row_bytes) {
        v = *reinterpret_cast<const uint4*>(src);
      } else {
        uint8_t tmp[16] = {};
        for (int e = 0; b0 + e < row_bytes; ++e) tmp[e] = src[e];
        v = *reinterpret_cast<const uint4*>(tmp);
      }
    }
    *reinterpret_cast<uint4*>(out + blk * block + r * 128 + cout * 16) = v;
  }
  const int G = K / group;
  const int per = nslots * TILE_P;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nblocks * per; i += step) {
    const int64_t blk = i / per;
    const int rem = static_cast<int>(i - blk * per), slot = rem / TILE_P, r = rem - slot * TILE_P;
    const int64_t t = blk / S, s = blk - t * S;
    const int64_t n = t * TILE_P + r;
    const int64_t g = group < 256 ? s * (256 / group) + slot : (s * 256) / group;
    const uint16_t val = (n < N && g < G) ? scales[n * G + g] : static_cast<uint16_t>(0);
    reinterpret_cast<uint16_t*>(out + blk * block + kRawBytes)[slot * TILE_P + r] = val;
  }
}

}  // namespace

int pre_slots(int group) { return group < 256 ? 256 / group : 1; }
size_t pre_block_bytes(int group) { return kRawBytes + static_cast<size_t>(pre_slots(group)) * TILE_P * 2; }
// 0: no pre-packed layout for these sizes (a group that is not positive, or
// sizes past the kernel's 32-bit row and column indices).
size_t pre_total_bytes(int64_t N, int64_t K, int group) {
  if (N <= 0 || K <= 0 || group <= 0 || N > INT32_MAX || K > INT32_MAX) return 0;
  return static_cast<size_t>((N + TILE_P - 1) / TILE_P) * static_cast<size_t>((K + 255) / 256) * pre_block_bytes(group);
}

cudaError_t launch_int4_prepack(const void* B, int64_t ldb, const void* scales, int64_t N, int64_t K, int group,
                                void* out, cudaStream_t stream) {
  if (pre_total_bytes(N, K, group) == 0) return cudaErrorInvalidValue;
  const int S = static_cast<int>((K + 255) / 256);
  const int64_t nblocks = (N + TILE_P - 1) / TILE_P * S;
  if (nblocks == 0) return cudaSuccess;
  const int64_t want = nblocks * 1024 / 256;
  const int grid = static_cast<int>(want < 65535 ? (want > 0 ? want : 1) : 65535);
  return launch_pdl(int4_prepack_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, stream,
                    static_cast<const uint8_t*>(B), ldb, static_cast<const uint16_t*>(scales), static_cast<int>(N),
                    static_cast<int>(K), group, S, static_cast<int>(pre_block_bytes(group)), pre_slots(group), nblocks,
                    static_cast<uint8_t*>(out));
}

cudaError_t launch_int4_prep(const void* A, int64_t lda, int a_mn, int M, int K, int group, void* Ap, float* agsum,
                             int sms, cudaStream_t stream) {
  const int64_t chunks = static_cast<int64_t>(M) * (K / 8);
  if (chunks == 0) return cudaSuccess;
  int64_t blocks = (chunks + 255) / 256;
  if (blocks > static_cast<int64_t>(sms) * 8) blocks = static_cast<int64_t>(sms) * 8;
  // the pre-pass sums groups itself when a group's chunks are 8, 16 or 32
  // consecutive lanes of a warp: K-contiguous A, 32 | K / 8, and a grid of
  // whole warps with every lane in range
  const int gc = group / 8;
  const bool fused = int4_prep_fused(a_mn, K, group);
  if (!a_mn) {
    const int vec = (lda % 8 == 0) && (reinterpret_cast<uintptr_t>(A) % 16 == 0);
    cudaError_t e = launch_pdl(int4_prep_kmajor_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                               static_cast<const uint16_t*>(A), lda, vec, M, K, fused ? gc : 0,
                               static_cast<uint16_t*>(Ap), agsum);
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e = launch_pdl(int4_prep_mmajor_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                               static_cast<const uint16_t*>(A), lda, M, K, static_cast<uint16_t*>(Ap));
    if (e != cudaSuccess) return e;
  }
  if (!fused) {
    const int64_t gm = static_cast<int64_t>(M) * (K / group);
    int64_t gblocks = (gm + 255) / 256;
    if (gblocks > static_cast<int64_t>(sms) * 8) gblocks = static_cast<int64_t>(sms) * 8;
    cudaError_t e = launch_pdl(int4_group_sum_kernel, dim3(static_cast<unsigned>(gblocks)), dim3(256), 0, stream,
                               static_cast<const uint16_t*>(Ap), M, K, group, agsum);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_int4_gemm(const Int4Args& args, int bn, int grid, cudaStream_t stream) {
  switch (bn) {
    case 16: return launch4<16>(args, grid, stream);
    case 32: return launch4<32>(args, grid, stream);
    case 64: return launch4<64>(args, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lgt
