// int4-weight GEMM with the dequantisation inside the mainloop.
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
// Expansion.  A 32-bit word of codes q0..q7 (and the word shifted right by
// 8) gives the fp16 pairs of codes (0,4), (1,5), (2,6), (3,7) with one LOP3
// each: a code in bits 0..3 of a half ORed into 0x6400 is the fp16 number
// 1024 + q, a code in bits 4..7 ORed into 0x5400 is 64 + q (the mantissa's
// unit there is 1/16).  One packed subtraction of that offset gives q
// exactly, and one packed FMA q * s + (-z * s) gives the weight: -z * s is
// rounded to fp16 once per (row, group), the FMA rounds once more, so the
// weight is within one fp16 rounding of z * s of (q - z) * s.
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
// row segments keep the TMA stream near the HBM rate) plus one activation box
// per K block.  The accumulator of a run is double-buffered in TMEM, so the
// epilogue of one run overlaps the next; a run's epilogue (C, or the split-K
// partial and the arrival protocol) is the one of the dense kernels.
//
// Warp roles (448 threads):
//   warp 0       TMA producer.
//   warp 1       TMEM allocator and MMA issuer: waits for an expanded slot,
//                issues the stage's MMAs, frees the slot.
//   warps 2..5   epilogue (TMEM lane quadrant warp % 4).
//   warps 6..13  expanders: two warps per TMEM lane quadrant, alternating
//                stages; each thread owns one weight row of the tile.
#include "kernels.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lgt {
namespace {

constexpr int kThreads4 = 448;
constexpr int kEpiWarp04 = 2;
constexpr int kExpWarp0 = 6;
constexpr int kQuadK = 4;                     // K blocks per stage
constexpr uint32_t kRawBytes = TILE_P * 128;  // 128 rows x 128 bytes (256 codes)
constexpr int kTSlots = 3;                    // TMEM A slots of 128 columns
constexpr uint32_t kASlotCol0 = 128;          // A slots at [128, 512); the accumulators below

template <int BN>
struct Cfg4 {
  static constexpr uint32_t ACT_TILE = BN * TILE_K * 2;  // one 64-deep activation box
  static constexpr uint32_t STAGE_BYTES = kRawBytes + kQuadK * ACT_TILE;
  static constexpr int STAGES_RAW = (192 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  // barriers: full[S], sfree[S], a_full[T], tfree[T], accf[2], acce[2], teardown
  static constexpr uint32_t EPI_OFF = STAGES * STAGE_BYTES;
  static constexpr uint32_t BAR_OFF = EPI_OFF + EPI_STAGING_BYTES;
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 2 * kTSlots + 5;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr uint32_t SMEM_ALLOC = MISC_OFF + 64 + 1024;  // slack for 1024-byte alignment
  static_assert(STAGE_BYTES % 1024 == 0 && ACT_TILE % 1024 == 0, "swizzled buffers stay 1024-byte aligned");
  static_assert(STAGES > kTSlots, "a stage buffer outlives the TMEM slot cycle (sfree protocol)");
  static_assert(2 * BN <= static_cast<int>(kASlotCol0), "accumulators fit below the A slots");
  static_assert(kASlotCol0 + kTSlots * 128 <= 512, "A slots fit in the TMEM allocation");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
  return d;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ void tc_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

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

// One weight row's scales and zero points, eight groups (16 bytes) at a time,
// the next eight loaded while the current ones are in use.
struct RowScales {
  const uint16_t* srow = nullptr;
  const uint16_t* zrow = nullptr;
  int groups = 0, win = -1;
  bool vec = true;  // rows readable 16 bytes at a time; otherwise one load per group
  uint4 s_cur, z_cur, s_nxt, z_nxt;
  __device__ void fetch(int w, uint4& sv, uint4& zv) const {
    if (w * 8 < groups) {
      sv = __ldg(reinterpret_cast<const uint4*>(srow) + w);
      if (zrow) zv = __ldg(reinterpret_cast<const uint4*>(zrow) + w);
    }
  }
  __device__ void reset(const uint16_t* s, const uint16_t* z, int ngroups, int first_group, bool vectors) {
    srow = s;
    zrow = z;
    groups = ngroups;
    vec = vectors;
    const uint4 eight = make_uint4(0x48004800u, 0x48004800u, 0x48004800u, 0x48004800u);  // fp16 8.0
    s_cur = s_nxt = make_uint4(0u, 0u, 0u, 0u);
    z_cur = z_nxt = eight;
    win = first_group >> 3;
    if (srow && vec) {
      fetch(win, s_cur, z_cur);
      fetch(win + 1, s_nxt, z_nxt);
    }
  }
  // fp16 bits of (s, z) of group g (g >= the previous call's group)
  __device__ void get(int g, uint16_t& sb, uint16_t& zb) {
    if (!vec) {
      sb = srow ? __ldg(srow + g) : static_cast<uint16_t>(0);
      zb = zrow ? __ldg(zrow + g) : (srow ? static_cast<uint16_t>(0x4800) : static_cast<uint16_t>(0));
      return;
    }
    const int w = g >> 3;
    if (w != win && srow) {
      if (w == win + 1) {
        s_cur = s_nxt;
        z_cur = z_nxt;
      } else {
        fetch(w, s_cur, z_cur);
      }
      win = w;
      fetch(w + 1, s_nxt, z_nxt);
    }
    const int j = g & 7;
    const uint32_t sw = (j >> 1) == 0 ? s_cur.x : (j >> 1) == 1 ? s_cur.y : (j >> 1) == 2 ? s_cur.z : s_cur.w;
    const uint32_t zw = (j >> 1) == 0 ? z_cur.x : (j >> 1) == 1 ? z_cur.y : (j >> 1) == 2 ? z_cur.z : z_cur.w;
    sb = static_cast<uint16_t>((j & 1) ? (sw >> 16) : (sw & 0xFFFFu));
    zb = static_cast<uint16_t>((j & 1) ? (zw >> 16) : (zw & 0xFFFFu));
  }
};

template <int BN>
__global__ void __launch_bounds__(kThreads4, 1) int4_gemm_kernel(const __grid_constant__ Int4Args A4) {
  using C = Cfg4<BN>;
  const TcArgs& a = A4.t;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = base + C::BAR_OFF;
  // full[s]: stage s's TMA bytes landed.  sfree[s]: stage s may be refilled
  // (its expanders read its raw bytes, and the expanders of the stage that
  // reuses its TMEM slot saw that slot freed, i.e. the MMAs that read its
  // activation completed; that saves the MMA issuer a commit per stage).
  // a_full[t]: the expanders wrote a stage's weights into TMEM A slot t.
  // tfree[t]: the MMAs reading slot t completed.  accf / acce: accumulator
  // buffer full / drained.
  auto full_bar = [&](int i) { return bar0 + 8u * i; };
  auto sfree_bar = [&](int i) { return bar0 + 8u * (C::STAGES + i); };
  auto a_full = [&](int t) { return bar0 + 8u * (2 * C::STAGES + t); };
  auto tfree_bar = [&](int t) { return bar0 + 8u * (2 * C::STAGES + kTSlots + t); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 * kTSlots + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 * kTSlots + 2 + b); };
  const uint32_t teardown_bar = bar0 + 8u * (2 * C::STAGES + 2 * kTSlots + 4);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  volatile int* consumed_slot = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 8);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(sfree_bar(i), 4 + 4);  // the stage's four expander warps + the four of the stage 3 later
    }
    for (int t = 0; t < kTSlots; ++t) {
      mbar_init(a_full(t), 4);
      mbar_init(tfree_bar(t), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), kEpiThreads / 32);
    }
    mbar_init(teardown_bar, 1);
    *abort_flag = 0;
    *consumed_slot = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&A4.tm_w);
    tma_prefetch_desc(&a.tm_q);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int issued = 0;  // producer lane: stages whose loads were issued

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      StageIter it(a);
      int kb0, nk, st = 0;
      bool nr;
      while (it.next(a, kb0, nk, nr)) {
        const int s = st % C::STAGES;
        if (!mbar_wait_bounded(sfree_bar(s), ((st / C::STAGES) & 1) ^ 1u, a.wait_limit_ns, abort_flag)) {
          if (!*abort_flag) record_timeout(a, abort_flag, 0 * 16 + 1);
          break;
        }
        int32_t tp, tq, m0, m1, n0, n1;
        tile_ranges(a, it.g.tile, BN, tp, tq, m0, m1, n0, n1);
        const uint32_t sb = base + s * C::STAGE_BYTES;
        const int32_t k0 = (it.g.kb0 + kb0) * TILE_K;
        mbar_arrive_expect_tx(full_bar(s), kRawBytes + nk * C::ACT_TILE);
        tma_load_2d(sb, &A4.tm_w, full_bar(s), k0 / 2, n0);
        for (int j = 0; j < nk; ++j)
          tma_load_2d(sb + kRawBytes + j * C::ACT_TILE, &a.tm_q, full_bar(s), k0 + j * TILE_K, m0);
        ++issued;
        ++st;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      StageIter it(a);
      int kb0, nk, st = 0, acc_iter = -1;
      bool nr, ok = true;
      uint32_t d_tmem = tmem_base;
      while (ok && it.next(a, kb0, nk, nr)) {
        const int s = st % C::STAGES, t = st % kTSlots;
        if (nr) {
          ++acc_iter;
          const int buf = acc_iter & 1;
          if (!mbar_wait_bounded(acce_bar(buf), ((acc_iter >> 1) & 1) ^ 1u, a.wait_limit_ns, abort_flag)) {
            if (!*abort_flag) record_timeout(a, abort_flag, 1 * 16 + 3);
            break;
          }
          d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        }
        if (!mbar_wait_bounded(a_full(t), (st / kTSlots) & 1, a.wait_limit_ns, abort_flag)) {
          if (!*abort_flag) record_timeout(a, abort_flag, 1 * 16 + 0);
          break;
        }
        *consumed_slot = st + 1;
        tc_fence_after();
        const uint64_t bd0 = sw128_desc(base + s * C::STAGE_BYTES + kRawBytes, 16u, 1024u);
        const uint32_t a0 = tmem_base + kASlotCol0 + static_cast<uint32_t>(t * 128);
#pragma unroll
        for (int j = 0; j < kQuadK; ++j) {
          if (j < nk) {
            const uint64_t bd = bd0 + static_cast<uint64_t>((j * C::ACT_TILE) >> 4);
            const uint32_t at = a0 + static_cast<uint32_t>(j * 32);
            // columns 8 per K = 16 (fp16 pairs), descriptor +32 bytes per K = 16
            tc_mma_f16_ts(d_tmem, at, bd, a.idesc, (kb0 + j) != 0 ? 1u : 0u);
            tc_mma_f16_ts(d_tmem, at + 8, bd + 2, a.idesc, 1u);
            tc_mma_f16_ts(d_tmem, at + 16, bd + 4, a.idesc, 1u);
            tc_mma_f16_ts(d_tmem, at + 24, bd + 6, a.idesc, 1u);
          }
        }
        tc_commit(tfree_bar(t));
        if (kb0 + nk == it.g.nkb) tc_commit(accf_bar(acc_iter & 1));
        ++st;
      }
      (void)ok;
    }
  } else if (warp >= kExpWarp0) {
    // ------------------------------------------------------------ expanders
    const int q4 = warp & 3;
    const int h = (warp - kExpWarp0) >> 2;  // stages with index % 2 == h
    const int r = q4 * 32 + lane;           // weight row within the tile (TMEM lane)
    StageIter it(a);
    RowScales rs;
    int kb0, nk, st = 0;
    bool nr;
    while (it.next(a, kb0, nk, nr)) {
      if (nr) {
        int32_t tp, tq, m0, m1, n0, n1;
        tile_ranges(a, it.g.tile, BN, tp, tq, m0, m1, n0, n1);
        const int n = n0 + r;
        const bool row_ok = n < n1;
        const int g0 = static_cast<int>(magic_div(static_cast<uint32_t>(it.g.kb0), A4.div_kb_per_group));
        rs.reset(row_ok ? A4.scales + static_cast<int64_t>(n) * A4.groups : nullptr,
                 (row_ok && A4.zeros) ? A4.zeros + static_cast<int64_t>(n) * A4.groups : nullptr, A4.groups, g0,
                 A4.vec_sz != 0);
      }
      if ((st & 1) == h) {
        const int s = st % C::STAGES, t = st % kTSlots;
        const bool got =
            mbar_wait_bounded(full_bar(s), (st / C::STAGES) & 1, a.wait_limit_ns, abort_flag) &&
            mbar_wait_bounded(tfree_bar(t), ((st / kTSlots) & 1) ^ 1u, a.wait_limit_ns, abort_flag);
        if (!got && !*abort_flag) record_timeout(a, abort_flag, 3 * 16 + 0);
        // the warp leaves together (tcgen05.st below needs every lane)
        if (!__all_sync(0xffffffffu, got)) break;
        tc_fence_after();
        // the MMAs of stage st - kTSlots completed: its stage buffer may be refilled
        if (st >= kTSlots && lane == 0) mbar_arrive(sfree_bar((st - kTSlots) % C::STAGES));
        // raw row r: eight 16-byte chunks, chunk c stored at c ^ (r mod 8) (128-byte swizzle)
        const uint8_t* rowp = smem + s * C::STAGE_BYTES + r * 128;
        uint4 raw[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) raw[c] = *reinterpret_cast<const uint4*>(rowp + ((c ^ (r & 7)) << 4));
        __syncwarp();
        if (lane == 0) mbar_arrive(sfree_bar(s));
        const uint32_t slot = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + kASlotCol0 +
                              static_cast<uint32_t>(t * 128);
        for (int j = 0; j < nk; ++j) {
          const int grp =
              static_cast<int>(magic_div(static_cast<uint32_t>(it.g.kb0 + kb0 + j), A4.div_kb_per_group));
          uint16_t sb, zb;
          rs.get(grp, sb, zb);
          const uint32_t s2 = static_cast<uint32_t>(sb) * 0x10001u;
          const uint32_t nzs2 = hmul2(static_cast<uint32_t>(zb) * 0x10001u, s2) ^ 0x80008000u;  // -z * s
          const uint32_t words[8] = {raw[2 * j].x, raw[2 * j].y, raw[2 * j].z, raw[2 * j].w,
                                     raw[2 * j + 1].x, raw[2 * j + 1].y, raw[2 * j + 1].z, raw[2 * j + 1].w};
          uint32_t vals[32];
#pragma unroll
          for (int w8 = 0; w8 < 8; ++w8) {
            const uint32_t lo = words[w8], hi = lo >> 8;
            // codes (p, p + 4) of the word for p = 0..3, then q * s - z * s
            const uint32_t q0 = hsub2(lop3_and_or(lo, 0x000F000Fu, 0x64006400u), 0x64006400u);
            const uint32_t q1 = hsub2(lop3_and_or(lo, 0x00F000F0u, 0x54005400u), 0x54005400u);
            const uint32_t q2 = hsub2(lop3_and_or(hi, 0x000F000Fu, 0x64006400u), 0x64006400u);
            const uint32_t q3 = hsub2(lop3_and_or(hi, 0x00F000F0u, 0x54005400u), 0x54005400u);
            vals[4 * w8 + 0] = hfma2(q0, s2, nzs2);
            vals[4 * w8 + 1] = hfma2(q1, s2, nzs2);
            vals[4 * w8 + 2] = hfma2(q2, s2, nzs2);
            vals[4 * w8 + 3] = hfma2(q3, s2, nzs2);
          }
          tc_st_32x32b_x32(slot + static_cast<uint32_t>(j * 32), vals);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(a_full(t));
      }
      ++st;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;
    const int et = threadIdx.x - kEpiWarp04 * 32;
    Sched sched(a);
    Group g;
    int acc_iter = 0, ring = 0;
    const uint32_t stage_smem = base + C::EPI_OFF + static_cast<uint32_t>(warp - kEpiWarp04) * 8192u;
    while (sched.next(a, g)) {
      if (!epilogue_group<BN, (BN < 32 ? BN : 32)>(a, g, tmem_base, accf_bar(0), acce_bar(0), acc_iter, abort_flag,
                                                   q4, lane, et, 0, stage_smem, ring))
        break;
    }
    if (lane == 0) bulk_wait_group<0>();
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // Let the loads still in flight land before the CTA exits.
    volatile int no_abort = 0;
    for (int c = *consumed_slot; c < issued; ++c)
      mbar_wait_bounded(full_bar(c % C::STAGES), (c / C::STAGES) & 1, a.wait_limit_ns, &no_abort);
  }
  if (warp == 1 && lane == 0) {
    volatile int no_abort = 0;
    tc_commit(teardown_bar);
    mbar_wait_bounded(teardown_bar, 0, a.wait_limit_ns, &no_abort);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// Activation pre-pass, K-contiguous activation: one thread per 8-element
// chunk (m, c), c fastest, so that loads and stores are coalesced 16-byte
// vectors (scalar loads when the rows are not 16-byte aligned); the chunk is
// stored with its elements reordered to (0,4,1,5,2,6,3,7).
__global__ void __launch_bounds__(256) int4_prep_kmajor_kernel(const uint16_t* __restrict__ A, int64_t lda, int vec,
                                                               int M, int K, uint16_t* __restrict__ Ap) {
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
    *reinterpret_cast<uint4*>(Ap + static_cast<int64_t>(m) * K + 8 * c) = o;
  }
}

// Same for an M-contiguous activation: one thread per (8-element K chunk, m),
// m fastest, so that each of the eight loads is coalesced across the warp.
__global__ void __launch_bounds__(256) int4_prep_mmajor_kernel(const uint16_t* __restrict__ A, int64_t lda, int M,
                                                               int K, uint16_t* __restrict__ Ap) {
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
    *reinterpret_cast<uint4*>(Ap + static_cast<int64_t>(m) * K + 8 * c) = o;
  }
}

template <int BN>
cudaError_t launch4(const Int4Args& args, int grid, cudaStream_t stream) {
  using C = Cfg4<BN>;
  cudaError_t e = cudaFuncSetAttribute(int4_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM_ALLOC));
  if (e != cudaSuccess) return e;
  int4_gemm_kernel<BN><<<grid, kThreads4, C::SMEM_ALLOC, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_int4_prep(const void* A, int64_t lda, int a_mn, int M, int K, void* Ap, int sms,
                             cudaStream_t stream) {
  const int64_t chunks = static_cast<int64_t>(M) * (K / 8);
  if (chunks == 0) return cudaSuccess;
  int64_t blocks = (chunks + 255) / 256;
  if (blocks > static_cast<int64_t>(sms) * 8) blocks = static_cast<int64_t>(sms) * 8;
  if (!a_mn) {
    const int vec = (lda % 8 == 0) && (reinterpret_cast<uintptr_t>(A) % 16 == 0);
    int4_prep_kmajor_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(static_cast<const uint16_t*>(A), lda, vec,
                                                                          M, K, static_cast<uint16_t*>(Ap));
  } else {
    int4_prep_mmajor_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(static_cast<const uint16_t*>(A), lda, M,
                                                                          K, static_cast<uint16_t*>(Ap));
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
