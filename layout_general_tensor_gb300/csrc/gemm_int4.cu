// int4-weight GEMM with the dequantisation inside the mainloop.
//
//   C[m,n] = sum_k A[m,k] * w(k,n),  w(k,n) = (q(n,k) - z(n,g)) * s(n,g),
//   g = k / group_size, codes two per byte (low nibble = even k).
//
// Within one quantisation group the scale and zero point are constants of the
// weight row, so the sum splits per group g:
//   sum_{k in g} A[m,k] (q(n,k) - z) s = s * ( D_g[n,m] - (1024 + z) * S_g[m] ),
//   D_g[n,m] = sum_{k in g} (1024 + q(n,k)) * A[m,k],  S_g[m] = sum_{k in g} A[m,k].
// 1024 + q is exactly the fp16 number whose bits are 0x6400 | q, so the
// mainloop expands nibbles to fp16 with one LOP3 per pair of codes and no
// floating-point work; the tensor cores form D_g (exact products, fp32 sums)
// and the epilogue applies s and z once per (row, group) in fp32.
//
// The weight is the large operand and the activation the skinny one, so the
// MMA runs swapped: 128 weight rows (n) on the MMA's M side, the activation
// rows (m) on its N side, the accumulator holding C^T in TMEM.
//
// A small pre-pass (int4_prep_kernel) copies the activation into the
// workspace K-contiguous, with the eight elements of every 8-element group
// of K reordered to match the order in which one 32-bit word of codes
// expands (codes 0,4 | 1,5 | 2,6 | 3,7), and writes the per-64-K row sums
// S used above.
//
// A pipeline stage is up to four 64-deep K blocks of one run: the packed
// weight arrives as one TMA box of 128 rows x 128 bytes (128-byte swizzle; wide
// row segments keep the TMA stream near the HBM rate, 32-byte ones cap it at a
// third of it) plus one activation box per K block.
//
// Warp roles of the main kernel (480 threads):
//   warp 0       TMA producer.
//   warp 1       MMA issuer (and TMEM allocator): the expanded weight tile is
//                the MMA's A operand *in TMEM*, the activation its B operand in
//                shared memory; one TMEM accumulator per group segment.
//   warps 2..9   expanders: two warps per TMEM lane quadrant, alternating
//                stages.  Each thread owns one weight row: eight 16-byte shared
//                loads (conflict-free thanks to the swizzle), 3 shifts and 4
//                LOP3 per 8 codes, one tcgen05.st of 32 columns per K block.
//   warps 10..13 epilogue: per group segment, tcgen05.ld the accumulator and
//                fold in s and z; at the end of a run, store C or add the fp32
//                partial to the split-K workspace (shared arrival protocol).
//   warp 14      waiter: performs every mbarrier wait the MMA issuer needs and
//                hands it each ready stage through a named barrier.  An
//                mbarrier wait executed while MMAs are in flight stalls until
//                they drain; the named barrier does not, so the issuer only
//                issues MMAs and commits and the tensor core stays fed.
//
// The dequantise copy of the BitBLAS TileLang page (the thread-level TIR
// listing in "Relevant Issues") decomposes a flat index into (vj, vk, vjj, vkk)
// to vectorise loads of the packed weight; here the TMA box does that
// addressing and each thread's loads are 128-bit.
#include "kernels.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lgt {
namespace {

constexpr int kThreads4 = 480;
constexpr int kDequantWarp0 = 2;
constexpr int kEpiWarp04 = 10;
constexpr int kWaiterWarp = 14;
constexpr int kQuadK = 4;                     // K blocks per stage
constexpr uint32_t kRawBytes = TILE_P * 128;  // 128 rows x 128 bytes (256 codes)
constexpr int kTSlots = 3;                    // TMEM A slots of 128 columns
constexpr uint32_t kASlotCol0 = 128;          // A slots at [128, 512); segment accumulators below
constexpr uint32_t kBarStage = 2;             // named barrier: waiter warp <-> MMA warp
constexpr int kGsumChunk = 64;                // groups of activation row sums staged in shared memory

template <int BN>
struct Cfg4 {
  static constexpr uint32_t ACT_TILE = BN * TILE_K * 2;  // one 64-deep activation box
  static constexpr uint32_t STAGE_BYTES = kRawBytes + kQuadK * ACT_TILE;
  static constexpr int STAGES_RAW = (192 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int NSEG = (128 / BN) > 8 ? 8 : (128 / BN);  // segment accumulators in TMEM
  // barriers: full[S], sfree[S], a_full[T], tfree[T], d_full[NSEG], d_empty[NSEG], teardown
  static constexpr uint32_t BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 2 * kTSlots + 2 * NSEG + 1;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr uint32_t GSUM_OFF = ((MISC_OFF + 64 + 15) / 16) * 16;  // staged group row sums
  static constexpr uint32_t SMEM_ALLOC = GSUM_OFF + kGsumChunk * BN * 4 + 1024;
  static_assert(STAGE_BYTES % 1024 == 0 && ACT_TILE % 1024 == 0, "swizzled buffers stay 1024-byte aligned");
  static_assert(STAGES >= 2, "at least two shared-memory stages");
  static_assert(NSEG * BN <= static_cast<int>(kASlotCol0), "accumulators fit below the A slots");
  static_assert(kASlotCol0 + kTSlots * 128 <= 512, "A slots fit in the TMEM allocation");
  static_assert(BN <= 64, "per-thread fp32 accumulators: at most 64 activation rows per tile");
};

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
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

// End (exclusive) of the run's K blocks that share the quantisation group of
// block kb.
__device__ __forceinline__ int segment_end(const Int4Args& A4, const Group& g, int kb) {
  const uint32_t grp = magic_div(static_cast<uint32_t>(g.kb0 + kb), A4.div_kb_per_group);
  const int next_group_kb = static_cast<int>((grp + 1) * A4.div_kb_per_group.d) - g.kb0;
  return min(g.nkb, next_group_kb);
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

// Group segments of the K blocks, in order: which TMEM accumulator buffer a
// block accumulates into and whether it opens / closes its segment.
template <int NSEG>
struct SegTracker {
  int seg_end = 0, nseg = 0, buf = 0;
  __device__ void new_run() { seg_end = 0; }
  __device__ void step(const Int4Args& A4, const Group& g, int kb, bool& start, bool& last, int& b, uint32_t& ph) {
    start = (kb == seg_end);
    ph = 0;
    if (start) {
      seg_end = segment_end(A4, g, kb);
      buf = nseg % NSEG;
      ph = static_cast<uint32_t>((nseg / NSEG) & 1);
      ++nseg;
    }
    b = buf;
    last = (kb + 1 == seg_end);
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
  // (its raw bytes were read by the expanders and the MMAs that read its
  // activation completed).  a_full[t]: the expanders wrote the stage's weights
  // into TMEM A slot t.  tfree[t]: the MMAs reading slot t completed.
  auto full_bar = [&](int i) { return bar0 + 8u * i; };
  auto sfree_bar = [&](int i) { return bar0 + 8u * (C::STAGES + i); };
  auto a_full = [&](int t) { return bar0 + 8u * (2 * C::STAGES + t); };
  auto tfree_bar = [&](int t) { return bar0 + 8u * (2 * C::STAGES + kTSlots + t); };
  auto d_full = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 * kTSlots + b); };
  auto d_empty = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 * kTSlots + C::NSEG + b); };
  const uint32_t teardown_bar = bar0 + 8u * (2 * C::STAGES + 2 * kTSlots + 2 * C::NSEG);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(sfree_bar(i), 4 + 1);  // the stage's four expander warps + the MMA's commit
    }
    for (int t = 0; t < kTSlots; ++t) {
      mbar_init(a_full(t), 4);
      mbar_init(tfree_bar(t), 1);
    }
    for (int b = 0; b < C::NSEG; ++b) {
      mbar_init(d_full(b), 1);
      mbar_init(d_empty(b), kEpiThreads / 32);
    }
    mbar_init(teardown_bar, 1);
    *abort_flag = 0;
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

  int issued = 0;

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
    StageIter it(a);
    SegTracker<C::NSEG> sg;
    int kb0, nk, st = 0;
    bool nr;
    while (it.next(a, kb0, nk, nr)) {
      // the waiter warp has checked every barrier of this stage
      if (named_bar_or(kBarStage, 64, false)) break;
      if (lane == 0) {
        if (nr) sg.new_run();
        const int s = st % C::STAGES, t = st % kTSlots;
        // operands of the stage's K blocks first, then the MMAs back to back
        // and the commits after them (segment hand-offs at the end of the
        // stage are only a few hundred cycles later)
        const uint64_t bd0 = sw128_desc(base + s * C::STAGE_BYTES + kRawBytes, 16u, 1024u);
        const uint32_t a0 = tmem_base + kASlotCol0 + static_cast<uint32_t>(t * 128);
        uint32_t dcol[kQuadK];
        uint32_t first = 0, closes = 0;  // bit j: K block j opens / closes its segment
#pragma unroll
        for (int j = 0; j < kQuadK; ++j) {
          if (j < nk) {
            bool start, last;
            int buf;
            uint32_t ph;
            sg.step(A4, it.g, kb0 + j, start, last, buf, ph);
            dcol[j] = static_cast<uint32_t>(buf * BN);
            first |= (start ? 1u : 0u) << j;
            closes |= (last ? 1u : 0u) << j;
          } else {
            dcol[j] = 0;
          }
        }
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < kQuadK; ++j) {
          if (j < nk) {
            const uint64_t bd = bd0 + static_cast<uint64_t>((j * C::ACT_TILE) >> 4);
            const uint32_t at = a0 + static_cast<uint32_t>(j * 32);
            const uint32_t d_tmem = tmem_base + dcol[j];
            tc_mma_f16_ts(d_tmem, at, bd, a.idesc, ((first >> j) & 1u) ? 0u : 1u);
            tc_mma_f16_ts(d_tmem, at + 8, bd + 2, a.idesc, 1u);
            tc_mma_f16_ts(d_tmem, at + 16, bd + 4, a.idesc, 1u);
            tc_mma_f16_ts(d_tmem, at + 24, bd + 6, a.idesc, 1u);
          }
        }
#pragma unroll
        for (int j = 0; j < kQuadK; ++j)
          if (j < nk && ((closes >> j) & 1u)) tc_commit(d_full(static_cast<int>(dcol[j] / BN)));
        tc_commit(sfree_bar(s));
        tc_commit(tfree_bar(t));
      }
      ++st;
    }
  } else if (warp == kWaiterWarp) {
    // ------------------------------------------------------------ waiter
    StageIter it(a);
    SegTracker<C::NSEG> sg;
    int kb0, nk, st = 0;
    bool nr;
    bool failed = false;
    while (it.next(a, kb0, nk, nr)) {
      if (lane == 0 && !failed) {
        if (nr) sg.new_run();
        const int t = st % kTSlots;
        bool ok = mbar_wait_bounded(a_full(t), (st / kTSlots) & 1, a.wait_limit_ns, abort_flag);
        for (int j = 0; j < nk && ok; ++j) {
          bool start, last;
          int buf;
          uint32_t ph;
          sg.step(A4, it.g, kb0 + j, start, last, buf, ph);
          if (start) ok = mbar_wait_bounded(d_empty(buf), ph ^ 1u, a.wait_limit_ns, abort_flag);
        }
        if (!ok) {
          if (!*abort_flag) record_timeout(a, abort_flag, 1 * 16 + 0);
          failed = true;
        }
      }
      // a_full implies the stage's TMA bytes landed: the expanders observed
      // full[s] before publishing a_full[t]
      if (named_bar_or(kBarStage, 64, failed)) break;
      ++st;
    }
  } else if (warp < kEpiWarp04) {
    // ------------------------------------------------------------ expanders
    const int q4 = warp & 3;
    const int h = (warp - kDequantWarp0) >> 2;  // stages with index % 2 == h
    const int r = q4 * 32 + lane;               // weight row within the tile (TMEM lane)
    StageIter it(a);
    int kb0, nk, st = 0;
    bool nr;
    while (it.next(a, kb0, nk, nr)) {
      if ((st & 1) == h) {
        const int s = st % C::STAGES, t = st % kTSlots;
        const bool got =
            mbar_wait_bounded(full_bar(s), (st / C::STAGES) & 1, a.wait_limit_ns, abort_flag) &&
            mbar_wait_bounded(tfree_bar(t), ((st / kTSlots) & 1) ^ 1u, a.wait_limit_ns, abort_flag);
        if (!got && !*abort_flag) record_timeout(a, abort_flag, 3 * 16 + 0);
        // the warp leaves together (tcgen05.st below needs every lane)
        if (!__all_sync(0xffffffffu, got)) break;
        tc_fence_after();
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
          const uint32_t words[8] = {raw[2 * j].x, raw[2 * j].y, raw[2 * j].z, raw[2 * j].w,
                                     raw[2 * j + 1].x, raw[2 * j + 1].y, raw[2 * j + 1].z, raw[2 * j + 1].w};
          uint32_t vals[32];
#pragma unroll
          for (int w8 = 0; w8 < 8; ++w8) {
            // codes (0,4), (1,5), (2,6), (3,7) of the word as fp16 pairs 1024 + q
            const uint32_t w = words[w8];
            vals[4 * w8 + 0] = lop3_and_or(w, 0x000F000Fu, 0x64006400u);
            vals[4 * w8 + 1] = lop3_and_or(w >> 4, 0x000F000Fu, 0x64006400u);
            vals[4 * w8 + 2] = lop3_and_or(w >> 8, 0x000F000Fu, 0x64006400u);
            vals[4 * w8 + 3] = lop3_and_or(w >> 12, 0x000F000Fu, 0x64006400u);
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
    const int r = q4 * 32 + lane;
    float* gs_smem = reinterpret_cast<float*>(smem + C::GSUM_OFF);  // [kGsumChunk][BN]
    const int kpg = static_cast<int>(A4.div_kb_per_group.d);
    Sched sched(a);
    Group g;
    int seg = 0;
    bool ok = true;
    int gs_first = -(1 << 30), gs_m0 = -1;  // staged chunk: groups [gs_first, +kGsumChunk) of rows m0..
    while (ok && sched.next(a, g)) {
      int32_t tp, tq, m0, m1, n0, n1;
      tile_ranges(a, g.tile, BN, tp, tq, m0, m1, n0, n1);
      const int n = n0 + r;
      const bool row_ok = n < n1;
      const uint16_t* srow = A4.scales + static_cast<int64_t>(row_ok ? n : 0) * A4.groups;
      const uint16_t* zrow = A4.zeros ? A4.zeros + static_cast<int64_t>(row_ok ? n : 0) * A4.groups : nullptr;
      float acc[BN];
#pragma unroll
      for (int j = 0; j < BN; ++j) acc[j] = 0.0f;
      // This row's scales and zero points, 8 groups (16 bytes) per load, the
      // next window loaded while the current one is in use.
      int win = -1, win_nxt = -1;
      uint4 s_cur = make_uint4(0, 0, 0, 0), s_nxt = s_cur;
      uint4 z_cur = make_uint4(0x48004800u, 0x48004800u, 0x48004800u, 0x48004800u), z_nxt = z_cur;  // fp16 8.0
      auto fetch_window = [&](int w, uint4& sv, uint4& zv) {
        if (row_ok && w * 8 < A4.groups) {
          sv = __ldg(reinterpret_cast<const uint4*>(srow) + w);
          if (zrow) zv = __ldg(reinterpret_cast<const uint4*>(zrow) + w);
        }
      };
      int kb = 0;
      while (kb < g.nkb) {
        const int end = segment_end(A4, g, kb);
        const uint32_t grp = magic_div(static_cast<uint32_t>(g.kb0 + kb), A4.div_kb_per_group);
        // scale and zero point of (row, group)
        uint16_t sb = 0, zb = 0x4800;
        if (A4.vec_sz) {
          const int w = static_cast<int>(grp >> 3);
          if (w != win) {
            if (w == win_nxt) {
              s_cur = s_nxt;
              z_cur = z_nxt;
            } else {
              fetch_window(w, s_cur, z_cur);
            }
            win = w;
            win_nxt = w + 1;
            fetch_window(win_nxt, s_nxt, z_nxt);
          }
          const uint32_t jj = grp & 7;
          const uint32_t sw = jj < 2 ? s_cur.x : jj < 4 ? s_cur.y : jj < 6 ? s_cur.z : s_cur.w;
          const uint32_t zw = jj < 2 ? z_cur.x : jj < 4 ? z_cur.y : jj < 6 ? z_cur.z : z_cur.w;
          sb = static_cast<uint16_t>((jj & 1) ? (sw >> 16) : (sw & 0xFFFFu));
          if (zrow) zb = static_cast<uint16_t>((jj & 1) ? (zw >> 16) : (zw & 0xFFFFu));
        } else if (row_ok) {
          sb = __ldg(srow + grp);
          if (zrow) zb = __ldg(zrow + grp);
        }
        const float sf = row_ok ? __half2float(*reinterpret_cast<const __half*>(&sb)) : 0.0f;
        const float zf = __half2float(*reinterpret_cast<const __half*>(&zb));
        // activation row sums of the segment
        float ssum[BN];
        const bool whole = (end - kb == kpg) && (static_cast<int>(grp) * kpg == g.kb0 + kb);
        if (whole) {
          if (static_cast<int>(grp) >= gs_first + kGsumChunk || static_cast<int>(grp) < gs_first || gs_m0 != m0) {
            // stage the next chunk of group sums (uniform across the 128 threads)
            named_bar_sync(1, kEpiThreads);
            gs_first = static_cast<int>(grp);
            gs_m0 = m0;
            const int cnt = min(kGsumChunk, A4.groups - gs_first) * BN;
            for (int i = et; i < cnt; i += kEpiThreads) {
              const int gi = i / BN, j = i - gi * BN;
              gs_smem[i] = A4.gsum[static_cast<int64_t>(gs_first + gi) * A4.asum_ld + m0 + j];
            }
            named_bar_sync(1, kEpiThreads);
          }
          const float4* sp = reinterpret_cast<const float4*>(gs_smem + (static_cast<int>(grp) - gs_first) * BN);
#pragma unroll
          for (int j4 = 0; j4 < BN / 4; ++j4) {
            const float4 f = sp[j4];
            ssum[4 * j4 + 0] = f.x;
            ssum[4 * j4 + 1] = f.y;
            ssum[4 * j4 + 2] = f.z;
            ssum[4 * j4 + 3] = f.w;
          }
        } else {
          // a split boundary cuts this group: add the per-block sums
#pragma unroll
          for (int j = 0; j < BN; ++j) ssum[j] = 0.0f;
          for (int k = kb; k < end; ++k) {
            const float4* sp =
                reinterpret_cast<const float4*>(A4.asum + static_cast<int64_t>(g.kb0 + k) * A4.asum_ld + m0);
#pragma unroll
            for (int j4 = 0; j4 < BN / 4; ++j4) {
              const float4 f = __ldg(sp + j4);
              ssum[4 * j4 + 0] += f.x;
              ssum[4 * j4 + 1] += f.y;
              ssum[4 * j4 + 2] += f.z;
              ssum[4 * j4 + 3] += f.w;
            }
          }
        }
        const int buf = seg % C::NSEG;
        const bool got = mbar_wait_bounded(d_full(buf), (seg / C::NSEG) & 1, a.wait_limit_ns, abort_flag);
        if (!got && !*abort_flag) record_timeout(a, abort_flag, 2 * 16 + 2);
        if (named_bar_or(1, kEpiThreads, !got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float bias = sf * (1024.0f + zf);
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + static_cast<uint32_t>(buf * BN);
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 16) {
          uint32_t v[16];
          tc_ld_32x32b_x16(t_row + c0, v);
          tc_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            acc[c0 + j] = fmaf(sf, __uint_as_float(v[j]), fmaf(-bias, ssum[c0 + j], acc[c0 + j]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(d_empty(buf));
        ++seg;
        kb = end;
      }
      if (!ok) break;
      const bool full_tile = (g.s0 == 0 && g.s1 == a.split);
      if (row_ok && g.nkb > 0) {
        if (full_tile) {
          uint16_t* cc = reinterpret_cast<uint16_t*>(a.c) + n;
#pragma unroll
          for (int j = 0; j < BN; ++j)
            if (m0 + j < m1) cc[static_cast<int64_t>(m0 + j) * a.ldc] = cvt1(acc[j], a.c_bf16);
        } else {
          float* wc = a.ws + n;
#pragma unroll
          for (int j = 0; j < BN; ++j)
            if (m0 + j < m1) red_add_f32(wc + static_cast<int64_t>(m0 + j) * a.N, acc[j]);
        }
      }
      if (!full_tile) arrive_split_tile(a, g, g.tile, m0, m1, n0, n1, et);
    }
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // Let the last loads issued into each stage land before the CTA exits.
    volatile int no_abort = 0;
    const int first = issued > C::STAGES ? issued - C::STAGES : 0;
    for (int c = first; c < issued; ++c)
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

// Activation pre-pass: one thread per (64-deep K block, row m).  Writes the
// row's 64 values to Ap (K-contiguous, pitch K) with each 8-element group
// reordered to (0,4,1,5,2,6,3,7), and their fp32 sum to asum[kb][m].
__global__ void int4_prep_kernel(const uint16_t* __restrict__ A, int64_t lda, int a_mn, int M, int K,
                                 uint16_t* __restrict__ Ap, float* __restrict__ asum, int asum_ld) {
  const int kb_count = K / TILE_K;
  const int64_t total = static_cast<int64_t>(kb_count) * M;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(i % M);
    const int kb = static_cast<int>(i / M);
    float sum = 0.0f;
#pragma unroll 2
    for (int j = 0; j < TILE_K / 8; ++j) {
      const int k0 = kb * TILE_K + 8 * j;
      uint16_t v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int64_t idx = a_mn ? static_cast<int64_t>(k0 + e) * lda + m : static_cast<int64_t>(m) * lda + k0 + e;
        v[e] = A[idx];
        sum += __half2float(*reinterpret_cast<const __half*>(&v[e]));
      }
      uint4 o;
      o.x = static_cast<uint32_t>(v[0]) | (static_cast<uint32_t>(v[4]) << 16);
      o.y = static_cast<uint32_t>(v[1]) | (static_cast<uint32_t>(v[5]) << 16);
      o.z = static_cast<uint32_t>(v[2]) | (static_cast<uint32_t>(v[6]) << 16);
      o.w = static_cast<uint32_t>(v[3]) | (static_cast<uint32_t>(v[7]) << 16);
      *reinterpret_cast<uint4*>(Ap + static_cast<int64_t>(m) * K + k0) = o;
    }
    asum[static_cast<int64_t>(kb) * asum_ld + m] = sum;
  }
}

// Activation pre-pass for a K-contiguous activation: one thread per
// 8-element chunk (m, c), c fastest, so that loads and stores are coalesced
// 16-byte vectors (scalar loads when the rows are not 16-byte aligned).  The
// chunk is stored with its elements reordered to (0,4,1,5,2,6,3,7); the 8
// chunks of a 64-deep block sit in 8 adjacent lanes (K is a multiple of 64)
// and their sum is reduced by shuffles into asum[kb][m]; when a quantisation
// group spans 8, 16 or 32 lanes (64, 128 or 256 elements), the group sum
// gsum[g][m] is reduced the same way (lanes_per_group = 0: not here).
__global__ void __launch_bounds__(256) int4_prep_kmajor_kernel(const uint16_t* __restrict__ A, int64_t lda, int vec,
                                                               int M, int K, uint16_t* __restrict__ Ap,
                                                               float* __restrict__ asum, float* __restrict__ gsum,
                                                               int asum_ld, int lanes_per_group) {
  const int chunks = K / 8;
  const int64_t total = static_cast<int64_t>(M) * chunks;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // base is a multiple of the block size: warps cover 32 consecutive chunks
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x; base < total; base += step) {
    const int64_t i = base + threadIdx.x;
    const bool act = i < total;
    int m = 0, c = 0;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (act) {
      m = static_cast<int>(i / chunks);
      c = static_cast<int>(i - static_cast<int64_t>(m) * chunks);
      const uint16_t* src = A + static_cast<int64_t>(m) * lda + 8 * c;
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
    }
    // elements e = 0..7 are the halves of w[e / 2]; the stored order is 0,4 | 1,5 | 2,6 | 3,7
    uint4 o;
    o.x = (w[0] & 0xFFFFu) | (w[2] << 16);
    o.y = (w[0] >> 16) | (w[2] & 0xFFFF0000u);
    o.z = (w[1] & 0xFFFFu) | (w[3] << 16);
    o.w = (w[1] >> 16) | (w[3] & 0xFFFF0000u);
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[e]);
      const float2 f = __half22float2(h);
      s += f.x + f.y;
    }
    if (act) *reinterpret_cast<uint4*>(Ap + static_cast<int64_t>(m) * K + 8 * c) = o;
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 4);
    if (act && (c & 7) == 0) asum[static_cast<int64_t>(c >> 3) * asum_ld + m] = s;
    if (lanes_per_group >= 16) s += __shfl_xor_sync(0xFFFFFFFFu, s, 8);
    if (lanes_per_group >= 32) s += __shfl_xor_sync(0xFFFFFFFFu, s, 16);
    if (lanes_per_group && act && c % lanes_per_group == 0)
      gsum[static_cast<int64_t>(c / lanes_per_group) * asum_ld + m] = s;
  }
}

// Per-group row sums from the per-block ones: gsum[g][m] = sum of asum over
// the group's 64-deep blocks (same fp32 values the epilogue would add).
__global__ void int4_group_sum_kernel(const float* __restrict__ asum, float* __restrict__ gsum, int asum_ld, int M,
                                      int groups, int kb_per_group) {
  const int64_t total = static_cast<int64_t>(groups) * M;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(i % M);
    const int g = static_cast<int>(i / M);
    float s = 0.0f;
    for (int k = 0; k < kb_per_group; ++k) s += asum[static_cast<int64_t>(g * kb_per_group + k) * asum_ld + m];
    gsum[static_cast<int64_t>(g) * asum_ld + m] = s;
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

cudaError_t launch_int4_prep(const void* A, int64_t lda, int a_mn, int M, int K, int group, void* Ap, float* asum,
                             float* gsum, int asum_ld, int sms, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(K / TILE_K) * M;
  if (total == 0) return cudaSuccess;
  if (!a_mn) {
    const int lanes = group / 8;
    const int lpg = (lanes == 8 || lanes == 16 || lanes == 32) ? lanes : 0;
    const int vec = (lda % 8 == 0) && (reinterpret_cast<uintptr_t>(A) % 16 == 0);
    const int64_t chunks = static_cast<int64_t>(M) * (K / 8);
    int64_t blocks = (chunks + 255) / 256;
    if (blocks > static_cast<int64_t>(sms) * 8) blocks = static_cast<int64_t>(sms) * 8;
    int4_prep_kmajor_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(A), lda, vec, M, K, static_cast<uint16_t*>(Ap), asum, gsum, asum_ld, lpg);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || lpg) return e;
  }
  const int threads = 128;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > static_cast<int64_t>(sms) * 16) blocks = static_cast<int64_t>(sms) * 16;
  if (a_mn) {
    int4_prep_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(static_cast<const uint16_t*>(A), lda, a_mn, M,
                                                                       K, static_cast<uint16_t*>(Ap), asum, asum_ld);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int groups = K / group;
  const int64_t gtotal = static_cast<int64_t>(groups) * M;
  int64_t gblocks = (gtotal + threads - 1) / threads;
  if (gblocks > static_cast<int64_t>(sms) * 16) gblocks = static_cast<int64_t>(sms) * 16;
  int4_group_sum_kernel<<<static_cast<int>(gblocks), threads, 0, stream>>>(asum, gsum, asum_ld, M, groups,
                                                                           group / TILE_K);
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
