// int4-weight GEMM with the dequantisation inside the mainloop.
//
//   C[m,n] = sum_k A[m,k] * w(k,n),  w(k,n) = (q(n,k) - z(n,g)) * s(n,g),
//   g = k / group_size, codes two per byte (low nibble = even k).
//
// The weight is the large operand and the activation the skinny one, so the
// MMA runs swapped: 128 weight rows (n) on the MMA's M side, the activation
// rows (m) on its N side, the accumulator holding C^T in TMEM.
//
// Warp roles (448 threads):
//   warp 0       TMA producer: raw int4 tile (128 rows x 32 bytes = 64 codes,
//                32-byte swizzle) and the activation tile (64 K, 128-byte
//                swizzle) of each 64-deep K block into a ring of stages.
//   warp 1       TMEM allocator and MMA issuer.  The dequantised weight tile
//                is the MMA's A operand *in TMEM*; the activation is read from
//                shared memory through a descriptor.
//   warps 2..9   dequantisers: two warps per TMEM lane quadrant, alternating K
//                blocks.  Each thread owns one weight row: it reads its 32 raw
//                bytes with two 16-byte shared loads (conflict-free thanks to
//                the swizzle), expands each byte to an fp16 pair with a byte
//                permute and one LOP3 (0x6400 | code is 1024 + code in fp16),
//                removes the zero point and applies the scale with two fp16x2
//                operations -- each weight is rounded once, exactly
//                RN((q - z) * s) -- and writes the 64 values (32 TMEM columns)
//                of its row with one tcgen05.st.
//   warps 10..13 epilogue, shared with the dense kernel (split-K reduction).
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

constexpr int kThreads4 = 448;
constexpr int kDequantWarp0 = 2;
constexpr int kEpiWarp04 = 10;
constexpr uint32_t kRawBytes = TILE_P * 32;   // 128 rows x 32 bytes (64 codes)
constexpr int kASlots = 8;                    // TMEM A-operand slots of 32 columns (64 fp16 per lane)
constexpr uint32_t kASlotCol0 = 256;          // first A-slot column (accumulators use [0, 256))

template <int BN>
struct Cfg4 {
  static constexpr uint32_t ACT_BYTES = BN * TILE_K * 2;
  static constexpr uint32_t STAGE_BYTES = kRawBytes + ACT_BYTES;
  static constexpr int STAGES_RAW = (192 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 24 ? 24 : STAGES_RAW;
  static constexpr int CH = BN < 32 ? BN : 32;
  // barriers: raw_full[S], raw_empty[S], a_full[T], a_empty[T], acc_full[2], acc_empty[2], teardown
  static constexpr uint32_t BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 2 * kASlots + 5;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr uint32_t SMEM_ALLOC = MISC_OFF + 64 + 1024;
  static_assert(STAGE_BYTES % 1024 == 0, "stage buffers stay 1024-byte aligned");
  static_assert(2 * BN <= kASlotCol0, "accumulators fit below the A slots");
};

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
  return d;
}

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t half2_bits(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Per (row, group) constants of the dequantisation.  Codes arrive as
// t = (1024 + q_even, 1024 + 16 q_odd) in fp16 (the odd code keeps its
// nibble position).  Exact path (integer zero point, s/16 exact):
//   w = (t - (1024 + z, 1024 + 16 z)) * (s, s/16).
// General path: d = (t - 1024) - (z, 16 z); w = (d * s) * (1, 1/16).
struct DqConst {
  uint32_t bias, mul;  // exact path
  uint32_t z2, s2;     // general path
  bool exact;
};

__device__ __forceinline__ DqConst make_dq(float s, float z) {
  DqConst c;
  const __half s16 = __float2half_rn(s * 0.0625f);
  const bool s16_exact = __half2float(s16) * 16.0f == s;
  c.exact = s16_exact && z == rintf(z) && fabsf(z) <= 512.0f;
  c.bias = half2_bits(1024.0f + z, 1024.0f + 16.0f * z);
  c.mul = half2_bits(s, 0.0f) & 0xFFFFu;
  c.mul |= static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&s16)) << 16;
  c.z2 = half2_bits(z, 16.0f * z);
  c.s2 = half2_bits(s, s);
  return c;
}

// One 32-bit word (8 codes, k = 8j..8j+7) -> four fp16x2 (k pairs).
__device__ __forceinline__ void dequant_word(uint32_t w, const DqConst& c, uint32_t (&out)[4]) {
  const uint32_t k1024 = 0x64006400u;
  const uint32_t one_16th = 0x2C003C00u;  // (1.0, 0.0625)
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t y = __byte_perm(w, 0u, 0x1111u * b);         // byte b in every byte
    const uint32_t t = lop3_and_or(y, 0x00F0000Fu, k1024);      // (1024 + q_lo, 1024 + 16 q_hi)
    if (c.exact) {
      out[b] = hmul2_u(hsub2_u(t, c.bias), c.mul);
    } else {
      const uint32_t d = hsub2_u(hsub2_u(t, k1024), c.z2);
      out[b] = hmul2_u(hmul2_u(d, c.s2), one_16th);
    }
  }
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
  auto raw_full = [&](int s) { return bar0 + 8u * s; };
  auto raw_empty = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto a_full = [&](int t) { return bar0 + 8u * (2 * C::STAGES + t); };
  auto a_empty = [&](int t) { return bar0 + 8u * (2 * C::STAGES + kASlots + t); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 * kASlots + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 * kASlots + 2 + b); };
  const uint32_t teardown_bar = bar0 + 8u * (2 * C::STAGES + 2 * kASlots + 4);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(raw_full(s), 1);
      mbar_init(raw_empty(s), 4 + 1);  // the four dequant warps of the stage + the MMA's commit
    }
    for (int t = 0; t < kASlots; ++t) {
      mbar_init(a_full(t), 4);
      mbar_init(a_empty(t), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), kEpiThreads / 32);
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
      Sched sched(a);
      Group g;
      int c = 0;
      bool ok = true;
      while (ok && sched.next(a, g)) {
        int32_t tp, tq, m0, m1, n0, n1;
        tile_ranges(a, g.tile, BN, tp, tq, m0, m1, n0, n1);
        for (int kb = 0; kb < g.nkb; ++kb, ++c) {
          const int s = c % C::STAGES;
          if (!mbar_wait_bounded(raw_empty(s), ((c / C::STAGES) & 1) ^ 1u, a.wait_limit_ns, abort_flag)) {
            if (!*abort_flag) record_timeout(a, abort_flag, 0 * 16 + 1);
            ok = false;
            break;
          }
          const uint32_t sraw = base + s * C::STAGE_BYTES;
          const uint32_t sact = sraw + kRawBytes;
          const int32_t k0 = (g.kb0 + kb) * TILE_K;
          mbar_arrive_expect_tx(raw_full(s), C::STAGE_BYTES);
          tma_load_2d(sraw, &A4.tm_w, raw_full(s), k0 / 2, n0);
          if (!a.q_mn) {
            tma_load_2d(sact, &a.tm_q, raw_full(s), k0, m0);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(sact + j * 8192u, &a.tm_q, raw_full(s), m0 + 64 * j, k0);
          }
          ++issued;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      Sched sched(a);
      Group g;
      int c = 0;
      int acc_iter = 0;
      bool ok = true;
      const uint32_t q_step = a.q_mn ? 2048u : 32u;
      const uint32_t q_lbo = a.q_mn ? 8192u : 16u;
      while (ok && sched.next(a, g)) {
        if (g.nkb == 0) continue;
        const int buf = acc_iter & 1;
        if (!mbar_wait_bounded(acce_bar(buf), ((acc_iter >> 1) & 1) ^ 1u, a.wait_limit_ns, abort_flag)) {
          if (!*abort_flag) record_timeout(a, abort_flag, 1 * 16 + 3);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < g.nkb; ++kb, ++c) {
          const int s = c % C::STAGES, t = c % kASlots;
          if (!mbar_wait_bounded(raw_full(s), (c / C::STAGES) & 1, a.wait_limit_ns, abort_flag) ||
              !mbar_wait_bounded(a_full(t), (c / kASlots) & 1, a.wait_limit_ns, abort_flag)) {
            if (!*abort_flag) record_timeout(a, abort_flag, 1 * 16 + 0);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sact = base + s * C::STAGE_BYTES + kRawBytes;
          const uint32_t a_tmem = tmem_base + kASlotCol0 + static_cast<uint32_t>(t * 32);
#pragma unroll
          for (int k = 0; k < TILE_K / 16; ++k) {
            const uint64_t bd = sw128_desc(sact + k * q_step, q_lbo, 1024u);
            tc_mma_f16_ts(d_tmem, a_tmem + k * 8, bd, a.idesc, (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(raw_empty(s));
          tc_commit(a_empty(t));
        }
        if (!ok) break;
        tc_commit(accf_bar(buf));
        ++acc_iter;
      }
    }
  } else if (warp < kEpiWarp04) {
    // ------------------------------------------------------------ dequantisers
    const int q4 = warp & 3;
    const int h = (warp - kDequantWarp0) >> 2;  // which K blocks: c % 2 == h
    const int r = q4 * 32 + lane;               // weight row within the tile (TMEM lane)
    Sched sched(a);
    Group g;
    int c = 0;
    bool ok = true;
    while (ok && sched.next(a, g)) {
      int32_t tp, tq, m0, m1, n0, n1;
      tile_ranges(a, g.tile, BN, tp, tq, m0, m1, n0, n1);
      const int n = n0 + r;
      const bool row_ok = n < a.N;
      const uint16_t* srow = A4.scales + static_cast<int64_t>(row_ok ? n : 0) * A4.groups;
      const uint16_t* zrow = A4.zeros ? A4.zeros + static_cast<int64_t>(row_ok ? n : 0) * A4.groups : nullptr;
      for (int kb = 0; kb < g.nkb; ++kb, ++c) {
        if ((c & 1) != h) continue;
        const int s = c % C::STAGES, t = c % kASlots;
        const uint32_t grp = magic_div(static_cast<uint32_t>(g.kb0 + kb), A4.div_kb_per_group);
        float sf = 0.0f, zf = 8.0f;
        if (row_ok) {
          const uint16_t sb = __ldg(srow + grp);
          sf = __half2float(*reinterpret_cast<const __half*>(&sb));
          if (zrow) {
            const uint16_t zb = __ldg(zrow + grp);
            zf = __half2float(*reinterpret_cast<const __half*>(&zb));
          }
        }
        const DqConst dq = make_dq(sf, zf);
        const bool got = mbar_wait_bounded(raw_full(s), (c / C::STAGES) & 1, a.wait_limit_ns, abort_flag) &&
                         mbar_wait_bounded(a_empty(t), ((c / kASlots) & 1) ^ 1u, a.wait_limit_ns, abort_flag);
        if (!got && !*abort_flag) record_timeout(a, abort_flag, 3 * 16 + 0);
        // the warp leaves together (tcgen05.st below needs every lane)
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // raw row r: two 16-byte chunks, chunk q stored at q ^ bit 2 of r (32-byte swizzle)
        const uint8_t* rowp = smem + s * C::STAGE_BYTES + r * 32;
        const int sw = (r >> 2) & 1;
        const uint4 lo = *reinterpret_cast<const uint4*>(rowp + (sw ? 16 : 0));
        const uint4 hi = *reinterpret_cast<const uint4*>(rowp + (sw ? 0 : 16));
        __syncwarp();
        if (lane == 0) mbar_arrive(raw_empty(s));
        const uint32_t words[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        uint32_t vals[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t o[4];
          dequant_word(words[j], dq, o);
#pragma unroll
          for (int b = 0; b < 4; ++b) vals[4 * j + b] = o[b];
        }
        const uint32_t taddr =
            tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + kASlotCol0 + static_cast<uint32_t>(t * 32);
        tc_st_32x32b_x32(taddr, vals);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(a_full(t));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;
    const int et = threadIdx.x - kEpiWarp04 * 32;
    Sched sched(a);
    Group g;
    int acc_iter = 0;
    while (sched.next(a, g)) {
      if (!epilogue_group<BN, C::CH>(a, g, tmem_base, accf_bar(0), acce_bar(0), acc_iter, abort_flag, q4, lane,
                                     et))
        break;
    }
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // Let the last loads issued into each stage land before the CTA exits.
    volatile int no_abort = 0;
    const int first = issued > C::STAGES ? issued - C::STAGES : 0;
    for (int c = first; c < issued; ++c)
      mbar_wait_bounded(raw_full(c % C::STAGES), (c / C::STAGES) & 1, a.wait_limit_ns, &no_abort);
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

cudaError_t launch_int4_gemm(const Int4Args& args, int bn, int grid, cudaStream_t stream) {
  switch (bn) {
    case 16: return launch4<16>(args, grid, stream);
    case 32: return launch4<32>(args, grid, stream);
    case 64: return launch4<64>(args, grid, stream);
    case 128: return launch4<128>(args, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lgt
