// int4-weight GEMM, e4m3 form: the codes go to the tensor core as exact
// 8-bit values, and every scale is applied in fp32 after the MMA.
//
//   C[m,n] = sum_k A[m,k] * w(k,n),  w(k,n) = (q(n,k) - z(n,g)) * s(n,g),
//   g = k / group_size, codes two per byte (low nibble = even k).
//
// Why e4m3.  The MMA runs swapped (128 weight rows n on its M side, the at
// most 16 activation rows m on its N side) with the expanded weight tile as
// its A operand in TMEM.  With so narrow an N the cost is the MMA issue and
// the TMEM traffic of the A operand, not arithmetic: one issuing warp
// completes about one 128 x N x K-step MMA per 165 cycles whatever N is
// (measured here), several issuing warps overlap, and kind::f8f6f4 covers 32
// of K per MMA against 16 for kind::f16 -- half the MMAs and half the TMEM
// bytes per weight.
//
// Exactness.  A code q placed in the low nibble of a byte *is* the e4m3
// number q * 2^-9 (codes 0..7 are the subnormals m * 2^-9, codes 8..15 the
// first binade (8 + m) * 2^-9), so expanding eight codes is one AND and one
// shift-and-AND.  The fp16 activation is split, per row and 128-deep block of
// K, into three e4m3 terms: with S_b = 2^e (the block's largest |a| times S_b
// in [224, 448)), b1 = e4m3(a S_b), b2 = e4m3(16 (a S_b - b1)),
// b3 = e4m3(16 (16 (a S_b - b1) - b2)) (each residual exact in fp32), and
// a S_b = b1 + b2/16 + b3/256 exactly for every element whose a S_b lies in
// e4m3's normal range (2^-6 and up: each rounding keeps four significant bits
// and an fp16 value has eleven); for the smaller elements the absolute error
// is at most 2^-18 / S_b, below 2^-25 of the block's largest |a|.  (Checked
// over every finite fp16 value and block maxima 2^-24 .. 2^16.)
// The MMA's N = 48 columns are the three terms of the 16 activation rows;
// products of e4m3 values are exact and accumulate in fp32.  So per 128-deep
// block ("segment") the accumulator holds
//   D[n, 16t + m] = sum_k q(n,k) 2^-9 b_t(m,k),
// and the epilogue forms, in fp32,
//   C[m,n] += s(n,g) 2^9 / S_b (D[n,m] + D[n,16+m]/16 + D[n,32+m]/256)
//             - s(n,g) z(n,g) Ag_b[m],
// with Ag_b[m] the block's sum of row m of the activation (the zero point
// enters through it, as the dequantised weight (q - z) s does).  Apart from
// fp32 accumulation, the only error against the exact sum of A (q - z) s is
// that of the activation's smallest elements above.
//
// The BitBLAS TileLang page's dequantise copy ("Relevant Issues") expands
// packed weights with vectorised loads into the operand layout; here the TMA
// box does the addressing, every thread's shared loads are 128-bit and the
// expansion writes the TMEM operand directly.  Split-K units and the fp32
// reduction of partial runs are those of the dense kernels (BitBLAS page,
// "SplitK Infer for dequantize cases"; IREE page, partial sums -> shared
// storage -> second reduction).
//
// Pipeline (one CTA per SM, persistent):
//   W stage   = 256 of K: the packed weights of 128 rows (one 128 x 128-byte
//               TMA box, 128-byte swizzle); two segments.
//   segment   = 128 of K (one K block of the e4m3 operand): its activation
//               box (48 rows x 128 bytes), its TMEM A slot (32 columns), its
//               four MMAs and its own 48-column accumulator.
// Warp roles (512 threads: 128 registers a thread, none spilled):
//   warp 0       TMA producer of the weight ring (one copy per W stage).
//   warp 1       TMA producer of the activation ring (one copy per segment).
//   warps 2, 3   MMA issuers: segment s goes to issuer s % 2, which issues its
//                four MMAs back to back into accumulator slot s % 4.  Warp 2
//                owns the TMEM.
//   warps 4..7   epilogue (TMEM lane quadrant warp % 4): per segment, read
//                the accumulator, free it, scale and add into the run's fp32
//                sums; at the end of a run store C or the split-K partial.
//   warps 8..15  expanders, two per lane quadrant: warp h of a quadrant
//                expands segment h of every W stage for its 32 weight rows.
// Every barrier that several threads wait on is waited on for each of its
// phases in order (no waiter can skip a phase and mistake an older one for
// the one it wants), and every wait is bounded.
#include <cuda_fp16.h>

#include "int4.h"
#include "kernels.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lgt {
namespace {

constexpr int kF8Threads = 512;
constexpr int kF8IssWarp0 = 2;
constexpr int kF8Issuers = 2;
constexpr int kF8EpiWarp0 = 4;
constexpr int kF8ExpWarp0 = 8;
constexpr int kF8N = 48;                       // MMA N: three e4m3 terms x 16 activation rows
constexpr uint32_t kF8WStage = 128 * 128;      // packed weights of one W stage
constexpr uint32_t kF8XStage = kF8N * 128;     // activation box of one segment: 6 KiB
constexpr int kF8WST = 8;                      // weight ring
constexpr int kF8XST = 4;                      // activation ring (a multiple of the issuers)
constexpr int kF8TSL = 8;                      // TMEM A slots (a multiple of the issuers)
constexpr int kF8ASL = 4;                      // accumulator slots (a multiple of the issuers)
constexpr uint32_t kF8ACol0 = 256;             // A slots at TMEM columns [256, 512); accumulators below
constexpr int kF8TabBlocks = 256;              // activation tables staged in shared memory up to this many blocks
constexpr uint32_t kF8TabBytes = 2 * kF8TabBlocks * 16 * 4;
constexpr uint32_t kF8XOff = kF8WST * kF8WStage;
constexpr uint32_t kF8TabOff = kF8XOff + kF8XST * kF8XStage;
constexpr uint32_t kF8BarOff = kF8TabOff + kF8TabBytes;
// full_w, wfree, full_x, xfree, a_full, tfree, accf, acce, teardown
constexpr uint32_t kF8NumBars = 2 * kF8WST + 2 * kF8XST + 2 * kF8TSL + 2 * kF8ASL + 1;
constexpr uint32_t kF8MiscOff = kF8BarOff + kF8NumBars * 8;
constexpr uint32_t kF8Smem = kF8MiscOff + 64 + 1024;
static_assert(kF8TSL % kF8Issuers == 0 && kF8XST % kF8Issuers == 0 && kF8ASL % kF8Issuers == 0,
              "one issuer per A slot, activation buffer and accumulator slot");
static_assert(kF8ASL * kF8N <= static_cast<int>(kF8ACol0) && kF8ACol0 + kF8TSL * 32 <= 512, "TMEM columns");
static_assert(kF8XStage % 1024 == 0 && kF8WStage % 1024 == 0, "swizzled buffers stay 1024-byte aligned");
static_assert(kF8Smem <= 227 * 1024, "shared memory budget");
static_assert(kF8Issuers >= 1 && kF8IssWarp0 + kF8Issuers <= kF8EpiWarp0, "issuer warps lie between the producers and the epilogue");

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f8f6f4 (e4m3 x e4m3, fp32 accumulate).
__device__ __forceinline__ void tc_mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ float half_bits_f32(uint32_t b) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
}

// One weight row's scales and zero points, in group order, for the
// epilogue: read 8 groups (16 bytes) at a time with the next window already
// in flight (rows 16-byte aligned, groups a multiple of 8), else one group at
// a time with the next group in flight.  Each load is issued a window (or a
// group) before it is needed, so its latency under the weight stream is
// hidden behind the segments in between.
struct RowParams {
  const uint16_t* srow = nullptr;  // null: row beyond N (scale 0)
  const uint16_t* zrow = nullptr;  // null: zero point 8
  int G = 0;
  bool vec = false;
  int wcur = -2;
  uint4 s_cur, z_cur, s_nxt, z_nxt;
  __device__ uint4 load(const uint16_t* row, int w, uint32_t dflt) const {
    if (!row || (vec ? w * 8 : w) >= G) return make_uint4(dflt, dflt, dflt, dflt);
    if (vec) return __ldg(reinterpret_cast<const uint4*>(row) + w);
    return make_uint4(static_cast<uint32_t>(__ldg(row + w)), 0u, 0u, 0u);  // scalar mode: "window" = one group
  }
  __device__ void reset(const uint16_t* s, const uint16_t* z, int groups, bool v, int g0) {
    srow = s;
    zrow = z;
    vec = v;
    G = groups;
    wcur = -2;
    fetch(g0);
  }
  __device__ int window_of(int g) const { return vec ? (g >> 3) : g; }
  __device__ void fetch(int g) {
    const int w = window_of(g);
    if (w == wcur) return;
    if (w == wcur + 1) {
      s_cur = s_nxt;
      z_cur = z_nxt;
    } else {
      s_cur = load(srow, w, 0u);
      z_cur = load(zrow, w, 0x48004800u);  // fp16 8.0 pairs
    }
    s_nxt = load(srow, w + 1, 0u);
    z_nxt = load(zrow, w + 1, 0x48004800u);
    wcur = w;
  }
  __device__ void get(int g, float& s, float& z) {
    fetch(g);
    uint32_t sb, zb;
    if (vec) {
      const int e = g & 7;
      const uint32_t sw = e < 4 ? (e < 2 ? s_cur.x : s_cur.y) : (e < 6 ? s_cur.z : s_cur.w);
      const uint32_t zw = e < 4 ? (e < 2 ? z_cur.x : z_cur.y) : (e < 6 ? z_cur.z : z_cur.w);
      sb = (e & 1) ? (sw >> 16) : (sw & 0xFFFFu);
      zb = (e & 1) ? (zw >> 16) : (zw & 0xFFFFu);
    } else {
      sb = s_cur.x & 0xFFFFu;
      zb = z_cur.x & 0xFFFFu;
    }
    s = half_bits_f32(sb);
    z = half_bits_f32(zb);
  }
};

// Segments of this CTA, in order: every run of (tile, splits) from the
// scheduler, cut into 128-deep segments, two per W stage.
struct SegRun {
  Sched sched;
  Group g;
  int nseg = 0;
  __device__ explicit SegRun(const TcArgs& a) : sched(a) {}
  __device__ bool next(const TcArgs& a) {
    while (sched.next(a, g)) {
      nseg = g.nkb >> 1;  // runs hold whole 128-deep blocks
      if (nseg > 0) return true;
    }
    return false;
  }
};

// e4m3 round to nearest (saturating at 448) of y, as a byte; and the exact
// value of an e4m3 byte.  (Both halves of the pair instructions get the same
// value, so the byte order within a pair does not matter.)
__device__ __forceinline__ uint32_t e4m3_rn(float y) {
  uint16_t p;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(p) : "f"(y));
  return p & 0xFFu;
}

__device__ __forceinline__ float e4m3_value(uint32_t b) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(b | (b << 8))));
  return half_bits_f32(h2 & 0xFFFFu);
}

// The three e4m3 terms of y (|y| < 448): y = b1 + b2 / 16 + b3 / 256,
// exactly when y is an fp16 value times a power of two and |y| >= 2^-6,
// else to within 2^-18 (each residual is exact in fp32).
__device__ __forceinline__ void split3(float y, uint32_t& b1, uint32_t& b2, uint32_t& b3) {
  b1 = e4m3_rn(y);
  const float r1 = 16.0f * (y - e4m3_value(b1));
  b2 = e4m3_rn(r1);
  const float r2 = 16.0f * (r1 - e4m3_value(b2));
  b3 = e4m3_rn(r2);
}

// Activation pre-pass of the e4m3 form (K-contiguous A, M <= 16, K a
// multiple of 128).  One thread per 8-element chunk (m, c) of a 16-row
// activation (rows m >= M are zero), c fastest; the 16 chunks of a 128-deep
// block are 16 consecutive lanes.  Writes, for block b = c / 16:
//   Xp[((b * 48 + 16 t + m) * 128 + 8 (c mod 16) + i] = term t of element
//     8c + perm(i), perm = (0, 2, 4, 6, 1, 3, 5, 7) (the expanders' byte order);
//   inv_scale[b * 16 + m] = 1 / S_b(m);  agsum[b * 16 + m] = sum of the block
//   (fp32, fixed butterfly order).
__global__ void __launch_bounds__(256) int4f8_prep_kernel(const uint16_t* __restrict__ A, int64_t lda, int vec, int M,
                                                          int K, uint8_t* __restrict__ Xp,
                                                          float* __restrict__ inv_scale, float* __restrict__ agsum) {
  pdl_launch_dependents();
  pdl_wait();
  const int chunks = K / 8;
  const int64_t total = static_cast<int64_t>(16) * chunks;  // a multiple of 32: every warp is full
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += step) {
    const int m = static_cast<int>(i / chunks);
    const int c = static_cast<int>(i - static_cast<int64_t>(m) * chunks);
    float x[8];
    if (m < M) {
      const uint16_t* src = A + static_cast<int64_t>(m) * lda + 8 * c;
      if (vec) {
        const uint4 q = *reinterpret_cast<const uint4*>(src);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[2 * e] = half_bits_f32(w[e] & 0xFFFFu);
          x[2 * e + 1] = half_bits_f32(w[e] >> 16);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = half_bits_f32(src[e]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = 0.0f;
    }
    // block maximum of |a| and block sum over the 16 lanes of the block
    float mx = 0.0f, sum = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      mx = fmaxf(mx, fabsf(x[e]));
      sum += x[e];
    }
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      sum += __shfl_xor_sync(0xffffffffu, sum, off);
    }
    // S = 2^e with mx * S in [224, 448): mx = f 2^E (1 <= f < 2) gives
    // e = 8 - E, or 7 - E when f >= 1.75
    int e = 0;
    if (mx > 0.0f) {
      const uint32_t bits = __float_as_uint(mx);
      const int E = static_cast<int>((bits >> 23) & 0xFFu) - 127;
      e = ((bits & 0x7FFFFFu) >= 0x600000u ? 7 : 8) - E;
    }
    const float S = ldexpf(1.0f, e);
    uint32_t t1[8], t2[8], t3[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) split3(x[k] * S, t1[k], t2[k], t3[k]);
    // byte order 0, 2, 4, 6 | 1, 3, 5, 7
    auto pack = [](const uint32_t (&t)[8]) {
      return make_uint2(t[0] | (t[2] << 8) | (t[4] << 16) | (t[6] << 24), t[1] | (t[3] << 8) | (t[5] << 16) | (t[7] << 24));
    };
    const int b = c >> 4;
    uint8_t* dst = Xp + (static_cast<int64_t>(b) * kF8N + m) * 128 + 8 * (c & 15);
    *reinterpret_cast<uint2*>(dst) = pack(t1);
    *reinterpret_cast<uint2*>(dst + 16 * 128) = pack(t2);
    *reinterpret_cast<uint2*>(dst + 32 * 128) = pack(t3);
    if ((c & 15) == 0) {
      inv_scale[b * 16 + m] = ldexpf(1.0f, -e);
      agsum[b * 16 + m] = sum;
    }
  }
}

__global__ void __launch_bounds__(kF8Threads, 1) int4f8_gemm_kernel(const __grid_constant__ Int4Args A4) {
  pdl_launch_dependents();
  const TcArgs& a = A4.t;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = base + kF8BarOff;
  // full_w[i] / full_x[i]: a weight / activation copy landed.  wfree[i]:
  // every thread of the eight expander warps read the W stage.  xfree[i]: the MMAs reading the
  // activation buffer completed.  a_full[t]: the four expander warps of a
  // segment wrote A slot t.  tfree[t]: the MMAs reading A slot t completed.
  // accf[i] / acce[i]: accumulator slot i complete / drained.
  auto full_w = [&](int i) { return bar0 + 8u * i; };
  auto wfree = [&](int i) { return bar0 + 8u * (kF8WST + i); };
  auto full_x = [&](int i) { return bar0 + 8u * (2 * kF8WST + i); };
  auto xfree = [&](int i) { return bar0 + 8u * (2 * kF8WST + kF8XST + i); };
  auto a_full = [&](int t) { return bar0 + 8u * (2 * kF8WST + 2 * kF8XST + t); };
  auto tfree = [&](int t) { return bar0 + 8u * (2 * kF8WST + 2 * kF8XST + kF8TSL + t); };
  auto accf = [&](int i) { return bar0 + 8u * (2 * kF8WST + 2 * kF8XST + 2 * kF8TSL + i); };
  auto acce = [&](int i) { return bar0 + 8u * (2 * kF8WST + 2 * kF8XST + 2 * kF8TSL + kF8ASL + i); };
  const uint32_t teardown_bar = bar0 + 8u * (2 * kF8WST + 2 * kF8XST + 2 * kF8TSL + 2 * kF8ASL);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kF8MiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kF8MiscOff + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kF8WST; ++i) {
      mbar_init(full_w(i), 1);
      mbar_init(wfree(i), 8 * 32);  // every expander thread, after its loads returned
    }
    for (int i = 0; i < kF8XST; ++i) {
      mbar_init(full_x(i), 1);
      mbar_init(xfree(i), 1);
    }
    for (int t = 0; t < kF8TSL; ++t) {
      mbar_init(a_full(t), 4);
      mbar_init(tfree(t), 1);
    }
    for (int i = 0; i < kF8ASL; ++i) {
      mbar_init(accf(i), 1);
      mbar_init(acce(i), kEpiThreads / 32);
    }
    mbar_init(teardown_bar, kF8Issuers);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&A4.tm_w);
    tma_prefetch_desc(&a.tm_q);
  }
  if (warp == kF8IssWarp0) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the pre-pass's output, C and the split-K workspace come from earlier kernels
  pdl_wait();

  int w_issued = 0, x_issued = 0;  // producer lanes: copies issued

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      SegRun it(a);
      bool ok = true;
      while (ok && it.next(a)) {
        int32_t tp, tq, m0, m1, n0, n1;
        tile_ranges(a, it.g.tile, 16, tp, tq, m0, m1, n0, n1);
        for (int j = 0; j < it.nseg; j += 2) {
          const int s = w_issued % kF8WST;
          if (!mbar_wait_bounded(wfree(s), ((w_issued / kF8WST) & 1) ^ 1u, a.wait_limit_ns, abort_flag)) {
            if (!*abort_flag) record_timeout(a, abort_flag, 0 * 16 + 1);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_w(s), kF8WStage);
          // byte column of the first code of segment j: 64 codes (32 bytes) per 64-deep K block
          tma_load_2d(base + s * kF8WStage, &A4.tm_w, full_w(s), (it.g.kb0 + 2 * j) * 32, n0);
          ++w_issued;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ activation producer
    if (lane == 0) {
      SegRun it(a);
      int ws = 0;
      bool ok = true;
      while (ok && it.next(a)) {
        for (int j = 0; ok && j < it.nseg; j += 2, ++ws) {
          for (int h = 0; h < 2; ++h) {
            const int sg = 2 * ws + h, s = sg % kF8XST;
            if (!mbar_wait_bounded(xfree(s), ((sg / kF8XST) & 1) ^ 1u, a.wait_limit_ns, abort_flag)) {
              if (!*abort_flag) record_timeout(a, abort_flag, 0 * 16 + 2);
              ok = false;
              break;
            }
            if (j + h < it.nseg) {
              mbar_arrive_expect_tx(full_x(s), kF8XStage);
              tma_load_3d(base + kF8XOff + s * kF8XStage, &a.tm_q, full_x(s), 0, 0, (it.g.kb0 >> 1) + j + h);
              x_issued = sg + 1;
            } else {
              mbar_arrive(full_x(s));  // the empty second segment of a run's last W stage
            }
          }
        }
      }
    }
  } else if (warp < kF8EpiWarp0) {
    // ------------------------------------------------------------ MMA issuers
    // Segment sg = 2 * (W stage) + h goes to issuer sg % 2 and uses A slot
    // sg % 8, activation buffer sg % 4 and accumulator slot sg % 4 (all
    // multiples of the issuer count, so every slot's and buffer's barriers
    // have one waiting issuer, which sees each of their phases in order).  An empty segment (the
    // second of a run's last W stage when the run has an odd number) issues
    // no MMA but keeps every barrier's phase count.
    const int iss = warp - kF8IssWarp0;
    if (lane == 0 && iss < kF8Issuers) {
      SegRun it(a);
      int ws = 0;
      bool ok = true;
      // B: 48 rows of 128 bytes (K-major, 128-byte swizzle, 8-row atoms 1 KiB
      // apart); +32 bytes per 32-deep step.  A: 8 TMEM columns per step.
      while (ok && it.next(a)) {
        for (int j = 0; ok && j < it.nseg; j += 2, ++ws) {
          for (int h = 0; h < 2; ++h) {
            const int sg = 2 * ws + h;
            if (sg % kF8Issuers != iss) continue;
            const int acc = sg % kF8ASL, t = sg % kF8TSL, x = sg % kF8XST;
            if (!mbar_wait_bounded(acce(acc), ((sg / kF8ASL) & 1) ^ 1u, a.wait_limit_ns, abort_flag) ||
                !mbar_wait_bounded(a_full(t), (sg / kF8TSL) & 1, a.wait_limit_ns, abort_flag) ||
                !mbar_wait_bounded(full_x(x), (sg / kF8XST) & 1, a.wait_limit_ns, abort_flag)) {
              if (!*abort_flag) record_timeout(a, abort_flag, 1 * 16 + 4);
              ok = false;
              break;
            }
            tc_fence_after();
            if (j + h < it.nseg) {
              const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kF8N);
              const uint32_t a0 = tmem_base + kF8ACol0 + static_cast<uint32_t>(t * 32);
              const uint64_t bd0 = sw128_desc(base + kF8XOff + x * kF8XStage, 16u, 1024u);
#pragma unroll
              for (int k = 0; k < 4; ++k) tc_mma_f8_ts(d, a0 + 8u * k, bd0 + 2u * k, a.idesc, k ? 1u : 0u);
            }
            tc_commit(tfree(t));
            tc_commit(xfree(x));
            tc_commit(accf(acc));
          }
        }
      }
    }
  } else if (warp >= kF8ExpWarp0) {
    // ------------------------------------------------------------ expanders
    // Warp h of each lane quadrant expands segment 2 * (W stage) + h, whose A
    // slot (sg % 8, so of this warp's parity) only its four warps write and
    // wait on, every phase in order.
    const int q4 = warp & 3;
    const int h = (warp - kF8ExpWarp0) >> 2;  // segment h of every W stage
    const int r = q4 * 32 + lane;             // weight row within the tile (TMEM lane)
    SegRun it(a);
    int ws = 0;  // W stages seen
    bool ok = true;
    while (ok && it.next(a)) {
      for (int j = 0; ok && j < it.nseg; j += 2, ++ws) {
        const bool real = j + h < it.nseg;
        const int sw = ws % kF8WST;
        bool got = mbar_wait_bounded(full_w(sw), (ws / kF8WST) & 1, a.wait_limit_ns, abort_flag);
        if (!got && !*abort_flag) record_timeout(a, abort_flag, 3 * 16 + 0);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        // row r: eight 16-byte chunks, chunk c stored at c ^ (r mod 8); this
        // warp's segment is chunks 4h .. 4h + 3
        uint4 raw[4] = {};
        if (real) {
          const uint8_t* rowp = smem + sw * kF8WStage + r * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) raw[c] = *reinterpret_cast<const uint4*>(rowp + (((4 * h + c) ^ (r & 7)) << 4));
        }
        // hand the stage back once this thread's loads have returned (the
        // arrive depends on their values)
        const uint32_t dep = raw[0].x ^ raw[0].y ^ raw[0].z ^ raw[0].w ^ raw[1].x ^ raw[1].y ^ raw[1].z ^ raw[1].w ^
                             raw[2].x ^ raw[2].y ^ raw[2].z ^ raw[2].w ^ raw[3].x ^ raw[3].y ^ raw[3].z ^ raw[3].w;
        mbar_arrive_after(wfree(sw), base + kF8MiscOff + 8u, dep);  // (misc word 2: the scratch sink)
        const int sg = 2 * ws + h, t = sg % kF8TSL;
        got = mbar_wait_bounded(tfree(t), ((sg / kF8TSL) & 1) ^ 1u, a.wait_limit_ns, abort_flag);
        if (!got && !*abort_flag) record_timeout(a, abort_flag, 3 * 16 + 1);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        if (real) {
          tc_fence_after();
          const uint32_t slot = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + kF8ACol0 +
                                static_cast<uint32_t>(t * 32);
          const uint32_t words[16] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w, raw[1].x, raw[1].y, raw[1].z, raw[1].w,
                                      raw[2].x, raw[2].y, raw[2].z, raw[2].w, raw[3].x, raw[3].y, raw[3].z, raw[3].w};
          uint32_t v[32];
#pragma unroll
          for (int w = 0; w < 16; ++w) {
            // codes k0..k7 of a word: even k in the low nibbles, odd k in the high ones
            v[2 * w] = words[w] & 0x0F0F0F0Fu;
            v[2 * w + 1] = (words[w] >> 4) & 0x0F0F0F0Fu;
          }
          tc_st_32x32b_x32_wait(slot, v);  // store and wait in one statement (source registers)
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(a_full(t));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;
    const int et = threadIdx.x - kF8EpiWarp0 * 32;
    const int row = q4 * 32 + lane;
    const int nblk = a.K >> 7;
    const float* inv_g = A4.inv_scale;
    const float* ag_g = A4.agsum;
    const uint32_t tab = base + kF8TabOff;
    const bool staged = nblk <= kF8TabBlocks;
    if (staged) {
      // the activation tables (1 / S_b and Ag_b, 16 rows each) once per CTA
      for (int i = et; i < nblk * 16; i += kEpiThreads) {
        st_shared_f32(tab + 4u * i, __ldg(inv_g + i));
        st_shared_f32(tab + 4u * (kF8TabBlocks * 16 + i), __ldg(ag_g + i));
      }
    }
    named_bar_sync(1, kEpiThreads);
    auto table4 = [&](int which, int b, int q) -> float4 {
      if (staged) return ld_shared_f32x4(tab + 4u * (which * kF8TabBlocks * 16 + b * 16 + 4 * q));
      return __ldg(reinterpret_cast<const float4*>((which ? ag_g : inv_g) + b * 16) + q);
    };
    // (every run, including runs of empty splits: those still count on the
    // tile's arrival counter, with a zero partial)
    Sched sched(a);
    Group g;
    RowParams rp;
    int ws = 0;  // W stages seen (segment sg = 2 ws + h)
    bool ok = true;
    while (ok && sched.next(a, g)) {
      const int nseg = g.nkb >> 1;
      int32_t tp, tq, m0, m1, n0, n1;
      tile_ranges(a, g.tile, 16, tp, tq, m0, m1, n0, n1);
      const int n = n0 + row;
      const bool live = n < n1;
      const int g_first = static_cast<int>(magic_div(static_cast<uint32_t>(g.kb0), A4.div_kb_per_group));
      rp.reset(live ? A4.scales + static_cast<int64_t>(n) * A4.groups : nullptr,
               (live && A4.zeros) ? A4.zeros + static_cast<int64_t>(n) * A4.groups : nullptr, A4.groups,
               A4.vec_sz != 0, g_first);
      float out[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) out[m] = 0.0f;
      int gcur = -1;
      float sg512 = 0.0f, szg = 0.0f;
      for (int j = 0; j < nseg + (nseg & 1); ++j) {
        const int sg = 2 * ws + (j & 1);
        if (j & 1) ++ws;
        const int blk = (g.kb0 >> 1) + j;  // 128-deep block of K
        if (j >= nseg) {
          // the empty second segment of the run's last W stage: its slot
          // holds nothing of this run; just pass it back
          const int acc = sg % kF8ASL;
          const bool got = mbar_wait_bounded(accf(acc), (sg / kF8ASL) & 1, a.wait_limit_ns, abort_flag);
          if (!got && !*abort_flag) record_timeout(a, abort_flag, 2 * 16 + 9);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(acce(acc));
          continue;
        }
        const int gi = static_cast<int>(magic_div(static_cast<uint32_t>(2 * blk), A4.div_kb_per_group));
        if (gi != gcur) {
          gcur = gi;
          float s, z;
          rp.get(gi, s, z);
          sg512 = 512.0f * s;
          szg = s * z;
        }
        const int acc = sg % kF8ASL;
        const bool got = mbar_wait_bounded(accf(acc), (sg / kF8ASL) & 1, a.wait_limit_ns, abort_flag);
        if (!got && !*abort_flag) record_timeout(a, abort_flag, 2 * 16 + 8);
        // (each warp decides on its own; the four agree at the end of the run)
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t0 = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + static_cast<uint32_t>(acc * kF8N);
        // the three terms: v = D[m] + D[16 + m] / 16 + D[32 + m] / 256 (two
        // loads in flight at a time keeps the registers below the cap of 18 warps)
        float v[16];
        {
          uint32_t d1[16], d2[16];
          tc_ld_32x32b_x16(t0, d1);
          tc_ld_32x32b_x16(t0 + 16u, d2);
          tc_wait_ld_regs(d1);
          tc_regs_after_wait(d2);
#pragma unroll
          for (int m = 0; m < 16; ++m) v[m] = fmaf(__uint_as_float(d2[m]), 0.0625f, __uint_as_float(d1[m]));
          tc_ld_32x32b_x16(t0 + 32u, d1);
          tc_wait_ld_regs(d1);
#pragma unroll
          for (int m = 0; m < 16; ++m) v[m] = fmaf(__uint_as_float(d1[m]), 0.00390625f, v[m]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce(acc));
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 iv = table4(0, blk, q), ag = table4(1, blk, q);
          const float ivs[4] = {iv.x, iv.y, iv.z, iv.w}, ags[4] = {ag.x, ag.y, ag.z, ag.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = 4 * q + e;
            out[m] = fmaf(v[m], sg512 * ivs[e], out[m]);
            out[m] = fmaf(-szg, ags[e], out[m]);
          }
        }
      }
      // all four epilogue warps leave together if any of them gave up a wait
      if (named_bar_or(1, kEpiThreads, !ok)) {
        ok = false;
        break;
      }
      // the run's total: C, or the split-K partial and the tile's arrival
      const bool full_tile = (g.s0 == 0 && g.s1 == a.split);
      if (a.det && !full_tile) {
        int first, nruns;
        tile_runs(a, g.tile, first, nruns);
        const int rr = static_cast<int>(blockIdx.x) - first;
        float* slot = a.slots + (static_cast<int64_t>(g.tile) * a.max_runs + rr) * (static_cast<int64_t>(TILE_P) * 16);
#pragma unroll
        for (int m = 0; m < 16; ++m) slot[static_cast<int64_t>(m) * TILE_P + row] = out[m];
      } else if (live) {
        if (full_tile) {
          uint16_t* cc = reinterpret_cast<uint16_t*>(a.c) + n;
#pragma unroll
          for (int m = 0; m < 16; ++m)
            if (m0 + m < m1) cc[static_cast<int64_t>(m0 + m) * a.ldc] = cvt1(out[m], a.c_bf16);
        } else {
          float* wc = a.ws + n;
#pragma unroll
          for (int m = 0; m < 16; ++m)
            if (m0 + m < m1) red_add_f32(wc + static_cast<int64_t>(m0 + m) * a.N, out[m]);
        }
      }
      if (!full_tile) {
        if (a.det)
          arrive_split_tile_det<16>(a, g, g.tile, m0, m1, n0, n1, et);
        else
          arrive_split_tile<4>(a, g, g.tile, m0, m1, n0, n1, et);  // (a 128 x 16 tile: one pass of 4 loads a thread)
      }
    }
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_flag && lane == 0 && (warp == 0 || warp == 1)) {
    // Let the copies still in flight land before the CTA exits: every buffer
    // use before its last one landed (its consumer waited for it before
    // freeing it), so only each ring's last round can be pending.
    volatile int no_abort = 0;
    if (warp == 0) {
      for (int c = w_issued > kF8WST ? w_issued - kF8WST : 0; c < w_issued; ++c)
        mbar_wait_bounded(full_w(c % kF8WST), (c / kF8WST) & 1, a.wait_limit_ns, &no_abort);
    } else {
      for (int c = x_issued > kF8XST ? x_issued - kF8XST : 0; c < x_issued; ++c)
        mbar_wait_bounded(full_x(c % kF8XST), (c / kF8XST) & 1, a.wait_limit_ns, &no_abort);
    }
  }
  // every issuer's MMAs completed before the TMEM is released
  if (warp >= kF8IssWarp0 && warp < kF8IssWarp0 + kF8Issuers && lane == 0) tc_commit(teardown_bar);
  if (warp == kF8IssWarp0 && lane == 0) {
    volatile int no_abort = 0;
    mbar_wait_bounded(teardown_bar, 0, a.wait_limit_ns, &no_abort);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kF8IssWarp0) tmem_dealloc(tmem_base, 512);
}

}  // namespace

bool int4f8_supported(int a_mn, int64_t M, int64_t K, int group) {
  return !a_mn && M >= 1 && M <= 16 && K % 128 == 0 && group % 128 == 0;
}

size_t int4f8_prep_bytes(int64_t K) { return static_cast<size_t>(K / 128) * kF8N * 128; }

cudaError_t launch_int4f8_prep(const void* A, int64_t lda, int M, int K, void* Xp, float* inv_scale, float* agsum,
                               int sms, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(16) * (K / 8);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > static_cast<int64_t>(sms) * 8) blocks = static_cast<int64_t>(sms) * 8;
  const int vec = (lda % 8 == 0) && (reinterpret_cast<uintptr_t>(A) % 16 == 0);
  return launch_pdl(int4f8_prep_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                    static_cast<const uint16_t*>(A), lda, vec, M, K, static_cast<uint8_t*>(Xp), inv_scale, agsum);
}

cudaError_t launch_int4f8_gemm(const Int4Args& args, int grid, cudaStream_t stream) {
  cudaError_t e = set_smem_once<int4f8_gemm_kernel>(static_cast<int>(kF8Smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(int4f8_gemm_kernel, dim3(static_cast<unsigned>(grid)), dim3(kF8Threads), kF8Smem, stream, args);
}

}  // namespace lgt
