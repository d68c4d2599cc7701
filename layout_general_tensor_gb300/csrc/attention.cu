// Fused attention forward: O = softmax(Q K^T * scale) V per head, the second
// product P.V taken with V as it is stored (contiguous along head_dim), an
// MN-major operand of the tensor core -- the non-TN second dot of Flash
// Attention that the Triton inThreadTranspose page names ("Introduction").
//
// One CTA per 128 queries of a head; the head's keys in blocks of 128.
//   S_j = Q K_j^T       tcgen05 MMA, both operands K-major (TMA, 128-byte
//                       swizzle), fp32 accumulator in tensor memory.
//   P_j, m, l           online softmax by eight warps, two per query row
//                       quadrant (half of the keys each), one row per
//                       thread, the logits held in registers: a
//                       reference maximum m (of the logits times
//                       scale * log2 e) moved only when a block's maximum
//                       exceeds it by more than 8, running sum l;
//                       P_j = 2^(s - m) (at most 2^8)
//                       rounded to the input type into tensor memory; the
//                       O accumulator rescaled by 2^(m_old - m) in the
//                       blocks where m moved.
//   O += P_j V_j        tcgen05 MMA with A = P_j from tensor memory and
//                       B = V_j MN-major from shared memory.
//   O / l               the softmax warps, then 16-byte stores.
// S is double-buffered, so S_{j+1} is computed while the softmax works on
// S_j; P is double-buffered, so P_j is written while P_{j-1} is multiplied.
//
// Warp roles (384 threads): warp 0 TMA producer (Q once, rings of K and V
// tiles), warp 1 S issuer (owns the tensor memory), warp 2 P.V issuer,
// warps 4..11 softmax
// and epilogue, two per tensor-memory lane quadrant (warp % 4), each taking
// half of a block's keys and half of O's columns.  Tensor memory: S at
// columns 0 and 128, P at 256 and 320 (bf16 / fp16 pairs), O at 384.
// Every wait is bounded; a wait that runs out records GEMM_ERR_TIMEOUT and
// the CTA winds down.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <new>

#include "attention.h"
#include "kernels.h"
#include "plan.h"
#include "ptx.cuh"

namespace lgt {
namespace {

constexpr int kAttnThreads = 384;
constexpr int kBM = 128;  // queries per CTA
constexpr int kBN = 128;  // keys per block
constexpr int kSoftWarp0 = 4;   // softmax warps 4..11: two per lane quadrant
constexpr int kAttnTimeout = 6;  // GEMM_ERR_TIMEOUT
constexpr uint32_t kTmemO = 384;

struct AttnArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // 3-D {head_dim, rows, heads}, box {64, 128, 1}
  void* o;
  DeviceStatus* status;
  uint64_t wait_limit_ns;
  int32_t heads, sq, sk;
  float cs;  // scale * log2(e)
  uint32_t idesc_s, idesc_pv;
  int32_t bf16;
};

template <int D>
struct AttnCfg {
  static constexpr uint32_t CHUNK = 128u * 128u;      // one 64-wide box of 128 rows: 16 KiB
  static constexpr uint32_t TILE = (D / 64) * CHUNK;  // a Q, K or V tile
  // K and V rings of their own: a K tile is free once S = Q K^T completed,
  // a V tile only once P.V completed, so K is loaded further ahead
  static constexpr int NSK = D == 128 ? 3 : 4;
  static constexpr int NSV = D == 128 ? 2 : 3;
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = TILE;
  static constexpr uint32_t V_OFF = K_OFF + NSK * TILE;
  static constexpr uint32_t BAR_OFF = V_OFF + NSV * TILE;
  // q_full, k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV], s_full[2], s_free[2], p_full[2], pv_done[2],
  // teardown
  static constexpr int NBARS = 1 + 2 * NSK + 2 * NSV + 8 + 1;
  // the two softmax halves of a row exchange their block maxima (by block
  // parity) and, at the end, their partial sums: fp32 [2][2][128]
  static constexpr uint32_t XCH_OFF = BAR_OFF + ((NBARS * 8 + 15) & ~15);
  static constexpr uint32_t MISC_OFF = XCH_OFF + 2 * 2 * 128 * 4;
  static constexpr uint32_t SMEM = MISC_OFF + 16 + 1024;  // slack for the 1024-byte alignment
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2^x (the hardware approximation; 2^-inf = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two floats as one word of 16-bit values (lo in the low half), rounded to nearest.
template <bool BF16>
__device__ __forceinline__ uint32_t pack_pair(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void attn_timeout(const AttnArgs& a, volatile int* abort_flag, int where) {
  *abort_flag = 1;
  if (atomicCAS(&a.status->code, 0, kAttnTimeout) == 0) a.status->where = where;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnArgs a) {
  using C = AttnCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int q0 = blockIdx.x * kBM;
  const int nb = (a.sk + kBN - 1) / kBN;

  const uint32_t bar0 = base + C::BAR_OFF;
  const uint32_t q_full = bar0;
  constexpr int kB = 1 + 2 * C::NSK + 2 * C::NSV;
  auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto k_empty = [&](int s) { return bar0 + 8u * (1 + C::NSK + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (1 + 2 * C::NSK + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (1 + 2 * C::NSK + C::NSV + s); };
  auto s_full = [&](int b) { return bar0 + 8u * (kB + b); };
  auto s_free = [&](int b) { return bar0 + 8u * (kB + 2 + b); };
  auto p_full = [&](int b) { return bar0 + 8u * (kB + 4 + b); };
  auto pv_done = [&](int b) { return bar0 + 8u * (kB + 6 + b); };
  const uint32_t teardown = bar0 + 8u * (kB + 8);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NSK; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < C::NSV; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(s_free(b), 8);  // the eight softmax warps
      mbar_init(p_full(b), 8);
      mbar_init(pv_done(b), 1);
    }
    mbar_init(teardown, 2);  // both MMA issuers
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&a.tm_q);
    tma_prefetch_desc(&a.tm_k);
    tma_prefetch_desc(&a.tm_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Q, K and V may come from the previous kernel, which may also read O
  pdl_wait();

  bool q_issued = false;
  int k_issued = 0, v_issued = 0;  // producer lane: K / V tiles whose loads were issued

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, C::TILE);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_load_3d(base + C::Q_OFF + c * C::CHUNK, &a.tm_q, q_full, c * 64, q0, h);
      q_issued = true;
      // the two rings, each fed as soon as its next buffer is free
      uint64_t stall_t0 = 0;
      while (k_issued < nb || v_issued < nb) {
        bool progress = false;
        if (k_issued < nb) {
          const int j = k_issued, s = j % C::NSK;
          if (j < C::NSK || mbar_test_wait(k_empty(s), ((j / C::NSK) - 1) & 1)) {
            const uint32_t kd = base + C::K_OFF + s * C::TILE;
            mbar_arrive_expect_tx(k_full(s), C::TILE);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tma_load_3d(kd + c * C::CHUNK, &a.tm_k, k_full(s), c * 64, j * kBN, h);
            ++k_issued;
            progress = true;
          }
        }
        if (v_issued < nb && v_issued < k_issued) {
          const int j = v_issued, s = j % C::NSV;
          if (j < C::NSV || mbar_test_wait(v_empty(s), ((j / C::NSV) - 1) & 1)) {
            const uint32_t vd = base + C::V_OFF + s * C::TILE;
            mbar_arrive_expect_tx(v_full(s), C::TILE);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tma_load_3d(vd + c * C::CHUNK, &a.tm_v, v_full(s), c * 64, j * kBN, h);
            ++v_issued;
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
          attn_timeout(a, abort_flag, 0);
          break;
        }
        __nanosleep(64);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    // One thread issues a tcgen05 MMA only every hundred-odd cycles, so the
    // two products have issuers of their own: this one S = Q K^T, warp 2
    // O += P V (disjoint accumulators; they meet only through barriers).
    if (lane == 0) {
      bool ok = mbar_wait_bounded(q_full, 0, a.wait_limit_ns, abort_flag);
      // S_j = Q K_j^T into S buffer j % 2 (once the softmax has read S_{j-2}).
      // K-major tiles: 128-byte rows of 64 elements, 8-row groups 1 KiB
      // apart; 16-deep step k is 32 bytes into 64-wide chunk k / 4.
      for (int j = 0; ok && j < nb; ++j) {
        const int b = j & 1, s = j % C::NSK;
        if ((j >= 2 && !mbar_wait_bounded(s_free(b), ((j >> 1) - 1) & 1, a.wait_limit_ns, abort_flag)) ||
            !mbar_wait_bounded(k_full(s), (j / C::NSK) & 1, a.wait_limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kb = base + C::K_OFF + s * C::TILE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = static_cast<uint32_t>(k >> 2) * C::CHUNK + static_cast<uint32_t>(k & 3) * 32u;
          tc_mma_f16_ss(tmem + static_cast<uint32_t>(b * 128), sw128_desc(base + C::Q_OFF + off, 16u, 1024u),
                        sw128_desc(kb + off, 16u, 1024u), a.idesc_s, k > 0 ? 1u : 0u);
        }
        tc_commit(s_full(b));
        tc_commit(k_empty(s));
      }
      if (!ok && !*abort_flag) attn_timeout(a, abort_flag, 1);
      tc_commit(teardown);  // every MMA of this thread completed before the tensor memory is freed
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ P.V issuer
    if (lane == 0) {
      bool ok = true;
      for (int j = 0; j < nb; ++j) {
        const int b = j & 1, s = j % C::NSV;
        if (!mbar_wait_bounded(p_full(b), (j >> 1) & 1, a.wait_limit_ns, abort_flag) ||
            !mbar_wait_bounded(v_full(s), (j / C::NSV) & 1, a.wait_limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // O += P_j V_j: A = P_j (8 columns of pairs per 16 keys), B = V_j
        // MN-major: 128-byte rows along head_dim, one per key, 8-key groups
        // 1 KiB apart, 64-wide head_dim chunks 16 KiB apart; 16 keys = 2 KiB.
        const uint32_t vb = base + C::V_OFF + s * C::TILE;
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)
          mma_ts(tmem + kTmemO, tmem + 256u + static_cast<uint32_t>(b * 64 + k * 8),
                 sw128_desc(vb + static_cast<uint32_t>(k) * 2048u, C::CHUNK, 1024u), a.idesc_pv,
                 (j | k) != 0 ? 1u : 0u);
        tc_commit(pv_done(b));
        tc_commit(v_empty(s));
      }
      if (!ok && !*abort_flag) attn_timeout(a, abort_flag, 1);
      tc_commit(teardown);
    }
  } else if (warp >= kSoftWarp0) {
    // ------------------------------------------------------------ softmax
    const int q4 = warp & 3;
    const int hh = (warp - kSoftWarp0) >> 2;  // this warp's half of a block's keys and of O's columns
    const int row = q4 * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q4 * 32) << 16);  // this warp's lane quadrant
    const uint32_t pair_bar = 1u + static_cast<uint32_t>(q4);            // named barrier of the two halves
    const uint32_t xch = base + C::XCH_OFF;
    // m: the reference maximum of this row's scaled logits (log2 units) that
    // P is taken against.  It moves only when a block's maximum exceeds it
    // by more than kLazy: P then stays at most 2^kLazy (safe in 16-bit and
    // in the fp32 sums), and O is rescaled -- after waiting for the P.V
    // before -- only in the blocks where some row of the warp moved.  The
    // result O / l does not depend on the reference.  The two halves of a
    // row see the same block maximum (exchanged) and so move m together; each
    // keeps the partial sum of its keys.  Every wait's outcome is agreed
    // between the two halves before they part, so both take the same path
    // to every named barrier.
    constexpr float kLazy = 8.0f;
    const float cs = a.cs;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      const int b = j & 1;
      // S_j, and P buffer b free (PV_{j-2} done), agreed by both halves at once
      bool got = mbar_wait_bounded(s_full(b), (j >> 1) & 1, a.wait_limit_ns, abort_flag);
      if (got && j >= 2) got = mbar_wait_bounded(pv_done(b), ((j >> 1) - 1) & 1, a.wait_limit_ns, abort_flag);
      if (named_bar_or(pair_bar, 64, !got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int valid = min(kBN, a.sk - j * kBN) - hh * 64;  // keys of this half inside the head
      const uint32_t sb = tl + static_cast<uint32_t>(b * 128 + hh * 64);
      // this half's 64 logits in registers, then the S buffer is free for S_{j+2}
      uint32_t sv[64];
      tc_ld_32x32b_x32(sb, *reinterpret_cast<uint32_t(*)[32]>(sv));
      tc_ld_32x32b_x32(sb + 32u, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
      tc_wait_ld_regs(sv);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(b));
      // (keys past the head's end, in its last block only, count as -inf)
      if (valid < 64) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i >= valid) sv[i] = __float_as_uint(-INFINITY);
      }
      // (eight independent partial maxima and sums: short dependency chains)
      float mp[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mp[u] = __uint_as_float(sv[u]);
#pragma unroll
      for (int i = 8; i < 64; ++i) mp[i & 7] = fmaxf(mp[i & 7], __uint_as_float(sv[i]));
      float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])), fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      // the block maximum of the whole row: exchange with the other half
      st_shared_f32(xch + static_cast<uint32_t>(((b * 2 + hh) * 128 + row) * 4), mx);
      named_bar_sync(pair_bar, 64);
      mx = fmaxf(mx, ld_shared_f32(xch + static_cast<uint32_t>(((b * 2 + (hh ^ 1)) * 128 + row) * 4))) * cs;
      float alpha = 1.0f;
      if (mx > m + kLazy) {  // always on the first block (m = -inf)
        alpha = ex2(m - mx);  // 0 on the first block
        m = mx;
      }
      // P = 2^(s cs - m) as pairs: 64 keys, 32 pair columns
      float sp[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) sp[u] = 0.0f;
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float e0 = ex2(fmaf(__uint_as_float(sv[2 * i]), cs, -m));  // -inf past the end: 0
        const float e1 = ex2(fmaf(__uint_as_float(sv[2 * i + 1]), cs, -m));
        sp[i & 7] += e0 + e1;
        pk[i] = pack_pair<BF16>(e0, e1);
      }
      tc_st_32x32b_x32_wait(tl + 256u + static_cast<uint32_t>(b * 64 + hh * 32), pk);
      const float sum = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
      l = l * alpha + sum;
      // O holds the sum up to block j - 1: rescale this half's columns (once
      // PV_{j-1} is done) where a row's reference moved (the same rows in
      // both halves)
      if (j >= 1 && __any_sync(0xffffffffu, alpha < 1.0f)) {
        got = mbar_wait_bounded(pv_done((j - 1) & 1), ((j - 1) >> 1) & 1, a.wait_limit_ns, abort_flag);
        if (named_bar_or(pair_bar, 64, !got)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          const uint32_t col = kTmemO + static_cast<uint32_t>(hh * (D / 2) + c * 32);
          uint32_t v[32];
          tc_ld_32x32b_x32(tl + col, v);
          tc_wait_ld_regs(v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tc_st_32x32b_x32_wait(tl + col, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(b));
    }
    if (ok) {
      // the last PV done: O / l (the two halves' sums added), rounded once,
      // 16-byte stores of this half of the row
      const bool got = mbar_wait_bounded(pv_done((nb - 1) & 1), ((nb - 1) >> 1) & 1, a.wait_limit_ns, abort_flag);
      if (!named_bar_or(pair_bar, 64, !got)) {
        tc_fence_after();
        st_shared_f32(xch + static_cast<uint32_t>((hh * 128 + row) * 4), l);
        named_bar_sync(pair_bar, 64);
        const float inv = 1.0f / (l + ld_shared_f32(xch + static_cast<uint32_t>(((hh ^ 1) * 128 + row) * 4)));
        const bool in = q0 + row < a.sq;
        uint16_t* orow = static_cast<uint16_t*>(a.o) + (static_cast<int64_t>(h) * a.sq + q0 + row) * D + hh * (D / 2);
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          uint32_t v[32];
          tc_ld_32x32b_x32(tl + kTmemO + static_cast<uint32_t>(hh * (D / 2) + c * 32), v);
          tc_wait_ld_regs(v);
          if (in) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = pack_pair<BF16>(__uint_as_float(v[8 * q + 2 * e]) * inv,
                                       __uint_as_float(v[8 * q + 2 * e + 1]) * inv);
              st_global_v4(orow + c * 32 + 8 * q, w[0], w[1], w[2], w[3]);
            }
          }
        }
      } else if (!*abort_flag) {
        attn_timeout(a, abort_flag, 2);
      }
    } else if (!*abort_flag) {
      attn_timeout(a, abort_flag, 2);
    }
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // let the loads still in flight land before the CTA exits
    volatile int no_abort = 0;
    if (q_issued) mbar_wait_bounded(q_full, 0, a.wait_limit_ns, &no_abort);
    for (int j = k_issued > C::NSK ? k_issued - C::NSK : 0; j < k_issued; ++j)
      mbar_wait_bounded(k_full(j % C::NSK), (j / C::NSK) & 1, a.wait_limit_ns, &no_abort);
    for (int j = v_issued > C::NSV ? v_issued - C::NSV : 0; j < v_issued; ++j)
      mbar_wait_bounded(v_full(j % C::NSV), (j / C::NSV) & 1, a.wait_limit_ns, &no_abort);
  }
  if (warp == 1 && lane == 0) {
    volatile int no_abort = 0;
    mbar_wait_bounded(teardown, 0, a.wait_limit_ns, &no_abort);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int D, bool BF16>
cudaError_t launch_attn(const AttnArgs& args, cudaStream_t stream) {
  using C = AttnCfg<D>;
  static const cudaError_t set = cudaFuncSetAttribute(attn_fwd_kernel<D, BF16>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                      static_cast<int>(C::SMEM));
  if (set != cudaSuccess) return set;
  const dim3 grid(static_cast<unsigned>((args.sq + kBM - 1) / kBM), static_cast<unsigned>(args.heads));
  return launch_pdl(attn_fwd_kernel<D, BF16>, grid, dim3(kAttnThreads), C::SMEM, stream, args);
}

// 3-D map over heads x rows x head_dim (16-bit, [head][row][d] contiguous):
// box {64, 128, 1}, 128-byte swizzle, zero fill past the rows of a head.
bool encode_attn(CUtensorMap* map, const void* ptr, int dtype, int64_t heads, int64_t rows, int64_t d) {
  auto enc = get_encoder();
  if (!enc) return false;
  const CUtensorMapDataType dt =
      dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(rows * d) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBN), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint64_t attn_wait_limit() {
  const char* s = std::getenv("LGT_GEMM_WAIT_LIMIT_MS");
  if (s && *s) {
    const double ms = std::atof(s);
    if (ms > 0) return static_cast<uint64_t>(ms * 1e6);
  }
  return 2000ull * 1000ull * 1000ull;  // 2 s
}

}  // namespace
}  // namespace lgt

struct attn_plan {
  attn_desc_t d;
  int device = -1;
  lgt::DeviceStatus* d_status = nullptr;
  uint64_t wait_limit_ns = 0;
  // arguments of the last run: the maps are re-encoded only when a pointer changes
  lgt::AttnArgs args;
  const void* q = nullptr;
  const void* k = nullptr;
  const void* v = nullptr;
  bool have = false;
};

extern "C" {

gemm_status_t attn_create(const attn_desc_t* desc, attn_plan_t** plan) {
  if (!desc || !plan) return GEMM_ERR_INVALID_ARG;
  *plan = nullptr;
  const attn_desc_t& d = *desc;
  if (d.heads < 1 || d.heads > 65535 || d.seq_q < 1 || d.seq_k < 1 || (d.head_dim != 64 && d.head_dim != 128) ||
      (d.dtype != GEMM_F16 && d.dtype != GEMM_BF16) || !(d.scale >= 0.0f) || std::isinf(d.scale))
    return GEMM_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  attn_plan* p = new (std::nothrow) attn_plan();
  if (!p) return GEMM_ERR_CUDA;
  p->d = d;
  p->device = dev;
  p->wait_limit_ns = lgt::attn_wait_limit();
  if (cudaMalloc(&p->d_status, 16) != cudaSuccess || cudaMemset(p->d_status, 0, 16) != cudaSuccess) {
    cudaGetLastError();
    if (p->d_status) cudaFree(p->d_status);
    delete p;
    return GEMM_ERR_CUDA;
  }
  *plan = p;
  return GEMM_OK;
}

gemm_status_t attn_run(attn_plan_t* plan, const void* Q, const void* K, const void* V, void* O, void* stream) {
  if (!plan || !Q || !K || !V || !O) return GEMM_ERR_INVALID_ARG;
  for (const void* ptr : {Q, K, V, static_cast<const void*>(O)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return GEMM_ERR_ALIGNMENT;
  const attn_desc_t& d = plan->d;
  lgt::AttnArgs& a = plan->args;
  if (!plan->have || plan->q != Q || plan->k != K || plan->v != V) {
    if (!lgt::encode_attn(&a.tm_q, Q, d.dtype, d.heads, d.seq_q, d.head_dim) ||
        !lgt::encode_attn(&a.tm_k, K, d.dtype, d.heads, d.seq_k, d.head_dim) ||
        !lgt::encode_attn(&a.tm_v, V, d.dtype, d.heads, d.seq_k, d.head_dim)) {
      plan->have = false;
      return GEMM_ERR_CUDA;
    }
    plan->q = Q;
    plan->k = K;
    plan->v = V;
    plan->have = true;
    const float scale = d.scale > 0.0f ? d.scale : 1.0f / std::sqrt(static_cast<float>(d.head_dim));
    a.cs = scale * 1.4426950408889634f;  // log2(e)
    a.heads = d.heads;
    a.sq = d.seq_q;
    a.sk = d.seq_k;
    a.bf16 = d.dtype == GEMM_BF16;
    a.idesc_s = lgt::idesc_f16(a.bf16, 0u, 0u, 128u, 128u);
    a.idesc_pv = lgt::idesc_f16(a.bf16, 0u, 1u, 128u, static_cast<uint32_t>(d.head_dim));
    a.status = plan->d_status;
    a.wait_limit_ns = plan->wait_limit_ns;
  }
  a.o = O;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = d.head_dim == 128 ? (a.bf16 ? lgt::launch_attn<128, true>(a, s) : lgt::launch_attn<128, false>(a, s))
                                          : (a.bf16 ? lgt::launch_attn<64, true>(a, s) : lgt::launch_attn<64, false>(a, s));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return GEMM_OK;
}

gemm_status_t attn_sync_status(attn_plan_t* plan, void* stream) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  if (plan->device < 0 || !plan->d_status) return GEMM_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GEMM_ERR_CUDA;
  lgt::DeviceStatus st;
  if (cudaMemcpy(&st, plan->d_status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
  if (st.code != 0) {
    if (cudaMemset(plan->d_status, 0, sizeof(st)) != cudaSuccess) return GEMM_ERR_CUDA;
    return static_cast<gemm_status_t>(st.code);
  }
  return GEMM_OK;
}

gemm_status_t attn_destroy(attn_plan_t* plan) {
  if (!plan) return GEMM_OK;
  if (plan->d_status) cudaFree(plan->d_status);
  delete plan;
  return GEMM_OK;
}

}  // extern "C"
