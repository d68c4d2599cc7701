// Device-side pieces shared by the tensor-core GEMM kernels: the (tile,
// split) work scheduler, output conversion, and the epilogue with the
// cross-CTA fp32 split-K reduction.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace lgt {
namespace {

constexpr int kEpiThreads = 128;
constexpr int kTimeoutCode = 6;  // GEMM_ERR_TIMEOUT

struct Group {
  int32_t tile;
  int32_t s0, s1;    // splits [s0, s1) of the tile
  int32_t kb0, nkb;  // K blocks
};

// Work assignment.  Two kinds of groups:
//  - round-robin tiles [0, rr_tiles): worker b takes tiles b, b+G, b+2G, ...
//    each as one whole group (all of its K blocks);
//  - contiguous units [rr_tiles * split, num_units), unit u = tile * split + s:
//    worker b takes [b*U/G, (b+1)*U/G) of the U units; a group is a maximal
//    run of one tile's units.
// Order for one worker: its first round-robin tile, then its contiguous
// units, then its other round-robin tiles.  split == 1 has round-robin tiles
// only; an explicit split > 1 has contiguous units only (consecutive splits
// of one tile then accumulate in TMEM).  The stream-K tail has both, with
// split = the K blocks of a tile: one whole wave first warms L2 with the
// operands, then the tail units run and their partial sums complete early,
// so that their conversion (by the fixup warps) overlaps the later waves.
// A worker is a CTA, or a CTA pair (both CTAs walk the same units).
struct Sched {
  int32_t u, u_end;          // contiguous-unit cursor
  int32_t r, r_end, r_step;  // round-robin cursor
  bool first;                // the first round-robin tile is still to come
  __device__ Sched(const TcArgs& a) {
    const int32_t G = gridDim.x >> a.pair, b = blockIdx.x >> a.pair;
    r = b;
    r_end = a.rr_tiles;
    r_step = G;
    first = true;
    const int64_t u0 = static_cast<int64_t>(a.rr_tiles) * a.split;
    const int64_t U = static_cast<int64_t>(a.num_units) - u0;
    u = static_cast<int32_t>(u0 + (static_cast<int64_t>(b) * U) / G);
    u_end = static_cast<int32_t>(u0 + (static_cast<int64_t>(b + 1) * U) / G);
  }
  __device__ bool next(const TcArgs& a, Group& g) {
    const bool rr_now = r < r_end && (first || u >= u_end);
    first = false;
    if (rr_now) {
      g.tile = r;
      g.s0 = 0;
      g.s1 = a.split;
      r += r_step;
    } else if (u < u_end) {
      uint32_t tile, s;
      magic_divmod(static_cast<uint32_t>(u), a.div_split, tile, s);
      const int32_t avail = u_end - u;
      const int32_t s1 = min(a.split, static_cast<int32_t>(s) + avail);
      g.tile = static_cast<int32_t>(tile);
      g.s0 = static_cast<int32_t>(s);
      g.s1 = s1;
      u += s1 - static_cast<int32_t>(s);
    } else {
      return false;
    }
    g.kb0 = g.s0 * a.kb_per_split;
    const int32_t kb1 = min(a.kb_total, g.s1 * a.kb_per_split);
    g.nkb = kb1 > g.kb0 ? kb1 - g.kb0 : 0;
    return true;
  }
};

__device__ __forceinline__ void record_timeout(const TcArgs& a, volatile int* abort_flag, int where) {
  *abort_flag = 1;
  if (atomicCAS(&a.status->code, 0, kTimeoutCode) == 0) a.status->where = where;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint16_t cvt1(float v, int bf16) {
  if (bf16) {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t*>(&h);
  }
  __half h = __float2half_rn(v);
  return *reinterpret_cast<uint16_t*>(&h);
}

// (m, n) ranges of a tile in C coordinates.  A pair tile is 256 rows high
// on the P side.
__device__ __forceinline__ void tile_ranges(const TcArgs& a, int32_t tile, int bn, int32_t& tp, int32_t& tq,
                                            int32_t& m0, int32_t& m1, int32_t& n0, int32_t& n1) {
  uint32_t q, r;
  magic_divmod(static_cast<uint32_t>(tile), a.div_tiles_p, q, r);
  tp = static_cast<int32_t>(r);
  tq = static_cast<int32_t>(q);
  const int32_t pt = TILE_P << a.pair;
  if (!a.swap) {
    m0 = tp * pt;
    n0 = tq * bn;
    m1 = min(a.M, m0 + pt);
    n1 = min(a.N, n0 + bn);
  } else {
    n0 = tp * pt;
    m0 = tq * bn;
    n1 = min(a.N, n0 + pt);
    m1 = min(a.M, m0 + bn);
  }
}

// The 128 P-side rows of a pair tile that CTA `half` of the pair holds in its
// TMEM (may be empty at a ragged edge).
__device__ __forceinline__ void narrow_to_half(const TcArgs& a, int half, int32_t& m0, int32_t& m1, int32_t& n0,
                                               int32_t& n1) {
  if (!a.swap) {
    m0 += half * TILE_P;
    m1 = max(m0, min(m1, m0 + TILE_P));
  } else {
    n0 += half * TILE_P;
    n1 = max(n0, min(n1, n0 + TILE_P));
  }
}

// Convert the fp32 sums of C rows [m0, m1) x columns [n0, n1) from the
// workspace (L2), store them to C and zero the workspace region again.  The
// 128 epilogue threads walk the region in 4-float vectors with U loads in
// flight per thread: a round trip to L2 costs microseconds on this GPU, so
// the loads of a whole region should be in flight together.
template <int U>
__device__ __noinline__ void finish_tile(const TcArgs& a, int m0, int m1, int n0, int n1, int et) {
  const int rows = m1 - m0, cols = n1 - n0;
  uint16_t* cbase = reinterpret_cast<uint16_t*>(a.c);
  if (a.ws_vec && a.c_vec && (cols & 3) == 0) {
    // c_vec: C rows and n0 are 16-byte aligned, so 4-element (8-byte) stores are aligned too
    const int cols4 = cols >> 2;
    const int total = rows * cols4;
    for (int i0 = et; i0 < total; i0 += kEpiThreads * U) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * kEpiThreads;
        if (i < total) {
          const int r = i / cols4, c4 = i - r * cols4;
          v[u] = __ldcg(reinterpret_cast<const float4*>(a.ws + static_cast<int64_t>(m0 + r) * a.N + n0) + c4);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * kEpiThreads;
        if (i < total) {
          const int r = i / cols4, c4 = i - r * cols4;
          __stcg(reinterpret_cast<float4*>(a.ws + static_cast<int64_t>(m0 + r) * a.N + n0) + c4,
                 make_float4(0.f, 0.f, 0.f, 0.f));
          uint2 o;
          o.x = pack2(v[u].x, v[u].y, a.c_bf16);
          o.y = pack2(v[u].z, v[u].w, a.c_bf16);
          *reinterpret_cast<uint2*>(cbase + static_cast<int64_t>(m0 + r) * a.ldc + n0 + 4 * c4) = o;
        }
      }
    }
    return;
  }
  const int total = rows * cols;
  constexpr int U1 = U < 8 ? U : 8;
  for (int i0 = et; i0 < total; i0 += kEpiThreads * U1) {
    float v[U1];
#pragma unroll
    for (int u = 0; u < U1; ++u) {
      const int i = i0 + u * kEpiThreads;
      if (i < total) {
        const int r = i / cols, cidx = i - r * cols;
        v[u] = __ldcg(a.ws + static_cast<int64_t>(m0 + r) * a.N + (n0 + cidx));
      }
    }
#pragma unroll
    for (int u = 0; u < U1; ++u) {
      const int i = i0 + u * kEpiThreads;
      if (i < total) {
        const int r = i / cols, cidx = i - r * cols;
        __stcg(a.ws + static_cast<int64_t>(m0 + r) * a.N + (n0 + cidx), 0.0f);
        cbase[static_cast<int64_t>(m0 + r) * a.ldc + (n0 + cidx)] = cvt1(v[u], a.c_bf16);
      }
    }
  }
}

// Deterministic split-K.  The worker (CTA or CTA pair) that owns unit u of
// the contiguous-unit phase: the largest b with floor(b*U/G) <= u - u0.
__device__ __forceinline__ int unit_owner(const TcArgs& a, int64_t u) {
  const int64_t G = gridDim.x >> a.pair;
  const int64_t u0 = static_cast<int64_t>(a.rr_tiles) * a.split;
  const int64_t U = static_cast<int64_t>(a.num_units) - u0;
  const int64_t v = u - u0;
  int64_t b = (v * G) / U;
  while (b + 1 < G && ((b + 1) * U) / G <= v) ++b;
  while (b > 0 && (b * U) / G > v) --b;
  return static_cast<int>(b);
}

// Runs of tile `tile` (one per worker its units meet) and the slot index of
// this worker's run.
__device__ __forceinline__ void tile_runs(const TcArgs& a, int tile, int& first_owner, int& nruns) {
  const int64_t u = static_cast<int64_t>(a.rr_tiles) * a.split + static_cast<int64_t>(tile - a.rr_tiles) * a.split;
  first_owner = unit_owner(a, u);
  nruns = unit_owner(a, u + a.split - 1) - first_owner + 1;
}

// Last arriver of a deterministic split tile: C = the sum of the tile's run
// slots in run order (rows x cols of C at m0 / n0; slot element (i, j) at
// i * cols_ld + j, i the C row within the strip).
template <int U>
__device__ __noinline__ void finish_tile_det(const TcArgs& a, const float* slot0, int64_t slot_elems, int nruns,
                                             int m0, int m1, int n0, int n1, int cols_ld, int et) {
  const int rows = m1 - m0, cols = n1 - n0;
  uint16_t* cbase = reinterpret_cast<uint16_t*>(a.c);
  const int total = rows * cols;
  for (int i0 = et; i0 < total; i0 += kEpiThreads * U) {
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = 0.0f;
    for (int r = 0; r < nruns; ++r) {
      const float* slot = slot0 + static_cast<int64_t>(r) * slot_elems;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * kEpiThreads;
        if (i < total) {
          const int rr = i / cols, cc = i - rr * cols;
          v[u] += __ldcg(slot + static_cast<int64_t>(rr) * cols_ld + cc);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * kEpiThreads;
      if (i < total) {
        const int rr = i / cols, cc = i - rr * cols;
        cbase[static_cast<int64_t>(m0 + rr) * a.ldc + (n0 + cc)] = cvt1(v[u], a.c_bf16);
      }
    }
  }
}

// After the 128 epilogue threads have added a run's fp32 partial into the
// workspace: count the run's splits on the tile's arrival counter, and if
// this arrival completes the tile, convert it (the CTA that arrives last
// reads the full sum from L2), then reset the counter.
// FU: loads in flight per thread in the conversion (registers permitting).
// Ordering: every thread's partial adds are fenced before the barrier; the
// counting thread fences again after it (so that its count, at GPU scope,
// follows the adds of the whole CTA it has synchronised with: a relaxed
// atomic after a CTA barrier alone does not publish other threads' writes)
// and after its atomic (so that the reads of a finishing CTA follow every
// count it has seen).
template <int FU = 8>
__device__ __forceinline__ void arrive_split_tile(const TcArgs& a, const Group& g, int counter, int m0, int m1, int n0,
                                                  int n1, int et) {
  __threadfence();
  named_bar_sync(1, kEpiThreads);
  if (a.tail_tiles) {
    // stream-K tail: count the arrival only; every CTA finishes a share of
    // the tail tiles at the end (finish_tail)
    if (et == 0) {
      __threadfence();
      atomicAdd(&a.counters[counter], g.s1 - g.s0);
    }
    return;
  }
  bool mine_last = false;
  if (et == 0) {
    __threadfence();
    const int old = atomicAdd(&a.counters[counter], g.s1 - g.s0);
    mine_last = (old + (g.s1 - g.s0) == a.split);
    __threadfence();
  }
  if (named_bar_or(1, kEpiThreads, mine_last)) {
    __threadfence();
    finish_tile<FU>(a, m0, m1, n0, n1, et);
    named_bar_sync(1, kEpiThreads);
    if (et == 0) a.counters[counter] = 0;
  }
}

// Conversion of split tiles by the 128 fixup threads of every CTA (their own
// warps, named barrier 2): the tiles [rr_tiles, rr_tiles + tail_tiles) --
// a stream-K tail, or every tile of a split-K plan.  Each tile is cut into
// strips (the two halves of a pair tile; the tile itself otherwise) of
// C rows (128, or BN when swapped), shared among the CTAs (see below): for
// each strip it serves, a CTA waits until all of the strip's K blocks have
// arrived (for a
// stream-K tail early in the kernel, behind the whole tiles' main loops;
// for split-K at the end, all CTAs at once), converts and stores its rows
// of C, zeroes them in the workspace, and counts them on the strip's second
// counter; the CTA completing a strip resets both counters for the next
// run.  Spreading the reads over all SMs matters: one CTA reading a whole
// tile competes with its own main loop for the SM's L2 bandwidth.
template <int BN>
__device__ __noinline__ bool finish_tail(const TcArgs& a, volatile int* abort_flag, int et) {
  constexpr int kBar = 2;
  const int halves = 1 + a.pair;
  const int strip_rows = a.swap ? BN : TILE_P;
  const int S = a.tail_tiles * halves;  // strips
  const int G = gridDim.x, c = blockIdx.x;
  // With at least as many CTAs as strips every CTA serves one strip (a
  // group of CTAs shares each strip's rows evenly); otherwise each CTA
  // serves whole strips.
  int s_begin, s_end;
  if (G >= S) {
    s_begin = static_cast<int>((static_cast<int64_t>(c) * S) / G);
    s_end = s_begin + 1;
  } else {
    s_begin = static_cast<int>((static_cast<int64_t>(c) * S) / G);
    s_end = static_cast<int>((static_cast<int64_t>(c + 1) * S) / G);
  }
  int32_t* done = a.counters + static_cast<int64_t>(a.tiles_p) * a.tiles_q * halves;
  for (int strip = s_begin; strip < s_end; ++strip) {
    int r0 = 0, r1 = strip_rows;
    if (G >= S) {
      // CTAs [first, last) share this strip: first = ceil(strip*G/S)
      const int first = static_cast<int>((static_cast<int64_t>(strip) * G + S - 1) / S);
      const int last = static_cast<int>((static_cast<int64_t>(strip + 1) * G + S - 1) / S);
      const int k = last - first, j = c - first;
      r0 = (j * strip_rows) / k;
      r1 = ((j + 1) * strip_rows) / k;
    }
    const int tile = a.rr_tiles + strip / halves;
    const int half = strip % halves;
    const int cidx = tile * halves + half;
    int32_t tp, tq, m0, m1, n0, n1;
    tile_ranges(a, tile, BN, tp, tq, m0, m1, n0, n1);
    if (!a.swap) m0 += half * TILE_P;  // pair halves are P rows = C rows
    const int ma = min(a.M, m0 + r0), mb = min(a.M, m0 + r1);
    bool ok = true;
    if (et == 0) {
      volatile int32_t* cnt = a.counters + cidx;
      if (*cnt < a.split) {
        const uint64_t t0 = global_timer_ns();
        while (*cnt < a.split) {
          if (*abort_flag || global_timer_ns() - t0 > a.wait_limit_ns) {
            ok = false;
            break;
          }
          __nanosleep(64);
        }
      }
      if (!ok && !*abort_flag) record_timeout(a, abort_flag, 2 * 16 + 5);
      __threadfence();
    }
    if (named_bar_or(kBar, kEpiThreads, !ok)) return false;
    if (mb > ma) finish_tile<8>(a, ma, mb, n0, n1, et);
    __threadfence();
    named_bar_sync(kBar, kEpiThreads);
    if (et == 0 && r1 > r0) {
      const int old = atomicAdd(&done[cidx], r1 - r0);
      if (old + (r1 - r0) == strip_rows) {
        a.counters[cidx] = 0;
        done[cidx] = 0;
      }
    }
  }
  return true;
}

// Deterministic split-K arrival: after the run's partial is in its slot,
// count the run's splits; the CTA completing the count sums the strip's run
// slots in run order (so the result does not depend on arrival order),
// converts and stores C, then resets the counter.  Slots are tile-shaped
// (TILE_P x BN fp32, rows = C rows of the strip) and are overwritten by every
// run, so nothing needs zeroing.
template <int BN>
__device__ __noinline__ void arrive_split_tile_det(const TcArgs& a, const Group& g, int counter, int m0, int m1,
                                                   int n0, int n1, int et) {
  __threadfence();
  named_bar_sync(1, kEpiThreads);
  bool mine_last = false;
  if (et == 0) {
    __threadfence();  // (see arrive_split_tile)
    const int old = atomicAdd(&a.counters[counter], g.s1 - g.s0);
    mine_last = (old + (g.s1 - g.s0) == a.split);
    __threadfence();
  }
  if (named_bar_or(1, kEpiThreads, mine_last)) {
    __threadfence();
    int first, nruns;
    tile_runs(a, g.tile, first, nruns);
    constexpr int64_t kSlotElems = static_cast<int64_t>(TILE_P) * BN;
    const float* slot0 = a.slots + static_cast<int64_t>(counter) * a.max_runs * kSlotElems;
    finish_tile_det<8>(a, slot0, kSlotElems, nruns, m0, m1, n0, n1, a.swap ? TILE_P : BN, et);
    named_bar_sync(1, kEpiThreads);
    if (et == 0) a.counters[counter] = 0;
  }
}

// The epilogue of one group, run by the 128 epilogue threads (TMEM lane
// quadrant q4, lane `lane`, index `et` among the 128).  Reads the fp32
// accumulator buffer of the group from TMEM (the sum of NACC partial
// accumulators, buffer b of them at columns [b * NACC * BN, (b + 1) * NACC * BN))
// and either converts and stores the tile of C, or adds it to the split-K
// workspace and, for the CTA whose arrival completes the tile, converts the
// total.  `fix(c0, v)` may adjust each block of accumulator values (columns
// c0.. of this thread's row) before it leaves.  Returns false when the CTA
// is aborting; all 128 threads return the same value.
// PAIR: the CTA holds P-side half `half` of a pair tile, and the buffer-free
// arrival goes to the pair's MMA CTA (acce_bar0 is a shared::cluster address).
//
// With a.tma_c / a.tma_ws (and BN a multiple of 32) tiles leave through
// shared memory: each warp writes a 32 x 32 block of C (its 32 TMEM lanes
// by 32 accumulator columns; rows are m, or n when swapped) into one of its
// two 4 KiB staging buffers (`stage_smem`, 1024-aligned; `ring` counts the
// blocks it has issued) and one lane hands the block to a bulk tile store
// (C) or bulk tile reduction (fp32 partials), so whole lines reach L2.
// Otherwise each thread stores its own values directly.
// The group's accumulator as NACC partial accumulators (one per MMA issuer,
// ST columns apart, added in index order): N columns from taddr of each.
// Only those whose bit is set in `mask` hold this group's sums (an issuer
// with no MMA in the group leaves its accumulator untouched); all are read,
// 32 / N of them per wait after the first (32 registers in flight).
template <int N, int NACC, int ST>
__device__ __forceinline__ void ld_acc(uint32_t taddr, uint32_t (&v)[N], uint32_t mask = (1u << NACC) - 1u) {
  static_assert(N == 16 || N == 32, "tcgen05.ld shapes used here");
  auto ld = [&](uint32_t addr, uint32_t (&r)[N]) {
    if constexpr (N == 32) tc_ld_32x32b_x32(addr, r); else tc_ld_32x32b_x16(addr, r);
  };
  ld(taddr, v);
  if constexpr (NACC > 1) {
    constexpr int CH = 32 / N;  // further accumulators per wait
    const bool v0 = mask & 1u;
#pragma unroll
    for (int i0 = 1; i0 < NACC; i0 += CH) {
      uint32_t w[CH][N];
#pragma unroll
      for (int c = 0; c < CH; ++c)
        if (i0 + c < NACC) ld(taddr + (i0 + c) * ST, w[c]);
      if (i0 == 1) {
        tc_wait_ld_regs(v);
        if (!v0) {
#pragma unroll
          for (int j = 0; j < N; ++j) v[j] = 0u;  // +0.0f: adding the valid ones to it is exact
        }
      } else {
        tc_wait_ld();
      }
#pragma unroll
      for (int c = 0; c < CH; ++c)
        if (i0 + c < NACC) tc_regs_after_wait(w[c]);
#pragma unroll
      for (int c = 0; c < CH; ++c)
        if (i0 + c < NACC && ((mask >> (i0 + c)) & 1u))
#pragma unroll
          for (int j = 0; j < N; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(w[c][j]));
    }
  } else {
    tc_wait_ld_regs(v);
  }
}

// Split-K within a cluster (a.cl_size > 1; single-CTA kernel, swapped
// tiles, BN <= 64): the cluster's CTAs are the K-split runs of one tile, in
// rank order, and CTA q finishes C rows [q W, (q + 1) W), W = BN / cl, of the
// tile (accumulator columns; TMEM lanes are the tile's C columns n).  Each
// CTA reads its fp32 partial from TMEM and stores the W columns that CTA q
// finishes straight into q's epilogue staging buffer (its own included),
// slot = the sender's rank: row r of slot p at p * 128 * 4W + r * 4W bytes.
// Then it arrives once on every peer's `ready` mbarrier (count cl - 1,
// release at cluster scope, after the stores), waits on its own, and sums
// its slots in rank order (so the result does not depend on timing),
// converts and stores its rows of C.  Nothing is read remotely, no fp32
// partial goes through L2 and no counter is polled: the IREE page's
// partials -> shared storage -> second reduction, with the cluster's shared
// memory as the storage.  No peer touches a CTA's shared memory after
// arriving on its `ready`, so a CTA may leave as soon as its own `ready`
// completes.  A run without K blocks sends zeros.  Returns false when the
// CTA is aborting (all 128 threads agree).
// Split-K inside a cluster of CL CTAs (one run each, the tile's K range cut
// CL ways): CTA `rank` ends up owning columns [rank * W, rank * W + W) of the
// tile (W = BN / CL activation rows of C).  Every CTA writes the slices of its
// partial that other CTAs own into its own shared memory (`out0`, its
// pipeline stages, idle once its MMAs have completed) and sends each with one
// bulk copy into slot `rank` of the owner's receive area (`stage0`, CL slots
// of 128 rows x W fp32), completing on the owner's receive barrier, which
// expects (CL - 1) slices from the start of the kernel.  Its own slice goes
// straight into its slot.  The owner then adds its CL slots in rank order and
// stores its W rows of C (through a 16-bit transpose in shared memory when C
// rows allow 16-byte stores).
// Byte offset of 16-byte chunk c of row `row` in a slice (rows of W fp32):
// with W = 16 (64-byte rows) the chunk index is XORed with (row / 2) mod 4,
// so that the 16-byte accesses of eight consecutive rows hit distinct banks.
template <int W>
__device__ __forceinline__ uint32_t slice_off(int row, int c) {
  const int cs = W == 16 ? (c ^ ((row >> 1) & 3)) : c;
  return static_cast<uint32_t>(row * 4 * W + cs * 16);
}

template <int BN, int CL>
__device__ __forceinline__ void cluster_send_slices(const uint32_t (&v)[BN], uint32_t stage0, uint32_t out0, int row) {
  constexpr int W = BN / CL;
  constexpr uint32_t SL = TILE_P * 4 * W;  // bytes of one slice
  static_assert(W >= 4 && W % 4 == 0, "whole 16-byte chunks per slice row");
  const uint32_t rank = cluster_ctarank();
#pragma unroll
  for (int q = 0; q < CL; ++q) {
    const uint32_t dst = q == static_cast<int>(rank) ? stage0 + rank * SL : out0 + q * SL;
#pragma unroll
    for (int c = 0; c < W; c += 4)
      st_shared_v4(dst + slice_off<W>(row, c / 4), v[q * W + c], v[q * W + c + 1], v[q * W + c + 2], v[q * W + c + 3]);
  }
}

template <int BN, int CL>
__device__ __forceinline__ void cluster_sum_store(const TcArgs& a, uint32_t stage0, uint32_t tr0, int row, int et,
                                                  int m0, int m1, int n0, int n1) {
  constexpr int W = BN / CL;
  constexpr uint32_t SL = TILE_P * 4 * W;
  const uint32_t rank = cluster_ctarank();
  const int n = n0 + row;
  const int mr = m0 + static_cast<int>(rank) * W;  // first C row of this CTA's slice
  float s[W];
#pragma unroll
  for (int j = 0; j < W; ++j) s[j] = 0.0f;
#pragma unroll
  for (int p = 0; p < CL; ++p) {
    const uint32_t src = stage0 + static_cast<uint32_t>(p) * SL;
#pragma unroll
    for (int c = 0; c < W; c += 4) {
      const float4 t = ld_shared_f32x4(src + slice_off<W>(row, c / 4));
      s[c] += t.x;
      s[c + 1] += t.y;
      s[c + 2] += t.z;
      s[c + 3] += t.w;
    }
  }
  uint16_t* cb = reinterpret_cast<uint16_t*>(a.c);
  if (!a.c_vec) {
    if (n < n1) {
#pragma unroll
      for (int j = 0; j < W; ++j)
        if (mr + j < m1) cb[static_cast<int64_t>(mr + j) * a.ldc + n] = cvt1(s[j], a.c_bf16);
    }
    return;
  }
  // [W rows][128 columns] of 16-bit C in shared memory, then 16-byte stores
  // (8 columns of one row each; a ragged last chunk column by column)
#pragma unroll
  for (int j = 0; j < W; ++j) st_shared_u16(tr0 + static_cast<uint32_t>(j * TILE_P * 2 + row * 2), cvt1(s[j], a.c_bf16));
  named_bar_sync(1, kEpiThreads);
  for (int c = et; c < W * (TILE_P / 8); c += kEpiThreads) {
    const int j = c / (TILE_P / 8), col = (c % (TILE_P / 8)) * 8;
    if (mr + j >= m1 || n0 + col >= n1) continue;
    const uint32_t src = tr0 + static_cast<uint32_t>(j * TILE_P * 2 + col * 2);
    uint16_t* dst = cb + static_cast<int64_t>(mr + j) * a.ldc + n0 + col;
    if (n0 + col + 8 <= n1) {
      const uint4 w = ld_shared_v4(src);
      *reinterpret_cast<uint4*>(dst) = w;
    } else {
      for (int e = 0; n0 + col + e < n1; ++e) dst[e] = ld_shared_u16(src + 2u * e);
    }
  }
}

template <int BN>
__device__ __noinline__ bool cluster_split_tile(const TcArgs& a, const Group& g, uint32_t tmem_base,
                                                uint32_t accf_bar0, uint32_t acce_bar0, int& acc_iter,
                                                volatile int* abort_flag, int q4, int lane, int et,
                                                uint32_t stage0, uint32_t out0, uint32_t recv_bar, int m0, int m1,
                                                int n0, int n1) {
  static_assert(BN <= 64, "128 rows of BN fp32 fit the 32 KiB of epilogue staging");
  const int row = q4 * 32 + lane;
  const uint32_t cl = static_cast<uint32_t>(a.cl_size), rank = cluster_ctarank();
  uint32_t v[BN];
#pragma unroll
  for (int j = 0; j < BN; ++j) v[j] = 0u;  // +0.0f: a run without K blocks sends zeros
  bool ok = true;
  if (g.nkb > 0) {
    const int buf = acc_iter & 1;
    const bool got = mbar_wait_bounded(accf_bar0 + 8u * buf, (acc_iter >> 1) & 1, a.wait_limit_ns, abort_flag);
    if (!got && !*abort_flag) record_timeout(a, abort_flag, 2 * 16 + 2);
    ok = !named_bar_or(1, kEpiThreads, !got);
    if (ok) {
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + static_cast<uint32_t>(buf * BN);
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t t[16];
        tc_ld_32x32b_x16(t_row + c0, t);
        tc_wait_ld_regs(t);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[c0 + j] = t[j];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar0 + 8u * buf);
      ++acc_iter;
    }
  }
  const uint32_t sl = TILE_P * 4u * (static_cast<uint32_t>(BN) / cl);  // bytes of one slice
  if (ok) {
    // (the planner takes cl <= BN / 4)
    if (cl == 2) {
      cluster_send_slices<BN, 2>(v, stage0, out0, row);
    } else if (cl == 4) {
      if constexpr (BN >= 16) cluster_send_slices<BN, 4>(v, stage0, out0, row);
    } else {
      if constexpr (BN >= 32) cluster_send_slices<BN, 8>(v, stage0, out0, row);
    }
    fence_proxy_async_smem();  // the slices are written before the bulk copies read them
  }
  named_bar_sync(1, kEpiThreads);
  if (et == 0 && ok)
    for (uint32_t q = 0; q < cl; ++q)
      if (q != rank)
        bulk_copy_to_cluster(mapa_shared(stage0 + rank * sl, q), out0 + q * sl, sl, mapa_shared(recv_bar, q));
  // wait for the peers' slices even on the abort path: none may land in this
  // CTA's shared memory after it has left
  const bool got = mbar_wait_bounded_cluster(recv_bar, 0, a.wait_limit_ns, abort_flag);
  if (!got && !*abort_flag) record_timeout(a, abort_flag, 2 * 16 + 6);
  ok = !named_bar_or(1, kEpiThreads, !got || !ok);
  if (ok) {
    // (the transpose buffer lies after the outgoing slices: those may still
    // be read by the copies)
    const uint32_t tr0 = out0 + cl * sl;
    if (cl == 2) {
      cluster_sum_store<BN, 2>(a, stage0, tr0, row, et, m0, m1, n0, n1);
    } else if (cl == 4) {
      if constexpr (BN >= 16) cluster_sum_store<BN, 4>(a, stage0, tr0, row, et, m0, m1, n0, n1);
    } else {
      if constexpr (BN >= 32) cluster_sum_store<BN, 8>(a, stage0, tr0, row, et, m0, m1, n0, n1);
    }
  }
  return ok;
}

// No change to the accumulator values.
struct NoFix {
  template <int N>
  __device__ __forceinline__ void operator()(int, uint32_t (&)[N]) const {}
};

template <int BN, int CH, bool PAIR = false, int NACC = 1, class Fix = NoFix>
__device__ __forceinline__ bool epilogue_group(const TcArgs& a, const Group& g, uint32_t tmem_base, uint32_t accf_bar0,
                                               uint32_t acce_bar0, int& acc_iter, volatile int* abort_flag, int q4,
                                               int lane, int et, int half, uint32_t stage_smem, int& ring,
                                               const Fix& fix = Fix(), uint32_t nacc_mask = (1u << NACC) - 1u,
                                               uint32_t cl_bar0 = 0u, uint32_t cl_stage0 = 0u, uint32_t cl_out0 = 0u) {
  const int row = q4 * 32 + lane;  // accumulator row (TMEM lane)
  int32_t tp, tq, m0, m1, n0, n1;
  tile_ranges(a, g.tile, BN, tp, tq, m0, m1, n0, n1);
  if (PAIR) narrow_to_half(a, half, m0, m1, n0, n1);
  const bool full_tile = (g.s0 == 0 && g.s1 == a.split);
  if constexpr (!PAIR && NACC == 1 && BN <= 64) {
    if (a.cl_size > 1 && !full_tile)
      return cluster_split_tile<BN>(a, g, tmem_base, accf_bar0, acce_bar0, acc_iter, abort_flag, q4, lane, et,
                                    cl_stage0, cl_out0, cl_bar0, m0, m1, n0, n1);
  }
  const int cidx = PAIR ? 2 * g.tile + half : g.tile;
  // deterministic split-K: this run's slot (tile-shaped, rows = C rows)
  float* det_slot = nullptr;
  if (a.det && !full_tile) {
    int first, nruns;
    tile_runs(a, g.tile, first, nruns);
    const int r = static_cast<int>(blockIdx.x >> a.pair) - first;
    det_slot = a.slots + (static_cast<int64_t>(cidx) * a.max_runs + r) * (static_cast<int64_t>(TILE_P) * BN);
  }
  if (g.nkb > 0) {
    const int buf = acc_iter & 1;
    const uint32_t acc_phase = (acc_iter >> 1) & 1;
    const bool got = mbar_wait_bounded(accf_bar0 + 8u * buf, acc_phase, a.wait_limit_ns, abort_flag);
    if (!got && !*abort_flag) record_timeout(a, abort_flag, 2 * 16 + 2);
    // all epilogue threads leave together if any of them gave up
    if (named_bar_or(1, kEpiThreads, !got)) return false;
    tc_fence_after();
    const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + static_cast<uint32_t>(buf * BN * NACC);
    const bool staged = (BN % EPI_BOX == 0) && (full_tile ? a.tma_c : (a.tma_ws && !a.det));
    if (staged && a.swap) {
      // Swapped: TMEM lane = n, column = m.  Block rows are m, each holding
      // the warp's 32 n; this lane writes column `lane` of every row.
      const int32_t xbox = n0 + q4 * 32;  // first n of this warp's blocks
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += EPI_BOX) {
        uint32_t v[EPI_BOX];
        ld_acc<EPI_BOX, NACC, BN>(t_row + c0, v, nacc_mask);
        fix(c0, v);
        const int32_t ybox = m0 + c0;
        if (xbox >= n1 || ybox >= m1) continue;  // block wholly outside C (warp-uniform)
        const uint32_t sbuf = stage_smem + static_cast<uint32_t>(ring & 1) * 4096u;
        if (ring >= 2) {
          if (lane == 0) bulk_wait_group_read<1>();
          __syncwarp();
        }
        if (full_tile) {
          // 16-bit C: 64-byte rows in the 64-byte swizzle (16-byte chunk c of
          // row j stored at chunk c ^ ((j >> 1) & 3)); one row per instruction
#pragma unroll
          for (int j = 0; j < EPI_BOX; ++j)
            st_shared_u16(sbuf + 64u * j + ((static_cast<uint32_t>(lane >> 3) ^ ((j >> 1) & 3)) << 4) +
                              2u * (lane & 7),
                          cvt1(__uint_as_float(v[j]), a.c_bf16));
        } else {
          // fp32: 128-byte rows in the 128-byte swizzle (16-byte chunk index XOR row & 7)
#pragma unroll
          for (int j = 0; j < EPI_BOX; ++j)
            st_shared_f32(sbuf + 128u * j + ((static_cast<uint32_t>(lane >> 2) ^ (j & 7)) << 4) + 4u * (lane & 3),
                          __uint_as_float(v[j]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (full_tile)
            tma_store_2d(&a.tm_c, sbuf, xbox, ybox);
          else
            tma_reduce_add_2d(&a.tm_ws, sbuf, xbox, ybox);
          bulk_commit_group();
        }
        ++ring;
      }
      if (!full_tile && lane == 0) {
        bulk_wait_group<0>();
        fence_proxy_async_global();
      }
    } else if (staged) {
      const int32_t ybox = m0 + q4 * 32;  // first C row of this warp's blocks
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += EPI_BOX) {
        uint32_t v[EPI_BOX];
        ld_acc<EPI_BOX, NACC, BN>(t_row + c0, v, nacc_mask);
        fix(c0, v);
        const int32_t xbox = n0 + c0;
        if (ybox >= m1 || xbox >= n1) continue;  // block wholly outside C (warp-uniform)
        const uint32_t sbuf = stage_smem + static_cast<uint32_t>(ring & 1) * 4096u;
        if (ring >= 2) {
          // the block issued two steps ago has been read out of this buffer
          if (lane == 0) bulk_wait_group_read<1>();
          __syncwarp();
        }
        if (full_tile) {
          // 16-bit C: row `lane` of the block is 64 bytes in the 64-byte
          // swizzle (chunk j stored at chunk j ^ ((lane >> 1) & 3)), so the
          // eight lanes of each quarter-warp store to eight distinct bank groups
          const uint32_t r = sbuf + static_cast<uint32_t>(lane) * 64u;
          const uint32_t sw = static_cast<uint32_t>(lane >> 1) & 3u;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            st_shared_v4(r + 16u * (static_cast<uint32_t>(j) ^ sw), pack2(__uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1]), a.c_bf16),
                         pack2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]), a.c_bf16),
                         pack2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]), a.c_bf16),
                         pack2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]), a.c_bf16));
        } else {
          // fp32 partials: row `lane` is 128 bytes in the 128-byte swizzle
          // (16-byte chunk j stored at chunk j ^ (row & 7)), conflict-free
          const uint32_t r = sbuf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_shared_v4(r + 16u * static_cast<uint32_t>(j ^ (lane & 7)), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                         v[4 * j + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (full_tile)
            tma_store_2d(&a.tm_c, sbuf, xbox, ybox);
          else
            tma_reduce_add_2d(&a.tm_ws, sbuf, xbox, ybox);
          bulk_commit_group();
        }
        ++ring;
      }
      if (!full_tile && lane == 0) {
        // the partial sums must be in L2 before the tile's arrival is counted
        bulk_wait_group<0>();
        fence_proxy_async_global();
      }
    }
#pragma unroll 1
    for (int c0 = 0; c0 < (staged ? 0 : BN); c0 += CH) {
      uint32_t v[CH];
      ld_acc<CH, NACC, BN>(t_row + c0, v, nacc_mask);
      fix(c0, v);
      if (det_slot) {
        // the run's fp32 partial into its slot (every row; the conversion clips)
        if (!a.swap) {
          float* srow = det_slot + static_cast<int64_t>(row) * BN + c0;
#pragma unroll
          for (int j = 0; j < CH; j += 4) st_global_v4(srow + j, v[j], v[j + 1], v[j + 2], v[j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < CH; ++j) det_slot[static_cast<int64_t>(c0 + j) * TILE_P + row] = __uint_as_float(v[j]);
        }
        continue;
      }
      if (!a.swap) {
        const int m = m0 + row;
        const int nb = n0 + c0;
        if (m < m1) {
          if (full_tile) {
            uint16_t* crow = reinterpret_cast<uint16_t*>(a.c) + static_cast<int64_t>(m) * a.ldc;
            if (a.c_vec && nb + CH <= n1) {
#pragma unroll
              for (int j = 0; j < CH; j += 8) {
                st_global_v4(crow + nb + j, pack2(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), a.c_bf16),
                             pack2(__uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]), a.c_bf16),
                             pack2(__uint_as_float(v[j + 4]), __uint_as_float(v[j + 5]), a.c_bf16),
                             pack2(__uint_as_float(v[j + 6]), __uint_as_float(v[j + 7]), a.c_bf16));
              }
            } else {
#pragma unroll
              for (int j = 0; j < CH; ++j)
                if (nb + j < n1) crow[nb + j] = cvt1(__uint_as_float(v[j]), a.c_bf16);
            }
          } else {
            float* wrow = a.ws + static_cast<int64_t>(m) * a.N;
            if (a.ws_vec && nb + CH <= n1) {
#pragma unroll
              for (int j = 0; j < CH; j += 4)
                red_add_v4_f32(wrow + nb + j, __uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                               __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
            } else {
#pragma unroll
              for (int j = 0; j < CH; ++j)
                if (nb + j < n1) red_add_f32(wrow + nb + j, __uint_as_float(v[j]));
            }
          }
        }
      } else {
        const int n = n0 + row;
        if (n < n1) {
          if (full_tile) {
            uint16_t* cc = reinterpret_cast<uint16_t*>(a.c) + n;
#pragma unroll
            for (int j = 0; j < CH; ++j) {
              const int m = m0 + c0 + j;
              if (m < m1) cc[static_cast<int64_t>(m) * a.ldc] = cvt1(__uint_as_float(v[j]), a.c_bf16);
            }
          } else {
            float* wc = a.ws + n;
#pragma unroll
            for (int j = 0; j < CH; ++j) {
              const int m = m0 + c0 + j;
              if (m < m1) red_add_f32(wc + static_cast<int64_t>(m) * a.N, __uint_as_float(v[j]));
            }
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (PAIR)
        mbar_arrive_cluster(acce_bar0 + 8u * buf);
      else
        mbar_arrive(acce_bar0 + 8u * buf);
    }
    ++acc_iter;
  } else if (det_slot) {
    // a run of empty splits contributes zeros
    for (int i = et; i < TILE_P * BN; i += kEpiThreads) det_slot[i] = 0.0f;
  }
  if (!full_tile) {
    if (a.det)
      arrive_split_tile_det<BN>(a, g, cidx, m0, m1, n0, n1, et);
    else
      arrive_split_tile<4>(a, g, cidx, m0, m1, n0, n1, et);  // (4 loads in flight: no spills at the int4 kernels' register caps)
  }
  return true;
}

}  // namespace
}  // namespace lgt
