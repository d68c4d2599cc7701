// In-kernel realigning loader: fills an operand's part of each pipeline stage
// when a TMA box cannot address the operand directly (rows not a multiple of
// 16 bytes apart, or a base that is not 16-byte aligned), so that no realigned
// copy of the operand has to be written first.
//
// Source passages: the hipBLASLt page, "Add support for permuting perpDim"
// (which rows a load instruction fetches: a stride permutation of the rows,
// forward on the global side, inverse on the local side) and "Add support for
// generalized NLC=1" (any row length); the inThreadTranspose page ("PR
// description": per-vector alignment, whole-vector stores to shared memory).
//
// Row classes.  With a row pitch of p bytes, row i starts at byte i p, whose
// offset within its 16-byte word, (i p) mod 16, repeats with period
// P = 16 / gcd(p, 16) (1, 2, 4 or 8).  The rows of class r (i = r mod P) are
// a tensor of their own: base = the 16-byte word holding row r's start, pitch
// P p (a multiple of 16), every row at the same byte offset d_r.  A TMA map
// per class loads boxes of 64 c + 8 elements (the 128 c bytes of c 64-wide
// segments from any offset d_r <= 14) by several class rows.  Taking a stage's rows
// class by class -- r, r + P, r + 2P, ..., then r + 1, ... -- is the perpDim
// permutation of the stage's rows with stride P (perm_fwd with block = rows,
// stride = rows / P): the forward mapping on the global side.
//
// Staging and the realigning pass.  The boxes land unswizzled in a staging
// slot, class-major; the loader warps then move each 16-byte output chunk of
// the stage: two aligned 16-byte loads of the staged row, a funnel shift by
// d_r, one 16-byte store to where a swizzled TMA box would have put it (the
// inverse mapping on the local side).  Elements outside the tensor are zero:
// the class maps end at the row ends and at the last row of their class.
//
// Stage layouts (128-byte swizzle: 16-byte chunk c of a 128-byte row goes to
// chunk c ^ (row mod 8)).  K-major operand (storage rows along M or N, K
// contiguous): stage row s = tile row s, elements k0 .. k0 + 63, at s * 128.
// MN-major (storage rows along K): stage row k of 64-wide chunk j = storage
// row k0 + k, elements row0 + 64 j .. + 63, at j * 8 KiB + k * 128.
#pragma once

#include <cstdint>

#include "intmath.h"
#include "kernels.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lgt {

constexpr int kRlMaxStg = 4;     // staging slots at most (barriers reserved for them)
// (kRlMaxClasses: kernels.h)

// Eight 2-byte elements starting at byte offset `off` (even, < 16) of the
// aligned 16-byte pair (a, b); branch-free (threads of a warp may hold
// different offsets).
__device__ __forceinline__ uint4 realign8(const uint4& a, const uint4& b, uint32_t off) {
  const uint32_t q = off >> 2;
  uint32_t w0 = a.x, w1 = a.y, w2 = a.z, w3 = a.w, w4 = b.x;
  if (q & 2u) {
    w0 = a.z;
    w1 = a.w;
    w2 = b.x;
    w3 = b.y;
    w4 = b.z;
  }
  if (q & 1u) {
    w0 = w1;
    w1 = w2;
    w2 = w3;
    w3 = w4;
    w4 = (q & 2u) ? b.w : b.y;
  }
  const uint32_t sh = (off & 3u) * 8u;  // 0 or 16 bits
  return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh), __funnelshift_r(w2, w3, sh),
                    __funnelshift_r(w3, w4, sh));
}

// Class count P for a row pitch of `pitch` bytes (even).
LGT_HD int rl_classes(int64_t pitch) {
  const int64_t m = pitch % 16;
  return m == 0 ? 1 : (m % 8 == 0 ? 2 : (m % 4 == 0 ? 4 : 8));
}

// Geometry of one realigned operand's stage (tile rows `rows` on the M / N
// side, P classes).  K-major: one box per class, 64 elements along K (+ 8
// for the offset) by rows / P class rows.  MN-major: 64-wide chunks of the
// tile's M / N rows, up to three per box (64 c + 8 elements, at most 200), by
// 64 / P class rows (the stage's K rows of the class).  A staged row is the
// box's inner extent; boxes are padded to 128 bytes (TMA destinations).
struct RlGeom {
  int chunks;      // 64-wide chunks along a storage row: 1 (K-major) or the tile's
  int per_box;     // chunks one box covers
  int boxes;       // boxes per class
  int box_rows;    // class rows of a box
  uint32_t row_bytes;  // bytes of a staged row: (64 per_box + 8) * 2
  uint32_t box_stride;
  uint32_t stage_bytes;
};
LGT_HD RlGeom rl_geom(int mn, int rows, int classes) {
  RlGeom g;
  g.chunks = mn ? (rows + 63) / 64 : 1;
  g.per_box = g.chunks <= 3 ? g.chunks : 2;
  g.boxes = (g.chunks + g.per_box - 1) / g.per_box;
  g.box_rows = (mn ? 64 : rows) / classes;
  g.row_bytes = static_cast<uint32_t>(64 * g.per_box + 8) * 2u;
  g.box_stride = (static_cast<uint32_t>(g.box_rows) * g.row_bytes + 127u) & ~127u;
  g.stage_bytes = static_cast<uint32_t>(classes * g.boxes) * g.box_stride;
  return g;
}
// Storage rows of one stage: K-major one per tile row, MN-major 64 per chunk.
LGT_HD int rl_stage_rows(int mn, int rows) { return mn ? 64 * ((rows + 63) / 64) : rows; }
LGT_HD uint32_t rl_stage_bytes(int mn, int rows, int classes) { return rl_geom(mn, rows, classes).stage_bytes; }
// Bytes the boxes of one stage deliver (the full boxes, zero fill included).
LGT_HD uint32_t rl_stage_tx(int mn, int rows, int classes) {
  const RlGeom g = rl_geom(mn, rows, classes);
  return static_cast<uint32_t>(classes * g.boxes * g.box_rows) * g.row_bytes;
}

// Staging ring carved from the last `take` pipeline stages: the fewest stages
// that hold two slots.  Returns false when fewer than two pipeline stages
// would be left (the plan then repacks instead).
LGT_HD bool rl_ring(int stages, uint32_t stage_bytes, uint32_t stg_bytes, int& take, int& nstg) {
  if (stg_bytes == 0) {
    take = 0;
    nstg = 0;
    return true;
  }
  take = static_cast<int>((2u * stg_bytes + stage_bytes - 1u) / stage_bytes);
  nstg = static_cast<int>((static_cast<uint64_t>(take) * stage_bytes) / stg_bytes);
  if (nstg > kRlMaxStg) nstg = kRlMaxStg;
  return stages - take >= 2;
}

// The class boxes of one operand for one stage, into staging at `dst`,
// completing on `bar`.  rows / row0: the tile's rows on the M / N side (row0
// a multiple of 8); k0: the stage's first K element.  The boxes are spread
// over the `nlanes` lanes of the calling warp (`lane` < nlanes issue), so
// that their issue latencies overlap.
__device__ __forceinline__ void rl_issue(const CUtensorMap* maps, int classes, int mn, int rows, int row0, int k0,
                                         uint32_t dst, uint32_t bar, int lane, int nlanes) {
  const RlGeom g = rl_geom(mn, rows, classes);
  for (int b = lane; b < classes * g.boxes; b += nlanes) {
    const int r = b % classes, jb = b / classes;  // class, box along the row
    if (!mn)  // class r: tile rows row0 + r + P i = class rows row0 / P + i
      tma_load_2d(dst + static_cast<uint32_t>(r) * g.box_stride, &maps[r], bar, k0, row0 / classes);
    else
      tma_load_2d(dst + static_cast<uint32_t>(jb * classes + r) * g.box_stride, &maps[r], bar,
                  row0 + 64 * g.per_box * jb, k0 / classes);
  }
}

// The CTA's K blocks in pipeline order (the producer's order), one at a time.
struct KbIter {
  Sched sched;
  Group g;
  int kb = 0;
  bool have = false;
  __device__ explicit KbIter(const TcArgs& a) : sched(a) {}
  __device__ bool next(const TcArgs& a, int& tile, int& kb_abs) {
    while (!have || kb >= g.nkb) {
      if (!sched.next(a, g)) return false;
      have = true;
      kb = 0;
    }
    tile = g.tile;
    kb_abs = g.kb0 + kb;
    ++kb;
    return true;
  }
};

// The realigning pass of one operand for one stage: from staging `stg` into
// the operand's part of the pipeline stage `out`, by `nthreads` threads (t:
// this thread's index among them).  d[r]: byte offset of class r's rows.
// Each thread takes output chunks t, t + nthreads, ...; their staged loads
// are issued kRlBatch at a time before any of them is used.
constexpr int kRlBatch = 8;
__device__ __forceinline__ void rl_pass(const int32_t* d, int classes, int mn, int rows, uint32_t stg, uint32_t out,
                                        int t, int nthreads) {
  const RlGeom g = rl_geom(mn, rows, classes);
  const int lg = classes == 1 ? 0 : (classes == 2 ? 1 : (classes == 4 ? 2 : 3));
  const int total = rl_stage_rows(mn, rows) * 8;  // 16-byte output chunks
  for (int base_idx = 0; base_idx < total; base_idx += kRlBatch * nthreads) {
    uint4 lo[kRlBatch], hi[kRlBatch];
    uint32_t dst[kRlBatch], off[kRlBatch];
#pragma unroll
    for (int u = 0; u < kRlBatch; ++u) {
      const int idx = base_idx + u * nthreads + t;
      const int s = idx >> 3, c = idx & 7;
      const int k = mn ? (s & 63) : s, j = mn ? (s >> 6) : 0;  // row within its 128-byte-row block, the block
      const int r = k & (classes - 1), i = k >> lg;
      const int jb = j / g.per_box, jc = j - jb * g.per_box;   // box along the row, chunk within it
      const uint32_t src = stg + static_cast<uint32_t>(jb * classes + r) * g.box_stride +
                           static_cast<uint32_t>(i) * g.row_bytes + static_cast<uint32_t>(jc * 128 + c * 16);
      const bool in = idx < total;
      lo[u] = in ? ld_shared_v4(src) : make_uint4(0u, 0u, 0u, 0u);
      hi[u] = in ? ld_shared_v4(src + 16u) : make_uint4(0u, 0u, 0u, 0u);
      off[u] = static_cast<uint32_t>(d[r]);
      dst[u] = in ? out + static_cast<uint32_t>(j) * 8192u + static_cast<uint32_t>(k) * 128u +
                        ((static_cast<uint32_t>(c) ^ static_cast<uint32_t>(k & 7)) << 4)
                  : 0xFFFFFFFFu;
    }
#pragma unroll
    for (int u = 0; u < kRlBatch; ++u) {
      if (dst[u] == 0xFFFFFFFFu) continue;
      const uint4 v = realign8(lo[u], hi[u], off[u]);
      st_shared_v4(dst[u], v.x, v.y, v.z, v.w);
    }
  }
}

}  // namespace lgt
