// Integer helpers shared by the planner (host) and the kernels (device):
// magic-number division, the perpendicular-dimension stride permutation and
// the SM-waste split-K rule.
#pragma once
#include <cstdint>

#if defined(__CUDACC__)
#define LGT_HD __host__ __device__ __forceinline__
#else
#define LGT_HD inline
#endif

namespace lgt {

// Division of 31-bit unsigned dividends by a divisor fixed when a plan is
// made (hipBLASLt DTL page, "Add support for generalized NLC=1": offsets are
// divided by static divisors through a magic multiply).  Method: Granlund &
// Montgomery, "Division by Invariant Integers using Multiplication" (1994),
// round-up variant with N = 31 dividend bits: for d >= 2 let l = ceil(log2 d)
// and m = ceil(2^(31+l) / d); then m*d - 2^(31+l) < d <= 2^l, so
// floor(n/d) = floor(n*m / 2^(31+l)) for all 0 <= n < 2^31, and m < 2^32.
// The quotient is the high 32 bits of n*m shifted right by l-1.  d = 1 is
// stored as mul = 0 and returns n.
struct MagicDiv {
  uint32_t d;
  uint32_t mul;
  uint32_t shr;
};

inline MagicDiv magic_encode(uint32_t d) {
  MagicDiv m{d, 0u, 0u};
  if (d <= 1) return m;
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;                 // l = ceil(log2 d), 1 <= l <= 31
  const unsigned __int128 num = static_cast<unsigned __int128>(1) << (31 + l);
  const unsigned __int128 q = (num + d - 1) / d;
  m.mul = static_cast<uint32_t>(q);
  m.shr = l - 1;
  return m;
}

LGT_HD uint32_t umulhi32(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
  return __umulhi(a, b);
#else
  return static_cast<uint32_t>((static_cast<uint64_t>(a) * b) >> 32);
#endif
}

LGT_HD uint32_t magic_div(uint32_t n, const MagicDiv& m) {
  return m.mul == 0u ? n : (umulhi32(n, m.mul) >> m.shr);
}

LGT_HD void magic_divmod(uint32_t n, const MagicDiv& m, uint32_t& q, uint32_t& r) {
  q = magic_div(n, m);
  r = n - q * m.d;
}

// Perpendicular-dimension stride permutation (hipBLASLt DTL page, "Add
// support for permuting perpDim").  Within each block of `block` indices,
// with S' = block / stride: forward i' = stride*(i mod S') + i div S' (used
// for global-read offsets) and inverse i = S'*(i' mod stride) + i' div stride
// (local-read offsets).  A trailing partial block maps to itself; `stride`
// must divide `block` (otherwise the index is returned unchanged).
LGT_HD uint32_t perm_fwd(uint32_t i, uint32_t count, uint32_t block, uint32_t stride) {
  if (block == 0 || stride == 0 || block % stride != 0) return i;
  const uint32_t base = (i / block) * block;
  if (base + block > count) return i;
  const uint32_t r = i - base, sp = block / stride;
  return base + stride * (r % sp) + r / sp;
}

LGT_HD uint32_t perm_inv(uint32_t ip, uint32_t count, uint32_t block, uint32_t stride) {
  if (block == 0 || stride == 0 || block % stride != 0) return ip;
  const uint32_t base = (ip / block) * block;
  if (base + block > count) return ip;
  const uint32_t r = ip - base, sp = block / stride;
  return base + sp * (r % stride) + r / stride;
}

// SM-waste split-K rule (BitBLAS TileLang page, "SplitK Infer for dequantize
// cases"): start at 1; stop once the share of idle SMs in the last wave,
// (tiles*f mod num_sms) / (tiles*f), is at most `threshold`, or once doubling
// would make f*block_K reach K; otherwise double.  Tile counts are ceiling
// divisions (the page floors them, which gives zero tiles when M < block_M).
inline int32_t splitk_auto(int64_t M, int64_t N, int64_t K, int32_t bm, int32_t bn, int32_t bk, int32_t num_sms,
                           double threshold) {
  if (M <= 0 || N <= 0 || K <= 0 || bm <= 0 || bn <= 0 || bk <= 0 || num_sms <= 0) return 1;
  const int64_t tiles = ((M + bm - 1) / bm) * ((N + bn - 1) / bn);
  int64_t f = 1;
  while (true) {
    const int64_t t = tiles * f;
    const int64_t waste = t - (t / num_sms) * num_sms;
    if (static_cast<double>(waste) / static_cast<double>(t) <= threshold) break;
    const int64_t doubled = f * 2;
    if (doubled * bk >= K) break;
    f = doubled;
  }
  return static_cast<int32_t>(f);
}

}  // namespace lgt
