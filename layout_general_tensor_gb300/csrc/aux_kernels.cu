// Small HBM-bound helper kernels: the stride-realigning operand copy, and
// the device-side runs of the integer helpers (magic-number division and the
// perpendicular-dimension stride permutation) over index arrays.
#include "kernels.h"
#include "ptx.cuh"
#include "realign.cuh"

namespace lgt {
namespace {

// Copy rows of 16-bit elements from a source whose row pitch (or base) is only
// 2-byte aligned into rows whose pitch is a multiple of 16 bytes, so the
// operand becomes describable by a TMA tensor map.  This is the pre-pass form
// of the hipBLASLt DTL page's generalised loads ("Add support for
// non-power of 2 MT when TLU=1" / "generalized NLC=1"): any number of
// elements per row, offsets split with a magic-number division by the
// (static) chunks-per-row count.  Each thread produces eight 2-byte elements
// as one aligned 16-byte store: it loads the one or two aligned 16-byte words
// that hold them (consecutive threads read consecutive words, so a warp's
// loads coalesce) and realigns them with funnel shifts.  Every word read
// holds at least one of the thread's elements, so it lies in the same page as
// valid data.
// (realign8: realign.cuh, shared with the kernels' in-kernel loader)

// One chunk per thread over a grid that covers all chunks (measured faster
// than grid-stride loops with several chunks in flight per thread).
__global__ void __launch_bounds__(256) repack_rows_kernel(const uint16_t* __restrict__ src, int64_t src_pitch,
                                                          uint16_t* __restrict__ dst, int64_t dst_pitch,
                                                          int64_t row_elems, MagicDiv chunks_div,
                                                          int64_t total_chunks) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total_chunks; i += stride) {
    int64_t r, c;
    if (total_chunks < (1ll << 31)) {
      uint32_t q, rem;
      magic_divmod(static_cast<uint32_t>(i), chunks_div, q, rem);
      r = q;
      c = rem;
    } else {
      r = i / chunks_div.d;
      c = i - r * chunks_div.d;
    }
    const int64_t e0 = c * 8;
    const uint16_t* s = src + r * src_pitch + e0;
    uint16_t* d = dst + r * dst_pitch + e0;
    if (e0 + 8 <= row_elems) {
      const uintptr_t addr = reinterpret_cast<uintptr_t>(s);
      const uint4* p = reinterpret_cast<const uint4*>(addr & ~static_cast<uintptr_t>(15));
      const uint32_t off = static_cast<uint32_t>(addr & 15);  // even: 2-byte elements
      const uint4 a = __ldg(p);
      const uint4 b = off ? __ldg(p + 1) : a;
      *reinterpret_cast<uint4*>(d) = realign8(a, b, off);
    } else {
      for (int64_t j = 0; e0 + j < row_elems; ++j) d[j] = s[j];
    }
  }
}

__global__ void magic_divmod_kernel(const uint32_t* __restrict__ n, size_t count, MagicDiv m, uint32_t* q,
                                    uint32_t* r) {
  pdl_launch_dependents();
  pdl_wait();
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count; i += stride) {
    uint32_t qq, rr;
    magic_divmod(n[i], m, qq, rr);
    q[i] = qq;
    r[i] = rr;
  }
}

// out[j] = the stride permutation (or its inverse) of in[j] over `count`
// indices in blocks of `block` -- the device instance of perm_fwd / perm_inv,
// the same code the loaders use.
__global__ void perm_kernel(const uint32_t* __restrict__ in, size_t n, uint32_t count, uint32_t block,
                            uint32_t stride, int inverse, uint32_t* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  const size_t step = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t j = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < n; j += step)
    out[j] = inverse ? perm_inv(in[j], count, block, stride) : perm_fwd(in[j], count, block, stride);
}

int grid_for(int64_t work, int threads) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_repack_rows(const void* src, int64_t src_pitch, void* dst, int64_t dst_pitch, int64_t rows,
                               int64_t row_bytes, cudaStream_t stream) {
  if (rows <= 0 || row_bytes <= 0) return cudaSuccess;
  const int64_t row_elems = row_bytes / 2;
  const int64_t chunks = (row_elems + 7) / 8;
  const int64_t total = rows * chunks;
  const MagicDiv cd = magic_encode(static_cast<uint32_t>(chunks));
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  return launch_pdl(repack_rows_kernel,
                    dim3(static_cast<unsigned>(blocks < (1ll << 31) - 1 ? blocks : (1ll << 31) - 1)), dim3(threads), 0,
                    stream, static_cast<const uint16_t*>(src), src_pitch / 2, static_cast<uint16_t*>(dst),
                    dst_pitch / 2, row_elems, cd, total);
}

cudaError_t launch_magic_divmod(const uint32_t* n, size_t count, MagicDiv m, uint32_t* q, uint32_t* r,
                                cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  const int threads = 256;
  return launch_pdl(magic_divmod_kernel, dim3(static_cast<unsigned>(grid_for(static_cast<int64_t>(count), threads))),
                    dim3(threads), 0, stream, n, count, m, q, r);
}

cudaError_t launch_perm(const uint32_t* in, size_t n, uint32_t count, uint32_t block, uint32_t stride, int inverse,
                        uint32_t* out, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  return launch_pdl(perm_kernel, dim3(static_cast<unsigned>(grid_for(static_cast<int64_t>(n), threads))),
                    dim3(threads), 0, stream, in, n, count, block, stride, inverse, out);
}

}  // namespace lgt
