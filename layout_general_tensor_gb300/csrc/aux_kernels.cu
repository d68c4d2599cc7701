// Small HBM-bound helper kernels: the stride-realigning operand copy and the
// device-side magic-division check.
#include "kernels.h"

namespace lgt {
namespace {

// Copy rows of 16-bit elements from a source whose row pitch (or base) is only
// 2-byte aligned into rows whose pitch is a multiple of 16 bytes, so the
// operand becomes describable by a TMA tensor map.  This is the pre-pass form
// of the hipBLASLt DTL page's generalised loads ("Add support for
// non-power of 2 MT when TLU=1" / "generalized NLC=1"): any number of
// elements per row, offsets split with a magic-number division by the
// (static) chunks-per-row count.  Each thread gathers eight 2-byte elements
// (consecutive threads read consecutive addresses, so a warp's loads
// coalesce) and writes one aligned 16-byte vector.
__global__ void repack_rows_kernel(const uint16_t* __restrict__ src, int64_t src_pitch, uint16_t* __restrict__ dst,
                                   int64_t dst_pitch, int64_t rows, int64_t row_elems, MagicDiv chunks_div,
                                   int64_t total_chunks) {
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
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = static_cast<uint32_t>(s[2 * j]) | (static_cast<uint32_t>(s[2 * j + 1]) << 16);
      *reinterpret_cast<uint4*>(d) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      for (int64_t j = 0; e0 + j < row_elems; ++j) d[j] = s[j];
    }
  }
}

__global__ void magic_divmod_kernel(const uint32_t* __restrict__ n, size_t count, MagicDiv m, uint32_t* q,
                                    uint32_t* r) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count; i += stride) {
    uint32_t qq, rr;
    magic_divmod(n[i], m, qq, rr);
    q[i] = qq;
    r[i] = rr;
  }
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
  repack_rows_kernel<<<grid_for(total, threads), threads, 0, stream>>>(
      static_cast<const uint16_t*>(src), src_pitch / 2, static_cast<uint16_t*>(dst), dst_pitch / 2, rows, row_elems,
      cd, total);
  return cudaGetLastError();
}

cudaError_t launch_magic_divmod(const uint32_t* n, size_t count, MagicDiv m, uint32_t* q, uint32_t* r,
                                cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  const int threads = 256;
  magic_divmod_kernel<<<grid_for(static_cast<int64_t>(count), threads), threads, 0, stream>>>(n, count, m, q, r);
  return cudaGetLastError();
}

}  // namespace lgt
