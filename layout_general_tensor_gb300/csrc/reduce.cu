// fp32 row reduction, out[r] = sum_c x[r, c] (include/reduce.h).
//
// The IREE page "[LLVMGPUVectorDistribute] Add support for inter-subgroup
// multi_reduction" distributes the reduced dimension over the subgroups of a
// workgroup: each subgroup reduces its share, the subgroups' partial results
// go through shared memory to a new distribution, and a second reduction
// finishes.  Here the same two steps run at two levels:
//   - inside a CTA: each thread sums its strided share of the row slice into
//     16 fp32 accumulators (float4 loads, 8 in flight), the accumulators and
//     then the 32 lanes of a warp are added by a shuffle tree, the 8 warp
//     sums go through shared memory and warp 0 adds them the same way;
//   - across CTAs, for rows too few to fill the GPU: a row is split into
//     `splits` contiguous chunks (one work unit each), each unit's total goes
//     to the workspace, and the CTA whose arrival on the row's counter is the
//     last adds the row's partials in split order and resets the counter.
// Every sum is taken in an order fixed by the shapes and the SM count, so the
// result is reproducible bit for bit.  The kernel streams x once: HBM-bound
// for large inputs, latency-bound for the page's 4096-element cases.
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "reduce.h"

namespace lgt {
namespace {

constexpr int kRedThreads = 256;
constexpr int kRedUnroll = 8;        // float4 loads in flight per thread
constexpr int kRedCtasPerSm = 4;     // resident CTAs per SM the grid assumes
constexpr int64_t kMinChunk = 4096;  // elements: a split never gets fewer

struct ReduceArgs {
  const float* x;
  int64_t ldx, cols, chunk;
  float* out;
  float* part;        // rows x splits partials (splits > 1)
  int32_t* counters;  // rows arrival counters (splits > 1)
  int32_t splits;
  uint32_t units;     // rows * splits
  MagicDiv div_splits;
};

__device__ __forceinline__ float4 ld_stream_f4(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum of p[0, n) by the whole CTA; the result is valid in thread 0.
__device__ __forceinline__ float cta_sum(const float* p, int64_t n, float* red_smem) {
  const int t = threadIdx.x;
  // elements before the first 16-byte boundary, and after the last whole float4
  int64_t head = static_cast<int64_t>(((16u - (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p)) & 15u)) & 15u) >> 2);
  if (head > n) head = n;
  const int64_t n4 = (n - head) >> 2;
  const int64_t tail0 = head + 4 * n4;
  float edge = 0.0f;
  if (t < head) edge = p[t];
  if (tail0 + t < n) edge += p[tail0 + t];
  const float4* q = reinterpret_cast<const float4*>(p + head);
  float4 acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int64_t kStep = static_cast<int64_t>(kRedThreads) * kRedUnroll;
  int64_t i = t;
  for (; i + (kRedUnroll - 1) * kRedThreads < n4; i += kStep) {
    float4 v[kRedUnroll];
#pragma unroll
    for (int u = 0; u < kRedUnroll; ++u) v[u] = ld_stream_f4(q + i + u * kRedThreads);
#pragma unroll
    for (int u = 0; u < kRedUnroll; ++u) {
      acc[u & 3].x += v[u].x;
      acc[u & 3].y += v[u].y;
      acc[u & 3].z += v[u].z;
      acc[u & 3].w += v[u].w;
    }
  }
#pragma unroll
  for (int u = 0; u < kRedUnroll; ++u) {
    if (i < n4) {
      const float4 v = ld_stream_f4(q + i);
      acc[u & 3].x += v.x;
      acc[u & 3].y += v.y;
      acc[u & 3].z += v.z;
      acc[u & 3].w += v.w;
    }
    i += kRedThreads;
  }
  const float4 s01 = make_float4(acc[0].x + acc[1].x, acc[0].y + acc[1].y, acc[0].z + acc[1].z, acc[0].w + acc[1].w);
  const float4 s23 = make_float4(acc[2].x + acc[3].x, acc[2].y + acc[3].y, acc[2].z + acc[3].z, acc[2].w + acc[3].w);
  const float4 s = make_float4(s01.x + s23.x, s01.y + s23.y, s01.z + s23.z, s01.w + s23.w);
  float v = ((s.x + s.y) + (s.z + s.w)) + edge;
  v = warp_sum(v);
  const int warp = t >> 5, lane = t & 31;
  if (lane == 0) red_smem[warp] = v;
  __syncthreads();
  float total = 0.0f;
  if (warp == 0) {
    total = lane < kRedThreads / 32 ? red_smem[lane] : 0.0f;
#pragma unroll
    for (int o = (kRedThreads / 64); o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  __syncthreads();  // red_smem is reused by the next unit
  return total;
}

__global__ void __launch_bounds__(kRedThreads) reduce_rows_kernel(const __grid_constant__ ReduceArgs a) {
  __shared__ float red_smem[kRedThreads / 32];
  __shared__ int last_flag;
  pdl_launch_dependents();
  pdl_wait();
  for (uint32_t u = blockIdx.x; u < a.units; u += gridDim.x) {
    uint32_t r, s;
    magic_divmod(u, a.div_splits, r, s);
    const int64_t c0 = static_cast<int64_t>(s) * a.chunk;
    const int64_t c1 = min(a.cols, c0 + a.chunk);
    const float total = cta_sum(a.x + static_cast<int64_t>(r) * a.ldx + c0, c1 > c0 ? c1 - c0 : 0, red_smem);
    if (a.splits == 1) {
      if (threadIdx.x == 0) a.out[r] = total;
      continue;
    }
    if (threadIdx.x == 0) {
      a.part[static_cast<int64_t>(r) * a.splits + s] = total;
      __threadfence();
      const int old = atomicAdd(&a.counters[r], 1);
      last_flag = (old == a.splits - 1);
    }
    __syncthreads();
    if (last_flag && threadIdx.x < 32) {
      // the row's partials, in split order: lane l adds splits l, l+32, ...
      // sequentially, then the lanes' sums by the shuffle tree
      __threadfence();
      const float* pr = a.part + static_cast<int64_t>(r) * a.splits;
      float v = 0.0f;
      for (int j = threadIdx.x; j < a.splits; j += 32) v += __ldcg(pr + j);
      v = warp_sum(v);
      if (threadIdx.x == 0) {
        a.out[r] = v;
        a.counters[r] = 0;
      }
    }
    __syncthreads();  // last_flag is rewritten by the next unit
  }
}

struct ReducePlan {
  int32_t splits;
  int64_t chunk;
  int64_t units;
  size_t ws_bytes;
};

// Rows fill the GPU on their own when there are at least as many as the
// resident CTAs; otherwise each row is cut into chunks of at least kMinChunk
// elements (a multiple of 4, so chunk starts keep a row's 16-byte alignment)
// until the units reach the resident CTAs.
ReducePlan plan_reduce(int64_t rows, int64_t cols, int num_sms) {
  ReducePlan p{1, cols, rows, 0};
  const int64_t target = static_cast<int64_t>(num_sms) * kRedCtasPerSm;
  if (rows < target && cols > kMinChunk) {
    int64_t want = (target + rows - 1) / rows;
    const int64_t most = (cols + kMinChunk - 1) / kMinChunk;
    if (want > most) want = most;
    int64_t chunk = (cols + want - 1) / want;
    chunk = (chunk + 3) & ~int64_t{3};
    p.splits = static_cast<int32_t>((cols + chunk - 1) / chunk);
    p.chunk = chunk;
  }
  p.units = rows * p.splits;
  if (p.splits > 1) {
    const size_t part = static_cast<size_t>(rows) * p.splits * sizeof(float);
    p.ws_bytes = ((part + 255) & ~size_t{255}) + static_cast<size_t>(rows) * sizeof(int32_t);
  }
  return p;
}

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

}  // namespace
}  // namespace lgt

extern "C" gemm_status_t reduce_rows_workspace_size(int64_t rows, int64_t cols, int32_t num_sms, size_t* bytes) {
  if (!bytes || rows < 0 || cols < 0 || num_sms < 0) return GEMM_ERR_INVALID_ARG;
  *bytes = 0;
  if (num_sms == 0) {
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    num_sms = lgt::device_sms();
    if (num_sms <= 0) return GEMM_ERR_CUDA;
  }
  if (rows == 0 || cols == 0) return GEMM_OK;
  if (rows * static_cast<int64_t>((cols + lgt::kMinChunk - 1) / lgt::kMinChunk) >= (int64_t{1} << 31))
    return GEMM_ERR_UNSUPPORTED;
  *bytes = lgt::plan_reduce(rows, cols, num_sms).ws_bytes;
  return GEMM_OK;
}

extern "C" gemm_status_t reduce_rows_f32(const float* x, int64_t rows, int64_t cols, int64_t ldx, float* out,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  if (rows < 0 || cols < 0 || ldx < 0) return GEMM_ERR_INVALID_ARG;
  if (ldx == 0) ldx = cols;
  if (ldx < cols) return GEMM_ERR_INVALID_ARG;
  if (rows == 0) return GEMM_OK;
  if (!out || (cols > 0 && !x)) return GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(out) & 3u) || (reinterpret_cast<uintptr_t>(x) & 3u)) return GEMM_ERR_ALIGNMENT;
  if (rows * static_cast<int64_t>((cols + lgt::kMinChunk - 1) / lgt::kMinChunk) >= (int64_t{1} << 31))
    return GEMM_ERR_UNSUPPORTED;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cols == 0)
    return cudaMemsetAsync(out, 0, static_cast<size_t>(rows) * sizeof(float), st) == cudaSuccess ? GEMM_OK
                                                                                                  : GEMM_ERR_CUDA;
  const int sms = lgt::device_sms();
  if (sms <= 0) return GEMM_ERR_CUDA;
  const lgt::ReducePlan p = lgt::plan_reduce(rows, cols, sms);
  lgt::ReduceArgs a{};
  a.x = x;
  a.ldx = ldx;
  a.cols = cols;
  a.chunk = p.chunk;
  a.out = out;
  a.splits = p.splits;
  a.units = static_cast<uint32_t>(p.units);
  a.div_splits = lgt::magic_encode(static_cast<uint32_t>(p.splits));
  if (p.splits > 1) {
    if (!workspace || workspace_bytes < p.ws_bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return GEMM_ERR_WORKSPACE;
    const size_t part = static_cast<size_t>(rows) * p.splits * sizeof(float);
    a.part = static_cast<float*>(workspace);
    a.counters = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + ((part + 255) & ~size_t{255}));
  }
  const int64_t cap = static_cast<int64_t>(sms) * lgt::kRedCtasPerSm;
  const unsigned grid = static_cast<unsigned>(p.units < cap ? p.units : cap);
  const cudaError_t e = lgt::launch_pdl(lgt::reduce_rows_kernel, dim3(grid), dim3(lgt::kRedThreads), 0, st, a);
  return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}
