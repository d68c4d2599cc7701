// Kernel argument blocks and launchers shared between the C ABI (api.cu) and
// the kernel translation units.
#pragma once
#include <cstdint>
#include <cstdlib>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "intmath.h"

namespace lgt {

// cudaFuncAttributeMaxDynamicSharedMemorySize for `Kernel` on the current
// device, set once per device (the attribute outlives the call).
template <auto Kernel>
cudaError_t set_smem_once(int bytes) {
  static unsigned long long done = 0;  // one bit per device ordinal below 64
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) __atomic_fetch_or(&done, bit, __ATOMIC_RELEASE);
  return e;
}

// Launch with programmatic stream serialization: the kernel's prologue
// (barrier set-up, TMEM allocation, descriptor prefetch) overlaps the end of
// the previous kernel in the stream; every kernel here calls pdl_wait()
// before its first global-memory access.  LGT_GEMM_PDL=0 launches plainly.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  static const bool pdl = [] {
    const char* v = std::getenv("LGT_GEMM_PDL");
    return !(v && v[0] == '0');
  }();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_pdl, as a grid of clusters of `cluster` CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                               unsigned cluster, Args&&... args) {
  static const bool pdl = [] {
    const char* v = std::getenv("LGT_GEMM_PDL");
    return !(v && v[0] == '0');
  }();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// MMA tile: 128 rows on the P side (the operand whose rows map to TMEM
// lanes), BN rows on the Q side, 64 elements of K per pipeline stage.
constexpr int TILE_P = 128;
constexpr int TILE_K = 64;

// Epilogue staging in shared memory: per epilogue warp, two 4 KiB buffers of
// one 32-row x 32-column output block (fp32 partials or 16-bit C).
constexpr int EPI_BOX = 32;
constexpr uint32_t EPI_STAGING_BYTES = 4 * 2 * 4096;

// Instruction descriptor, kind::f16, fp32 accumulator, dense.
//   bits 4-5 D format (1 = f32); 7-9 A format, 10-12 B format (0 = f16,
//   1 = bf16); 15 / 16 A / B major (0 = K-major, 1 = MN-major);
//   17-22 N >> 3; 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t ab_bf16, uint32_t a_mn, uint32_t b_mn, uint32_t M,
                                                 uint32_t N) {
  return (1u << 4) | (ab_bf16 << 7) | (ab_bf16 << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}

// Status word written by kernels that give up a bounded wait.
struct DeviceStatus {
  int32_t code;   // 0 or GEMM_ERR_TIMEOUT
  int32_t where;  // role * 16 + barrier kind of the first wait that gave up
};

// Tensor-core GEMM over (tile, split) work units.  P is the MMA's M-side
// operand, Q its N-side operand.  Normal mode: P = A (rows m), Q = B
// (rows n).  Swapped mode (skinny M): P = B (rows n), Q = A (rows m), and the
// accumulator holds C^T.
constexpr int kRlMaxClasses = 8;  // realigning loader: row classes at most (16 / gcd(pitch, 16))

struct TcArgs {
  CUtensorMap tm_p;
  CUtensorMap tm_q;
  CUtensorMap tm_c;     // C, box 32 x 32, for bulk tile stores (valid if tma_c)
  CUtensorMap tm_ws;    // fp32 partial sums, box 32 x 32, for bulk reductions (valid if tma_ws)
  void* c;
  float* ws;            // fp32 partial sums [M][N] (split > 1)
  int32_t* counters;    // per-tile arrival counters (split > 1)
  DeviceStatus* status;
  uint64_t wait_limit_ns;
  int64_t ldc;
  int32_t M, N, K;
  int32_t tiles_p, tiles_q;
  int32_t split, kb_per_split, kb_total;
  int32_t num_units;
  int32_t rr_tiles;      // tiles dealt whole, round-robin, after the contiguous unit ranges
  float* slots;          // deterministic split-K: one fp32 partial slot per (strip, run); see det
  int32_t det;           // 1: runs store partials into slots, summed in run order by the last arriver
  int32_t max_runs;      // slots per strip
  int32_t tail_tiles;    // split tiles [rr_tiles, rr_tiles + tail_tiles) converted by the fixup warps of all CTAs
                         // (a stream-K tail, or every tile of a split-K plan); 0: the last arriver converts
  MagicDiv div_split;    // unit -> (tile, split)
  MagicDiv div_tiles_p;  // tile -> (tile_p, tile_q)
  int32_t p_mn, q_mn;    // 1: operand tile is MN-major in shared memory
  int32_t swap;
  int32_t c_bf16;
  int32_t c_vec;         // C rows allow 16-byte vector stores
  int32_t ws_vec;        // workspace rows allow 16-byte vector reductions
  int32_t pair;          // 1: CTA-pair kernel, 256-row P tiles split over the pair
  int32_t tma_c;         // full tiles leave through shared memory and bulk tile stores
  int32_t tma_ws;        // partial tiles leave through shared memory and bulk reductions
  int32_t cl_size;       // > 1: the split-K runs of a tile are the CTAs of one cluster of this size,
                         // reduced through distributed shared memory (single-CTA kernel, swapped, BN <= 64)
  int32_t withhold;      // test aid (single-CTA kernel): CTA 0 never fills its first pipeline stage
  // In-kernel realigning loader (realign.cuh) for operands TMA cannot address
  // directly, [0] = P, [1] = Q: one TMA map per row class (rows whose starts
  // share their offset within a 16-byte word), a staging ring, and a
  // realigning pass by the fixup warps (plans without fixup work).
  CUtensorMap tm_rl[2][kRlMaxClasses];
  int32_t rl_on[2];                  // 1: the operand goes through the loader
  int32_t rl_cls[2];                 // row classes P (1, 2, 4 or 8)
  int32_t rl_d[2][kRlMaxClasses];    // byte offset of class r's rows in their 16-byte words
  uint32_t idesc;
};

// Returns a cudaError_t; `bn` selects the kernel instance.
cudaError_t launch_tc_gemm(const TcArgs& args, int bn, int grid, cudaStream_t stream);
size_t tc_gemm_smem_bytes(int bn);
// Whether the realigning loader's staging ring fits beside at least two
// pipeline stages for tile width bn (p_cls / q_cls: row classes of a
// realigned P / Q, 0 when that operand is loaded by TMA directly).
bool tc_gemm_rl_fits(int bn, int p_mn, int q_mn, int p_cls, int q_cls);
bool tc_gemm_pair_rl_fits(int bn, int p_mn, int q_mn, int p_cls, int q_cls);
// Clusters of `cluster` CTAs of the single-CTA kernel (tile width bn <= 64)
// that can be resident at once on the current device (0 if none).
cudaError_t tc_gemm_max_clusters(int bn, int cluster, int* clusters);

// CTA-pair kernel (clusters of two CTAs, one cta_group::2 MMA per pair):
// tiles of 256 P rows x `bn` Q rows; `grid` CTAs (even).  args.pair must be 1.
bool tc_gemm_pair_supports(int bn);
cudaError_t launch_tc_gemm_pair(const TcArgs& args, int bn, int grid, cudaStream_t stream);
// Clusters of the pair kernel that can be resident at once on the current
// device (0 if it cannot run there).
cudaError_t tc_gemm_pair_max_clusters(int* clusters);

// Copy `rows` rows of `row_bytes` bytes from a source with row pitch
// `src_pitch` (any 2-byte alignment) into a destination with a 16-byte
// aligned pitch `dst_pitch`.
cudaError_t launch_repack_rows(const void* src, int64_t src_pitch, void* dst, int64_t dst_pitch, int64_t rows,
                               int64_t row_bytes, cudaStream_t stream);

cudaError_t launch_magic_divmod(const uint32_t* n, size_t count, MagicDiv m, uint32_t* q, uint32_t* r,
                                cudaStream_t stream);

// out[j] = perm_fwd (inverse = 0) or perm_inv (inverse != 0) of in[j].
cudaError_t launch_perm(const uint32_t* in, size_t n, uint32_t count, uint32_t block, uint32_t stride, int inverse,
                        uint32_t* out, cudaStream_t stream);

}  // namespace lgt
