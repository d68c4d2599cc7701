// gemm_run_static_scratch: run a plan with no device memory from the caller.
//
// Who needs this.  gemm_run takes a caller-provided workspace (the fp32
// split-K partial sums and per-tile counters).  Some callers cannot provide
// one at the moment they run the GEMM: an inference-engine plugin whose
// enqueue callback is not allowed to allocate, a service loop that must not
// stall on cudaMalloc / cudaFree (cudaFree can synchronise the whole device),
// or code running after another allocator has reserved all free device
// memory.  For them this entry point uses a fixed scratch array that lives in
// the library's own device memory, so nothing is allocated per call.
//
// Cost of that choice: every GPU on which the library is loaded holds the
// array (kStaticScratchBytes) until the process exits, and every call on a
// device shares the same array.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "plan.h"

namespace {

constexpr size_t kStaticScratchBytes = 8u << 20;  // 8 MiB: fp32 partials + tile counters
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a host-side stand-in:
// its device address is looked up per device with cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Once per device (with that device current): resolve the array's device
// address.  Returns nullptr on failure.
void* scratch_address(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_addr[device] = p;
  }
  return g_scratch_addr[device];
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" gemm_status_t gemm_run_static_scratch(const gemm_plan_t* plan, const void* A, const void* B, void* C,
                                                 void* stream_ptr) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  const gemm_desc_t& d = plan->d;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (plan->kernel != 0) return GEMM_ERR_UNSUPPORTED;
  if (d.M == 0 || d.N == 0) return GEMM_OK;
  if (!C) return GEMM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(C) % 2) return GEMM_ERR_ALIGNMENT;
  if (plan->device < 0 || !plan->d_status) return GEMM_ERR_CUDA;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != plan->device) return GEMM_ERR_INVALID_ARG;
  if (d.K == 0) {
    return cudaMemset2DAsync(C, plan->ldc * 2, 0, d.N * 2, d.M, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
  }
  if (!A || !B) return GEMM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(A) % 2 || reinterpret_cast<uintptr_t>(B) % 2) return GEMM_ERR_ALIGNMENT;
  // Operands must be addressable by TMA in place: there is no room reserved
  // for realigned copies.
  if (plan->repack_a || plan->repack_b || reinterpret_cast<uintptr_t>(A) % 16 ||
      reinterpret_cast<uintptr_t>(B) % 16)
    return GEMM_ERR_UNSUPPORTED;

  // Scratch layout: [tile counters][fp32 partial sums M x N].
  const size_t tiles = static_cast<size_t>(plan->tiles_p) * plan->tiles_q;
  const size_t counters_bytes = plan->split > 1 ? align256(tiles * sizeof(int32_t)) : 0;
  const size_t partial_bytes = plan->split > 1 ? static_cast<size_t>(d.M) * d.N * sizeof(float) : 0;
  if (counters_bytes + partial_bytes > kStaticScratchBytes) return GEMM_ERR_WORKSPACE;

  uint8_t* scratch = static_cast<uint8_t*>(scratch_address(plan->device));
  if (!scratch) return GEMM_ERR_CUDA;
  if (plan->split > 1) {
    // The array keeps whatever the previous call left; the counters and the
    // partial sums must start at zero.
    if (cudaMemsetAsync(scratch, 0, counters_bytes + partial_bytes, stream) != cudaSuccess) return GEMM_ERR_CUDA;
  }

  lgt::TcArgs args;
  std::memset(&args, 0, sizeof(args));
  const bool a_is_p = !plan->swap;
  const void* p_ptr = a_is_p ? A : B;
  const void* q_ptr = a_is_p ? B : A;
  const int p_mn = a_is_p ? plan->a_mn : plan->b_mn;
  const int q_mn = a_is_p ? plan->b_mn : plan->a_mn;
  const int64_t p_ext = a_is_p ? d.M : d.N;
  const int64_t q_ext = a_is_p ? d.N : d.M;
  const int64_t p_ld = a_is_p ? plan->lda : plan->ldb;
  const int64_t q_ld = a_is_p ? plan->ldb : plan->lda;
  if (!lgt::encode_operand(&args.tm_p, p_ptr, d.a_dtype, p_mn, p_ext, d.K, p_ld, lgt::TILE_P)) return GEMM_ERR_CUDA;
  if (!lgt::encode_operand(&args.tm_q, q_ptr, d.a_dtype, q_mn, q_ext, d.K, q_ld, plan->bn)) return GEMM_ERR_CUDA;
  args.c = C;
  args.ldc = plan->ldc;
  if (plan->split > 1) {
    args.counters = reinterpret_cast<int32_t*>(scratch);
    args.ws = reinterpret_cast<float*>(scratch + counters_bytes);
  }
  args.status = plan->d_status;
  args.wait_limit_ns = plan->wait_limit_ns;
  args.M = static_cast<int32_t>(d.M);
  args.N = static_cast<int32_t>(d.N);
  args.K = static_cast<int32_t>(d.K);
  args.tiles_p = plan->tiles_p;
  args.tiles_q = plan->tiles_q;
  args.split = plan->split;
  args.kb_per_split = plan->kb_per_split;
  args.kb_total = plan->kb_total;
  args.num_units = plan->num_units;
  args.div_split = lgt::magic_encode(static_cast<uint32_t>(plan->split));
  args.div_tiles_p = lgt::magic_encode(static_cast<uint32_t>(plan->tiles_p));
  args.p_mn = p_mn;
  args.q_mn = q_mn;
  args.swap = plan->swap;
  args.c_bf16 = d.c_dtype == GEMM_BF16;
  args.c_vec = (reinterpret_cast<uintptr_t>(C) % 16 == 0) && (plan->ldc % 8 == 0);
  args.ws_vec = (d.N % 4 == 0);
  args.idesc = lgt::idesc_f16(d.a_dtype == GEMM_BF16 ? 1u : 0u, static_cast<uint32_t>(p_mn),
                              static_cast<uint32_t>(q_mn), lgt::TILE_P, static_cast<uint32_t>(plan->bn));
  const int grid = plan->num_units < plan->sms_grid ? plan->num_units : plan->sms_grid;
  return lgt::launch_tc_gemm(args, plan->bn, grid, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}
