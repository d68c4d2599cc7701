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
  // Operands must be addressable in place, by TMA or by the kernel's
  // realigning loader: there is no room reserved for realigned copies.
  if (plan->det) return GEMM_ERR_UNSUPPORTED;  // per-run slots are not kept in the static array
  if (plan->repack_a || plan->repack_b) return GEMM_ERR_UNSUPPORTED;
  {
    const bool a_mis = reinterpret_cast<uintptr_t>(A) % 16 != 0, b_mis = reinterpret_cast<uintptr_t>(B) % 16 != 0;
    const bool rl_a = a_mis || (plan->lda * 2) % 16 != 0, rl_b = b_mis || (plan->ldb * 2) % 16 != 0;
    if ((a_mis || b_mis) && !(plan->rl_ok && lgt::rl_fits(*plan, rl_a, rl_b))) return GEMM_ERR_UNSUPPORTED;
  }

  // Scratch layout: [tile counters][fp32 partial sums M x N].  A stream-K
  // tail that does not fit is dropped (whole tiles only).
  const gemm_plan no_tail = lgt::plan_without_tail(*plan);
  if (plan->tail_tiles &&
      align256(static_cast<size_t>(plan->num_counters) * sizeof(int32_t)) + static_cast<size_t>(d.M) * d.N * 4 >
          kStaticScratchBytes)
    plan = &no_tail;
  // (split-K in a cluster adds its partials in shared memory: no region)
  const bool split_region = plan->split > 1 && plan->cl_size <= 1;
  const size_t counters_bytes =
      split_region ? align256(static_cast<size_t>(plan->num_counters) * sizeof(int32_t)) : 0;
  const size_t partial_bytes = split_region ? static_cast<size_t>(d.M) * d.N * sizeof(float) : 0;
  if (counters_bytes + partial_bytes > kStaticScratchBytes) return GEMM_ERR_WORKSPACE;

  uint8_t* scratch = static_cast<uint8_t*>(scratch_address(plan->device));
  if (!scratch) return GEMM_ERR_CUDA;
  if (split_region) {
    // The array keeps whatever the previous call left; the counters and the
    // partial sums must start at zero.
    if (cudaMemsetAsync(scratch, 0, counters_bytes + partial_bytes, stream) != cudaSuccess) return GEMM_ERR_CUDA;
  }

  float* partial = split_region ? reinterpret_cast<float*>(scratch + counters_bytes) : nullptr;
  int32_t* counters = split_region ? reinterpret_cast<int32_t*>(scratch) : nullptr;
  return lgt::launch_dense(plan, A, plan->lda, B, plan->ldb, C, partial, counters, stream);
}
