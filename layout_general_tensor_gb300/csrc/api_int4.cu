// C ABI, int4-weight plans: the choice between the two kernel forms, the
// workspace layout of the prepared activation, tensor-map encoding and the
// launches (pre-pass, then the GEMM).  gemm_create and gemm_run in api.cu
// call in here for b_dtype = GEMM_INT4.
//
// Forms.  Plans run the fp16 form (gemm_int4.cu), the faster of the two on
// the shapes measured so far.  LGT_GEMM_INT4_FORM=e4m3 at gemm_create selects
// the e4m3 form (gemm_int4_f8.cu) where it applies: activations of up to 16
// rows, K-contiguous, with K and the group size multiples of 128 and split
// ranges of whole 128-deep blocks.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>

#include "gemm.h"
#include "int4.h"
#include "kernels.h"
#include "plan.h"

namespace lgt {

// The int4 kernels' launch arguments of a plan's last run, keyed by the
// buffers they depend on (see ArgCache).
struct Int4Cache {
  int busy;
  int valid;
  const void* B;
  void* C;
  const void* scales;
  const void* zeros;
  const uint8_t* ws;
  float* partial;
  int32_t* counters;
  Int4Args args;
};

namespace {

constexpr int kBlockK = 64;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Packed int4 weights: N rows of `ld_bytes` bytes (K/2 used), box 128 bytes
// (256 codes) x 128 rows, 128-byte swizzle so that the threads' 16-byte row
// reads fall in different bank groups.
bool encode_int4_weights(CUtensorMap* map, const void* ptr, int64_t N, int64_t ld_bytes) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(ld_bytes), static_cast<cuuint64_t>(N)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_bytes)};
  cuuint32_t box[2] = {128, static_cast<cuuint32_t>(TILE_P)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp16 form's prepared activation, K-block-major fp16 (element (m, k) at
// ((k / 64) * M + m) * 64 + k % 64): a 3-D map {64, M, K / 64}, box
// {64, bn, kb_box}, 128-byte swizzle, so one copy brings a stage's K blocks
// as kb_box consecutive bn x 128-byte tiles.
bool encode_int4_activation(CUtensorMap* map, const void* ptr, int64_t M, int64_t K, int bn, int kb_box) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
  cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(M) * 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(bn), static_cast<cuuint32_t>(kb_box)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// e4m3 form's prepared activation, Xp[K / 128][48][128] bytes (the three
// terms of 16 rows per 128-deep block): a 3-D map {128, 48, K / 128}, box
// {128, 48, 1} (one segment), 128-byte swizzle.
bool encode_int4f8_activation(CUtensorMap* map, const void* ptr, int64_t K) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, 48, static_cast<cuuint64_t>(K / 128)};
  cuuint64_t strides[2] = {128, 48 * 128};
  cuuint32_t box[3] = {128, 48, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool build_int4_args(const gemm_plan* plan, const void* B, void* C, const void* scales, const void* zeros,
                     const uint8_t* ws, float* partial, int32_t* counters, Int4Args& a4) {
  const gemm_desc_t& d = plan->d;
  std::memset(&a4, 0, sizeof(a4));
  TcArgs& args = a4.t;
  const bool f8 = plan->int4_form == 2;
  const void* ap = ws + plan->off_aprep;
  if (f8) {
    if (!encode_int4f8_activation(&args.tm_q, ap, d.K)) return false;
  } else if (!encode_int4_activation(&args.tm_q, ap, d.M, d.K, plan->bn,
                                     d.K / 64 < 4 ? static_cast<int>(d.K / 64) : 4)) {
    return false;
  }
  if (d.flags & GEMM_FLAG_INT4_PREPACKED) {
    // B is the pre-packed buffer (gemm_int4_prepack): bulk copies, no map
    a4.wpre = static_cast<const uint8_t*>(B);
    a4.pre_block = static_cast<int32_t>(pre_block_bytes(static_cast<int>(plan->group)));
    a4.pre_stages = static_cast<int32_t>((d.K + 255) / 256);
    a4.pre_kbpg = static_cast<int32_t>(plan->group / kBlockK);
  } else if (!encode_int4_weights(&a4.tm_w, B, d.N, plan->ldb)) {
    return false;
  }
  args.c = C;
  args.ldc = plan->ldc;
  args.ws = partial;
  args.counters = counters;
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
  args.rr_tiles = plan->rr_tiles;
  args.det = plan->det;
  args.max_runs = plan->max_runs;
  if (plan->det) args.slots = partial;
  args.div_split = magic_encode(static_cast<uint32_t>(plan->split));
  args.div_tiles_p = magic_encode(static_cast<uint32_t>(plan->tiles_p));
  args.swap = plan->swap;
  args.c_bf16 = d.c_dtype == GEMM_BF16;
  args.c_vec = (reinterpret_cast<uintptr_t>(C) % 16 == 0) && (plan->ldc % 8 == 0);
  args.ws_vec = (d.N % 4 == 0);
  args.q_mn = 0;
  // MMA A operand: the expanded weight in TMEM (K-major); B: the activation.
  // The fp16 form's descriptor (f16 x f16) and the e4m3 form's (e4m3 x e4m3,
  // N = 48: three terms of 16 rows) have the same fields, all type codes 0.
  args.idesc = idesc_f16(0u, 0u, 0u, TILE_P, f8 ? 48u : static_cast<uint32_t>(plan->bn));
  a4.agsum = reinterpret_cast<const float*>(ws + plan->off_agsum);
  a4.inv_scale = f8 ? reinterpret_cast<const float*>(ws + plan->off_inv) : nullptr;
  a4.scales = static_cast<const uint16_t*>(scales);
  a4.zeros = static_cast<const uint16_t*>(zeros);
  a4.groups = static_cast<int32_t>(d.K / plan->group);
  a4.div_kb_per_group = magic_encode(static_cast<uint32_t>(plan->group / kBlockK));
  a4.x_box_kb = d.K / 64 < 4 ? static_cast<int32_t>(d.K / 64) : 4;
  a4.vec_sz = (a4.groups % 8 == 0) && reinterpret_cast<uintptr_t>(scales) % 16 == 0 &&
              reinterpret_cast<uintptr_t>(zeros) % 16 == 0;
  return true;
}

}  // namespace

void int4_plan(gemm_plan& p, size_t off) {
  const gemm_desc_t& d = p.d;
  const char* form = std::getenv("LGT_GEMM_INT4_FORM");
  // (pre-packed weights are the fp16 form's layout)
  const bool want_f8 = form && std::strcmp(form, "e4m3") == 0 && !(d.flags & GEMM_FLAG_INT4_PREPACKED);
  p.int4_form = (want_f8 && int4f8_supported(p.a_mn, d.M, d.K, p.group) && p.kb_per_split % 2 == 0) ? 2 : 1;
  p.off_aprep = off;
  if (p.int4_form == 2) {
    // three e4m3 terms of 16 rows per 128-deep block, then 1 / S_b and the
    // block sums, fp32 [K / 128][16] each
    const size_t tab = static_cast<size_t>(d.K / 128) * 16 * sizeof(float);
    p.off_agsum = align_up(off + int4f8_prep_bytes(d.K), 256);
    p.off_inv = align_up(p.off_agsum + tab, 256);
    p.ws_bytes = align_up(p.off_inv + tab, 256);
  } else {
    // the K-block-major, pair-ordered fp16 activation and its per-group sums
    p.off_agsum = align_up(off + static_cast<size_t>(d.M) * d.K * 2, 256);
    p.off_inv = 0;
    p.ws_bytes = align_up(p.off_agsum + static_cast<size_t>(d.M) * (d.K / p.group) * sizeof(float), 256);
  }
  p.ws_bytes_misaligned = p.ws_bytes;
}

void int4_cache_free(gemm_plan* plan) {
  delete plan->cache4;
  plan->cache4 = nullptr;
}

gemm_status_t run_int4(gemm_plan* plan, const void* A, const void* B, void* C, const void* scales, const void* zeros,
                       uint8_t* ws, float* partial, int32_t* counters, cudaStream_t stream) {
  const gemm_desc_t& d = plan->d;
  // pre-pass: the activation in the layout the kernel's map reads
  if (plan->int4_form == 2) {
    if (launch_int4f8_prep(A, plan->lda, static_cast<int>(d.M), static_cast<int>(d.K), ws + plan->off_aprep,
                           reinterpret_cast<float*>(ws + plan->off_inv), reinterpret_cast<float*>(ws + plan->off_agsum),
                           plan->sms_grid, stream) != cudaSuccess)
      return GEMM_ERR_CUDA;
  } else if (launch_int4_prep(A, plan->lda, plan->a_mn, static_cast<int>(d.M), static_cast<int>(d.K),
                              static_cast<int>(plan->group), ws + plan->off_aprep,
                              reinterpret_cast<float*>(ws + plan->off_agsum), plan->sms_grid, stream) != cudaSuccess) {
    return GEMM_ERR_CUDA;
  }
  if (!plan->cache4) plan->cache4 = new (std::nothrow) Int4Cache();
  Int4Cache* cache = plan->cache4;
  const bool mine = cache && __atomic_exchange_n(&cache->busy, 1, __ATOMIC_ACQUIRE) == 0;
  Int4Args a4;
  if (mine && cache->valid && cache->B == B && cache->C == C && cache->scales == scales && cache->zeros == zeros &&
      cache->ws == ws && cache->partial == partial && cache->counters == counters) {
    a4 = cache->args;
  } else {
    if (!build_int4_args(plan, B, C, scales, zeros, ws, partial, counters, a4)) {
      if (mine) __atomic_store_n(&cache->busy, 0, __ATOMIC_RELEASE);
      return GEMM_ERR_CUDA;
    }
    if (mine) {
      cache->valid = 1;
      cache->B = B;
      cache->C = C;
      cache->scales = scales;
      cache->zeros = zeros;
      cache->ws = ws;
      cache->partial = partial;
      cache->counters = counters;
      cache->args = a4;
    }
  }
  if (mine) __atomic_store_n(&cache->busy, 0, __ATOMIC_RELEASE);
  const cudaError_t e = plan->int4_form == 2 ? launch_int4f8_gemm(a4, plan->grid, stream)
                                             : launch_int4_gemm(a4, plan->bn, plan->grid, stream);
  return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace lgt
