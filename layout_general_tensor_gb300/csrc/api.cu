// C ABI: planning (tile, swap, split-K factor, workspace), validation, TMA
// descriptor encoding and kernel launch.  See include/gemm.h for the contract.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "gemm.h"
#include "kernels.h"
#include "realign.cuh"
#include "int4.h"
#include "plan.h"

using lgt::MagicDiv;


namespace {

constexpr int kBlockK = 64;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int next_pow2_at_least16(int64_t v) {
  int p = 16;
  while (p < v && p < 256) p <<= 1;
  return p;
}

bool is_half(int t) { return t == GEMM_F16 || t == GEMM_BF16; }

gemm_status_t validate(const gemm_desc_t& d) {
  const int64_t lim = (1ll << 31) - 1;
  if (d.M < 0 || d.N < 0 || d.K < 0 || d.M > lim || d.N > lim || d.K > lim) return GEMM_ERR_INVALID_ARG;
  if ((d.a_layout != GEMM_K_CONTIG && d.a_layout != GEMM_MN_CONTIG) ||
      (d.b_layout != GEMM_K_CONTIG && d.b_layout != GEMM_MN_CONTIG))
    return GEMM_ERR_INVALID_ARG;
  if (!is_half(d.c_dtype)) return GEMM_ERR_INVALID_ARG;
  if (d.b_dtype == GEMM_INT4) {
    if (d.a_dtype != GEMM_F16 || d.b_layout != GEMM_K_CONTIG) return GEMM_ERR_INVALID_ARG;
  } else if (!is_half(d.a_dtype) || d.a_dtype != d.b_dtype) {
    return GEMM_ERR_INVALID_ARG;
  }
  if (d.split_k < 0 || d.split_k > 65536 || d.num_sms < 0 || d.group_size < 0 ||
      (d.flags & ~(GEMM_FLAG_DETERMINISTIC | GEMM_FLAG_INT4_PREPACKED | GEMM_FLAG_TEST_WITHHOLD_STAGE)) != 0)
    return GEMM_ERR_INVALID_ARG;
  if (d.lda < 0 || d.ldb < 0 || d.ldc < 0) return GEMM_ERR_INVALID_ARG;
  const int64_t a_min = d.a_layout == GEMM_K_CONTIG ? d.K : d.M;
  const int64_t c_min = d.N;
  if (d.lda && d.lda < a_min) return GEMM_ERR_INVALID_ARG;
  if (d.ldc && d.ldc < c_min) return GEMM_ERR_INVALID_ARG;
  if (d.b_dtype != GEMM_INT4) {
    const int64_t b_min = d.b_layout == GEMM_K_CONTIG ? d.K : d.N;
    if (d.ldb && d.ldb < b_min) return GEMM_ERR_INVALID_ARG;
  }
  return GEMM_OK;
}

// Resident clusters of the CTA-pair kernel on each device (queried once).
int pair_clusters(int device) {
  constexpr int kMaxDevices = 64;
  static int cached[kMaxDevices];
  static std::once_flag once[kMaxDevices];
  if (device < 0 || device >= kMaxDevices) return 0;
  std::call_once(once[device], [device] {
    int c = 0;
    if (lgt::tc_gemm_pair_max_clusters(&c) != cudaSuccess) {
      cudaGetLastError();
      c = 0;
    }
    cached[device] = c;
  });
  return cached[device];
}

// Integer value of an environment variable, or `dflt` when unset / empty.
int env_int(const char* name, int dflt) {
  const char* s = std::getenv(name);
  if (!s || !*s) return dflt;
  return std::atoi(s);
}

// Time model of a persistent tile kernel (relative units: microseconds of a
// 4096-deep K loop on this GPU).  A full wave is paced by the operand stream
// from L2 into shared memory: measured 18.2 us for pair tiles of width 128,
// 21.2 us for width 256 (about w + 650 column-units), 25.2 us for single-CTA
// 128 x 256 tiles.  A partial last wave competes with fewer CTAs and runs
// faster, but a tile never beats its pure MMA time (17 us for 256 columns).
double waves_cost(int64_t tiles, int64_t workers, double wave_us, double mma_us) {
  const int64_t full = tiles / workers, rest = tiles % workers;
  double t = static_cast<double>(full) * wave_us;
  if (rest) {
    const double frac = static_cast<double>(rest) / static_cast<double>(workers) * wave_us;
    t += frac > mma_us ? frac : mma_us;
  }
  return t;
}
double pair_wave_us(int w) { return (w + 650.0) / 906.0 * 21.2; }
double mma_tile_us(int w) { return w / 256.0 * 17.0; }
constexpr double kSingleWave256Us = 25.2;
constexpr int kPairWidths[] = {256, 224, 192, 160, 128};

uint64_t wait_limit_from_env() {
  const char* s = std::getenv("LGT_GEMM_WAIT_LIMIT_MS");
  if (s && *s) {
    const double ms = std::atof(s);
    if (ms > 0) return static_cast<uint64_t>(ms * 1e6);
  }
  return 2000ull * 1000ull * 1000ull;  // 2 s
}

}  // namespace

namespace lgt {

// cuTensorMapEncodeTiled, resolved once through the runtime (no link-time
// dependency on the driver library); null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D tensor map over a 16-bit operand.  K-major: dims {K, rows}, box
// {64, box_rows}.  MN-major: dims {mn, K}, box {64, 64}.  128-byte swizzle,
// zero fill outside the tensor (ragged M / N / K tails).
bool encode_operand(CUtensorMap* map, const void* ptr, int dtype, bool mn_major, int64_t rows_or_mn, int64_t K,
                    int64_t ld, int box_rows) {
  auto enc = get_encoder();
  if (!enc) return false;
  const CUtensorMapDataType dt =
      dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t dims[2];
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2];
  cuuint32_t estr[2] = {1, 1};
  if (!mn_major) {
    dims[0] = static_cast<cuuint64_t>(K);
    dims[1] = static_cast<cuuint64_t>(rows_or_mn);
    box[0] = kBlockK;
    box[1] = static_cast<cuuint32_t>(box_rows);
  } else {
    dims[0] = static_cast<cuuint64_t>(rows_or_mn);
    dims[1] = static_cast<cuuint64_t>(K);
    box[0] = 64;
    box[1] = kBlockK;
  }
  CUresult r = enc(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output-side maps for the staged epilogue: a row-major rows x cols matrix
// (row pitch `pitch_bytes`), box 32 x 32.  fp32 partials use the 128-byte
// swizzle (32 floats = one 128-byte row), 16-bit C the 64-byte swizzle (32
// halves = one 64-byte row), matching the epilogue's shared-memory writes.
bool encode_output(CUtensorMap* map, void* ptr, bool fp32, int c_dtype, int64_t rows, int64_t cols,
                   int64_t pitch_bytes) {
  auto enc = get_encoder();
  if (!enc) return false;
  const CUtensorMapDataType dt = fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                      : (c_dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(EPI_BOX), static_cast<cuuint32_t>(EPI_BOX)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dt, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   fp32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Realigning loader (realign.cuh): one map per row class of an operand TMA
// cannot address directly.  Class r: the rows r, r + P, ... (P = 16 /
// gcd(pitch, 16)), from the 16-byte word holding row r's start, pitch P times
// the row pitch; boxes of 72 elements by the class rows of a stage.
bool encode_classes(TcArgs& args, int o, const void* ptr, int dtype, int mn, int64_t ext, int64_t K, int64_t ld,
                    int tile_rows) {
  auto enc = get_encoder();
  if (!enc) return false;
  const int64_t pitch = ld * 2;
  const int P = rl_classes(pitch);
  const int64_t nrows = mn ? K : ext;   // storage rows
  const int64_t rowlen = mn ? ext : K;  // elements along a storage row
  if (nrows < P) return false;
  const CUtensorMapDataType dt = dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  for (int r = 0; r < P; ++r) {
    const uintptr_t start = reinterpret_cast<uintptr_t>(ptr) + static_cast<uintptr_t>(r * pitch);
    const uintptr_t word = start & ~static_cast<uintptr_t>(15);
    const int64_t dr = static_cast<int64_t>(start - word);  // even
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(rowlen + dr / 2), static_cast<cuuint64_t>((nrows - r + P - 1) / P)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(P * pitch)};
    const RlGeom geo = rl_geom(mn, tile_rows, P);
    cuuint32_t box[2] = {static_cast<cuuint32_t>(64 * geo.per_box + 8), static_cast<cuuint32_t>(geo.box_rows)};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&args.tm_rl[o][r], dt, 2, reinterpret_cast<void*>(word), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
    args.rl_d[o][r] = static_cast<int32_t>(dr);
  }
  args.rl_on[o] = 1;
  args.rl_cls[o] = P;
  return true;
}

// Whether the realigning loader's staging fits the plan's kernel when A
// (rl_a) and / or B (rl_b) go through it.
bool rl_fits(const gemm_plan& p, bool rl_a, bool rl_b) {
  const bool a_is_p = !p.swap;
  const int a_cls = rl_a ? rl_classes(p.lda * 2) : 0, b_cls = rl_b ? rl_classes(p.ldb * 2) : 0;
  const int p_cls = a_is_p ? a_cls : b_cls, q_cls = a_is_p ? b_cls : a_cls;
  const int p_mn = a_is_p ? p.a_mn : p.b_mn, q_mn = a_is_p ? p.b_mn : p.a_mn;
  return p.pair ? tc_gemm_pair_rl_fits(p.bn, p_mn, q_mn, p_cls, q_cls)
                : tc_gemm_rl_fits(p.bn, p_mn, q_mn, p_cls, q_cls);
}

// The dense kernels' arguments for one run (tensor maps encoded here).
bool build_dense_args(const gemm_plan* plan, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                      float* partial, int32_t* counters, TcArgs& args) {
  const gemm_desc_t& d = plan->d;
  std::memset(&args, 0, sizeof(args));
  // P operand: the MMA's M side (128-row tiles, 256 for a CTA pair whose
  // CTAs load 128 each).  Q operand: bn-row tiles (128 per CTA for a pair).
  const bool a_is_p = !plan->swap;
  const void* p_ptr = a_is_p ? A : B;
  const void* q_ptr = a_is_p ? B : A;
  const int p_mn = a_is_p ? plan->a_mn : plan->b_mn;
  const int q_mn = a_is_p ? plan->b_mn : plan->a_mn;
  const int64_t p_ext = a_is_p ? d.M : d.N;
  const int64_t q_ext = a_is_p ? d.N : d.M;
  const int64_t p_ld = a_is_p ? lda : ldb;
  const int64_t q_ld = a_is_p ? ldb : lda;
  const int q_box = plan->pair ? plan->bn / 2 : plan->bn;
  // an operand TMA cannot address (pitch or base not 16-byte aligned) goes to
  // the kernel's realigning loader (the plan allows it, else it was repacked)
  auto tma_ok = [](const void* ptr, int64_t ld) {
    return reinterpret_cast<uintptr_t>(ptr) % 16 == 0 && (ld * 2) % 16 == 0;
  };
  const bool rl_p = plan->rl_ok && !tma_ok(p_ptr, p_ld);
  const bool rl_q = plan->rl_ok && !tma_ok(q_ptr, q_ld);
  if (!rl_p && !encode_operand(&args.tm_p, p_ptr, d.a_dtype, p_mn, p_ext, d.K, p_ld, TILE_P)) return false;
  if (!rl_q && !encode_operand(&args.tm_q, q_ptr, d.a_dtype, q_mn, q_ext, d.K, q_ld, q_box)) return false;
  if (rl_p || rl_q) {
    // (gemm_run falls back to repacking when the staging does not fit)
    const int pc = rl_p ? rl_classes(p_ld * 2) : 0, qc = rl_q ? rl_classes(q_ld * 2) : 0;
    if (!(plan->pair ? tc_gemm_pair_rl_fits(plan->bn, p_mn, q_mn, pc, qc) : tc_gemm_rl_fits(plan->bn, p_mn, q_mn, pc, qc)))
      return false;
  }
  if (rl_p && !encode_classes(args, 0, p_ptr, d.a_dtype, p_mn, p_ext, d.K, p_ld, TILE_P)) return false;
  if (rl_q && !encode_classes(args, 1, q_ptr, d.a_dtype, q_mn, q_ext, d.K, q_ld, q_box)) return false;
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
  args.tail_tiles = plan->fin_tiles;
  args.det = plan->det;
  args.max_runs = plan->max_runs;
  if (plan->det) args.slots = partial;
  args.div_split = magic_encode(static_cast<uint32_t>(plan->split));
  args.div_tiles_p = magic_encode(static_cast<uint32_t>(plan->tiles_p));
  args.p_mn = p_mn;
  args.q_mn = q_mn;
  args.swap = plan->swap;
  args.c_bf16 = d.c_dtype == GEMM_BF16;
  args.c_vec = (reinterpret_cast<uintptr_t>(C) % 16 == 0) && (plan->ldc % 8 == 0);
  args.ws_vec = (d.N % 4 == 0);
  args.pair = plan->pair;
  args.cl_size = plan->cl_size;
  // Staged epilogue: whole-line bulk stores of C and bulk reductions of the
  // fp32 partials, where the pointers and pitches allow them (16 bytes).
  static const bool tma_epi = env_int("LGT_GEMM_TMA_EPI", 1) != 0;
  if (tma_epi) {
    args.tma_c = args.c_vec && encode_output(&args.tm_c, C, false, d.c_dtype, d.M, d.N, plan->ldc * 2);
    args.tma_ws = partial && !plan->det && (d.N % 4 == 0) &&
                  encode_output(&args.tm_ws, partial, true, 0, d.M, d.N, d.N * 4);
  }
  args.idesc = idesc_f16(d.a_dtype == GEMM_BF16 ? 1u : 0u, static_cast<uint32_t>(p_mn), static_cast<uint32_t>(q_mn),
                         static_cast<uint32_t>(TILE_P << plan->pair), static_cast<uint32_t>(plan->bn));
  return true;
}

gemm_status_t launch_dense(const gemm_plan* plan, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                           float* partial, int32_t* counters, cudaStream_t stream, int withhold) {
  ArgCache* cache = plan->cache;
  const bool mine = cache && __atomic_exchange_n(&cache->busy, 1, __ATOMIC_ACQUIRE) == 0;
  TcArgs args;
  if (mine && cache->valid && cache->A == A && cache->B == B && cache->C == C && cache->partial == partial &&
      cache->counters == counters && cache->lda == lda && cache->ldb == ldb) {
    args = cache->args;
  } else {
    if (!build_dense_args(plan, A, lda, B, ldb, C, partial, counters, args)) {
      if (mine) __atomic_store_n(&cache->busy, 0, __ATOMIC_RELEASE);
      return GEMM_ERR_CUDA;
    }
    if (mine) {
      cache->valid = 1;
      cache->A = A;
      cache->B = B;
      cache->C = C;
      cache->partial = partial;
      cache->counters = counters;
      cache->lda = lda;
      cache->ldb = ldb;
      cache->args = args;
    }
  }
  if (mine) __atomic_store_n(&cache->busy, 0, __ATOMIC_RELEASE);
  args.withhold = withhold;
  const cudaError_t e = plan->pair ? launch_tc_gemm_pair(args, plan->bn, plan->grid, stream)
                                   : launch_tc_gemm(args, plan->bn, plan->grid, stream);
  return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

gemm_plan plan_without_tail(const gemm_plan& p) {
  gemm_plan q = p;
  q.cache = nullptr;  // the copy's arguments differ from the plan's
  q.withhold_armed = 0;
  if (!q.tail_tiles) return q;
  q.split = 1;
  q.kb_per_split = q.kb_total;
  q.rr_tiles = q.tiles_p * q.tiles_q;
  q.tail_tiles = 0;
  q.fin_tiles = 0;
  q.num_units = q.rr_tiles;
  const int workers = q.pair ? q.grid / 2 : q.sms_grid;
  q.grid = (q.pair ? 2 : 1) * (q.num_units < workers ? q.num_units : workers);
  return q;
}

}  // namespace lgt

extern "C" {

const char* gemm_status_string(gemm_status_t s) {
  switch (s) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED";
    case GEMM_ERR_ALIGNMENT: return "GEMM_ERR_ALIGNMENT";
    case GEMM_ERR_WORKSPACE: return "GEMM_ERR_WORKSPACE";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
    default: return "GEMM_ERR_UNKNOWN";
  }
}

int32_t gemm_splitk_auto(int64_t M, int64_t N, int64_t K, int32_t bm, int32_t bn, int32_t bk, int32_t num_sms,
                         double threshold) {
  return lgt::splitk_auto(M, N, K, bm, bn, bk, num_sms, threshold);
}

uint32_t gemm_perm_fwd(uint32_t i, uint32_t count, uint32_t block, uint32_t stride) {
  return lgt::perm_fwd(i, count, block, stride);
}

uint32_t gemm_perm_inv(uint32_t i, uint32_t count, uint32_t block, uint32_t stride) {
  return lgt::perm_inv(i, count, block, stride);
}

gemm_status_t gemm_perm_device(const uint32_t* in, size_t n, uint32_t count, uint32_t block, uint32_t stride,
                               int32_t inverse, uint32_t* out, void* stream) {
  if (n && (!in || !out)) return GEMM_ERR_INVALID_ARG;
  return lgt::launch_perm(in, n, count, block, stride, inverse, out, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? GEMM_OK
             : GEMM_ERR_CUDA;
}

size_t gemm_int4_prepack_bytes(int64_t N, int64_t K, int32_t group_size) {
  const int group = group_size ? group_size : 128;
  if (N <= 0 || K <= 0 || K % 64 != 0 || group % 64 != 0 || K % group != 0 ||
      !(group == 64 || group == 128 || group % 256 == 0))
    return 0;
  return lgt::pre_total_bytes(N, K, group);
}

gemm_status_t gemm_int4_prepack(const void* B, int64_t ldb, const void* scales, int64_t N, int64_t K,
                                int32_t group_size, void* out, void* stream) {
  const int group = group_size ? group_size : 128;
  if (gemm_int4_prepack_bytes(N, K, group) == 0) return GEMM_ERR_INVALID_ARG;
  if (!B || !scales || !out) return GEMM_ERR_INVALID_ARG;
  const int64_t ld = ldb ? ldb : K / 2;
  if (ld < K / 2) return GEMM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(B) % 16 || ld % 16 || reinterpret_cast<uintptr_t>(out) % 16 ||
      reinterpret_cast<uintptr_t>(scales) % 2)
    return GEMM_ERR_ALIGNMENT;
  return lgt::launch_int4_prepack(B, ld, scales, N, K, group, out, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GEMM_OK
             : GEMM_ERR_CUDA;
}

gemm_status_t gemm_magic_divmod_host(const uint32_t* n, size_t count, uint32_t divisor, uint32_t* q, uint32_t* r) {
  if (divisor == 0 || (count && (!n || !q || !r))) return GEMM_ERR_INVALID_ARG;
  const MagicDiv m = lgt::magic_encode(divisor);
  for (size_t i = 0; i < count; ++i) {
    if (n[i] >= (1u << 31)) return GEMM_ERR_INVALID_ARG;
    lgt::magic_divmod(n[i], m, q[i], r[i]);
  }
  return GEMM_OK;
}

gemm_status_t gemm_magic_divmod_device(const uint32_t* n, size_t count, uint32_t divisor, uint32_t* q, uint32_t* r,
                                       void* stream) {
  if (divisor == 0 || (count && (!n || !q || !r))) return GEMM_ERR_INVALID_ARG;
  const MagicDiv m = lgt::magic_encode(divisor);
  return lgt::launch_magic_divmod(n, count, m, q, r, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GEMM_OK
             : GEMM_ERR_CUDA;
}

gemm_status_t gemm_create(const gemm_desc_t* desc, gemm_plan_t** out) {
  if (!out) return GEMM_ERR_INVALID_ARG;
  *out = nullptr;
  if (!desc) return GEMM_ERR_INVALID_ARG;
  const gemm_status_t v = validate(*desc);
  if (v != GEMM_OK) return v;
  const bool int4 = desc->b_dtype == GEMM_INT4;
  if (int4) {
    // group: a multiple of the 64-deep K block that divides K; rows of packed
    // bytes must be TMA-addressable (16-byte multiples)
    const int64_t g = desc->group_size ? desc->group_size : 128;
    if (g % kBlockK != 0 || desc->K % g != 0 || desc->K % 2 != 0) return GEMM_ERR_INVALID_ARG;
    const int64_t ldb = desc->ldb ? desc->ldb : desc->K / 2;
    if (ldb < desc->K / 2) return GEMM_ERR_INVALID_ARG;
    if (ldb % 16 != 0) return GEMM_ERR_UNSUPPORTED;
  }

  gemm_plan p;
  std::memset(&p, 0, sizeof(p));
  p.d = *desc;
  const gemm_desc_t& d = p.d;
  p.device = -1;
  p.wait_limit_ns = wait_limit_from_env();

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) {
    ndev = 0;
    cudaGetLastError();
  }
  if (ndev > 0) {
    if (cudaGetDevice(&p.device) != cudaSuccess) return GEMM_ERR_CUDA;
    if (cudaDeviceGetAttribute(&p.sms_grid, cudaDevAttrMultiProcessorCount, p.device) != cudaSuccess)
      return GEMM_ERR_CUDA;
  }
  p.sms_rule = d.num_sms > 0 ? d.num_sms : p.sms_grid;
  if (p.sms_rule <= 0) return GEMM_ERR_CUDA;  // rule needs an SM count and there is no device

  p.lda = d.lda ? d.lda : (d.a_layout == GEMM_K_CONTIG ? d.K : d.M);
  p.ldb = d.ldb ? d.ldb : (d.b_layout == GEMM_K_CONTIG ? d.K : d.N);
  p.ldc = d.ldc ? d.ldc : d.N;
  if (p.lda == 0) p.lda = 1;
  if (p.ldb == 0) p.ldb = 1;
  if (p.ldc == 0) p.ldc = 1;
  p.a_mn = d.a_layout == GEMM_MN_CONTIG;
  p.b_mn = d.b_layout == GEMM_MN_CONTIG;
  if (int4) {
    p.kernel = 1;
    p.group = d.group_size ? d.group_size : 128;
    p.ldb = d.ldb ? d.ldb : d.K / 2;  // bytes
  }

  // Tile shape.  Skinny M runs swapped: the 128-row MMA side walks N and the
  // MMA's N extent covers all of M.
  p.swap = ((d.M <= 64 && d.N > d.M) || int4) ? 1 : 0;
  // (the int4 path reads a prepared K-contiguous copy of the activation)
  const bool q_mn = int4 ? false : (p.swap ? p.a_mn : p.b_mn);
  const int64_t q_extent = p.swap ? d.M : d.N;
  // 256-wide tiles halve the L2 -> shared-memory bytes per FLOP of 128-wide
  // ones; narrow problems use the smallest power of two covering them.
  // They are used only while the problem still has a tile for every SM.
  const int64_t p_tiles = ceil_div(p.swap ? d.N : d.M, lgt::TILE_P);
  const int sms = p.sms_grid > 0 ? p.sms_grid : p.sms_rule;
  int bn = q_extent >= 128 ? 128 : next_pow2_at_least16(q_extent);
  if (q_extent >= 256 && p_tiles * ceil_div(q_extent, 256) >= sms) bn = 256;
  if (int4 && bn > 64) bn = 64;  // the int4 epilogue holds a tile row's fp32 sums in registers
  if (q_mn && bn < 64) bn = 64;  // MN-major tiles come in 64-element swizzle atoms
  if (!p.swap) {
    // tuning override of the tile width for large problems
    const char* e = std::getenv("LGT_GEMM_BN");
    const int o = e ? std::atoi(e) : 0;
    if ((o == 64 || o == 128 || o == 192 || o == 256) && q_extent >= o) bn = o;
  }
  // CTA pairs (one cta_group::2 MMA over a 256 x w tile, w in 128..256):
  // where the single-CTA plan has at least a wave of 256-wide tiles, take the
  // pair width with the lowest modelled time if it beats the single-CTA plan.
  // LGT_GEMM_PAIR=0 / 1 disables / forces pairs, LGT_GEMM_PAIR_BN forces w.
  p.pair = 0;
  const int clusters = (!int4 && !p.swap && p.device >= 0) ? pair_clusters(p.device) : 0;
  if (clusters > 0) {
    const int mode = env_int("LGT_GEMM_PAIR", -1);
    const int forced_w = env_int("LGT_GEMM_PAIR_BN", 0);
    const int64_t pair_rows = ceil_div(d.M, 2 * lgt::TILE_P);
    int best_w = 0;
    double best = 0;
    for (int w : kPairWidths) {
      if (forced_w && w != forced_w) continue;
      const double c = waves_cost(pair_rows * ceil_div(q_extent, w), clusters, pair_wave_us(w), mma_tile_us(w));
      if (!best_w || c < best) {
        best_w = w;
        best = c;
      }
    }
    const double single = waves_cost(p_tiles * ceil_div(q_extent, bn), sms, kSingleWave256Us, mma_tile_us(bn));
    if (best_w && (mode == 1 || (mode != 0 && bn == 256 && best < single))) {
      p.pair = 1;
      bn = best_w;
    }
  }
  p.bn = bn;
  p.tiles_p = static_cast<int>(ceil_div(p.swap ? d.N : d.M, lgt::TILE_P << p.pair));
  p.tiles_q = static_cast<int>(ceil_div(q_extent, bn));

  // Split-K factor: the SM-waste rule on the logical M x N with 128 x 128 x 64
  // tiles, or the caller's factor.
  p.kb_total = static_cast<int>(ceil_div(d.K, kBlockK));
  if (d.K == 0) {
    p.split = 1;
  } else if (d.split_k == 0) {
    p.split = lgt::splitk_auto(d.M, d.N, d.K, 128, 128, kBlockK, p.sms_rule, 0.05);
  } else {
    p.split = d.split_k;
  }
  p.kb_per_split = p.kb_total > 0 ? static_cast<int>(ceil_div(p.kb_total, p.split)) : 0;
  if ((d.flags & GEMM_FLAG_INT4_PREPACKED) && d.split_k == 0 && p.split > 1 && p.kb_per_split % 4 != 0) {
    // pre-packed weights come in 256-deep stages: the rule's split ranges
    // are rounded up to whole stages
    p.kb_per_split = (p.kb_per_split + 3) / 4 * 4;
    p.split = static_cast<int>(ceil_div(p.kb_total, p.kb_per_split));
  }
  p.det = (d.flags & GEMM_FLAG_DETERMINISTIC) && p.split > 1;
  p.split_req = p.split;
  const int64_t tiles = static_cast<int64_t>(p.tiles_p) * p.tiles_q;
  if (tiles * (p.kb_total > 0 ? p.kb_total : 1) >= (1ll << 31)) return GEMM_ERR_UNSUPPORTED;
  const int workers = p.pair ? pair_clusters(p.device) : p.sms_grid;
  p.rr_tiles = p.split == 1 ? static_cast<int>(tiles) : 0;
  p.tail_tiles = 0;
  // Stream-K tail: with no K split, whole waves of tiles run as they are and
  // the K blocks of a last partial wave (at most 3/4 full) are spread evenly
  // over all workers, their fp32 partials reduced like split-K partials.
  // Off with GEMM_FLAG_DETERMINISTIC or LGT_GEMM_STREAMK=0.
  // (a plan with a tail keeps its fixup warps for it: operands TMA cannot
  // address are then repacked rather than realigned in the kernel)
  // (opt-in: on the shapes measured so far the repacking pre-pass is faster,
  // since it realigns each operand once while the loader pays per stage)
  const bool realign = !int4 && env_int("LGT_GEMM_REALIGN", 0) != 0;
  if (!int4 && !p.swap && p.split == 1 && !(d.flags & GEMM_FLAG_DETERMINISTIC) && p.kb_total >= 2 && workers > 0 &&
      env_int("LGT_GEMM_STREAMK", 1) != 0) {
    const int64_t full = tiles / workers, rest = tiles % workers;
    // (at least three whole waves: the tail's conversion runs behind the
    // whole tiles that follow it and needs two of them to stay hidden)
    if (full >= 3 && rest > 0 && rest * 4 <= static_cast<int64_t>(workers) * 3) {
      p.rr_tiles = static_cast<int>(full * workers);
      p.tail_tiles = static_cast<int>(rest);
      p.split = p.kb_total;  // a tail tile's units are its single K blocks
      p.kb_per_split = 1;
    }
  }
  p.num_units = static_cast<int>(tiles * p.split);
  // Split tiles of the tensor-core kernels are converted at the end by all
  // CTAs together (their fixup warps), not by each tile's last arriver: a
  // single CTA converting a whole tile is bound by its own L2 round trips.
  p.fin_tiles = int4 ? 0 : (p.tail_tiles ? p.tail_tiles : (p.split > 1 ? static_cast<int>(tiles) : 0));
  // arrival counters per tile (per half-tile for pairs); converted tiles
  // also keep a finished-rows counter per strip after them
  p.num_counters = static_cast<int>(tiles) * (1 + p.pair) * (p.fin_tiles ? 2 : 1);
  if (p.pair) {
    p.grid = 2 * (p.num_units < workers ? p.num_units : workers);
  } else {
    p.grid = p.num_units < p.sms_grid ? p.num_units : p.sms_grid;
  }

  // Storage rows of each operand and whether TMA can address them in place.
  p.a_rows = p.a_mn ? d.K : d.M;
  p.a_row_elems = p.a_mn ? d.M : d.K;
  p.b_rows = p.b_mn ? d.K : d.N;
  p.b_row_elems = p.b_mn ? d.N : d.K;
  p.rl_ok = realign && p.fin_tiles == 0 && d.M >= 8 && d.N >= 8 && d.K >= 8 &&
            lgt::rl_fits(p, (p.lda * 2) % 16 != 0, (p.ldb * 2) % 16 != 0);
  p.repack_a = !int4 && !p.rl_ok && (p.lda * 2) % 16 != 0;
  p.repack_b = !int4 && !p.rl_ok && (p.ldb * 2) % 16 != 0;
  p.a_pack_ld = align_up(static_cast<size_t>(p.a_row_elems), 8);
  p.b_pack_ld = align_up(static_cast<size_t>(p.b_row_elems), 8);

  // Split-K through a cluster's shared memory: when the tiles are few (a
  // skinny, swapped problem, BN <= 64) and a cluster of c CTAs per tile still
  // covers at least 3/4 of the SMs, each tile's K range is split over the c
  // CTAs of one cluster (c divides the split factor, so CTA b's contiguous
  // unit range is exactly split / c units of tile b / c) and their partials
  // are added on chip: no fp32 partial through L2, no counter, no fixup
  // pass.  Needs a device (the cluster occupancy query).  LGT_GEMM_CLUSTER=0
  // turns it off.
  p.cl_size = 0;
  if (!int4 && !p.pair && p.swap && !p.det && p.split > 1 && p.tail_tiles == 0 && p.bn <= 64 && p.device >= 0 &&
      env_int("LGT_GEMM_CLUSTER", 1) != 0) {
    for (int c : {8, 4, 2}) {
      if (c > p.bn / 4 || p.split % c != 0) continue;
      const int64_t g = tiles * c;
      if (g > p.sms_grid || g * 4 < static_cast<int64_t>(p.sms_grid) * 3) continue;
      int resident = 0;
      if (lgt::tc_gemm_max_clusters(p.bn, c, &resident) != cudaSuccess) {
        cudaGetLastError();
        continue;
      }
      if (resident < tiles) continue;
      p.cl_size = c;
      p.grid = static_cast<int>(g);
      p.fin_tiles = 0;
      break;
    }
  }

  if (p.det) {
    // Deterministic split-K: the tiles' runs (one per worker a tile's units
    // meet) each own a tile-shaped fp32 slot; max_runs is the most runs of
    // any tile.  Worker b owns units [b*U/G, (b+1)*U/G).
    p.fin_tiles = 0;
    const int64_t G = p.pair ? p.grid / 2 : p.grid;
    const int64_t U = static_cast<int64_t>(p.num_units);
    auto owner = [&](int64_t v) {
      int64_t b = G > 0 ? (v * G) / U : 0;
      while (b + 1 < G && ((b + 1) * U) / G <= v) ++b;
      while (b > 0 && (b * U) / G > v) --b;
      return b;
    };
    p.max_runs = 1;
    for (int64_t t = 0; G > 0 && t < tiles; ++t) {
      const int64_t r = owner((t + 1) * p.split - 1) - owner(t * p.split) + 1;
      if (r > p.max_runs) p.max_runs = static_cast<int>(r);
    }
  }
  size_t off = 0;
  // (split-K in a cluster adds its partials in shared memory: no region)
  if (p.split > 1 && p.cl_size <= 1) {
    p.off_partial = off;
    const size_t region = p.det ? static_cast<size_t>(tiles) * (1 + p.pair) * p.max_runs * lgt::TILE_P * p.bn *
                                      sizeof(float)
                                : static_cast<size_t>(d.M) * d.N * sizeof(float);
    off = align_up(off + region, 256);
    p.off_counters = off;
    off = align_up(off + static_cast<size_t>(p.num_counters) * sizeof(int32_t), 256);
  }
  const size_t pack_a_bytes = align_up(static_cast<size_t>(p.a_rows) * p.a_pack_ld * 2, 256);
  const size_t pack_b_bytes = int4 ? 0 : align_up(static_cast<size_t>(p.b_rows) * p.b_pack_ld * 2, 256);
  size_t off_aligned = off;
  p.off_pack_a = off;
  if (p.repack_a) off_aligned += pack_a_bytes;
  p.off_pack_b = off_aligned;
  if (p.repack_b) off_aligned += pack_b_bytes;
  p.ws_bytes = off_aligned;
  // When a base pointer is not 16-byte aligned the operand is repacked too.
  p.ws_bytes_misaligned = off + pack_a_bytes + pack_b_bytes;
  if (d.flags & GEMM_FLAG_INT4_PREPACKED) {
    // pre-packed weights: int4 only, whole 256-deep stages per split range,
    // groups of 64 or 128 or a multiple of 256 (the fp16 form: int4_plan)
    const bool group_ok = p.group == 64 || p.group == 128 || p.group % 256 == 0;
    if (!int4 || !group_ok || (p.split > 1 && p.kb_per_split % 4 != 0)) return GEMM_ERR_UNSUPPORTED;
  }
  if (int4) lgt::int4_plan(p, off);  // form, prepared-activation region and tables

  if (d.flags & GEMM_FLAG_TEST_WITHHOLD_STAGE) {
    // the test aid needs a kernel in which no CTA waits on another
    if (int4 || p.pair || p.cl_size > 1 || p.split != 1 || p.tail_tiles || p.fin_tiles) return GEMM_ERR_UNSUPPORTED;
    p.withhold_armed = 1;
  }

  if (p.device >= 0) {
    if (cudaMalloc(&p.d_status, sizeof(lgt::DeviceStatus)) != cudaSuccess) return GEMM_ERR_CUDA;
    if (cudaMemset(p.d_status, 0, sizeof(lgt::DeviceStatus)) != cudaSuccess) {
      cudaFree(p.d_status);
      return GEMM_ERR_CUDA;
    }
  }
  p.cache = new (std::nothrow) lgt::ArgCache();
  gemm_plan* h = p.cache ? new (std::nothrow) gemm_plan(p) : nullptr;
  if (!h) {
    delete p.cache;
    if (p.d_status) cudaFree(p.d_status);
    return GEMM_ERR_INVALID_ARG;
  }
  *out = h;
  return GEMM_OK;
}

gemm_status_t gemm_workspace_size(const gemm_plan_t* plan, size_t* bytes) {
  if (!plan || !bytes) return GEMM_ERR_INVALID_ARG;
  *bytes = plan->ws_bytes;
  return GEMM_OK;
}

gemm_status_t gemm_query(const gemm_plan_t* plan, gemm_info_t* info) {
  if (!plan || !info) return GEMM_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof(*info));
  info->split_k = plan->split_req;
  info->tile_m = plan->swap ? plan->bn : (lgt::TILE_P << plan->pair);
  info->tile_n = plan->swap ? lgt::TILE_P : plan->bn;
  info->tile_k = kBlockK;
  info->swap_ab = plan->swap;
  info->num_units = plan->num_units;
  // (a stream-K tail's units are single K blocks; the whole tiles take all of K)
  info->k_per_split = static_cast<int32_t>((plan->tail_tiles ? plan->kb_total : plan->kb_per_split) * kBlockK);
  info->streamk_tiles = plan->tail_tiles;
  info->cluster_size = plan->cl_size;
  info->repack_a = plan->repack_a;
  info->repack_b = plan->repack_b;
  info->kernel = plan->kernel == 0 && plan->pair ? 2 : plan->kernel;
  info->dequant_form = plan->kernel == 1 ? plan->int4_form : 0;
  info->realign = plan->rl_ok;
  return GEMM_OK;
}

gemm_status_t gemm_run(gemm_plan_t* plan, const void* A, const void* B, void* C, const void* scales,
                       const void* zeros, void* workspace, size_t workspace_bytes, void* stream_ptr) {
  (void)scales;
  (void)zeros;
  if (!plan) return GEMM_ERR_INVALID_ARG;
  const gemm_desc_t& d = plan->d;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (d.M == 0 || d.N == 0) return GEMM_OK;
  if (!C) return GEMM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(C) % 2) return GEMM_ERR_ALIGNMENT;
  if (plan->device < 0) return GEMM_ERR_CUDA;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != plan->device) return GEMM_ERR_INVALID_ARG;
  if (d.K == 0) {
    return cudaMemset2DAsync(C, plan->ldc * 2, 0, d.N * 2, d.M, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
  }
  if (!A || !B) return GEMM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(A) % 2 || reinterpret_cast<uintptr_t>(B) % 2) return GEMM_ERR_ALIGNMENT;
  const bool int4 = plan->kernel == 1;
  if (int4) {
    // packed weights are read by TMA in place; scales (and zeros) are fp16
    if (reinterpret_cast<uintptr_t>(B) % 16) return GEMM_ERR_ALIGNMENT;
    if (!scales) return GEMM_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(scales) % 2 || reinterpret_cast<uintptr_t>(zeros) % 2) return GEMM_ERR_ALIGNMENT;
  }

  const bool a_mis = !int4 && reinterpret_cast<uintptr_t>(A) % 16 != 0;
  const bool b_mis = !int4 && reinterpret_cast<uintptr_t>(B) % 16 != 0;
  // Operands TMA cannot address: read in place by the kernel's realigning
  // loader when the plan has it and its staging ring fits for this run's
  // set of such operands, else repacked first.
  const bool a_tma = !a_mis && (plan->lda * 2) % 16 == 0, b_tma = !b_mis && (plan->ldb * 2) % 16 == 0;
  bool rl_a = !int4 && plan->rl_ok && !a_tma, rl_b = !int4 && plan->rl_ok && !b_tma;
  if ((rl_a || rl_b) && !lgt::rl_fits(*plan, rl_a, rl_b)) rl_a = rl_b = false;
  const bool pack_a = !int4 && !a_tma && !rl_a;
  const bool pack_b = !int4 && !b_tma && !rl_b;
  // (the plan's own repacks are in ws_bytes; a base pointer that must be
  // repacked at run time needs the larger size)
  const bool pack_mis = (pack_a && !plan->repack_a) || (pack_b && !plan->repack_b);
  const size_t need = pack_mis ? plan->ws_bytes_misaligned : plan->ws_bytes;
  if (need > 0 && (!workspace || workspace_bytes < need)) return GEMM_ERR_WORKSPACE;
  if (need > 0 && reinterpret_cast<uintptr_t>(workspace) % 256) return GEMM_ERR_ALIGNMENT;
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  // Operand addresses and leading dimensions the kernel sees.
  const void* a_eff = A;
  const void* b_eff = B;
  int64_t lda = plan->lda, ldb = plan->ldb;
  size_t next_pack = plan->off_pack_a;  // repacked copies follow the split-K region
  if (pack_a) {
    void* dst = ws + next_pack;
    if (lgt::launch_repack_rows(A, plan->lda * 2, dst, plan->a_pack_ld * 2, plan->a_rows, plan->a_row_elems * 2,
                                stream) != cudaSuccess)
      return GEMM_ERR_CUDA;
    a_eff = dst;
    lda = plan->a_pack_ld;
    next_pack += align_up(static_cast<size_t>(plan->a_rows) * plan->a_pack_ld * 2, 256);
  }
  if (pack_b) {
    void* dst = ws + next_pack;
    if (lgt::launch_repack_rows(B, plan->ldb * 2, dst, plan->b_pack_ld * 2, plan->b_rows, plan->b_row_elems * 2,
                                stream) != cudaSuccess)
      return GEMM_ERR_CUDA;
    b_eff = dst;
    ldb = plan->b_pack_ld;
  }

  const bool split_region = plan->split > 1 && plan->cl_size <= 1;
  float* partial = split_region ? reinterpret_cast<float*>(ws + plan->off_partial) : nullptr;
  int32_t* counters = split_region ? reinterpret_cast<int32_t*>(ws + plan->off_counters) : nullptr;
  if (!int4) {
    const int withhold = plan->withhold_armed ? __atomic_exchange_n(&plan->withhold_armed, 0, __ATOMIC_ACQ_REL) : 0;
    return lgt::launch_dense(plan, a_eff, lda, b_eff, ldb, C, partial, counters, stream, withhold);
  }

  return lgt::run_int4(plan, A, B, C, scales, zeros, ws, partial, counters, stream);
}

gemm_status_t gemm_sync_status(gemm_plan_t* plan, void* stream) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  if (plan->device < 0 || !plan->d_status) return GEMM_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GEMM_ERR_CUDA;
  lgt::DeviceStatus st;
  if (cudaMemcpy(&st, plan->d_status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
  if (st.code != 0) {
    if (cudaMemset(plan->d_status, 0, sizeof(st)) != cudaSuccess) return GEMM_ERR_CUDA;
    return static_cast<gemm_status_t>(st.code);
  }
  return GEMM_OK;
}

gemm_status_t gemm_destroy(gemm_plan_t* plan) {
  if (!plan) return GEMM_OK;
  if (plan->d_status) cudaFree(plan->d_status);
  delete plan->cache;
  lgt::int4_cache_free(plan);
  delete plan;
  return GEMM_OK;
}

}  // extern "C"
