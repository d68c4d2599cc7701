// Host-side plan of the GEMM (the object behind gemm_plan_t) and helpers
// shared by the C-ABI translation units.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <cstdint>

#include "gemm.h"
#include "kernels.h"

namespace lgt {
struct ArgCache;
struct Int4Cache;
}

struct gemm_plan {
  gemm_desc_t d;
  int device;        // device current at create time, -1 if none was queried
  int sms_rule;      // SM count fed to the split-K rule
  int sms_grid;      // persistent grid size (device SMs), 0 without a device
  int kernel;        // 0: tensor-core any-layout, 1: int4 dequant
  int group;         // int4 quantisation group along K
  int swap;
  int bn;
  int pair;          // 1: CTA-pair kernel (256 x 256 tiles, clusters of two CTAs)
  int grid;          // CTAs launched by the tensor-core kernels
  int num_counters;  // split-K arrival counters (one per tile, per half-tile for pairs)
  int split, kb_per_split, kb_total;  // split: units per tile in the kernel's unit space
  int split_req;     // split-K factor of the SM-waste rule or of the caller
  int rr_tiles;      // tiles dealt whole before the contiguous unit ranges
  int tail_tiles;    // stream-K tail: tiles whose K blocks are spread over all workers
  int fin_tiles;     // split tiles converted by the fixup warps of all CTAs (the tail, or all tiles when split > 1)
  int cl_size;       // > 1: each tile's split-K runs are one cluster of this many CTAs, reduced on chip
  int det;           // deterministic split-K: per-run partial slots summed in run order
  int max_runs;      // slots per strip (det)
  int tiles_p, tiles_q, num_units;
  int64_t lda, ldb, ldc;
  int a_mn, b_mn;
  // operand repacking (leading dimension not a multiple of 16 bytes)
  int repack_a, repack_b;
  // Operands TMA cannot address (unaligned row pitch, or an unaligned base at
  // run time) are realigned by the kernel's loader warps when the plan leaves
  // them free (no fixup work); else they are repacked by a pre-pass.
  int rl_ok;
  int64_t a_rows, a_row_elems, b_rows, b_row_elems;  // storage rows of each operand
  int64_t a_pack_ld, b_pack_ld;
  size_t off_partial, off_counters, off_pack_a, off_pack_b, ws_bytes;
  size_t ws_bytes_misaligned;
  int int4_form;      // int4: 1 = fp16 form, 2 = e4m3 form (gemm_info_t.dequant_form)
  size_t off_aprep;  // int4: the prepared activation
  size_t off_agsum;  // int4: activation sums (fp16 form: [groups][M]; e4m3 form: [K / 128][16]), fp32
  size_t off_inv;    // int4, e4m3 form: 1 / S_b per 128-deep block and row, fp32 [K / 128][16]
  lgt::DeviceStatus* d_status;
  uint64_t wait_limit_ns;
  int withhold_armed;  // GEMM_FLAG_TEST_WITHHOLD_STAGE: the next run withholds a stage (one shot)
  lgt::ArgCache* cache;  // launch arguments of the last run (owned; null in copies made by plan_without_tail)
  lgt::Int4Cache* cache4;  // the same for the int4 kernels (owned; made on first use)
};


namespace lgt {

// The dense kernels' launch arguments of a plan's last run, keyed by what
// the tensor maps and pointers depend on, so that a run with the same
// buffers as the one before it encodes no tensor map (an encode costs about
// a microsecond of host time).  A plan may be used from several threads: a
// run that finds the cache busy encodes its own arguments.
struct ArgCache {
  int busy;  // 0 / 1, taken with an atomic exchange
  int valid;
  const void* A;
  const void* B;
  void* C;
  float* partial;
  int32_t* counters;
  int64_t lda, ldb;
  TcArgs args;
};

// cuTensorMapEncodeTiled (see api.cu); null if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 get_encoder();
// Whether the realigning loader's staging fits the plan's kernel when A
// (rl_a) and / or B (rl_b) go through it.
bool rl_fits(const gemm_plan& p, bool rl_a, bool rl_b);

// Encode a 2-D TMA map over a 16-bit operand (see api.cu).
bool encode_operand(CUtensorMap* map, const void* ptr, int dtype, bool mn_major, int64_t rows_or_mn, int64_t K,
                    int64_t ld, int box_rows);

// int4 plans (api_int4.cu): choose the form and lay out the prepared
// activation and its tables after the split-K region at `off`; run a plan;
// free its argument cache.
void int4_plan(gemm_plan& p, size_t off);
gemm_status_t run_int4(gemm_plan* plan, const void* A, const void* B, void* C, const void* scales, const void* zeros,
                       uint8_t* ws, float* partial, int32_t* counters, cudaStream_t stream);
void int4_cache_free(gemm_plan* plan);

// Launch the dense tensor-core kernel of `plan` on operands TMA can address
// in place (16-byte aligned bases and pitches `lda` / `ldb` in elements),
// with the split-K partial sums and counters at `partial` / `counters`
// (zero-filled; unused when split == 1).
// A copy of `p` that runs every tile whole (no stream-K tail).
gemm_plan plan_without_tail(const gemm_plan& p);

// withhold: the test aid of GEMM_FLAG_TEST_WITHHOLD_STAGE for this run.
gemm_status_t launch_dense(const gemm_plan* plan, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                           float* partial, int32_t* counters, cudaStream_t stream, int withhold = 0);

}  // namespace lgt
