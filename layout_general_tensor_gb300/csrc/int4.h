// int4-weight GEMM: argument block and launchers shared between the C ABI
// (api_int4.cu) and the int4 kernels (gemm_int4.cu, gemm_int4_f8.cu).
#pragma once
#include "kernels.h"

namespace lgt {

// int4-weight GEMM (always swapped: P = the weight rows n, Q = the activation
// rows m).  `t` carries the scheduler, the map over the prepared activation
// (tm_q) and the epilogue fields; tm_p is unused.
struct Int4Args {
  TcArgs t;
  CUtensorMap tm_w;          // packed weight bytes: dims {ldb bytes, N}, box {128, 128}, 128-byte swizzle
  // fp16 form: per-group sums of the activation, fp32 [groups][M];
  // e4m3 form: per-128-block sums, fp32 [K / 128][16]
  const float* agsum;
  const float* inv_scale;    // e4m3 form: 1 / S_b of each 128-deep block and row, fp32 [K / 128][16]
  const uint16_t* scales;    // fp16 [N][groups]
  const uint16_t* zeros;     // fp16 [N][groups], or null for z = 8
  int32_t groups;
  MagicDiv div_kb_per_group; // 64-deep K block -> quantisation group
  int32_t x_box_kb;          // fp16 form: K blocks per activation box (min(4, K / 64)); t.tm_q is 3-D {64, M, K / 64}
  int32_t vec_sz;            // fp16 form: scale / zero rows readable 8 groups (16 bytes) at a time
  // fp16 form with pre-packed weights (gemm_int4_prepack): one block per
  // 128-row tile and 256-deep stage, [tile][stage]; null: the plain layout
  const uint8_t* wpre;
  int32_t pre_block;         // bytes of a block (codes + scale slots)
  int32_t pre_stages;        // blocks per tile (ceil(K / 256))
  int32_t pre_kbpg;          // 64-deep K blocks per group (scale slot of K block j: j / kbpg, 0 when >= 4)
};

// Pre-packed int4 weights (the fp16 form's offline layout).  For each
// 128-row tile t and 256-deep stage s, a block at (t * S + s) * block bytes:
// the 128 rows x 128 bytes of codes, row r at r * 128, its 16-byte chunk c
// (codes 32 c .. 32 c + 31 of the stage) at chunk c ^ (r mod 8) -- where a
// 128-byte-swizzled TMA box of the plain layout puts them -- then the
// stage's scale slots, 128 fp16 each (row r at 2 r): one per group for groups
// of 64 or 128 (4 or 2 slots), one for groups of 256 or more.  Rows past N
// and K past K are zero.
int pre_slots(int group);
size_t pre_block_bytes(int group);
size_t pre_total_bytes(int64_t N, int64_t K, int group);
cudaError_t launch_int4_prepack(const void* B, int64_t ldb, const void* scales, int64_t N, int64_t K, int group,
                                void* out, cudaStream_t stream);

// ---- fp16 form (any M <= 64, any activation layout, any group multiple of 64)

cudaError_t launch_int4_gemm(const Int4Args& args, int bn, int grid, cudaStream_t stream);

// Activation pre-pass of the fp16 form: copy of A (M x K, any layout,
// 2-byte aligned) into Ap, K-block-major: the 64 elements of row m in K block
// kb at Ap + (kb * M + m) * 64, each 8-element group of K reordered to
// (0,4,1,5,2,6,3,7); and agsum[g * M + m] = the fp32 sum (fixed order) of row
// m's elements in group g (group elements of K).  K and group must be
// multiples of 64.
cudaError_t launch_int4_prep(const void* A, int64_t lda, int a_mn, int M, int K, int group, void* Ap, float* agsum,
                             int sms, cudaStream_t stream);

// ---- e4m3 form (M <= 16, K-contiguous activation, K and group multiples of 128)

bool int4f8_supported(int a_mn, int64_t M, int64_t K, int group);
// Bytes of the e4m3 form's prepared activation (three terms of 16 rows per 128-deep block).
size_t int4f8_prep_bytes(int64_t K);
// Pre-pass: the three e4m3 terms of A (K-contiguous, lda elements per row) in
// the layout the kernel's activation map reads, Xp[K / 128][48][128], and per
// block and row 1 / S_b (inv_scale) and the block sum (agsum), fp32 [K / 128][16].
cudaError_t launch_int4f8_prep(const void* A, int64_t lda, int M, int K, void* Xp, float* inv_scale, float* agsum,
                               int sms, cudaStream_t stream);
// The GEMM: args.t.tm_q is the 3-D map {128 bytes, 48, K / 128} over Xp, box
// {128, 48, 1}; args.t.idesc the kind::f8f6f4 descriptor (e4m3 x e4m3, M 128, N 48).
cudaError_t launch_int4f8_gemm(const Int4Args& args, int grid, cudaStream_t stream);

}  // namespace lgt
