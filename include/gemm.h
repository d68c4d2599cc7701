/*
 * gemm.h -- C ABI of the any-layout half-precision GEMM for GB300 (sm_103a).
 *
 *   C = A . B,  A logically M x K, B logically K x N, C row-major M x N,
 *   products accumulated in fp32, C written once (round to nearest even).
 *
 * Operand layouts.  The two storage orders of each operand are the cases the
 * Triton inThreadTranspose page ("[AMD] inThreadTranspose ...", "Feature
 * description" and "PR description") distinguishes: a dot operand that is
 * contiguous along K, and a "non-KContig" one that is contiguous along M
 * (for A) or N (for B).
 *   A, GEMM_K_CONTIG : row-major M x K, element (m,k) at A[m*lda + k]
 *   A, GEMM_MN_CONTIG: column-major M x K, element (m,k) at A[k*lda + m]
 *   B, GEMM_K_CONTIG : stored N x K row-major, element (k,n) at B[n*ldb + k]
 *   B, GEMM_MN_CONTIG: stored K x N row-major, element (k,n) at B[k*ldb + n]
 *   C                : element (m,n) at C[m*ldc + n]
 * Leading dimensions are in elements; 0 means dense (K, M, K, N, N).
 *
 * Split-K.  split_k = 0 selects the SM-waste rule of the BitBLAS TileLang
 * page ("SplitK Infer for dequantize cases"), evaluated on the 128 x 128 x 64
 * tile and a 0.05 threshold; split z covers k in [z*Ks, min(K,(z+1)*Ks)) with
 * Ks = ceil(K / (split_k*64)) * 64, following the page's per-split K offset
 * in its T.Parallel / T.copy example.  Partial sums are reduced across CTAs
 * in fp32 (the reduction-across-workers pattern of the IREE page,
 * "[LLVMGPUVectorDistribute] Add support for inter-subgroup multi_reduction").
 *
 * int4 weights (b_dtype = GEMM_INT4).  B is N rows of K/2 bytes, code q(n,k)
 * in the low nibble of byte k/2 for even k and the high nibble for odd k;
 * w(k,n) = (q(n,k) - z(n,k/g)) * s(n,k/g) with g = group_size and fp16
 * scales / zeros stored [N, K/g] row-major (zeros NULL means z = 8).  The
 * weight is dequantised inside the GEMM mainloop (BitBLAS TileLang page,
 * "Relevant Issues": dequantize layout transformations).  A must be fp16.
 *
 * Errors: every entry point returns a status code; nothing aborts or prints.
 * All pointers passed to gemm_run are device pointers owned by the caller.
 */
#ifndef LGT_GEMM_H
#define LGT_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = 1, /* bad shape, enum, leading dimension or NULL pointer */
  GEMM_ERR_UNSUPPORTED = 2, /* valid request this library does not implement */
  GEMM_ERR_ALIGNMENT = 3,   /* an operand pointer is not aligned to its element size */
  GEMM_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than gemm_workspace_size */
  GEMM_ERR_CUDA = 5,        /* a CUDA runtime / driver call failed, or no device */
  GEMM_ERR_TIMEOUT = 6      /* a kernel gave up waiting (bounded waits); output invalid */
} gemm_status_t;

typedef enum { GEMM_K_CONTIG = 0, GEMM_MN_CONTIG = 1 } gemm_layout_t;

typedef enum { GEMM_F16 = 0, GEMM_BF16 = 1, GEMM_INT4 = 2, GEMM_F32 = 3 } gemm_dtype_t;

/* Problem description.  Enum-valued fields are int32_t so the struct has the
 * same layout from every language. */
typedef struct {
  int64_t M, N, K;
  int32_t a_layout, b_layout; /* gemm_layout_t; int4 B must be GEMM_K_CONTIG */
  int64_t lda, ldb, ldc;      /* elements (bytes for int4 B: ldb = K/2 or 0); 0 = dense */
  int32_t a_dtype, b_dtype, c_dtype; /* F16 / BF16 (A and B alike), or B = INT4 with A = F16; C = F16 / BF16 */
  int32_t split_k;            /* 0 = SM-waste rule; >= 1 explicit factor */
  int32_t group_size;         /* int4 quantisation group along K (0 = 128); must divide K and the split length */
  int32_t num_sms;            /* SM count the split-K rule uses: 0 = the current device's */
  int32_t flags;              /* GEMM_FLAG_* bits (below); 0 for none */
} gemm_desc_t;

/* Bitwise-reproducible results.  No stream-K tail (below); with a split-K
 * factor above 1 each run of consecutive splits stores its fp32 partial sum
 * into a slot of its own (no atomics) and the tile's slots are added in a
 * fixed order before the conversion.  The workspace then holds the slots
 * instead of an M x N region.  gemm_run_static_scratch does not support
 * this mode with a split factor above 1 (GEMM_ERR_UNSUPPORTED). */
#define GEMM_FLAG_DETERMINISTIC 1

/* int4 weights pre-packed by gemm_int4_prepack: gemm_run's B is the packed
 * buffer (scales and zeros are still passed in their plain [N][groups]
 * layout: the zero-point term reads them).  Needs b_dtype = GEMM_INT4, a
 * group size of 64 or 128 or a multiple of 256, and split ranges of whole
 * 256-deep stages: with split_k = 0 the planner rounds the SM-waste rule's
 * ranges up to whole stages; a caller's split_k whose ranges
 * (ceil(ceil(K / 64) / split_k) K blocks) are not a multiple of 4 blocks, or
 * any other shape outside these, gets GEMM_ERR_UNSUPPORTED from gemm_create.  Plans with this flag
 * use the fp16 form; the results are the same bits as with the plain layout. */
#define GEMM_FLAG_INT4_PREPACKED 4

/* Test aid for the failure path (not for production use).  The plan's first
 * gemm_run withholds the first pipeline stage of one CTA: no copy is issued
 * for it, so the MMA issuer's bounded wait on it runs out, the kernel records
 * GEMM_ERR_TIMEOUT (read by gemm_sync_status) and that CTA's tile of C is
 * left unwritten; every later run of the plan is normal.  Every copy that was
 * issued still lands before the CTA exits.  Accepted only where the plan uses
 * the single-CTA tensor-core kernel with whole tiles (no split-K, no stream-K
 * tail, no cluster, no CTA pair; gemm_create returns GEMM_ERR_UNSUPPORTED
 * otherwise), so that no other CTA waits on the withheld one.  The wait limit
 * is the plan's (LGT_GEMM_WAIT_LIMIT_MS at gemm_create, 2 s by default). */
#define GEMM_FLAG_TEST_WITHHOLD_STAGE (1 << 30)

/* What a plan decided. */
typedef struct {
  int32_t split_k;     /* factor in use */
  int32_t tile_m, tile_n, tile_k; /* output tile of one work unit (M x N x K) */
  int32_t swap_ab;     /* 1: the MMA runs C^T = B^T A^T (skinny M) */
  int32_t num_units;   /* (tile, split) work units */
  int32_t k_per_split; /* Ks in elements */
  int32_t repack_a, repack_b; /* operand copied into the workspace first by a pre-pass (a stride TMA cannot
                                 express, where the kernel's realigning loader is not available) */
  int32_t kernel;      /* 0 = tensor-core any-layout, 1 = int4 dequant,
                          2 = tensor-core any-layout on CTA pairs (256 x 256 tiles) */
  int32_t streamk_tiles; /* tiles of the stream-K tail (0 = none), see gemm_create */
  int32_t cluster_size;  /* > 1: each tile's split-K runs are the CTAs of one cluster of this size and
                            their fp32 partials are added in shared memory (0 = split-K through the workspace) */
  int32_t dequant_form;  /* int4 weights: 1 = fp16 form (each weight expanded to fp16 q*s, the zero point
                            through the activation's group sums), 2 = e4m3 form (codes as exact e4m3 values,
                            the activation split into three e4m3 terms per 128-deep block, scales, zero
                            points and activation scales applied in fp32 after the MMA: activations of at
                            most 16 rows, K-contiguous, K and group_size multiples of 128); 0 otherwise */
  int32_t realign;       /* 1: operands TMA cannot address (a leading dimension that is not a multiple of
                            8 elements, or an A / B pointer not 16-byte aligned at gemm_run) are loaded by
                            the kernel's realigning loader warps, which read them in place; 0: such
                            operands are repacked by a pre-pass into the workspace (the default).
                            LGT_GEMM_REALIGN=1 at gemm_create selects the loader where it applies: not
                            for plans whose tensor-core CTAs convert split tiles at the end (split-K
                            through the workspace, stream-K tails), tiny shapes (M, N or K below 8) or
                            plans whose staging does not fit beside two pipeline stages.  The loader copies the rows of each row class (rows
                            whose starts share their offset within a 16-byte word: the perpDim
                            permutation of the rows with stride 16 / gcd(pitch, 16)) with TMA into a
                            staging ring and realigns them in shared memory. */
} gemm_info_t;

typedef struct gemm_plan gemm_plan_t;

/* Validate `desc`, choose tiles and the split factor, and return a plan.
 *
 * Stream-K tail.  With split factor 1 (given, or from the rule) the tiles
 * are dealt to the persistent CTAs in whole waves; when the last wave would
 * leave at least a quarter of the CTAs idle, the K blocks of its tiles are
 * spread evenly over all CTAs instead and their fp32 partial sums reduced as
 * split-K partials are (so those tiles' rounding order depends on timing).
 * The workspace then holds an M x N fp32 region.  GEMM_FLAG_DETERMINISTIC
 * turns it off; gemm_info_t.streamk_tiles reports it.
 *
 * Split-K in a cluster.  For a skinny problem (M <= 64, run as C^T) with a
 * split factor above 1 whose tiles are few, when c CTAs per tile (c in 8, 4,
 * 2, dividing the factor) still cover at least 3/4 of the SMs and the
 * device can hold the clusters at once, each tile's K range is split over
 * the c CTAs of one cluster and their fp32 partials are added in shared
 * memory, in a fixed order (results are then reproducible run to run); the
 * workspace then holds no split-K region (gemm_workspace_size is 0 unless an
 * operand is repacked).  gemm_info_t.cluster_size reports it.  Chosen only
 * with a device (num_sms given and no device: never).
 *
 * Needs a CUDA device only when desc->num_sms == 0 (to count its SMs); the
 * plan's kernels run on the device current at gemm_create.  The plan is
 * immutable and may be used from several streams, each with its own
 * workspace.  *out is NULL on error. */
gemm_status_t gemm_create(const gemm_desc_t* desc, gemm_plan_t** out);

/* Bytes of device workspace gemm_run needs (0 if none).  The workspace holds
 * the fp32 split-K partial sums and per-tile arrival counters, and repacked
 * operand copies.  It must be zero-filled before its first use; every
 * successful gemm_run leaves it zero-filled again (a run that returns or
 * records GEMM_ERR_TIMEOUT does not). */
gemm_status_t gemm_workspace_size(const gemm_plan_t* plan, size_t* bytes);

gemm_status_t gemm_query(const gemm_plan_t* plan, gemm_info_t* info);

/* Enqueue C = A.B on `stream` (a cudaStream_t; NULL = legacy default stream).
 * A, B, C: device pointers in the plan's layouts; A and B are read only, C is
 * written only.  scales / zeros: int4 only (zeros may be NULL).  The call is
 * asynchronous; errors found on the host are returned at once, a device-side
 * timeout is reported by gemm_sync_status.  Concurrent runs of one plan must
 * use distinct workspaces. */
gemm_status_t gemm_run(gemm_plan_t* plan, const void* A, const void* B, void* C, const void* scales,
                       const void* zeros, void* workspace, size_t workspace_bytes, void* stream);

/* Run a plan without any caller-provided device memory.  (No counterpart on
 * the source pages: this is an interface addition of this library.)
 *
 * For callers that cannot allocate device memory when they run the GEMM --
 * e.g. an inference-engine plugin whose enqueue call must not allocate, a
 * serving loop that cannot afford a cudaMalloc / cudaFree stall, or code that
 * runs after another allocator has reserved all free device memory -- and so
 * cannot hand gemm_run a workspace.  The split-K partial sums and tile
 * counters then live in a fixed 8 MiB array in the library's own device
 * memory, held on every GPU that loads the library until the process exits.
 *
 * - Nothing is allocated by this call (no cudaMalloc / cudaFree); the plan
 *   itself is made beforehand with gemm_create.
 * - The first call on a device resolves the array's address on that device
 *   (cudaGetSymbolAddress), so make that first call before any stream
 *   capture.  The plan's device must be current.
 * - Plans whose split-K region (M*N*4 bytes plus the tile counters) exceeds
 *   8 MiB are rejected with GEMM_ERR_WORKSPACE.  Plans that need a realigned
 *   operand copy (a leading dimension that is not a multiple of 16 bytes) or
 *   operands not 16-byte aligned are rejected with GEMM_ERR_UNSUPPORTED.
 * - All calls on a device share the array; each call clears the part it uses
 *   (cudaMemsetAsync on `stream`) before its kernel.  Calls whose work
 *   overlaps on the GPU (different streams, no ordering between them) race
 *   on the array and give wrong results.
 * - A device-side timeout is reported by gemm_sync_status, as for gemm_run. */
gemm_status_t gemm_run_static_scratch(const gemm_plan_t* plan, const void* A, const void* B, void* C, void* stream);

/* Wait for `stream`, then read and clear the plan's device status word:
 * GEMM_OK, or GEMM_ERR_TIMEOUT if a kernel of this plan gave up a wait. */
gemm_status_t gemm_sync_status(gemm_plan_t* plan, void* stream);

gemm_status_t gemm_destroy(gemm_plan_t* plan);

/* The split-K rule on its own (host computation, no device needed). */
int32_t gemm_splitk_auto(int64_t M, int64_t N, int64_t K, int32_t block_m, int32_t block_n, int32_t block_k,
                         int32_t num_sms, double threshold);

/* Perpendicular-dimension stride permutation of the hipBLASLt DTL page ("Add
 * support for permuting perpDim"), over `count` indices in blocks of `block`
 * with stride `stride` (must divide `block`; a trailing partial block and an
 * invalid stride map indices to themselves).  Host computation. */
uint32_t gemm_perm_fwd(uint32_t index, uint32_t count, uint32_t block, uint32_t stride);
uint32_t gemm_perm_inv(uint32_t index, uint32_t count, uint32_t block, uint32_t stride);

/* Offline pre-pack of int4 weights for GEMM_FLAG_INT4_PREPACKED (the BitBLAS
 * page's "Relevant Issues": a ladder-based basic layout, so that the
 * dequantising producer's accesses are whole vectors without bank
 * conflicts; here the layout is the kernel's stage).  For each 128-row tile t
 * and 256-deep stage s (S = ceil(K / 256) stages), a block of
 * gemm_int4_prepack_bytes(N, K, group) / (ceil(N / 128) * S) bytes at block
 * index t * S + s: the tile's 128 rows x 128 bytes of codes of the stage, row
 * r at r * 128, its 16-byte chunk c (codes 32c .. 32c + 31 of the stage) at
 * chunk c ^ (r mod 8) (the 128-byte swizzle), then the stage's scales as slots
 * of 128 fp16 (row r at 2r): one slot per group for groups of 64 or 128, one
 * for groups of 256 or more.  Rows past N and codes past K are zero.
 *   B: N rows of ldb bytes (ldb = 0: K / 2), codes as for gemm_run; device,
 *      16-byte aligned, ldb a multiple of 16.  scales: fp16 [N][K / group].
 *   out: device, 16-byte aligned, gemm_int4_prepack_bytes bytes, caller-owned.
 * gemm_int4_prepack_bytes returns 0 for shapes it does not take (K a multiple
 * of 64 and of the group, group 64, 128 or a multiple of 256). */
size_t gemm_int4_prepack_bytes(int64_t N, int64_t K, int32_t group_size);
gemm_status_t gemm_int4_prepack(const void* B, int64_t ldb, const void* scales, int64_t N, int64_t K,
                                int32_t group_size, void* out, void* stream);

/* The same permutation computed on the device by the routine the kernels'
 * loaders use: out[j] = gemm_perm_fwd(in[j], count, block, stride) (inverse
 * == 0) or gemm_perm_inv(...) (inverse != 0) for j < n.  `in` and `out` are
 * device arrays of n uint32 owned by the caller (they may be the same array);
 * the call is asynchronous on `stream` (a cudaStream_t).  Returns
 * GEMM_ERR_INVALID_ARG for a NULL array with n > 0, GEMM_ERR_CUDA if the
 * launch fails.  Same rules as the host functions: `stride` must divide
 * `block`, a trailing partial block and an invalid stride map to themselves. */
gemm_status_t gemm_perm_device(const uint32_t* in, size_t n, uint32_t count, uint32_t block, uint32_t stride,
                               int32_t inverse, uint32_t* out, void* stream);

/* Magic-number division by a divisor fixed in advance (hipBLASLt DTL page,
 * "Add support for generalized NLC=1": static divisors use a magic multiply).
 * gemm_magic_divmod_host runs the kernels' own quotient routine on the host
 * over `count` dividends (< 2^31); gemm_magic_divmod_device runs it on the
 * device over device arrays on `stream`.  divisor must be >= 1. */
gemm_status_t gemm_magic_divmod_host(const uint32_t* n, size_t count, uint32_t divisor, uint32_t* q, uint32_t* r);
gemm_status_t gemm_magic_divmod_device(const uint32_t* n, size_t count, uint32_t divisor, uint32_t* q, uint32_t* r,
                                       void* stream);

const char* gemm_status_string(gemm_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* LGT_GEMM_H */
