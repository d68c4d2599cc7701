/*
 * attention.h -- C ABI of the fused attention forward (same library as gemm.h).
 *
 *   O[h] = softmax(Q[h] K[h]^T * scale) V[h],   h < heads,
 *
 * Q: heads x seq_q x head_dim, K and V: heads x seq_k x head_dim, O: heads x
 * seq_q x head_dim, all stored [head][row][head_dim] contiguous, fp16 or
 * bf16 (one type for all four), fp32 accumulation, the softmax in fp32, the
 * probabilities rounded to the input type for the second product, O written
 * once.  Non-causal.
 *
 * This is the setting of the Triton inThreadTranspose page ("Introduction"):
 * the second dot of Flash Attention, P.V, whose V operand is contiguous along
 * the output dimension (head_dim), not along the reduction dimension (the
 * keys) -- a non-TN dot.  Here V's tiles are read by TMA as they are stored
 * and handed to the tensor core as an MN-major operand (128-byte swizzle), so
 * no transpose is made; P never leaves the SM (tensor memory).
 *
 * Errors are status codes (gemm_status_t); nothing aborts or prints.
 */
#ifndef LGT_ATTENTION_H
#define LGT_ATTENTION_H

#include <stddef.h>
#include <stdint.h>

#include "gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct attn_desc {
  int32_t heads;     /* >= 1 (at most 65535) */
  int32_t seq_q;     /* >= 1 */
  int32_t seq_k;     /* >= 1 */
  int32_t head_dim;  /* 64 or 128 */
  int32_t dtype;     /* GEMM_F16 or GEMM_BF16, for Q, K, V and O */
  float scale;       /* > 0; 0 = 1 / sqrt(head_dim) */
} attn_desc_t;

typedef struct attn_plan attn_plan_t;

/* Validate `desc` and make a plan (host state and a 16-byte device status
 * word on the current device).  GEMM_ERR_INVALID_ARG for a shape or type
 * outside the above, GEMM_ERR_CUDA when no device is usable. */
gemm_status_t attn_create(const attn_desc_t* desc, attn_plan_t** plan);

/* Enqueue the forward pass on `stream` (a cudaStream_t; NULL = legacy default
 * stream).  Q, K, V, O: device pointers, 16-byte aligned, caller-owned; O
 * must not overlap the inputs.  One CTA per 128 queries of a head walks that
 * head's keys in blocks of 128.  GEMM_ERR_INVALID_ARG (NULL pointer),
 * GEMM_ERR_ALIGNMENT, GEMM_ERR_CUDA (launch failure).  A kernel whose
 * bounded wait ran out records GEMM_ERR_TIMEOUT in the plan's status word
 * (attn_sync_status); O is then invalid. */
gemm_status_t attn_run(attn_plan_t* plan, const void* Q, const void* K, const void* V, void* O, void* stream);

/* Synchronise `stream`, read and clear the plan's status word: GEMM_OK or
 * GEMM_ERR_TIMEOUT. */
gemm_status_t attn_sync_status(attn_plan_t* plan, void* stream);

gemm_status_t attn_destroy(attn_plan_t* plan);

#ifdef __cplusplus
}
#endif

#endif /* LGT_ATTENTION_H */
