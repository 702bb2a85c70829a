/*
 * moe_mx.h -- C ABI of the MX-quantised routed-expert forward: MXFP8 tokens
 * with MXFP8 weights (A8W8-FP) or MXFP4 weights (A8W4-FP), and MXFP4 tokens
 * with MXFP4 weights (A4W4-FP).
 *
 * What the calls compute ("MegaMoE", ops-transformer operator doc):
 *  - "A8W8-FP 量化场景", stage 1: the tokens gathered per expert are quantised
 *    with Q_MX: groups of 32 consecutive elements along the row share one
 *    FLOAT8_E8M0 scale (an exponent), the elements are FLOAT8_E4M3FN or
 *    FLOAT8_E5M2 (moe_permute_mx, moe_mx_quantize);
 *  - stage 2: G_e = DQ(X_e) DQ(W1_e^G), U_e = DQ(X_e) DQ(W1_e^U), gate = the
 *    first N/2 output channels of weight1, up = the last N/2;
 *    A_e = Activation(G_e, U_e), then Q_MX(A_e) in the same element type as
 *    stage 1 (gmm_forward_mx with an activation);
 *  - stage 3: O_e = DQ(A_e) DQ(W2_e), bf16 (gmm_forward_mx, no activation);
 *  - stage 4: Y[i] = sum_k W[i, k] O[pi(i, k)] (the A16W16 combine,
 *    moe_unpermute).  moe_layer_forward_mx runs the four stages.
 *  - "A8W4-FP 量化场景": the same stages with FLOAT4_E2M1 weights for both
 *    matmuls (w_format MOE_FP4_E2M1) and E4M3 tokens and activations.
 *  - "A4W4-FP 量化场景": the tokens are quantised to FLOAT4_E2M1 too
 *    (x_format MOE_FP4_E2M1), and the activation to FLOAT8_E4M3FN, so the
 *    second matmul is A8W4.  In general the activation takes the tokens' fp8
 *    type, or E4M3 after E2M1 tokens; any pairing of token and weight types
 *    is accepted.
 *  - "约束说明", MXFP: weight1 is (E, 2I, H) and weight2 (E, H, I): each
 *    output channel is a row of K contiguous elements; weightScales1 is
 *    (E, 2I, ceil(H/64), 2) and weightScales2 (E, H, ceil(I/64), 2), i.e. one
 *    E8M0 code per 32 elements of K, row-major; the scales of x are
 *    (rows, ceil(H/32)).
 *
 * Quantisation rule (the pages say "extract a shared exponent"; this is the
 * usual MX rule): for a group with largest magnitude amax, the scale is
 * X = 2^(floor(log2 amax) - emax), emax = 8 for E4M3, 15 for E5M2 and 2 for
 * E2M1, never below 2^-127 (amax = 0 gives code 0); a group holding an
 * infinity or NaN gets scale code 0xFF (E2M1, which has no NaN, then codes
 * every element 7).  Each element is x / X rounded to nearest even,
 * saturating at +-448 (E4M3), +-57344 (E5M2) or +-6 (E2M1).  The gate / up products are
 * rounded to bf16 before the activation; the activation is quantised from
 * fp32.
 *
 * Layouts: every fp8 tensor is row-major uint8 codes, every E2M1 tensor
 * row-major packed codes (K/2 bytes a row); every scale tensor is row-major
 * uint8 E8M0 codes with K/32 per row.  K of both matmuls (H, I)
 * must be a multiple of 128 and N a multiple of 128 (2I a multiple of 256
 * with an activation); pointers 16-byte aligned.  Errors and workspaces as in
 * moe_gmm.h (status block first, zeroed once by moe_workspace_init).
 */
#ifndef MOE_MX_H
#define MOE_MX_H

#include "moe_gmm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Element formats: FLOAT8_E4M3FN, FLOAT8_E5M2 and FLOAT4_E2M1 ("MegaMoE",
 * A8W4-FP and A4W4-FP 量化场景).  E2M1 codes are packed two per byte, element
 * 2i in the low nibble: an E2M1 w_q is [E, N, K/2] bytes, an E2M1 x_q
 * [M, K/2]; an E2M1 operand of gmm_forward_mx is 32-byte aligned. */
typedef enum { MOE_FP8_E4M3 = 0, MOE_FP8_E5M2 = 1, MOE_FP4_E2M1 = 5 } moe_fp8_format_t;

/* Workspace bytes for moe_mx_quantize (the status block only). */
MOE_API size_t moe_mx_quantize_workspace_size(void);

/* Q_MX of each row of x [rows, K] (K a multiple of 32):
 *   q [rows, K] fp8 codes ([rows, K/2] packed E2M1), scales [rows, K/32] E8M0
 *   codes. */
MOE_API moe_status_t moe_mx_quantize(const moe_bf16* x, int64_t rows, int64_t K, int32_t format,
                                     uint8_t* q, uint8_t* scales, void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_permute (moe_gmm.h) whose gathered rows leave quantised (stage 1):
 *   x_q [T*k, H] fp8 ([T*k, H/2] packed E2M1) and x_scales [T*k, H/32]
 *   instead of bf16 x_perm, in the same row order; group_list, row_id_map
 *   and sorted_flat as moe_permute.
 *   H a multiple of 32; workspace moe_permute_workspace_size. */
MOE_API moe_status_t moe_permute_mx(const moe_bf16* x, const int32_t* topk_ids, int64_t T, int64_t H, int64_t k,
                                    int64_t E, int32_t format, uint8_t* x_q, uint8_t* x_scales,
                                    int64_t* group_list, int32_t* row_id_map, int32_t* sorted_flat,
                                    void* ws, size_t ws_bytes, moe_stream_t stream);

/* Workspace bytes for gmm_forward_mx. */
MOE_API size_t gmm_mx_workspace_size(int64_t M, int64_t K, int64_t N, int64_t E);

/* Block-scaled grouped matmul per expert e with rows [off_e, off_e + group_list[e]):
 *   P = DQ(x_q, x_scales)[rows] @ DQ(w_q[e], w_scales[e])^T
 *   x_q [M, K] fp8 or [M, K/2] packed E2M1 (x_format), x_scales [M, K/32];
 *   w_q [E, N, K] fp8 or [E, N, K/2] packed E2M1 (w_format),
 *   w_scales [E, N, K/32]; group_list [E] int64 counts summing to M.
 *   activation NULL: y [M, N] bf16 = P.
 *   activation given (N = 2I): H = bf16(P), A = activation(H[:, :I], H[:, I:]),
 *     a_q [M, I] fp8 (x_format, or E4M3 when x_format is E2M1) and
 *     a_scales [M, I/32] = Q_MX(A); h_save [M, N] bf16 receives H when not
 *     NULL (y unused).
 *   A bad group_list sets MOE_ERR_DEVICE in the status word. */
MOE_API moe_status_t gmm_forward_mx(const uint8_t* x_q, const uint8_t* x_scales, const uint8_t* w_q,
                                    const uint8_t* w_scales, const int64_t* group_list,
                                    int64_t M, int64_t K, int64_t N, int64_t E, int32_t x_format, int32_t w_format,
                                    const moe_activation_t* activation, moe_bf16* y, uint8_t* a_q, uint8_t* a_scales,
                                    moe_bf16* h_save, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Workspace bytes for moe_layer_forward_mx. */
MOE_API size_t moe_layer_mx_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k);

/* The A8W8-FP / A8W4-FP / A4W4-FP layer forward (x_format and w_format as
 * gmm_forward_mx takes them, E2M1 weights packed): moe_permute_mx (x_format)
 * -> gmm_forward_mx with the activation (w1_q [E, 2I, H],
 * w1_scales [E, 2I, H/32]) -> gmm_forward_mx
 * (w2_q [E, H, I], w2_scales [E, H, I/32]) -> combine with topk_w into
 * y [T, H] bf16.  Intermediates live in ws (32-byte aligned with E2M1
 * tokens). */
MOE_API moe_status_t moe_layer_forward_mx(const moe_bf16* x, const int32_t* topk_ids, const float* topk_w,
                                          const uint8_t* w1_q, const uint8_t* w1_scales, const uint8_t* w2_q,
                                          const uint8_t* w2_scales, int64_t T, int64_t H, int64_t I, int64_t E,
                                          int64_t k, int32_t x_format, int32_t w_format,
                                          const moe_activation_t* activation, moe_bf16* y,
                                          void* ws, size_t ws_bytes, moe_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* MOE_MX_H */
