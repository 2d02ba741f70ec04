/*
 * moe_testing.h -- test hooks and measurement utilities of libmoe (not for production use).
 *
 * These entry points exist so that the failure-detection paths of the kernels can be exercised on a
 * GPU without faulting it, and so that benchmarks can measure the tensor-core peak their roofline
 * divides by.  They have no counterpart in the DeepSeek-V4-Flash pages.
 */
#ifndef MOE_TESTING_H_
#define MOE_TESTING_H_

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * enable != 0: in later moe_forward / moe_expert_ffn calls on this handle, the load warp of the
 * grouped GEMMs issues no copies.  The MMA warp's bounded wait for the first pipeline stage then
 * runs out (after the handle's wait budget, see moe_set_wait_budget), the kernel records
 * MOE_ERR_TIMEOUT in the handle's status and returns without touching the output; moe_check reports
 * it and the CUDA context stays usable.  enable = 0 restores normal operation.
 */
MOE_API moe_status_t moe_testing_stall_loads(moe_experts_t experts, int32_t enable);

/*
 * enable != 0: later calls on this handle run batches with 128-row tiles (MXFP8 activations) on the
 * CTA-pair grouped GEMMs -- two SMs per work item, one M = 256 tcgen05.mma.cta_group::2 per K step, each
 * SM holding half the weight tile -- instead of the one-SM kernels (the default); enable = 0 restores
 * the default.  Both give the same results (bit for bit in the tests); the pair kernel pads every expert
 * group to an even number of row tiles, which costs more than it gains on skewed routing with many
 * single-tile experts.  Tests compare the two; benchmarks measure one against the other.
 * Errors: MOE_ERR_INVALID_ARG (NULL handle).
 */
MOE_API moe_status_t moe_testing_set_pair_gemm(moe_experts_t experts, int32_t enable);

/*
 * Reads back the SwiGLU output h of the last moe_forward / moe_expert_ffn on this handle, as the
 * down projection consumed it: *n_rows receives its row count (the call's routed rows in permuted
 * order, then one shared row per token in token order; 0 if there was none), h_q [n_rows, d_ff]
 * E4M3 codes (or [n_rows, d_ff/2] packed E2M1 codes with MOE_ACT_MXFP4) and h_s [n_rows, d_ff/32]
 * E8M0 bytes, both device buffers (h_s 4-byte aligned) that the caller sizes for n_rows; pass NULL
 * for both to learn n_rows only.  Asynchronous on `stream`; valid until the next call on the handle.
 * Tests use it to compare the kernels' h codes with the oracle's and to check the down projection on
 * the kernels' own h.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_WORKSPACE, MOE_ERR_CUDA.
 */
MOE_API moe_status_t moe_testing_read_h(moe_experts_t experts, uint8_t* h_q, uint8_t* h_s, int32_t* n_rows,
                                        moe_stream_t stream);

/*
 * Reads back the layer output of the last moe_forward on this handle before its rounding to bf16:
 * y32 fp32 [T, d_model] (device, 16-byte aligned, sized by the caller) receives, per token, the same
 * fixed-order fp32 sum that the combine rounds once to bf16 (routing slots 0..top_k-1, then the shared
 * row; a stack layer's residual is not included).  *T receives the forward's row count; y32 = NULL
 * asks for it only.  It re-runs the sum from the expert rows the forward left in the workspace, so it
 * is valid until the next moe_forward on the handle.  Tests use it to check the arithmetic before the
 * output rounding against the layer's tolerance, and that the bf16 output is exactly that sum rounded
 * to nearest even.  Asynchronous on `stream`.  Errors: MOE_ERR_INVALID_ARG (NULL handle or T, no
 * forward since the last one started, misaligned y32), MOE_ERR_WORKSPACE, MOE_ERR_CUDA.
 */
MOE_API moe_status_t moe_testing_read_y32(moe_experts_t experts, float* y32, int32_t* T, moe_stream_t stream);

/*
 * Measures the throughput of the block-scaled MMA the grouped GEMMs are built on (tcgen05.mma
 * kind::mxf8f6f4.block_scale.scale_vec::1X, E4M3 activations x E2M1 weights with E8M0 scales,
 * M = 128, N = 256, K = 32) on the current device: one CTA per SM issues n_stages x 4 MMAs back to
 * back, operands rotating through six shared-memory stages, scale atoms copied into tensor memory
 * two stages ahead.  *tflops receives 2 * M * N * K * MMAs / (slowest SM's time), in TFLOP/s (dense;
 * the product of the MMA shape, not of any model workload).  Synchronous: it launches two kernels on
 * the default stream and waits for them; it allocates and frees a few bytes of device memory.
 * n_stages must be in [8, 262144] (a few thousand give a stable figure in about a millisecond).
 * Returns MOE_ERR_INVALID_ARG, MOE_ERR_CUDA, or MOE_ERR_TIMEOUT if the kernel's bounded wait ran out.
 */
MOE_API moe_status_t moe_measure_mxf8f6f4_peak(int32_t n_stages, double* tflops);

/*
 * The same measurement for the MMA of the MXFP4-activation variant (moe_experts_set_activation_format
 * with MOE_ACT_MXFP4): tcgen05.mma kind::mxf4.block_scale.scale_vec::2X, E2M1 x E2M1 with E8M0
 * scales, M = 128, N = 256, K = 64; n_stages x 2 MMAs per SM, operands packed in 64-byte rows.
 * Arguments, result and errors as moe_measure_mxf8f6f4_peak.
 */
MOE_API moe_status_t moe_measure_mxf4_peak(int32_t n_stages, double* tflops);

#ifdef __cplusplus
}
#endif

#endif /* MOE_TESTING_H_ */
