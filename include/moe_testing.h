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

#ifdef __cplusplus
}
#endif

#endif /* MOE_TESTING_H_ */
