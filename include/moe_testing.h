/*
 * moe_testing.h -- test hooks of libmoe (not for production use).
 *
 * These entry points exist so that the failure-detection paths of the kernels can be exercised on a
 * GPU without faulting it.  They have no counterpart in the DeepSeek-V4-Flash pages.
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

#ifdef __cplusplus
}
#endif

#endif /* MOE_TESTING_H_ */
