// moe_route_noalloc: the learned router (fp32 logits, sqrt-softplus scores, biased top-k) for callers
// that cannot allocate device memory.  Some callers can't call cudaMalloc: plug-ins whose host
// framework owns every device allocation, and latency-critical paths that must never enter the
// allocator (an allocation may synchronise the device or wait on a lock).  They have no expert handle
// and no workspace, so the router's split-K partial sums live in a fixed array in the library's own
// device memory instead.
#include <cstdio>

#include "moe.h"
#include "moe_internal.h"

namespace {

// Scratch of the router partial sums, [ksplit, T, E] fp32.  Every GPU that loads the library holds
// these 4 MiB until the process exits.
constexpr size_t kScratchFloats = size_t(1) << 20;
static __device__ __align__(256) float g_router_scratch[kScratchFloats];

// Device address of the scratch array in the current context.  The name g_router_scratch in host code
// is only a host-side stand-in: a kernel must receive this address.  It is looked up on every call
// rather than cached: the lookup is a host-side table read once the library's device code is loaded,
// and a cached address would go stale when the context is destroyed and recreated (cudaDeviceReset,
// or a released primary context), which may load the device code at another address.
cudaError_t scratch_on_current_device(float** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_router_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<float*>(p);
  return cudaSuccess;
}

moe_status_t reject(moe_status_t st, const char* msg) {
  moe::set_last_error(msg);
  return st;
}

}  // namespace

extern "C" moe_status_t moe_route_noalloc(const moe_config_t* cfg, const moe_input_t* x, const float* router_w,
                                          const float* router_bias, int32_t* topk_ids, float* topk_w,
                                          moe_stream_t stream) {
  char msg[256];
  if (!cfg || !x) return reject(MOE_ERR_INVALID_ARG, "moe_route_noalloc: config or input is NULL");
  const int T = x->T, E = cfg->n_experts, k = cfg->top_k, d = cfg->d_model;
  if (d <= 0 || d % 128 || E < 1 || E > 512 || k < 1 || k > 16 || k > E) {
    snprintf(msg, sizeof(msg), "moe_route_noalloc: unsupported shape d_model=%d n_experts=%d top_k=%d", d, E, k);
    return reject(MOE_ERR_UNSUPPORTED, msg);
  }
  if (T < 0 || x->token_ids)
    return reject(MOE_ERR_INVALID_ARG, "moe_route_noalloc: T < 0, or token_ids given (hash routing needs no scratch)");
  if (T == 0) return MOE_OK;
  if (!x->x_bf16 || !router_w || !router_bias || !topk_ids || !topk_w)
    return reject(MOE_ERR_INVALID_ARG, "moe_route_noalloc: a pointer argument is NULL");
  if ((reinterpret_cast<uintptr_t>(x->x_bf16) | reinterpret_cast<uintptr_t>(router_w)) % 16)
    return reject(MOE_ERR_INVALID_ARG, "moe_route_noalloc: x and router_w must be 16-byte aligned");
  if ((size_t)T * (size_t)E > kScratchFloats) {
    snprintf(msg, sizeof(msg),
             "moe_route_noalloc: T * n_experts = %zu exceeds the fixed scratch of %zu fp32 values (T <= %zu at %d "
             "experts); use moe_route with a workspace",
             (size_t)T * E, kScratchFloats, kScratchFloats / (size_t)E, E);
    return reject(MOE_ERR_WORKSPACE, msg);
  }
  int ks = moe::router_ksplit(T, E, d);
  while (ks > 1 && (size_t)ks * T * E > kScratchFloats) ks /= 2;
  float* scratch = nullptr;
  cudaError_t e = scratch_on_current_device(&scratch);
  if (e == cudaSuccess) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    e = moe::launch_router_logits(static_cast<const __nv_bfloat16*>(x->x_bf16), router_w, T, d, E, ks, scratch, s);
    if (e == cudaSuccess)
      e = moe::launch_router_topk(scratch, ks, router_bias, T, E, k, cfg->route_scale, topk_ids, topk_w, s);
  }
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "moe_route_noalloc: %s", cudaGetErrorString(e));
    return reject(MOE_ERR_CUDA, msg);
  }
  return MOE_OK;
}
