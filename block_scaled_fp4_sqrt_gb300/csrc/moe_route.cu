// Router: fp32 logits x . Wr^T, score s = sqrt(softplus(l)), top-k on s + bias, weights
// route_scale * s_j / sum of the selected s (sqrt-softplus routing of the DeepSeek-V4 MoE, TensorSharp
// page "How TensorSharp runs it"; top-k = 6 and route_scale = 1.5 from the model card's "Speeds,
// Sizes, Times").  Hash layers replace the router by a token-id -> expert-ids table.
#include <float.h>

#include "moe_device.cuh"

namespace moe {

namespace {

constexpr int kTT = 64;   // tokens per block
constexpr int kTE = 64;   // experts per block
constexpr int kTK = 32;   // K chunk

// partial[z][t][e] = sum over k in split z of x[t][k] * w[e][k] (fp32, fixed order within a split).
__global__ void __launch_bounds__(256) router_logits_kernel(const __nv_bfloat16* __restrict__ x,
                                                            const float* __restrict__ w, int T, int d, int E,
                                                            int k_per_split, float* __restrict__ partial) {
  __shared__ float xs[kTK][kTT + 4];
  __shared__ float ws[kTK][kTE + 4];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kTT, e0 = blockIdx.y * kTE, z = blockIdx.z;
  const int kbeg = z * k_per_split, kend = kbeg + k_per_split;
  const int tx = tid % 16, ty = tid / 16;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int kc = kbeg; kc < kend; kc += kTK) {
    {  // x tile: 64 tokens x 32 k, one 8-element vector per thread
      int r = tid / 4, c = (tid % 4) * 8;
      int t = t0 + r;
      float v[8];
      if (t < T) {
        uint4 raw = *reinterpret_cast<const uint4*>(x + (size_t)t * d + kc + c);
        const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __bfloat162float(h[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[c + i][r] = v[i];
    }
    {  // w tile: 64 experts x 32 k, two 4-element vectors per thread
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        int idx = tid + h * 256;
        int r = idx / 8, c = (idx % 8) * 4;
        int e = e0 + r;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < E) v = *reinterpret_cast<const float4*>(w + (size_t)e * d + kc + c);
        ws[c + 0][r] = v.x;
        ws[c + 1][r] = v.y;
        ws[c + 2][r] = v.z;
        ws[c + 3][r] = v.w;
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kTK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int e = e0 + tx * 4 + j;
      if (e < E) partial[((size_t)z * T + t) * E + e] = acc[i][j];
    }
  }
}

constexpr int kMaxPerLane = 16;  // E <= 512
constexpr int kMaxTopK = 16;


// Block of 8 warps per 8 tokens.  Phase 1: every thread sums the split partials of some (token,
// expert) pairs in a fixed order (coalesced over experts) and stores s = sqrt(softplus(l)) and
// s + bias in shared memory.  Phase 2: warp w selects the k largest s + bias of token w (ties to the
// lower expert id) and reports ids ascending with weights route_scale * s_j / sum_j s_j.
constexpr int kTopkTokens = 8;


// KS = the number of split-K partials, a template argument so that the KS loads of a sum are issued
// unconditionally and back to back (a runtime-bounded loop serialises them on the L2 latency).
template <int KS, int NPL>
__global__ void __launch_bounds__(512) router_topk_kernel(const float* __restrict__ partial,
                                                          const float* __restrict__ bias, int T, int E, int k,
                                                          float route_scale, int32_t* __restrict__ ids,
                                                          float* __restrict__ wts) {
  pdl_trigger();
  pdl_wait();
  __shared__ float s_s[kTopkTokens][32 * kMaxPerLane];
  __shared__ float s_sel[kTopkTokens][32 * kMaxPerLane];
  const int t0 = blockIdx.x * kTopkTokens;
  for (int idx = threadIdx.x; idx < kTopkTokens * E; idx += blockDim.x) {
    const int i = idx / E, e = idx - i * E;
    const int t = t0 + i;
    if (t >= T) continue;
    float v[KS];
#pragma unroll
    for (int z = 0; z < KS; ++z) v[z] = __ldg(&partial[((size_t)z * T + t) * E + e]);
    float l = 0.f;
#pragma unroll
    for (int z = 0; z < KS; ++z) l += v[z];
    const float sv = sqrtf(softplus_f(l));
    s_s[i][e] = sv;
    s_sel[i][e] = sv + bias[e];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int t = t0 + w;
  if (w >= kTopkTokens || t >= T) return;
  float sc[NPL], sel[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    sc[i] = e < E ? s_s[w][e] : 0.f;
    sel[i] = e < E ? s_sel[w][e] : -FLT_MAX;
  }
  warp_route_topk<NPL>(sc, sel, E, k, route_scale, ids + (size_t)t * k, wts + (size_t)t * k);
}

// Hash routing: ids = the token's table row (ascending), weights route_scale / k.  Out-of-range token
// ids or table entries raise a device status bit and are replaced by valid values so that no later
// kernel indexes out of bounds.
__global__ void hash_route_kernel(const int32_t* __restrict__ tok, const int32_t* __restrict__ table, int V, int T,
                                  int E, int k, float route_scale, int32_t* __restrict__ ids, float* __restrict__ wts,
                                  int* status) {
  pdl_trigger();
  pdl_wait();
  int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int v = tok[t];
  if (v < 0 || v >= V) {
    set_status(status, DEV_BAD_TOKEN_ID);
    v = 0;
  }
  int row[kMaxTopK];
  for (int j = 0; j < k; ++j) {
    int e = table[(size_t)v * k + j];
    if (e < 0 || e >= E) {
      set_status(status, DEV_BAD_EXPERT_ID);
      e = 0;
    }
    row[j] = e;
  }
  for (int a = 1; a < k; ++a) {
    int c = row[a], b = a - 1;
    while (b >= 0 && row[b] > c) { row[b + 1] = row[b]; --b; }
    row[b + 1] = c;
  }
  float w = route_scale / (float)k;
  for (int j = 0; j < k; ++j) {
    ids[(size_t)t * k + j] = row[j];
    wts[(size_t)t * k + j] = w;
  }
}

}  // namespace

int router_ksplit(int T, int E, int d) {
  int base = ((T + kTT - 1) / kTT) * ((E + kTE - 1) / kTE);
  int ks = 1;
  while (ks < kRouterKSplitMax && base * ks < 2 * 152 && (d / kTK) % (ks * 2) == 0) ks *= 2;
  return ks;
}

cudaError_t launch_router_logits(const __nv_bfloat16* x, const float* w, int T, int d, int E, int ksplit,
                                 float* partial, cudaStream_t s) {
  dim3 grid((T + kTT - 1) / kTT, (E + kTE - 1) / kTE, ksplit);
  router_logits_kernel<<<grid, 256, 0, s>>>(x, w, T, d, E, d / ksplit, partial);
  return cudaGetLastError();
}

cudaError_t launch_router_topk(const float* partial, int ksplit, const float* bias, int T, int E, int k,
                               float route_scale, int32_t* ids, float* wts, cudaStream_t s) {
  const int blocks = (T + kTopkTokens - 1) / kTopkTokens;
  switch (ksplit) {
#define MOE_TOPK_CASE(KS) \
  case KS:                                                                                                \
    return E <= 256 ? launch_pdl(router_topk_kernel<KS, 8>, dim3(blocks), dim3(512), 0, s, partial, bias, T, E, k, \
                                 route_scale, ids, wts)                                                  \
                    : launch_pdl(router_topk_kernel<KS, 16>, dim3(blocks), dim3(512), 0, s, partial, bias, T, E, k, \
                                 route_scale, ids, wts);
    MOE_TOPK_CASE(1)
    MOE_TOPK_CASE(2)
    MOE_TOPK_CASE(4)
    MOE_TOPK_CASE(8)
    MOE_TOPK_CASE(16)
    MOE_TOPK_CASE(32)
#undef MOE_TOPK_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_hash_route(const int32_t* tok, const int32_t* table, int V, int T, int E, int k, float route_scale,
                              int32_t* ids, float* wts, int* status, cudaStream_t s) {
  return launch_pdl(hash_route_kernel, dim3((T + 127) / 128), dim3(128), 0, s, tok, table, V, T, E, k, route_scale, ids,
                    wts, status);
}

}  // namespace moe
