// Router: fp32 logits x . Wr^T, score s = sqrt(softplus(l)), top-k on s + bias, weights
// route_scale * s_j / sum of the selected s (sqrt-softplus routing of the DeepSeek-V4 MoE, TensorSharp
// page "How TensorSharp runs it"; top-k = 6 and route_scale = 1.5 from the model card's "Speeds,
// Sizes, Times").  Hash layers replace the router by a token-id -> expert-ids table.
#include <float.h>

#include "moe_device.cuh"
#include "moe_dispatch_state.cuh"

static_assert(moe::kRouterDispatchMaxT <= moe::kDispatchStateMaxT, "router-written dispatch state: batch size");

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

// Router for small batches (T <= 32), one kernel.  A 128-token tensor-core tile would leave most of
// the GPU idle while one cluster streams the weights; here every CTA takes two experts and computes their
// full fp32 dot products with all T tokens, so the 4 * E * d bytes of router weights are read by E / 2
// SMs at once.  Warp w sums K range [w d/8, (w+1) d/8) (lane-strided, then a shuffle tree), the CTA adds
// the eight warp sums in order and stores the logits; the last CTA to finish (an atomic count, fenced on
// both sides) computes s = sqrt(softplus(l)) and runs the same warp top-k as the other routers for every
// token, and resets the count for the next call.
// early_params: the weights and bias are the handle's resident copies (written only by
// moe_experts_set_router's copies, never by the kernel this one may overlap), so a lane loads its first
// weight vectors and its bias values before the programmatic-dependency wait, hiding their HBM latency
// behind the previous kernel's tail; only x waits.
template <int TMAX, int NPL>
__global__ void __launch_bounds__(256) router_small_kernel(const __nv_bfloat16* __restrict__ x,
                                                           const float* __restrict__ w, const float* __restrict__ bias,
                                                           int T, int d, int E, int k, float route_scale,
                                                           float* __restrict__ logits, int* __restrict__ done,
                                                           int32_t* __restrict__ ids, float* __restrict__ wts,
                                                           int early_params, SmallDispatch disp) {
  pdl_trigger();
  __shared__ float red[8][2][TMAX];
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = 2 * blockIdx.x;
  const bool has1 = e0 + 1 < E;
  const int kw = d / 8, kb = warp * kw;
  const float* w0p = w + (size_t)e0 * d;
  const float* w1p = w + (size_t)(has1 ? e0 + 1 : e0) * d;
  float acc0[TMAX], acc1[TMAX];
#pragma unroll
  for (int t = 0; t < TMAX; ++t) acc0[t] = acc1[t] = 0.f;
  float4 wa[4], wb[4];
  auto load_w = [&](int base) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kk = base + 128 * j + 4 * lane;
      const bool in = kk < kb + kw;
      wa[j] = in ? __ldg(reinterpret_cast<const float4*>(w0p + kk)) : make_float4(0.f, 0.f, 0.f, 0.f);
      wb[j] = in ? __ldg(reinterpret_cast<const float4*>(w1p + kk)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  float bv[NPL];  // the bias values this lane's selection reads, if this CTA turns out to be the last
  auto load_bias = [&]() {
#pragma unroll
    for (int i = 0; i < NPL; ++i) bv[i] = lane + 32 * i < E ? __ldg(&bias[lane + 32 * i]) : 0.f;
  };
  if (early_params) {
    load_w(kb);
    load_bias();
  }
  pdl_wait();
  if (!early_params) {
    load_w(kb);
    load_bias();
  }
  // the warp's K range in pieces of 4 x 128: a lane holds its 4 weight vectors of both experts, then loads
  // all tokens' activation vectors of the piece, so that a piece costs one memory round trip
  for (int base = kb; base < kb + kw; base += 4 * 128) {
    if (base != kb) load_w(base);
    // tokens in groups of 8: all 32 activation vectors of a group are loaded before their FMAs
#pragma unroll
    for (int tg = 0; tg < TMAX; tg += 8) {
      uint2 raw[8][4];
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int kk = base + 128 * j + 4 * lane;
          raw[u][j] = (tg + u < T && kk < kb + kw)
                          ? __ldg(reinterpret_cast<const uint2*>(x + (size_t)(tg + u) * d + kk))
                          : make_uint2(0u, 0u);
        }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int t = tg + u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[u][j].x));
          const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[u][j].y));
          acc0[t] = fmaf(wa[j].x, lo.x, acc0[t]);
          acc0[t] = fmaf(wa[j].y, lo.y, acc0[t]);
          acc0[t] = fmaf(wa[j].z, hi.x, acc0[t]);
          acc0[t] = fmaf(wa[j].w, hi.y, acc0[t]);
          acc1[t] = fmaf(wb[j].x, lo.x, acc1[t]);
          acc1[t] = fmaf(wb[j].y, lo.y, acc1[t]);
          acc1[t] = fmaf(wb[j].z, hi.x, acc1[t]);
          acc1[t] = fmaf(wb[j].w, hi.y, acc1[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TMAX; ++t) {
    float v0 = acc0[t], v1 = acc1[t];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, off);
      v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, off);
    }
    if (lane == 0) {
      red[warp][0][t] = v0;
      red[warp][1][t] = v1;
    }
  }
  __syncthreads();
  if (threadIdx.x < 2 * TMAX) {
    const int e = threadIdx.x / TMAX, t = threadIdx.x - e * TMAX;
    if (t < T && (e == 0 || has1)) {
      float l = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) l += red[q][e][t];
      logits[(size_t)t * E + e0 + e] = l;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(done, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) *done = 0;  // every CTA of this call has counted
  for (int t = warp; t < T; t += 8) {
    float sc[NPL], sel[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        const float sv = sqrtf(softplus_f(__ldcg(&logits[(size_t)t * E + e])));
        sc[i] = sv;
        sel[i] = sv + bv[i];
      } else {
        sc[i] = 0.f;
        sel[i] = -FLT_MAX;
      }
    }
    warp_route_topk<NPL>(sc, sel, E, k, route_scale, ids + (size_t)t * k, wts + (size_t)t * k);
  }
  if (!disp.counts) return;
  // Dispatch state of this batch (the ids above are this block's own global writes, visible after the
  // barrier).  Rows per group <= T <= 32, so a non-empty group is one tile and the lone 32-token chunk's
  // bases are all 0.  Groups are scanned in thread-contiguous runs of kGPer, then across the block.
  constexpr int kGPer = 3;  // 256 threads x 3 >= 513 groups
  __shared__ int s_cnt[256 * kGPer];
  __shared__ int s_wsum[2][8];
  const int G = disp.G;
  __syncthreads();
  for (int g = threadIdx.x; g < G; g += blockDim.x) s_cnt[g] = (disp.has_shared && g == E) ? T : 0;
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) atomicAdd(&s_cnt[ids[i]], 1);
  __syncthreads();
  int c[kGPer], nt[kGPer], run_r = 0, run_t = 0;
#pragma unroll
  for (int j = 0; j < kGPer; ++j) {
    const int g = threadIdx.x * kGPer + j;
    c[j] = g < G ? s_cnt[g] : 0;
    nt[j] = (c[j] + disp.bn - 1) / disp.bn;
    run_r += c[j];
    run_t += nt[j];
  }
  // exclusive prefix of (run_r, run_t) over the block's threads
  int ir = run_r, it = run_t;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int orr = __shfl_up_sync(0xFFFFFFFFu, ir, off), ott = __shfl_up_sync(0xFFFFFFFFu, it, off);
    if (lane >= off) {
      ir += orr;
      it += ott;
    }
  }
  if (lane == 31) {
    s_wsum[0][warp] = ir;
    s_wsum[1][warp] = it;
  }
  __syncthreads();
  int br = 0, bt = 0, tot_r = 0, tot_t = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (q < warp) {
      br += s_wsum[0][q];
      bt += s_wsum[1][q];
    }
    tot_r += s_wsum[0][q];
    tot_t += s_wsum[1][q];
  }
  int off_r = br + ir - run_r, off_t = bt + it - run_t;
#pragma unroll
  for (int j = 0; j < kGPer; ++j) {
    const int g = threadIdx.x * kGPer + j;
    if (g < G) {
      disp.chunk_hist[g] = 0;
      disp.counts[g] = c[j];
      disp.offsets[g] = off_r;
      disp.tile_off[g] = off_t;
      for (int i = 0; i < nt[j]; ++i)
        if (off_t + i < disp.max_tiles) {
          RowTile rt;
          rt.group = g;
          rt.row0 = off_r + i * disp.bn;
          rt.nrows = min(disp.bn, c[j] - i * disp.bn);
          rt.pad = 0;
          disp.tiles[off_t + i] = rt;
        }
    }
    off_r += c[j];
    off_t += nt[j];
  }
  if (threadIdx.x == 0) {
    disp.offsets[G] = tot_r;
    disp.tile_off[G] = tot_t;
    *disp.n_tiles = min(tot_t, disp.max_tiles);
  }
}

// Hash routing: ids = the token's table row (ascending), weights route_scale / k.  Out-of-range token
// ids or table entries raise a device status bit and are replaced by valid values so that no later
// kernel indexes out of bounds.
// With disp.counts set, the last block to finish also writes the batch's dispatch state (dynamic shared
// memory: dispatch_state_smem_ints(G, T) ints).
__global__ void hash_route_kernel(const int32_t* __restrict__ tok, const int32_t* __restrict__ table, int V, int T,
                                  int E, int k, float route_scale, int32_t* __restrict__ ids, float* __restrict__ wts,
                                  int* status, int* done, DispatchOut disp) {
  pdl_trigger();
  pdl_wait();
  int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < T) {
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
  if (!disp.counts) return;
  extern __shared__ int dsm[];
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(done, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) *done = 0;
  write_dispatch_state(ids, T, k, E, disp, dsm);
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

cudaError_t launch_router_small(const __nv_bfloat16* x, const float* w, const float* bias, int T, int d, int E, int k,
                                float route_scale, float* logits, int* done, int32_t* ids, float* wts,
                                int early_params, const SmallDispatch* disp, cudaStream_t s) {
  if (T < 1 || T > kRouterSmallMaxT || E > 512) return cudaErrorInvalidValue;
  if (disp && (disp->G > 256 * 3 || disp->bn < kRouterSmallMaxT)) return cudaErrorInvalidValue;
  SmallDispatch dd{};
  if (disp) dd = *disp;
  const dim3 grid((E + 1) / 2), block(256);
#define MOE_SMALL(TM, NP) \
  launch_pdl(router_small_kernel<TM, NP>, grid, block, 0, s, x, w, bias, T, d, E, k, route_scale, logits, done, ids, wts, \
             early_params, dd)
  if (E <= 256) return T <= 8 ? MOE_SMALL(8, 8) : (T <= 16 ? MOE_SMALL(16, 8) : MOE_SMALL(32, 8));
  return T <= 8 ? MOE_SMALL(8, 16) : (T <= 16 ? MOE_SMALL(16, 16) : MOE_SMALL(32, 16));
#undef MOE_SMALL
}

cudaError_t launch_hash_route(const int32_t* tok, const int32_t* table, int V, int T, int E, int k, float route_scale,
                              int32_t* ids, float* wts, int* status, cudaStream_t s, int* done,
                              const DispatchOut* disp) {
  DispatchOut dd{};
  size_t smem = 0;
  if (disp) {
    if (!done || T > kDispatchStateMaxT) return cudaErrorInvalidValue;
    dd = *disp;
    smem = (size_t)dispatch_state_smem_ints(dd.G, T) * 4;
    if (smem > 48 * 1024) return cudaErrorInvalidValue;
  }
  // with the dispatch state to write, wider blocks give its one writer block more warps
  const int threads = disp ? 512 : 128;
  return launch_pdl(hash_route_kernel, dim3((T + threads - 1) / threads), dim3(threads), smem, s, tok, table, V, T, E,
                    k, route_scale, ids, wts, status, done, dd);
}

}  // namespace moe
