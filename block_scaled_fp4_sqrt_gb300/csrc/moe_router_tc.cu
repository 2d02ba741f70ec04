// Router logits on the tensor cores: l = x . Wr^T with x bf16 [T, d] and Wr fp32 [E, d].
//
// x is exactly bf16 and each fp32 weight splits exactly into three bf16 terms, w = hi + mid + lo
// (hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid) cover its 24-bit significand), so three
// bf16 x bf16 MMAs per K step, accumulated in fp32 in tensor memory, give the fp32 logits the
// sqrt-softplus router needs (TensorSharp page, "How TensorSharp runs it") at tensor-core rate.  Each
// CTA computes a 128-token x 256-expert tile over one K slice and writes fp32 partial sums
// [split, T, E]; the top-k kernel adds the splits in a fixed order.
#include <algorithm>

#include "moe_device.cuh"
#include "moe_dispatch_state.cuh"

namespace moe {

namespace {

constexpr int kRM = 128;       // tokens per tile
constexpr int kRN = 256;       // experts per tile
constexpr int kRK = 64;        // bf16 elements per stage (one 128-byte swizzle row)
constexpr int kRStages = 2;
constexpr int kRATile = kRM * 128;       // 16 KB
constexpr int kRBTile = kRN * 128;       // 32 KB per split
constexpr int kRStage = kRATile + 3 * kRBTile;
constexpr int kRSmem = kRStages * kRStage + 1024 + 64;
static_assert(kRSmem <= 232448, "router shared memory");

// kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t bf16_idesc(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Wr fp32 [E, d] -> three bf16 planes hi, mid, lo (rows E .. Epad-1 zero), stored tile-contiguous:
// plane p, K chunk kc (64 elements), expert tile et (256 rows) is one [256 x 64] block of 32 KB, at
// block index (p * d/64 + kc) * Epad/256 + et.  A router pipeline stage then loads three contiguous
// 32 KB boxes; boxes of 128-byte rows 8 KB apart streamed at about 28 GB/s per SM (measured).  Four
// weights per thread and step (d is a multiple of 256, so a group of four stays inside one chunk).
__device__ __forceinline__ size_t router_plane_offset(int p, int e, int k, int d, int Epad) {
  const int kc = k >> 6, kk = k & 63, et = e >> 8, er = e & 255;
  return ((((size_t)p * (d >> 6) + kc) * (Epad >> 8) + et) * 256 + er) * 64 + kk;
}

__global__ void split_router_kernel(const float4* __restrict__ w, int E, int Epad, int d,
                                    __nv_bfloat16* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const size_t total = (size_t)Epad * d, quads = total / 4;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < quads; i += (size_t)gridDim.x * blockDim.x) {
    const int e = (int)(i * 4 / d), k = (int)(i * 4 - (size_t)e * d);
    const float4 v4 = e < E ? __ldg(&w[i]) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float v[4] = {v4.x, v4.y, v4.z, v4.w};
    __nv_bfloat16 hi[4], mid[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      hi[j] = __float2bfloat16_rn(v[j]);
      const float r1 = v[j] - __bfloat162float(hi[j]);
      mid[j] = __float2bfloat16_rn(r1);
      lo[j] = __float2bfloat16_rn(r1 - __bfloat162float(mid[j]));
    }
    *reinterpret_cast<uint2*>(out + router_plane_offset(0, e, k, d, Epad)) = *reinterpret_cast<const uint2*>(hi);
    *reinterpret_cast<uint2*>(out + router_plane_offset(1, e, k, d, Epad)) = *reinterpret_cast<const uint2*>(mid);
    *reinterpret_cast<uint2*>(out + router_plane_offset(2, e, k, d, Epad)) = *reinterpret_cast<const uint2*>(lo);
  }
}

// Row coordinate of the [256 x 64] box of plane p, K chunk kc, expert tile et in the packed planes viewed
// as a [blocks * 256, 64] bf16 matrix.
__device__ __forceinline__ int router_box_row(int p, int kc, int et, int d, int Epad) {
  return ((p * (d >> 6) + kc) * (Epad >> 8) + et) * 256;
}

struct RouterArgs {
  float* partial;  // [split, T, E]
  int T, E, Epad, d;
  int k_per_split;  // multiple of kRK
  int* status;
  uint64_t budget_ns;
};

// grid (ceil(T / 128), Epad / 256, split); warps: 0 TMA, 1 MMA, 2..5 epilogue
__global__ void __launch_bounds__(192, 1) router_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                           const __grid_constant__ CUtensorMap tm_w,
                                                           const RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRStages * kRStage);
  uint64_t* empty = full + kRStages;
  uint64_t* acc_full = empty + kRStages;
  __shared__ uint32_t tmem_slot;
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRM, e0 = blockIdx.y * kRN, z = blockIdx.z;
  const int k0 = z * a.k_per_split, n_stages = a.k_per_split / kRK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_w);
  }
  if (warp == 1) tmem_alloc(&tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  pdl_wait();  // x and the split weights come from earlier kernels
  bool acc_ok = true;

  if (warp == 0 && lane == 0) {
    const uint64_t pol = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, last_par = 0;
    bool ok = true;
    for (int s = 0; s < n_stages; ++s) {
      if (!mbar_wait(&empty[stage], phase ^ 1u, a.budget_ns)) {
        ok = false;
        break;
      }
      uint8_t* st = smem + stage * kRStage;
      mbar_arrive_expect_tx(&full[stage], kRStage);
      const int kk = k0 + s * kRK;
      tma_load_2d(st, &tm_x, kk, t0, &full[stage], pol);
      for (int p = 0; p < 3; ++p)
        tma_load_2d(st + kRATile + p * kRBTile, &tm_w, 0, router_box_row(p, kk >> 6, blockIdx.y, a.d, a.Epad),
                    &full[stage], pol);
      issued |= 1u << stage;
      last_par = (last_par & ~(1u << stage)) | (phase << stage);
      if (++stage == kRStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {
      set_status(a.status, DEV_TIMEOUT);
      for (int s = 0; s < kRStages; ++s)
        if ((issued >> s) & 1u) (void)mbar_wait(&full[s], (last_par >> s) & 1u, 20000000ull);
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = bf16_idesc(kRM, kRN);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int s = 0; s < n_stages; ++s) {
      if (!mbar_wait(&full[stage], phase, a.budget_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint8_t* st = smem + stage * kRStage;
      const uint32_t a_addr = smem_addr(st);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t ad = smem_desc(a_addr + k * 32, 16, 1024, 2);
#pragma unroll
        for (int p = 0; p < 3; ++p)
          tc_mma_bf16(tbase, ad, smem_desc(smem_addr(st + kRATile + p * kRBTile) + k * 32, 16, 1024, 2), idesc,
                      (s | k | p) ? 1u : 0u);
      }
      tc_commit(&empty[stage]);
      if (++stage == kRStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) set_status(a.status, DEV_TIMEOUT);
    tc_commit(acc_full);  // also retires every MMA issued so far
  } else if (warp >= 2) {
    const int q = warp & 3;
    acc_ok = mbar_wait(acc_full, 0, a.budget_ns);
    acc_ok = __all_sync(0xFFFFFFFFu, acc_ok);
    tc_fence_after();
    if (!acc_ok) {
      if (lane == 0) set_status(a.status, DEV_TIMEOUT);
    } else if (t0 + q * 32 < a.T) {
      const int t = t0 + q * 32 + lane;
      const uint32_t tl = tbase + ((uint32_t)(q * 32) << 16);
      for (int c = 0; c < kRN / 32; ++c) {
        if (e0 + c * 32 >= a.E) break;
        float v[32];
        tmem_ld32(tl + (uint32_t)(c * 32), v);
        if (t < a.T) {
          float* dst = a.partial + ((size_t)z * a.T + t) * a.E + e0 + c * 32;
          if (e0 + c * 32 + 32 <= a.E && (a.E & 3) == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              reinterpret_cast<float4*>(dst)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (e0 + c * 32 + i < a.E) dst[i] = v[i];
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 256);
}

// ---------------------------------------------------------------------------------------------------
// Fused router for up to 256 experts: the logits above, reduced over the K split inside a thread-block
// cluster, then sqrt-softplus and top-k, in one kernel.  The S CTAs of a cluster compute partial logits
// of the same 128-token tile over S slices of K; each drains its [128 x 256] partial from tensor
// memory into its own shared memory, and after a cluster barrier CTA z sums rows z*128/S .. of all S
// partials through distributed shared memory in the fixed order 0..S-1 and selects the token's experts.
// No partial reaches global memory.
constexpr int kFThreads = 384;                 // warps 0 TMA, 1 MMA, 2..5 TMEM drain; all 12 select
constexpr int kFStride = kRN + 4;              // partial row stride in floats (1040 B: conflict-free)
static_assert(kRM * kFStride * 4 + (kFThreads / 32) * kRN * 4 <= kRStages * kRStage,
              "partials and the per-warp logit rows fit in the drained pipeline buffers");

struct FusedArgs {
  const float* bias;
  int32_t* ids;
  float* wts;
  int T, E, Epad, d, k;
  float route_scale;
  int k_per_split;  // multiple of kRK
  int* status;
  uint64_t budget_ns;
  int* done;         // CTAs finished (zero between calls), when the last one writes the dispatch state
  DispatchOut disp;  // disp.counts == NULL: no dispatch state
};

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Volatile (kept in order after the cluster barrier, which is a compiler barrier too) but without a
// memory clobber, so that a run of these loads issues back to back before their sum consumes them.
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

// grid (ceil(T / 128), S), cluster (1, S); blockIdx.y = the CTA's rank in its cluster = its K slice
template <int S>
__global__ void __launch_bounds__(kFThreads, 1) router_fused_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                                    const __grid_constant__ CUtensorMap tm_w,
                                                                    const FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRStages * kRStage);
  uint64_t* empty = full + kRStages;
  uint64_t* acc_full = empty + kRStages;
  __shared__ uint32_t tmem_slot;
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int z = blockIdx.y, t0 = blockIdx.x * kRM;
  const int k0 = z * a.k_per_split, n_stages = a.k_per_split / kRK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_w);
  }
  if (warp == 1) tmem_alloc(&tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  pdl_wait();  // x and the split weights come from earlier kernels

  if (warp == 0 && lane == 0) {
    const uint64_t pol = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, last_par = 0;
    bool ok = true;
    for (int s = 0; s < n_stages; ++s) {
      if (!mbar_wait(&empty[stage], phase ^ 1u, a.budget_ns)) {
        ok = false;
        break;
      }
      uint8_t* st = smem + stage * kRStage;
      mbar_arrive_expect_tx(&full[stage], kRStage);
      const int kk = k0 + s * kRK;
      tma_load_2d(st, &tm_x, kk, t0, &full[stage], pol);
      for (int p = 0; p < 3; ++p)
        tma_load_2d(st + kRATile + p * kRBTile, &tm_w, 0, router_box_row(p, kk >> 6, 0, a.d, a.Epad), &full[stage], pol);
      issued |= 1u << stage;
      last_par = (last_par & ~(1u << stage)) | (phase << stage);
      if (++stage == kRStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {
      set_status(a.status, DEV_TIMEOUT);
      for (int s = 0; s < kRStages; ++s)
        if ((issued >> s) & 1u) (void)mbar_wait(&full[s], (last_par >> s) & 1u, 20000000ull);
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = bf16_idesc(kRM, kRN);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int s = 0; s < n_stages; ++s) {
      if (!mbar_wait(&full[stage], phase, a.budget_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint8_t* st = smem + stage * kRStage;
      const uint32_t a_addr = smem_addr(st);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t ad = smem_desc(a_addr + k * 32, 16, 1024, 2);
#pragma unroll
        for (int p = 0; p < 3; ++p)
          tc_mma_bf16(tbase, ad, smem_desc(smem_addr(st + kRATile + p * kRBTile) + k * 32, 16, 1024, 2), idesc,
                      (s | k | p) ? 1u : 0u);
      }
      tc_commit(&empty[stage]);
      if (++stage == kRStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) set_status(a.status, DEV_TIMEOUT);
    tc_commit(acc_full);  // also retires every MMA issued so far
  } else if (warp >= 2 && warp < 6) {
    // drain the partial [128 x 256] into shared memory (the pipeline buffers are idle once every MMA
    // has retired, which acc_full signals): thread = token row, 256 fp32 per row
    const int q = warp & 3;
    bool acc_ok = mbar_wait(acc_full, 0, a.budget_ns);
    acc_ok = __all_sync(0xFFFFFFFFu, acc_ok);
    tc_fence_after();
    if (!acc_ok) {
      if (lane == 0) set_status(a.status, DEV_TIMEOUT);
    } else {
      const uint32_t tl = tbase + ((uint32_t)(q * 32) << 16);
      float4* prow = reinterpret_cast<float4*>(reinterpret_cast<float*>(smem) + (q * 32 + lane) * kFStride);
      for (int c = 0; c < kRN / 32; ++c) {
        float v[32];
        tmem_ld32(tl + (uint32_t)(c * 32), v);
#pragma unroll
        for (int i = 0; i < 8; ++i) prow[c * 8 + i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    }
  }
  // the selection's bias values, loaded before the cluster barrier so that their latency hides behind it
  float bv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) bv[i] = lane + 32 * i < a.E ? __ldg(&a.bias[lane + 32 * i]) : 0.f;
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();  // every partial of the cluster is in shared memory

  // CTA z: rows z * 128/S .. of the tile, one warp per token, summing the S partials in rank order
  constexpr int rows_per = kRM / S;
  uint32_t remote[S];  // each cluster CTA's partial buffer in the cluster's shared window
  const uint32_t part_addr = smem_addr(smem);
#pragma unroll
  for (int src = 0; src < S; ++src) remote[src] = cluster_map(part_addr, (uint32_t)src);
  // the warp's logit row, re-read in the one-expert-per-lane layout of the selection
  float* lrow = reinterpret_cast<float*>(smem + kRM * kFStride * 4) + warp * kRN;
  // lane l sums experts 4l..4l+3 and 128+4l..+3 of a row over the S partials, in rank order.  With few
  // partials (S <= 4: long token loops per warp) both halves of the warp's next row are loaded while the
  // current row is selected; with more, per half, S 16-byte loads are in flight at once.
  constexpr bool kAhead = S <= 4;
  constexpr int kNext = kAhead ? 2 * S : 1;
  constexpr int kWarps = kFThreads / 32;
  float4 nxt[kNext];
  auto fetch = [&](int rr) {
    const int r = z * rows_per + rr;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int src = 0; src < S; ++src)
        nxt[(h * S + src) % kNext] = ld_cluster_f4(remote[src] + (uint32_t)((r * kFStride + 128 * h + 4 * lane) * 4));
  };
  if (kAhead && warp < rows_per && t0 + z * rows_per + warp < a.T) fetch(warp);
  for (int rr = warp; rr < rows_per; rr += kWarps) {
    const int r = z * rows_per + rr, t = t0 + r;
    if (t >= a.T) continue;  // warp-uniform
    if (kAhead) {
      float4 cur[kNext];
#pragma unroll
      for (int i = 0; i < kNext; ++i) cur[i] = nxt[i];
      if (rr + kWarps < rows_per && t + kWarps < a.T) fetch(rr + kWarps);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int src = 0; src < S; ++src) {
          const float4 v = cur[(h * S + src) % kNext];
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        reinterpret_cast<float4*>(lrow + 128 * h)[lane] = acc;
      }
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t off = (uint32_t)((r * kFStride + 128 * h + 4 * lane) * 4);
        float4 v[S];
#pragma unroll
        for (int src = 0; src < S; ++src) v[src] = ld_cluster_f4(remote[src] + off);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int src = 0; src < S; ++src) {
          acc.x += v[src].x;
          acc.y += v[src].y;
          acc.z += v[src].z;
          acc.w += v[src].w;
        }
        reinterpret_cast<float4*>(lrow + 128 * h)[lane] = acc;
      }
    }
    __syncwarp();
    float sc[8], sel[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      const float sv = sqrtf(softplus_f(lrow[e]));
      sc[i] = e < a.E ? sv : 0.f;
      sel[i] = e < a.E ? sv + bv[i] : -FLT_MAX;
    }
    __syncwarp();
    warp_route_topk<8>(sc, sel, a.E, a.k, a.route_scale, a.ids + (size_t)t * a.k, a.wts + (size_t)t * a.k);
  }
  cluster_sync_all();  // no CTA leaves while another still reads its partial
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 256);
  if (a.disp.counts) {
    // the last CTA of the grid to finish writes the batch's dispatch state from the ids every CTA wrote
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(a.done, 1) == (int)(gridDim.x * gridDim.y) - 1;
    __syncthreads();
    if (s_last) {
      __threadfence();
      if (threadIdx.x == 0) *a.done = 0;  // every CTA of this call has counted
      write_dispatch_state(a.ids, a.T, a.k, a.E, a.disp, reinterpret_cast<int*>(smem));
    }
  }
}

}  // namespace

int router_tc_split(int T, int E, int d) {
  const int mt = (T + kRM - 1) / kRM, nt = (E + kRN - 1) / kRN;
  int s = 1;
  while (s < 32 && mt * nt * s * 2 <= 152 && (d / kRK) % (s * 2) == 0) s *= 2;
  return s;
}

int router_tc_epad(int E) { return (E + kRN - 1) / kRN * kRN; }

// Cluster size of the fused router: as many K slices as keep the grid within one wave of CTAs and
// divide K into whole 64-element stages, up to 16 where the device can co-schedule 16-CTA clusters
// (a non-portable size; checked once with the occupancy query) and 8 otherwise.
template <int S>
static cudaError_t configure_fused() {
  static PerDeviceOnce once;
  return once.run([] {
    cudaError_t e = cudaFuncSetAttribute(router_fused_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem);
    if (e == cudaSuccess && S > 8)
      e = cudaFuncSetAttribute(router_fused_kernel<S>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
  });
}

static int max_fused_cluster() {
  static std::atomic<int> cached[64];  // per device; 0 = not queried yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
  if (const int c = cached[dev].load(std::memory_order_relaxed)) return c;
  int best = 8;
  if (configure_fused<16>() == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 16, 1);
    cfg.blockDim = dim3(kFThreads, 1, 1);
    cfg.dynamicSmemBytes = kRSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 16;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, router_fused_kernel<16>, &cfg) == cudaSuccess && n >= 1) best = 16;
  }
  (void)cudaGetLastError();
  cached[dev].store(best, std::memory_order_relaxed);
  return best;
}

int router_fused_split(int T, int d) {
  const int mt = (T + kRM - 1) / kRM;
  const int cap = max_fused_cluster();
  int s = 1;
  while (s < cap && mt * s * 2 <= 152 && (d / kRK) % (s * 2) == 0) s *= 2;
  return s;
}

template <int S>
static cudaError_t launch_fused_S(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const FusedArgs& a, cudaStream_t s) {
  cudaError_t e = configure_fused<S>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.T + kRM - 1) / kRM, S, 1);
  cfg.blockDim = dim3(kFThreads, 1, 1);
  cfg.dynamicSmemBytes = kRSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = S;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, router_fused_kernel<S>, tm_x, tm_w, a);
}

cudaError_t launch_router_fused(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const float* bias, int T, int E,
                                int d, int k, float route_scale, int split, int32_t* ids, float* wts, int* status,
                                uint64_t budget_ns, cudaStream_t s, int* done, const DispatchOut* disp) {
  if (E > kRN) return cudaErrorInvalidValue;
  if (disp && (!done || T > kDispatchStateMaxT || dispatch_state_smem_ints(disp->G, T) * 4 > kRStages * kRStage))
    return cudaErrorInvalidValue;
  FusedArgs a{bias, ids, wts, T, E, router_tc_epad(E), d, k, route_scale, d / split, status, budget_ns, done, {}};
  if (disp) a.disp = *disp;
  switch (split) {
    case 1: return launch_fused_S<1>(tm_x, tm_w, a, s);
    case 2: return launch_fused_S<2>(tm_x, tm_w, a, s);
    case 4: return launch_fused_S<4>(tm_x, tm_w, a, s);
    case 8: return launch_fused_S<8>(tm_x, tm_w, a, s);
    case 16: return launch_fused_S<16>(tm_x, tm_w, a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_split_router(const float* w, int E, int d, __nv_bfloat16* out, cudaStream_t s) {
  const int Epad = router_tc_epad(E);
  const size_t total = (size_t)Epad * d;
  const int blocks = (int)std::min<size_t>((total / 4 + 255) / 256, 152 * 8);
  return launch_pdl(split_router_kernel, dim3(blocks), dim3(256), 0, s, reinterpret_cast<const float4*>(w), E, Epad,
                    d, out);
}

cudaError_t launch_router_tc(const CUtensorMap& tm_x, const CUtensorMap& tm_w, int T, int E, int d, int split,
                             float* partial, int* status, uint64_t budget_ns, cudaStream_t s) {
  static PerDeviceOnce smem_optin;
  const cudaError_t e =
      smem_optin.run([] { return cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem); });
  if (e != cudaSuccess) return e;
  RouterArgs a{partial, T, E, router_tc_epad(E), d, d / split, status, budget_ns};
  dim3 grid((T + kRM - 1) / kRM, a.Epad / kRN, split);
  return launch_pdl(router_tc_kernel, grid, dim3(192), kRSmem, s, tm_x, tm_w, a);
}

}  // namespace moe
