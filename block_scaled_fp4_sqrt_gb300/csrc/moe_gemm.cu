// Grouped expert GEMMs on 5th-generation tensor cores (tcgen05, kind::mxf8f6f4 with E8M0 block
// scales): MXFP4 expert weights x MXFP8 activations, fp32 accumulation in tensor memory.
//
//  * gate-up:  G = A . W1^T, U = A . W3^T per expert group; epilogue h = silu(min(G, L)) *
//    clamp(U, -L, L) (Ops.SiLUMulClamp, swiglu_limit = 10), re-quantised to MXFP8 along the FFN
//    dimension ("expert FFN (fused dequant + GEMM)", FaStar README "Features"; TensorSharp page
//    "How TensorSharp runs it").
//  * down:     Y = w_row * (H . W2^T) per permuted row, fp32 (summed by the combine kernel, the
//    weighted-sum epilogue moe_scatter_add of the TensorSharp page, "DSpark and MoE CPU offload") or
//    bf16 (the standalone grouped FFN call).
//
// Tile shape ("swap-AB"): the 128 weight rows of one output tile are the MMA's M side, the token
// rows of one expert group (up to 32) are its N side, so a verify batch with ~12 rows per expert
// streams each weight byte from HBM exactly once.  One persistent CTA per SM walks a device-built
// list of (row tile, output tile) work items.  Warp roles: warp 0 issues TMA loads, warp 1 issues
// tcgen05 copies/MMAs, warps 2..5 drain the TMEM accumulators (double buffered) and run the
// epilogue.  Every wait is bounded; on timeout the kernel records DEV_TIMEOUT and unwinds.
#include "moe_device.cuh"

namespace moe {

namespace {

constexpr int kBN = kDecodeBN;  // token rows per MMA (tcgen05 N)

__host__ __device__ constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int NMAT, int STAGES>
struct Cfg {
  static constexpr int kATile = kMmaM * 128;       // one 128 x 128 weight tile, FP4 padded to bytes in smem
  static constexpr int kBTile = kBN * 128;         // 32 token rows x 128 FP8
  static constexpr int kSfBytes = (NMAT + 1) * kSfAtomBytes;
  static constexpr int kStageRaw = NMAT * kATile + kBTile + kSfBytes;
  static constexpr int kStage = (kStageRaw + 1023) / 1024 * 1024;
  static constexpr int kBarBytes = (2 * STAGES + 5) * 8;
  static constexpr int kSmem = STAGES * kStage + 1024 + kBarBytes;
  // bytes delivered per stage: packed FP4 boxes count 64 bytes per row
  static constexpr uint32_t kTx = NMAT * (kMmaM * 64) + kBTile + kSfBytes;
  static constexpr int kAccCols = 2 * NMAT * kBN;  // two accumulator buffers
  static constexpr int kSfCols = (NMAT + 1) * 4;   // per stage
  static constexpr int kTmemCols = pow2_at_least(kAccCols + STAGES * kSfCols);
};

struct GemmArgs {
  const uint8_t* sf_routed;  // weight scale atoms [E, w_mblocks, KG, 512]
  const uint8_t* sf_shared;  // [1, w_mblocks, KG, 512]
  const uint8_t* act_sf;     // activation scale atoms [tile, KG, 512]
  const RowTile* tiles;
  const int32_t* n_tiles;
  int max_tiles;
  int E;                // group E is the shared expert
  int KG;               // K / 128
  int m_tiles;          // output tiles of 128 per row tile
  int rows_per_expert;  // weight rows per expert in the tensor map
  int up_row_offset;    // gate-up: rows f .. 2f-1 are the up projection
  int w_mblocks;        // rows_per_expert / 128
  // gate-up epilogue
  float limit;
  uint8_t* h_q;
  uint8_t* h_sf;
  int f;
  // down epilogue: exactly one of y_f32 / y_bf16 is set
  const float* row_w;
  float* y_f32;
  __nv_bfloat16* y_bf16;
  int d;
  int* status;
  uint64_t budget_ns;
  int stall_loads;  // test hook: issue no loads, so the consumers' bounded waits run out
};

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

template <int NMAT, int STAGES>
__global__ void __launch_bounds__(192, 1)
    grouped_mx_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_w_shared,
                           const __grid_constant__ CUtensorMap tm_act, const GemmArgs a) {
  using C = Cfg<NMAT, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStage);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;   // [2]
  uint64_t* drain = acc_empty + 2;      // [1]
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n_tiles = *reinterpret_cast<const volatile int32_t*>(a.n_tiles);
  if (n_tiles > a.max_tiles) n_tiles = a.max_tiles;
  const int total = n_tiles * a.m_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(drain, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    prefetch_tensormap(&tm_w);
    prefetch_tensormap(&tm_w_shared);
    prefetch_tensormap(&tm_act);
  }
  if (warp == 1) tmem_alloc(&tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      const uint64_t pol_w = l2_policy_evict_first();  // weights: streamed once
      const uint64_t pol_a = l2_policy_evict_last();   // activations: re-read by every output tile
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_par = 0;  // per-stage bits: ever issued, parity of the last issue
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok && !a.stall_loads; w += gridDim.x) {
        const int ti = w / a.m_tiles, mt = w - ti * a.m_tiles;
        const RowTile rt = a.tiles[ti];
        const bool sh = rt.group == a.E;
        const CUtensorMap* tw = sh ? &tm_w_shared : &tm_w;
        const int e = sh ? 0 : rt.group;
        const int wrow = e * a.rows_per_expert + mt * kMmaM;
        const uint8_t* sfw = (sh ? a.sf_shared : a.sf_routed) + (size_t)e * a.w_mblocks * a.KG * kSfAtomBytes;
        const uint8_t* sf_gate = sfw + (size_t)mt * a.KG * kSfAtomBytes;
        const uint8_t* sf_up = sfw + (size_t)(a.up_row_offset / kMmaM + mt) * a.KG * kSfAtomBytes;
        const uint8_t* sf_act = a.act_sf + (size_t)ti * a.KG * kSfAtomBytes;
        for (int kg = 0; kg < a.KG; ++kg) {
          if (abort_flag || !mbar_wait(&empty[stage], phase ^ 1u, a.budget_ns)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * C::kStage;
          mbar_arrive_expect_tx(&full[stage], C::kTx);
          tma_load_2d(st, tw, kg * kKGroup, wrow, &full[stage], pol_w);
          if (NMAT == 2) tma_load_2d(st + C::kATile, tw, kg * kKGroup, wrow + a.up_row_offset, &full[stage], pol_w);
          tma_load_2d(st + NMAT * C::kATile, &tm_act, kg * kKGroup, rt.row0, &full[stage], pol_a);
          uint8_t* sf = st + NMAT * C::kATile + C::kBTile;
          bulk_load(sf, sf_gate + kg * kSfAtomBytes, kSfAtomBytes, &full[stage]);
          if (NMAT == 2) bulk_load(sf + kSfAtomBytes, sf_up + kg * kSfAtomBytes, kSfAtomBytes, &full[stage]);
          bulk_load(sf + NMAT * kSfAtomBytes, sf_act + kg * kSfAtomBytes, kSfAtomBytes, &full[stage]);
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        set_status(a.status, DEV_TIMEOUT);
        abort_flag = 1;
        // let copies already in flight land before the CTA's shared memory is released
        for (int s = 0; s < STAGES; ++s)
          if ((issued >> s) & 1u) (void)mbar_wait(&full[s], (last_par >> s) & 1u, 20000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      const uint32_t idesc_k[4] = {mma_idesc(5, 0, kMmaM, kBN, 0, 0), mma_idesc(5, 0, kMmaM, kBN, 1, 1),
                                   mma_idesc(5, 0, kMmaM, kBN, 2, 2), mma_idesc(5, 0, kMmaM, kBN, 3, 3)};
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true, any = false;
      int it = 0;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_par = (uint32_t)(it >> 1) & 1u;
        if (abort_flag || !mbar_wait(&acc_empty[acc], acc_par ^ 1u, a.budget_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tbase + (uint32_t)(acc * NMAT * kBN);
        for (int kg = 0; kg < a.KG; ++kg) {
          if (abort_flag || !mbar_wait(&full[stage], phase, a.budget_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint8_t* st = smem + stage * C::kStage;
          const uint8_t* sf = st + NMAT * C::kATile + C::kBTile;
          const uint32_t sf_t = tbase + (uint32_t)(C::kAccCols + stage * C::kSfCols);
#pragma unroll
          for (int m = 0; m <= NMAT; ++m)
            tc_copy_sf(sf_t + 4 * m, smem_desc(smem_addr(sf + m * kSfAtomBytes), 128, 128, 0));
          const uint32_t a_addr = smem_addr(st), b_addr = smem_addr(st + NMAT * C::kATile);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t bdesc = smem_desc(b_addr + k * 32, 16, 1024, 2);
            const uint32_t accumulate = (kg | k) ? 1u : 0u;
            tc_mma_mx(d0, smem_desc(a_addr + k * 32, 16, 1024, 2), bdesc, idesc_k[k], sf_t, sf_t + 4 * NMAT,
                      accumulate);
            if (NMAT == 2)
              tc_mma_mx(d0 + kBN, smem_desc(a_addr + C::kATile + k * 32, 16, 1024, 2), bdesc, idesc_k[k], sf_t + 4,
                        sf_t + 4 * NMAT, accumulate);
          }
          any = true;
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);
      }
      if (!ok) {
        set_status(a.status, DEV_TIMEOUT);
        abort_flag = 1;
      }
      if (any) {  // all issued MMAs must retire before TMEM is released
        tc_commit(drain);
        if (!mbar_wait(drain, 0, a.budget_ns)) set_status(a.status, DEV_TIMEOUT);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int m = q * 32 + lane;
    int it = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t acc_par = (uint32_t)(it >> 1) & 1u;
      bool got = !abort_flag && mbar_wait(&acc_full[acc], acc_par, a.budget_ns);
      got = __all_sync(0xFFFFFFFFu, got);
      if (!got) {
        if (lane == 0) {
          set_status(a.status, DEV_TIMEOUT);
          abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const int ti = w / a.m_tiles, mt = w - ti * a.m_tiles;
      const RowTile rt = a.tiles[ti];
      const uint32_t tl = tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * NMAT * kBN);
      float g[kBN];
      tmem_ld32(tl, g);
      if (NMAT == 2) {
        float u[kBN];
        tmem_ld32(tl + kBN, u);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        const float L = a.limit;
        const int fcol = mt * kMmaM + m;
        uint8_t* hq_base = a.h_q + fcol;
        uint8_t* hsf_base = a.h_sf + ((size_t)ti * (a.f / kKGroup) + mt) * kSfAtomBytes + q;
#pragma unroll
        for (int n = 0; n < kBN; ++n) {
          const float gc = fminf(g[n], L);
          const float uc = fminf(fmaxf(u[n], -L), L);
          const float h = silu_f(gc) * uc;
          const uint32_t amax_bits = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(h)));
          const int se = mxfp8_block_exp(__uint_as_float(amax_bits));
          const uint8_t code = (uint8_t)(e4m3x2(h * exp2_neg_int(se), 0.0f) & 0xFF);
          if (n < rt.nrows) {
            hq_base[(size_t)(rt.row0 + n) * a.f] = code;
            if (lane == 0) hsf_base[(n & 31) * 16 + (n >> 5) * 4] = (uint8_t)(se + 127);
          }
        }
      } else {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        const int dcol = mt * kMmaM + m;
#pragma unroll
        for (int n = 0; n < kBN; ++n) {
          if (n < rt.nrows) {
            const int r = rt.row0 + n;
            const float wr = a.row_w ? __ldg(&a.row_w[r]) : 1.0f;
            if (a.y_f32)
              a.y_f32[(size_t)r * a.d + dcol] = g[n] * wr;
            else
              a.y_bf16[(size_t)r * a.d + dcol] = __float2bfloat16_rn(g[n] * wr);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, C::kTmemCols);
}

template <int NMAT, int STAGES>
cudaError_t launch_grouped(const CUtensorMap& w, const CUtensorMap& w_sh, const CUtensorMap& act, const GemmArgs& a,
                           int num_sms, cudaStream_t s) {
  using C = Cfg<NMAT, STAGES>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(grouped_mx_gemm_kernel<NMAT, STAGES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  grouped_mx_gemm_kernel<NMAT, STAGES><<<num_sms, 192, C::kSmem, s>>>(w, w_sh, act, a);
  return cudaGetLastError();
}

constexpr int kStagesGateUp = 5;
constexpr int kStagesDown = 8;

}  // namespace

cudaError_t launch_gemm_gate_up(const CUtensorMap& w_routed, const CUtensorMap& w_shared, const uint8_t* sf_routed,
                                const uint8_t* sf_shared, const CUtensorMap& act, const uint8_t* act_sf,
                                const RowTile* tiles, const int32_t* n_tiles, int max_tiles, int E, int d, int f,
                                float limit, uint8_t* h_q, uint8_t* h_sf, int* status, uint64_t wait_budget_ns,
                                int stall_loads, int num_sms, cudaStream_t s) {
  GemmArgs a{};
  a.sf_routed = sf_routed;
  a.sf_shared = sf_shared ? sf_shared : sf_routed;
  a.act_sf = act_sf;
  a.tiles = tiles;
  a.n_tiles = n_tiles;
  a.max_tiles = max_tiles;
  a.E = E;
  a.KG = d / kKGroup;
  a.m_tiles = f / kMmaM;
  a.rows_per_expert = 2 * f;
  a.up_row_offset = f;
  a.w_mblocks = 2 * f / kMmaM;
  a.limit = limit;
  a.h_q = h_q;
  a.h_sf = h_sf;
  a.f = f;
  a.status = status;
  a.budget_ns = wait_budget_ns;
  a.stall_loads = stall_loads;
  return launch_grouped<2, kStagesGateUp>(w_routed, w_shared, act, a, num_sms, s);
}

cudaError_t launch_gemm_down(const CUtensorMap& w_routed, const CUtensorMap& w_shared, const uint8_t* sf_routed,
                             const uint8_t* sf_shared, const CUtensorMap& act, const uint8_t* act_sf,
                             const RowTile* tiles, const int32_t* n_tiles, int max_tiles, int E, int d, int f,
                             const float* row_w, float* y_f32, __nv_bfloat16* y_bf16, int* status,
                             uint64_t wait_budget_ns, int stall_loads, int num_sms, cudaStream_t s) {
  GemmArgs a{};
  a.sf_routed = sf_routed;
  a.sf_shared = sf_shared ? sf_shared : sf_routed;
  a.act_sf = act_sf;
  a.tiles = tiles;
  a.n_tiles = n_tiles;
  a.max_tiles = max_tiles;
  a.E = E;
  a.KG = f / kKGroup;
  a.m_tiles = d / kMmaM;
  a.rows_per_expert = d;
  a.up_row_offset = 0;
  a.w_mblocks = d / kMmaM;
  a.row_w = row_w;
  a.y_f32 = y_f32;
  a.y_bf16 = y_bf16;
  a.d = d;
  a.status = status;
  a.budget_ns = wait_budget_ns;
  a.stall_loads = stall_loads;
  return launch_grouped<1, kStagesDown>(w_routed, w_shared, act, a, num_sms, s);
}

}  // namespace moe
