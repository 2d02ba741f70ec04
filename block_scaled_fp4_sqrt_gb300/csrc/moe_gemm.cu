// Grouped expert GEMMs on 5th-generation tensor cores (tcgen05, kind::mxf8f6f4 with E8M0 block
// scales): MXFP8 activations x MXFP4 expert weights, fp32 accumulation in tensor memory.
//
//  * gate-up:  G = A . W1^T, U = A . W3^T per expert group; epilogue h = silu(min(G, L)) *
//    clamp(U, -L, L) (Ops.SiLUMulClamp, swiglu_limit = 10), re-quantised to MXFP8 along the FFN
//    dimension ("expert FFN (fused dequant + GEMM)", FaStar README "Features"; TensorSharp page
//    "How TensorSharp runs it").
//  * down:     Y = w_row * (H . W2^T) per permuted row, as fp16 with one power-of-two scale per 32
//    columns (summed in fp32 by the combine kernel, the weighted-sum epilogue moe_scatter_add of the
//    TensorSharp page, "DSpark and MoE CPU offload") or bf16 (the standalone grouped FFN call).
//
// Tile shape.  One MMA (M = 128, N <= 256, K = 32) takes the same time for any N, so the weights sit
// on the N side: 256 weight rows per MMA (gate 128 + up 128 of one 128-wide FFN slice, or 256 rows of
// the down projection), the token rows of one expert group (up to 128) on the M side.  Each MMA then
// consumes 4 KB of MXFP4 weights, enough to stream HBM at full rate even for a handful of tokens.
// The weights are stored tile-contiguous (see moe_api.cu), so every pipeline stage is one contiguous
// 16 KB TMA box.
//
// Two shapes of the pipeline: row tiles of up to 128 token rows with 4 stages, and -- for verify
// batches, whose expert groups hold a handful of rows -- row tiles of up to 32 rows whose activation
// slots are only 32 rows high, which leaves room for 6 stages.  The MMA still has M = 128: its rows
// 32..127 then read the following slots, whose products land in accumulator rows nobody stores (the
// activation ring sits in front of the weight ring, so those reads stay inside the CTA's smem).
//
// One persistent CTA per SM walks a device-built list of (row tile, output tile) work items.  Warp 0
// issues TMA loads, warp 1 the tcgen05 scale copies and MMAs, warps 2..17 drain the accumulator:
// four warps per 32-lane TMEM quadrant, each owning a quarter of the 256 columns, so one thread holds
// one token row of one MX block and needs no shuffles.  The accumulator is released as soon as it is
// in registers.  Every wait is bounded; on timeout the kernel records DEV_TIMEOUT and unwinds.
//
// MXFP4-activation variant (FP4 = true): activations and h are MXFP4 too, and the MMA is kind::mxf4
// (E2M1 x E2M1, K = 64, two scales per row and MMA).  Both operands stay packed in shared memory: a
// stage's K = 128 is one 64-byte row per operand row (64-byte swizzle), two MMAs per stage, so the
// weight ring takes half the shared memory and the tensor pipe does twice the work per instruction.
// The weights, their scale atoms and the activation scale atoms are the same as in the MXFP8 path.
#include <atomic>

#include "moe_device.cuh"

namespace moe {

namespace {

constexpr int kN = 256;         // weight rows per MMA (tcgen05 N)
constexpr int kBM = kTileRows;  // token rows per MMA (tcgen05 M) = 128
constexpr int kSmallRows = 32;  // groups this small load a 32-row activation box
constexpr int kEpiWarps = 16;
constexpr int kThreads = 64 + 32 * kEpiWarps;  // the CTA-pair kernel: producer, issuer, 16 epilogue warps

// The one-SM kernel's warps.  A warp reaches the TMEM lanes of quadrant (warp % 4) only, and warps with the
// same index mod 4 share one of the SM's four sub-partitions (issue slots).  Warp 1 issues the MMAs.
// In the 32-row shape only quadrant 0's four epilogue warps work, so the producer sits on another
// sub-partition: warp 2 produces, warp 16 idles, and the epilogue warps are four per quadrant
//   q0: 0 4 8 12   q1: 5 9 13 17   q2: 6 10 14 18   q3: 3 7 11 15   (column quarter = position in the list);
// that took the verify512 step from 0.628 to 0.618 ms (A/B on one box).  With 128-row tiles every quadrant
// works and both that placement and a 19th (idle) warp measured 0.5-1 % slower at T = 8192, so there the
// CTA keeps 18 warps: warp 0 produces and warps 2..17 drain (column quarter (warp - 2) / 4).
template <int AROWS>
struct Roles1 {
  static constexpr bool kSmall = AROWS == 32;
  static constexpr int kThreads = kSmall ? 19 * 32 : 18 * 32;
  static constexpr int kProducer = kSmall ? 2 : 0;
  static constexpr int kIdle = kSmall ? 16 : -1;
  __device__ static int quarter(int warp) {
    if (!kSmall) return (warp - 2) >> 2;
    const int q = warp & 3;
    return (warp - (q == 0 ? 0 : q == 1 ? 5 : q == 2 ? 6 : 3)) >> 2;
  }
};

// Staging buffer of one epilogue warp for coalesced expert-row stores: 8 rows of 128 bytes (the warp's 32
// rows pass through it 8 at a time), rows 144 B apart (36 words) so that the row-per-lane writes and the
// line-per-quarter-warp reads are both free of bank conflicts.  8 rows rather than 32 leave the shared
// memory to one more pipeline stage of the down GEMM.
// 128-row shape: the epilogue pauses every 8 h elements (gate-up) or after each staged pass (down).  Its 16
// warps share the SM's issue slots with the single MMA-issuing thread (warp 1, the sub-partition of
// quadrant 1's warps) and the TMA producer (warp 0, quadrant 0's); spreading their work over the item
// instead of running it in one burst after each handoff shortens the items.  Measured on the prefill step
// (A/B on one box): no pause 1.404 ms; 300 ns for every warp 1.398; 400 ns beside the producer and the
// issuer with 100 ns elsewhere 1.383 (600 / 0 ns: 1.391).  A down item leaves about 3 us of slack for its
// epilogue.
constexpr uint32_t kEpiNapNear = 400;  // quadrants 0 and 1
constexpr uint32_t kEpiNapFar = 100;   // quadrants 2 and 3

constexpr int kStageStride = 36;
constexpr int kStageRows = 8;
constexpr int kStageFloats = kStageRows * kStageStride;

// EPI = 1: the down projection's expert rows leave through a per-warp shared-memory transpose (full
// 128-byte lines per quarter warp) instead of 16-byte stores to 32 different rows per instruction.
// FP4: packed MXFP4 operands (64-byte rows, kind::mxf4) instead of E4M3 x byte-expanded E2M1.
template <int STAGES, int AROWS, int EPI = 0, bool FP4 = false>
struct Cfg {
  static constexpr int kRowBytes = FP4 ? 64 : 128;   // one operand row of a stage (K = 128) in smem
  static constexpr uint32_t kSwizzle = FP4 ? 4 : 2;  // descriptor layout: 64- or 128-byte swizzle
  static constexpr uint32_t kSbo = 8 * kRowBytes;    // stride of the 8-row core groups
  static constexpr int kASlot = AROWS * kRowBytes;   // activation rows x 128 FP8 (or FP4)
  static constexpr int kBSlot = kN * kRowBytes;      // 256 weight rows x 128 FP4 (padded to bytes, or packed)
  static constexpr int kSfSlot = 3 * kSfAtomBytes;   // activation atom + two weight atoms
  static constexpr int kAOff = 0;                    // [activation ring | weight ring | scale ring]
  static constexpr int kBOff = STAGES * kASlot;
  static constexpr int kSfOff = kBOff + STAGES * kBSlot;
  static constexpr int kEpiOff = kSfOff + STAGES * kSfSlot;  // [ ... | scale ring | staging | barriers]
  static constexpr int kEpiBytes = EPI ? kEpiWarps * kStageFloats * 4 : 0;
  static constexpr int kBarOff = kEpiOff + kEpiBytes;
  static constexpr int kBarBytes = (2 * STAGES + 3) * 8;
  static constexpr int kSmem = kBarOff + 1024 + kBarBytes;
  static constexpr uint32_t kTxB = kN * 64 + 2 * kSfAtomBytes;  // packed FP4 box (64 B per row) + weight atoms
  static constexpr int kAccCols = kN;                           // one fp32 accumulator [128 x 256]
  static constexpr int kSfCols = 12;                            // per stage: A atom 4 columns, B atoms 8
  static constexpr int kTmemCols = 512;
  // warps that drain the accumulator: with rows only in TMEM lanes 0..31, the four warps of quadrant 0
  static constexpr int kDrainWarps = AROWS == kSmallRows ? kEpiWarps / 4 : kEpiWarps;
  static_assert(kBOff % 1024 == 0 && kSfOff % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(AROWS == kBM || kBOff >= (kBM - AROWS) * kRowBytes, "M = 128 reads past a short activation slot");
  static_assert(kAccCols + STAGES * kSfCols <= kTmemCols, "TMEM budget");
  static_assert(kEpiOff % 16 == 0, "staging rows are float4-aligned");
  static_assert(kSmem <= 232448 - 64, "shared memory budget");
};

struct GemmArgs {
  const uint8_t* sf_routed;  // weight scale atoms [E, KG, m_tiles, 2, 512]
  const uint8_t* sf_shared;  // [1, KG, m_tiles, 2, 512]
  const uint8_t* act_sf;     // activation scale atoms [tile, KG, 512]
  const RowTile* tiles;
  const int32_t* n_tiles;
  int max_tiles;
  int E;        // group E is the shared expert
  int KG;       // K / 128
  int m_tiles;  // 256-wide output tiles per row tile (f/128 gate-up slices, or d/256)
  int gate_up;  // 1: SwiGLU + MXFP8 epilogue; 0: weighted rows (scaled fp16, or bf16)
  // gate-up epilogue
  float limit;
  uint8_t* h_q;
  uint8_t* h_sf;
  int f;
  // down epilogue: exactly one of y16.val / y_bf16 is set
  const float* row_w;
  ExpertRows y16;
  __nv_bfloat16* y_bf16;
  int d;
  int* status;
  uint64_t budget_ns;
  int stall_loads;  // test hook: issue no loads, so the consumers' bounded waits run out
};

// silu(z) = z / (1 + e^-z) with the hardware exponential and reciprocal (__expf, __fdividef): a few
// instructions instead of the IEEE-exact sequences.  Their relative error (about 1e-6) is far below the
// MXFP8 step of h (2^-3), so it moves an h code only where h sits within that distance of a rounding
// midpoint.  The epilogue warps share the SM's issue slots with the MMA-issuing thread, whose issue rate
// bounds the grouped GEMMs, so fewer epilogue instructions mean faster MMA issue.  For z below about -88,
// e^-z overflows to infinity and the quotient is -0, the limit of silu.
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// The epilogue of one work item for one warp: the warp's 32 token rows (TMEM lane quadrant q) and its
// column quarter c of the accumulator, already in registers (v0, v1), for row tile `ti` (rows rt) and
// output tile mt.  Gate-up: SwiGLU with clamp, then the MX requantisation of h; down: the routing-weighted
// rows, as scaled fp16 (ExpertRows) through the warp's staging buffer stg (EPI) or direct, or as bf16.
template <int EPI, bool FP4>
__device__ __forceinline__ void epilogue_rows(const GemmArgs& a, const RowTile& rt, int ti, int mt, int q, int c,
                                              int lane, float* stg, bool active, float (&v0)[32], float (&v1)[32],
                                              uint32_t nap = 0) {
  const int lr = q * 32 + lane;  // token row inside the tile
  if (EPI && !a.gate_up) {
    // scaled fp16 rows through the warp's staging buffer
    if (active) {
      const bool row_ok = lr < rt.nrows;
      const float wr = !row_ok ? 0.f : (a.row_w ? __ldg(&a.row_w[rt.row0 + lr]) : 1.0f);
      // this lane's row: 64 columns, 128 bytes, packed into v0[0..15] and v1[0..15]
      const uint32_t e0 = row16_encode32(v0, wr), e1 = row16_encode32(v1, wr);
      __half* ybase = a.y16.val + (size_t)rt.row0 * a.d + (size_t)mt * kN + 64 * c;
      // lanes 8p .. 8p+7 write their rows' 128 bytes into the buffer; then each quarter warp stores one
      // buffered row (four rows per pass and instruction, two instructions per pass)
#pragma unroll
      for (int p = 0; p < 32 / kStageRows; ++p) {
        if ((lane >> 3) == p) {
          uint4* srow = reinterpret_cast<uint4*>(stg + (lane & 7) * kStageStride);
#pragma unroll
          for (int i = 0; i < 4; ++i) srow[i] = row16_words(v0, i);
#pragma unroll
          for (int i = 0; i < 4; ++i) srow[4 + i] = row16_words(v1, i);
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int br = 4 * i + (lane >> 3);  // buffered row
          const int rr = q * 32 + 8 * p + br;  // row inside the tile
          const uint4 val = reinterpret_cast<const uint4*>(stg + br * kStageStride)[lane & 7];
          if (rr < rt.nrows) reinterpret_cast<uint4*>(ybase + (size_t)rr * a.d)[lane & 7] = val;
        }
        __syncwarp();
        if (nap) __nanosleep(nap);
      }
      if (row_ok)
        *reinterpret_cast<uint16_t*>(a.y16.exp + (size_t)(rt.row0 + lr) * (a.d / 32) + mt * (kN / 32) + 2 * c) =
            (uint16_t)(e0 | (e1 << 8));
    }
    return;
  }
  if (!active || lr >= rt.nrows) return;
  const int r = rt.row0 + lr;
  if (a.gate_up) {
    const float L = a.limit;
    float* h = v0;  // h overwrites the gate values in place
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float gc = fminf(v0[j], L);
      const float uc = fminf(fmaxf(v1[j], -L), L);
      h[j] = silu_f(gc) * uc;
      amax = fmaxf(amax, fabsf(h[j]));
      if (nap && (j & 7) == 7) __nanosleep(nap);
    }
    const int se = FP4 ? mxfp4_block_exp(amax) : mxfp8_block_exp(amax);
    const float mul = exp2_neg_int(se);
    if (FP4) {  // 32 E2M1 codes: 16 bytes at h column mt * 128 + 32 c of a row of f / 2 bytes
      *reinterpret_cast<uint4*>(a.h_q + (size_t)r * (a.f / 2) + mt * (kKGroup / 2) + 16 * c) = e2m1_block(v0, mul);
    } else {
      uint32_t packed[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t lo = e4m3x2(h[4 * i] * mul, h[4 * i + 1] * mul);
        const uint32_t hi = e4m3x2(h[4 * i + 2] * mul, h[4 * i + 3] * mul);
        packed[i] = lo | (hi << 16);
      }
      uint4* dst = reinterpret_cast<uint4*>(a.h_q + (size_t)r * a.f + mt * kKGroup + 32 * c);
      dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    }
    a.h_sf[((size_t)ti * (a.f / kKGroup) + mt) * kSfAtomBytes + (lr & 31) * 16 + (lr >> 5) * 4 + c] =
        (uint8_t)(se + 127);
  } else {
    const float wr = a.row_w ? __ldg(&a.row_w[r]) : 1.0f;
    const size_t col0 = (size_t)mt * kN + 64 * c;
    if (a.y16.val) {
      const uint32_t e0 = row16_encode32(v0, wr), e1 = row16_encode32(v1, wr);
      uint4* dst = reinterpret_cast<uint4*>(a.y16.val + (size_t)r * a.d + col0);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = row16_words(v0, i);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[4 + i] = row16_words(v1, i);
      *reinterpret_cast<uint16_t*>(a.y16.exp + (size_t)r * (a.d / 32) + col0 / 32) = (uint16_t)(e0 | (e1 << 8));
    } else {
      uint4* dst = reinterpret_cast<uint4*>(a.y_bf16 + (size_t)r * a.d + col0);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float* src = i < 4 ? &v0[8 * i] : &v1[8 * (i - 4)];
        uint4 o;
        __nv_bfloat162* ov = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
        for (int p = 0; p < 4; ++p) ov[p] = __floats2bfloat162_rn(src[2 * p] * wr, src[2 * p + 1] * wr);
        dst[i] = o;
      }
    }
  }
}

template <int STAGES, int AROWS, int EPI, bool FP4>
__global__ void __launch_bounds__(Roles1<AROWS>::kThreads, 1)
    grouped_mx_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_w_shared,
                           const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_act_small,
                           const GemmArgs a) {
  using C = Cfg<STAGES, AROWS, EPI, FP4>;
  // The accumulator handoff: the issuer polls acc_empty in both shapes (one thread, nothing else to do).
  // The epilogue warps poll acc_full in the 32-row shape: there only the issuer and four epilogue warps
  // run, and polling took 4 % off the T = 8 step (measured).  With 128-row tiles the 16 polling epilogue
  // warps took issue slots from the producer and issuer (the T = 8192 step 2 % slower), so they suspend.
  constexpr bool kPollHandoff = AROWS == kSmallRows;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  // No pdl_trigger() here: letting the next kernel's CTAs in while the GEMM still runs slowed the
  // T = 8192 step by 4 % (measured); they launch when the GEMM completes.
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, C::kDrainWarps);
    mbar_init(drain, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    prefetch_tensormap(&tm_w);
    prefetch_tensormap(&tm_w_shared);
    prefetch_tensormap(&tm_act);
    prefetch_tensormap(&tm_act_small);
  }
  if (warp == 1) tmem_alloc(&tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  // the work list and the activations come from earlier kernels
  pdl_wait();
  int n_tiles = *reinterpret_cast<const volatile int32_t*>(a.n_tiles);
  if (n_tiles > a.max_tiles) n_tiles = a.max_tiles;
  const int total = n_tiles * a.m_tiles;

  using R = Roles1<AROWS>;
  if (warp == R::kProducer) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      // weights: streamed once by the 32-row (verify) shape; with 128-row tiles an expert's slab is read by
      // each of its row tiles, which the CTAs walk at about the same time, so let those reads hit in L2
      const uint64_t pol_w = AROWS == kSmallRows ? l2_policy_evict_first() : l2_policy_evict_normal();
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
        const bool small = AROWS == kSmallRows || rt.nrows <= kSmallRows;
        const CUtensorMap* ta = small ? &tm_act_small : &tm_act;
        const uint32_t tx = C::kTxB + (small ? kSmallRows : kBM) * C::kRowBytes + kSfAtomBytes;
        // packed weights are [expert][K group][output tile][256 rows]: slab (e, kg, mt)
        const int wrow0 = (e * a.KG * a.m_tiles + mt) * kN;
        const int wrow_kg = a.m_tiles * kN;
        const uint8_t* sfw = (sh ? a.sf_shared : a.sf_routed) + ((size_t)e * a.KG * a.m_tiles + mt) * 2 * kSfAtomBytes;
        const size_t sfw_kg = (size_t)a.m_tiles * 2 * kSfAtomBytes;
        const uint8_t* sfa = a.act_sf + (size_t)ti * a.KG * kSfAtomBytes;
        for (int kg = 0; kg < a.KG; ++kg) {
          if (abort_flag || !mbar_wait(&empty[stage], phase ^ 1u, a.budget_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], tx);
          tma_load_2d(smem + C::kBOff + stage * C::kBSlot, tw, 0, wrow0 + kg * wrow_kg, &full[stage], pol_w);
          tma_load_2d(smem + C::kAOff + stage * C::kASlot, ta, kg * C::kRowBytes, rt.row0, &full[stage], pol_a);
          uint8_t* sf = smem + C::kSfOff + stage * C::kSfSlot;
          bulk_load(sf, sfa + kg * kSfAtomBytes, kSfAtomBytes, &full[stage]);
          bulk_load(sf + kSfAtomBytes, sfw + kg * sfw_kg, 2 * kSfAtomBytes, &full[stage]);
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
      // A = activations (E4M3, or E2M1), B = weights (E2M1).  The tensor pipe queues only a couple of MMAs, so
      // this thread's instruction stream is on the critical path: descriptors are precomputed,
      // slots and phases advance incrementally (the same stage sequence as the producer's), and the
      // stage's four MMAs, its commit and a barrier test are one fused instruction block.  A scale
      // copy or a barrier wait right in front of the MMAs that depend on it also leaves the pipe idle,
      // so the scale atoms of a stage are copied into TMEM as soon as the stage is seen to have
      // landed (tested inside the MMA block of an earlier stage, up to kAhead stages ahead); only a
      // stage that has not landed by the time its MMAs are due is waited for in front of them.
      constexpr uint32_t kIdesc0 = FP4 ? mma_idesc(kMxf4E2M1, kMxf4E2M1, kBM, kN, 0, 0) : mma_idesc(0, 5, kBM, kN, 0, 0);
      constexpr int kAhead = 2;
      static_assert(STAGES > kAhead, "scale copies run up to kAhead stages ahead of the MMAs");
      const uint64_t a_desc0 = smem_desc(smem_addr(smem + C::kAOff), 16, C::kSbo, C::kSwizzle);
      const uint64_t b_desc0 = smem_desc(smem_addr(smem + C::kBOff), 16, C::kSbo, C::kSwizzle);
      const uint64_t sf_desc0 = smem_desc(smem_addr(smem + C::kSfOff), 128, 128, 0);
      const uint32_t sf_tmem0 = tbase + (uint32_t)C::kAccCols;
      auto copy_sf = [&](int slot) {  // activation atom, then the two weight atoms (512 B apart)
        const uint64_t dsc = sf_desc0 + (uint64_t)((slot * C::kSfSlot) >> 4);
        const uint32_t t = sf_tmem0 + (uint32_t)(slot * C::kSfCols);
        tc_copy_sf(t, dsc);
        tc_copy_sf(t + 4, dsc + (kSfAtomBytes >> 4));
        tc_copy_sf(t + 8, dsc + 2 * (kSfAtomBytes >> 4));
      };
      const int n_items = total > (int)blockIdx.x ? (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
      const int n_st = n_items * a.KG;
      bool ok = true, any = false;
      int cs = 0;          // slot of the stage being consumed
      uint32_t cph = 0;    // its phase
      int lg = 0, ls = 0;  // first stage whose scales are not in TMEM yet, and its slot / phase
      uint32_t lph = 0;
      int g = 0, kg = 0, item = 0;
      // The inner loop issues stages back to back and holds no branch with a wait loop inside: such a
      // branch, even never taken, slowed the MMA issue by a fifth (measured).  A work item's start (the
      // accumulator handoff) and a stage whose scales are not in TMEM yet leave it for the outer loop.
      while (g < n_st) {
        if (kg == 0) {  // a new work item: the epilogue must have drained the accumulator
          const uint32_t par = ((uint32_t)item & 1u) ^ 1u;
          if (abort_flag || !mbar_spin(acc_empty, par, a.budget_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (lg == g) {  // this stage has not been seen yet: wait for it
          if (abort_flag || !mbar_wait(&full[ls], lph, a.budget_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          copy_sf(ls);
          ++lg;
          if (++ls == STAGES) {
            ls = 0;
            lph ^= 1u;
          }
        }
        for (;;) {
          const bool look = lg < n_st && lg <= g + kAhead;
          // with nothing to look ahead for, the test re-reads this stage's own (completed) barrier
          const uint64_t ad = a_desc0 + (uint64_t)((cs * C::kASlot) >> 4);
          const uint64_t bd = b_desc0 + (uint64_t)((cs * C::kBSlot) >> 4);
          const uint32_t sfa = sf_tmem0 + (uint32_t)(cs * C::kSfCols);
          const bool landed =
              FP4 ? tc_stage2_mxf4_commit_poll(tbase, ad, bd, kIdesc0, sfa, sfa + 4, kg != 0 ? 1u : 0u, &empty[cs],
                                               look ? &full[ls] : &full[cs], look ? lph : cph)
                  : tc_stage4_mx_commit_poll(tbase, ad, bd, kIdesc0, sfa, sfa + 4, kg != 0 ? 1u : 0u, &empty[cs],
                                             look ? &full[ls] : &full[cs], look ? lph : cph);
          any = true;
          if (look && landed) {
            tc_fence_after();
            copy_sf(ls);
            ++lg;
            if (++ls == STAGES) {
              ls = 0;
              lph ^= 1u;
            }
          }
          if (++cs == STAGES) {
            cs = 0;
            cph ^= 1u;
          }
          ++g;
          if (++kg == a.KG) {
            tc_commit(acc_full);
            kg = 0;
            ++item;
            break;
          }
          if (lg == g) break;
        }
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
  } else if (warp != R::kIdle) {
    // ------------------------------------------------------------------ epilogue (16 warps)
    const int q = warp & 3;         // TMEM lane quadrant: token rows 32q .. 32q+31
    const int c = R::quarter(warp); // column quarter
    const int lr = q * 32 + lane;       // token row inside the tile
    int it = 0;
    // 32-row tiles keep their rows in TMEM lanes 0..31: the other quadrants' warps have nothing to do
    const int my_total = (AROWS == kSmallRows && q != 0) ? 0 : total;
    for (int w = blockIdx.x; w < my_total; w += gridDim.x, ++it) {
      bool got = !abort_flag && (kPollHandoff ? mbar_spin(acc_full, (uint32_t)it & 1u, a.budget_ns)
                                              : mbar_wait(acc_full, (uint32_t)it & 1u, a.budget_ns));
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
      const bool active = q * 32 < rt.nrows;  // warp-uniform
      const uint32_t tl = tbase + ((uint32_t)(q * 32) << 16);
      float v0[32], v1[32];
      if (active) {
        // gate-up: gate columns 32c.., up columns 128+32c..; down: columns 64c .. 64c+63
        tmem_ld32(tl + (uint32_t)(a.gate_up ? 32 * c : 64 * c), v0);
        tmem_ld32(tl + (uint32_t)(a.gate_up ? 128 + 32 * c : 64 * c + 32), v1);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      epilogue_rows<EPI, FP4>(a, rt, ti, mt, q, c, lane,
                              reinterpret_cast<float*>(smem + C::kEpiOff) + (4 * q + c) * kStageFloats, active, v0,
                              v1, AROWS == kBM ? (q <= 1 ? kEpiNapNear : kEpiNapFar) : 0u);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, C::kTmemCols);
}

// ---------------------------------------------------------------------------------------------------
// CTA-pair shape for large expert groups (the prefill chunk): a cluster of two CTAs on two SMs runs every
// work item as one M = 256 tcgen05.mma.cta_group::2 per K step.  The even CTA (the leader) issues the
// MMAs; each CTA holds 128 of the 256 token rows (two consecutive 128-row tiles of one expert group) and
// 128 of the 256 weight rows (gate 128 | up 128 of one FFN slice, or 256 down rows), and receives its own
// 128 rows of the [256 x 256] fp32 accumulator in its tensor memory.  Against the one-SM kernel each SM
// stores and reads half the weight tile per stage (16 KB instead of 32 KB of byte-expanded FP4), which
// leaves room for 6 stages instead of 4, and pulls half the weight bytes from L2.
//
// Both CTAs' TMA loads of a stage (weights, activations, and the scale atoms through 2-D maps of
// 256-byte rows) count their bytes on the leader's `full` barrier (the .cta_group::2 form of the copy);
// the leader's commits arrive on both CTAs' `empty` and `acc_full` barriers (multicast); the peer's
// epilogue warps arrive on the leader's `acc_empty` barrier across the cluster.  Every tcgen05 operation
// of the kernel uses cta_group::2.  Each CTA's tensor memory holds the scale atoms of the whole N = 256
// (both weight atoms) and of its own 128 activation rows.  The work list pads every expert group to an
// even number of row tiles, so the two tiles of a pair always belong to the same group.
template <int STAGES, int EPI>
struct PairCfg {
  static constexpr int kRowBytes = 128;                   // one operand row of a stage (K = 128) in smem
  static constexpr uint32_t kSbo = 8 * kRowBytes;
  static constexpr int kASlot = kBM * kRowBytes;          // this CTA's 128 token rows
  static constexpr int kBSlot = (kN / 2) * kRowBytes;     // this CTA's 128 weight rows (FP4 expanded to bytes)
  static constexpr int kSfSlot = 3 * kSfAtomBytes;        // activation atom, then the two weight atoms
  static constexpr int kAOff = 0;
  static constexpr int kBOff = STAGES * kASlot;
  static constexpr int kSfOff = kBOff + STAGES * kBSlot;
  static constexpr int kEpiOff = kSfOff + STAGES * kSfSlot;
  static constexpr int kEpiBytes = EPI ? kEpiWarps * kStageFloats * 4 : 0;
  static constexpr int kBarOff = kEpiOff + kEpiBytes;
  static constexpr int kBarBytes = (2 * STAGES + 3) * 8;
  static constexpr int kSmem = kBarOff + 1024 + kBarBytes;
  // bytes one CTA's loads of a stage move (global side): packed FP4 weights, activations, three atoms
  static constexpr uint32_t kTxCta = (kN / 2) * 64 + kBM * kRowBytes + 3 * kSfAtomBytes;
  static constexpr int kAccCols = kN;
  static constexpr int kSfCols = 12;
  static constexpr int kTmemCols = 512;
  static_assert(kBOff % 1024 == 0 && kSfOff % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(kAccCols + STAGES * kSfCols <= kTmemCols, "TMEM budget");
  static_assert(kEpiOff % 16 == 0, "staging rows are float4-aligned");
  static_assert(kSmem <= 232448 - 64, "shared memory budget");
};

template <int STAGES, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_mx_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_w_shared,
                                const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_sfw,
                                const __grid_constant__ CUtensorMap tm_sfw_shared,
                                const __grid_constant__ CUtensorMap tm_sfa, const GemmArgs a) {
  using C = PairCfg<STAGES, EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = (int)(blockIdx.x >> 1), n_pairs = (int)(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);  // the leader's producer (expect_tx of both CTAs' bytes); unused in the peer
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * kEpiWarps);  // drain warps of both CTAs; only the leader's is used
    mbar_init(drain, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    prefetch_tensormap(&tm_w);
    prefetch_tensormap(&tm_w_shared);
    prefetch_tensormap(&tm_act);
    prefetch_tensormap(&tm_sfw);
    prefetch_tensormap(&tm_sfw_shared);
    prefetch_tensormap(&tm_sfa);
  }
  if (warp == 1) tmem_alloc_pair(&tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  pdl_wait();
  int n_tiles = *reinterpret_cast<const volatile int32_t*>(a.n_tiles);
  if (n_tiles > a.max_tiles) n_tiles = a.max_tiles;
  const int total = (n_tiles >> 1) * a.m_tiles;  // work items: (tile pair, output tile)
  const int n_items = total > pair ? (total - pair + n_pairs - 1) / n_pairs : 0;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer (both CTAs)
      const uint64_t pol_w = l2_policy_evict_normal();  // an expert's slab is read by each of its tile pairs
      const uint64_t pol_a = l2_policy_evict_last();
      const uint32_t full0 = mapa_shared(smem_addr(&full[0]), 0);  // the leader's barriers
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_par = 0;
      bool ok = true;
      for (int w = pair; w < total && ok && !a.stall_loads; w += n_pairs) {
        const int pi = w / a.m_tiles, mt = w - pi * a.m_tiles;
        const int ti = 2 * pi + (int)rank;  // this CTA's row tile
        const RowTile rt = a.tiles[ti];
        const int g = a.tiles[2 * pi].group;
        const bool sh = g == a.E;
        const CUtensorMap* tw = sh ? &tm_w_shared : &tm_w;
        const CUtensorMap* tsw = sh ? &tm_sfw_shared : &tm_sfw;
        const int e = sh ? 0 : g;
        const int slab = e * a.KG * a.m_tiles + mt;  // packed weights [expert][K group][output tile]
        for (int kg = 0; kg < a.KG; ++kg) {
          if (abort_flag || !mbar_wait(&empty[stage], phase ^ 1u, a.budget_ns)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * C::kTxCta);
          const uint32_t fb = full0 + (uint32_t)(stage * 8);
          const int sl = slab + kg * a.m_tiles;
          tma_load_2d_pair(smem + C::kBOff + stage * C::kBSlot, tw, 0, sl * kN + (int)rank * (kN / 2), fb, pol_w);
          tma_load_2d_pair(smem + C::kAOff + stage * C::kASlot, &tm_act, kg * C::kRowBytes, rt.row0, fb, pol_a);
          uint8_t* sf = smem + C::kSfOff + stage * C::kSfSlot;
          tma_load_2d_pair(sf, &tm_sfa, 0, 2 * (ti * a.KG + kg), fb, pol_a);  // one atom: 2 rows of 256 B
          tma_load_2d_pair(sf + kSfAtomBytes, tsw, 0, 4 * sl, fb, pol_w);     // two atoms: 4 rows
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
        // the leader's barriers count both CTAs' copies: let those in flight land before shared memory goes
        if (leader)
          for (int s = 0; s < STAGES; ++s)
            if ((issued >> s) & 1u) (void)mbar_wait(&full[s], (last_par >> s) & 1u, 20000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------------- MMA issuer (leader only)
      // The one-SM issuer's structure (fused stage blocks, scale copies up to kAhead stages early) with the
      // pair's forms: M = 256, commits multicast to both CTAs.
      constexpr uint32_t kIdesc0 = mma_idesc(0, 5, 2 * kBM, kN, 0, 0);
      constexpr int kAhead = 2;
      static_assert(STAGES > kAhead, "scale copies run up to kAhead stages ahead of the MMAs");
      const uint64_t a_desc0 = smem_desc(smem_addr(smem + C::kAOff), 16, C::kSbo, 2);
      const uint64_t b_desc0 = smem_desc(smem_addr(smem + C::kBOff), 16, C::kSbo, 2);
      const uint64_t sf_desc0 = smem_desc(smem_addr(smem + C::kSfOff), 128, 128, 0);
      const uint32_t sf_tmem0 = tbase + (uint32_t)C::kAccCols;
      auto copy_sf = [&](int slot) {
        const uint64_t dsc = sf_desc0 + (uint64_t)((slot * C::kSfSlot) >> 4);
        const uint32_t t = sf_tmem0 + (uint32_t)(slot * C::kSfCols);
        tc_copy_sf_pair(t, dsc);
        tc_copy_sf_pair(t + 4, dsc + (kSfAtomBytes >> 4));
        tc_copy_sf_pair(t + 8, dsc + 2 * (kSfAtomBytes >> 4));
      };
      const int n_st = n_items * a.KG;
      bool ok = true, any = false;
      int cs = 0;
      uint32_t cph = 0;
      int lg = 0, ls = 0;
      uint32_t lph = 0;
      int g = 0, kg = 0, item = 0;
      while (g < n_st) {  // the one-SM issuer's loop structure: waits only in the outer loop
        if (kg == 0) {  // both CTAs' epilogues must have drained the accumulator
          if (abort_flag || !mbar_wait_cluster(acc_empty, ((uint32_t)item & 1u) ^ 1u, a.budget_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (lg == g) {
          if (abort_flag || !mbar_wait(&full[ls], lph, a.budget_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          copy_sf(ls);
          ++lg;
          if (++ls == STAGES) {
            ls = 0;
            lph ^= 1u;
          }
        }
        for (;;) {
          const bool look = lg < n_st && lg <= g + kAhead;
          const uint64_t ad = a_desc0 + (uint64_t)((cs * C::kASlot) >> 4);
          const uint64_t bd = b_desc0 + (uint64_t)((cs * C::kBSlot) >> 4);
          const uint32_t sfa = sf_tmem0 + (uint32_t)(cs * C::kSfCols);
          const bool landed = tc_stage4_mx_pair_commit_poll(tbase, ad, bd, kIdesc0, sfa, sfa + 4, kg != 0 ? 1u : 0u,
                                                            &empty[cs], look ? &full[ls] : &full[cs],
                                                            look ? lph : cph);
          any = true;
          if (look && landed) {
            tc_fence_after();
            copy_sf(ls);
            ++lg;
            if (++ls == STAGES) {
              ls = 0;
              lph ^= 1u;
            }
          }
          if (++cs == STAGES) {
            cs = 0;
            cph ^= 1u;
          }
          ++g;
          if (++kg == a.KG) {
            tc_commit_pair(acc_full);
            kg = 0;
            ++item;
            break;
          }
          if (lg == g) break;
        }
      }
      if (!ok) {
        set_status(a.status, DEV_TIMEOUT);
        abort_flag = 1;
      }
      if (any) {  // all issued MMAs must retire before either CTA releases its tensor memory
        tc_commit_pair(drain);
        if (!mbar_wait(drain, 0, a.budget_ns)) set_status(a.status, DEV_TIMEOUT);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..17, both CTAs)
    const int q = warp & 3;
    const int c = (warp - 2) >> 2;
    const uint32_t acc_empty_leader = mapa_shared(smem_addr(acc_empty), 0);
    int it = 0;
    for (int w = pair; w < total; w += n_pairs, ++it) {
      bool got = !abort_flag && mbar_wait(acc_full, (uint32_t)it & 1u, a.budget_ns);
      got = __all_sync(0xFFFFFFFFu, got);
      if (!got) {
        if (lane == 0) {
          set_status(a.status, DEV_TIMEOUT);
          abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const int pi = w / a.m_tiles, mt = w - pi * a.m_tiles;
      const int ti = 2 * pi + (int)rank;
      const RowTile rt = a.tiles[ti];
      const bool active = q * 32 < rt.nrows;  // warp-uniform
      const uint32_t tl = tbase + ((uint32_t)(q * 32) << 16);
      float v0[32], v1[32];
      if (active) {
        tmem_ld32(tl + (uint32_t)(a.gate_up ? 32 * c : 64 * c), v0);
        tmem_ld32(tl + (uint32_t)(a.gate_up ? 128 + 32 * c : 64 * c + 32), v1);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(acc_empty);
        else
          mbar_arrive_remote(acc_empty_leader);
      }
      epilogue_rows<EPI, false>(a, rt, ti, mt, q, c, lane,
                                reinterpret_cast<float*>(smem + C::kEpiOff) + (warp - 2) * kStageFloats, active, v0,
                                v1);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA releases its tensor or shared memory while the pair still uses them
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tbase, C::kTmemCols);
}

template <int STAGES, int AROWS, int EPI, bool FP4>
cudaError_t launch_shape(const CUtensorMap& w, const CUtensorMap& w_sh, const CUtensorMap& act,
                         const CUtensorMap& act_small, const GemmArgs& a, int num_sms, cudaStream_t s) {
  using C = Cfg<STAGES, AROWS, EPI, FP4>;
  static PerDeviceOnce smem_optin;
  const cudaError_t e = smem_optin.run([] {
    return cudaFuncSetAttribute(grouped_mx_gemm_kernel<STAGES, AROWS, EPI, FP4>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(grouped_mx_gemm_kernel<STAGES, AROWS, EPI, FP4>, dim3(num_sms), dim3(Roles1<AROWS>::kThreads),
                    C::kSmem, s, w, w_sh, act, act_small, a);
}

// CTA-pair launch: clusters of two CTAs with programmatic dependent launch.  The grid is as many pairs as
// the device co-schedules at one CTA per SM (the occupancy query, once per device), at most num_sms / 2.
template <int STAGES, int EPI>
cudaError_t launch_pair(const PairMaps& pm, const CUtensorMap& act, const GemmArgs& a, int num_sms, cudaStream_t s) {
  using C = PairCfg<STAGES, EPI>;
  auto kernel = grouped_mx_gemm_pair_kernel<STAGES, EPI>;
  static PerDeviceOnce smem_optin;
  cudaError_t e = smem_optin.run(
      [&] { return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem); });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  static std::atomic<int> pairs_cached[64];  // per device; 0 = not queried yet
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int pairs = dev >= 0 && dev < 64 ? pairs_cached[dev].load(std::memory_order_relaxed) : 0;
  if (pairs == 0) {
    cfg.gridDim = dim3(2 * (num_sms / 2));
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) return e;
    pairs = n < 1 ? 1 : (n > num_sms / 2 ? num_sms / 2 : n);
    if (dev >= 0 && dev < 64) pairs_cached[dev].store(pairs, std::memory_order_relaxed);
  }
  cfg.gridDim = dim3(2 * pairs);
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, pm.w, pm.w_shared, act, pm.sfw, pm.sfw_shared, pm.sfa, a);
}

// tile_rows 32: 6 stages of 32-row activation slots.  tile_rows 128: 4 stages of 128-row slots, also for
// the down projection's expert rows next to the epilogue's staging buffers (the 16-byte scattered
// stores of a direct epilogue bounded that GEMM at the 8192-token shape: 835 us with them, 373 us
// without any stores).
// FP4: the packed weight ring is half as large, so every shape holds more stages.
// pair (128-row tiles, MXFP8 activations): the CTA-pair kernel, 6 stages for gate-up and for the down
// projection's expert rows (next to their staging buffers); 5 stages for bf16 down rows (the grouped FFN
// call).
cudaError_t launch_grouped(const CUtensorMap& w, const CUtensorMap& w_sh, const CUtensorMap& act,
                           const CUtensorMap& act_small, const GemmArgs& a, int tile_rows, int act_fp4, int num_sms,
                           cudaStream_t s, const PairMaps* pair) {
  if (pair && tile_rows == kBM && !act_fp4) {
    if (a.gate_up) return launch_pair<6, 0>(*pair, act, a, num_sms, s);
    if (a.y16.val) return launch_pair<6, 1>(*pair, act, a, num_sms, s);
    return launch_pair<5, 0>(*pair, act, a, num_sms, s);
  }
  if (act_fp4) {
    if (tile_rows == kSmallRows) return launch_shape<8, kSmallRows, 0, true>(w, w_sh, act, act_small, a, num_sms, s);
    if (!a.gate_up && a.y16.val) return launch_shape<8, kBM, 1, true>(w, w_sh, act, act_small, a, num_sms, s);
    return launch_shape<8, kBM, 0, true>(w, w_sh, act, act_small, a, num_sms, s);
  }
  if (tile_rows == kSmallRows) return launch_shape<6, kSmallRows, 0, false>(w, w_sh, act, act_small, a, num_sms, s);
  if (!a.gate_up && a.y16.val) return launch_shape<4, kBM, 1, false>(w, w_sh, act, act_small, a, num_sms, s);
  return launch_shape<4, kBM, 0, false>(w, w_sh, act, act_small, a, num_sms, s);
}

}  // namespace

cudaError_t launch_gemm_gate_up(const CUtensorMap& w_routed, const CUtensorMap& w_shared, const uint8_t* sf_routed,
                                const uint8_t* sf_shared, const CUtensorMap& act, const CUtensorMap& act_small,
                                const uint8_t* act_sf, const RowTile* tiles, const int32_t* n_tiles, int max_tiles,
                                int E, int d, int f, float limit, uint8_t* h_q, uint8_t* h_sf, int* status,
                                uint64_t wait_budget_ns, int stall_loads, int tile_rows, int act_fp4, int num_sms,
                                cudaStream_t s, const PairMaps* pair) {
  GemmArgs a{};
  a.sf_routed = sf_routed;
  a.sf_shared = sf_shared ? sf_shared : sf_routed;
  a.act_sf = act_sf;
  a.tiles = tiles;
  a.n_tiles = n_tiles;
  a.max_tiles = max_tiles;
  a.E = E;
  a.KG = d / kKGroup;
  a.m_tiles = f / kKGroup;
  a.gate_up = 1;
  a.limit = limit;
  a.h_q = h_q;
  a.h_sf = h_sf;
  a.f = f;
  a.d = d;
  a.status = status;
  a.budget_ns = wait_budget_ns;
  a.stall_loads = stall_loads;
  return launch_grouped(w_routed, w_shared, act, act_small, a, tile_rows, act_fp4, num_sms, s, pair);
}

cudaError_t launch_gemm_down(const CUtensorMap& w_routed, const CUtensorMap& w_shared, const uint8_t* sf_routed,
                             const uint8_t* sf_shared, const CUtensorMap& act, const CUtensorMap& act_small,
                             const uint8_t* act_sf, const RowTile* tiles, const int32_t* n_tiles, int max_tiles, int E,
                             int d, int f, const float* row_w, ExpertRows y16, __nv_bfloat16* y_bf16, int* status,
                             uint64_t wait_budget_ns, int stall_loads, int tile_rows, int act_fp4, int num_sms,
                             cudaStream_t s, const PairMaps* pair) {
  GemmArgs a{};
  a.sf_routed = sf_routed;
  a.sf_shared = sf_shared ? sf_shared : sf_routed;
  a.act_sf = act_sf;
  a.tiles = tiles;
  a.n_tiles = n_tiles;
  a.max_tiles = max_tiles;
  a.E = E;
  a.KG = f / kKGroup;
  a.m_tiles = d / kN;
  a.gate_up = 0;
  a.row_w = row_w;
  a.y16 = y16;
  a.y_bf16 = y_bf16;
  a.d = d;
  a.f = f;
  a.status = status;
  a.budget_ns = wait_budget_ns;
  a.stall_loads = stall_loads;
  return launch_grouped(w_routed, w_shared, act, act_small, a, tile_rows, act_fp4, num_sms, s, pair);
}

}  // namespace moe
