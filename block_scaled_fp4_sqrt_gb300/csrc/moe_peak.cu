// Measured peaks of the block-scaled tensor-core MMAs the grouped GEMMs use -- tcgen05.mma
// kind::mxf8f6f4.block_scale.scale_vec::1X (E4M3 x E2M1, M = 128, N = 256, K = 32) and, for the
// MXFP4-activation variant, kind::mxf4.block_scale.scale_vec::2X (E2M1 x E2M1, K = 64): the
// denominators of the tensor-bound roofline.  One CTA per SM issues MMAs back to back with its
// operands rotating through six shared-memory stages laid out like the GEMM's (so the tensor pipe
// reads fresh operands every stage) and the scale atoms copied into TMEM two stages ahead.  The
// operands are fixed pseudo-random finite codes; the result is discarded.
#include <algorithm>
#include <vector>

#include "moe_device.cuh"
#include "moe_testing.h"

namespace moe {

namespace {

constexpr int kPS = 6;  // stages

// FP4 = false: E4M3 rows of 128 bytes and byte-expanded E2M1 weights (128-byte swizzle);
// FP4 = true: packed E2M1 rows of 64 bytes for both operands (64-byte swizzle).
template <bool FP4>
struct PeakCfg {
  static constexpr int kRowBytes = FP4 ? 64 : 128;
  static constexpr int kASlot = 4096;  // activation slot (the MMA's 128 rows read on into the next slots)
  static constexpr int kBSlot = 256 * kRowBytes;
  static constexpr int kSfSlot = 3 * 512;  // scale atoms
  static constexpr int kAOff = 0, kBOff = kPS * kASlot, kSfOff = kBOff + kPS * kBSlot;
  static constexpr int kUsed = kSfOff + kPS * kSfSlot;
  static constexpr int kSmem = kUsed + 1024;
  static_assert(kAOff + (kPS - 1) * kASlot + 128 * kRowBytes <= kBOff + kPS * kBSlot, "activation reads stay in smem");
  static_assert(kSmem <= 232448 - 64, "shared memory budget");
  // per stage: four K = 32 MMAs, or two K = 64 MMAs; either way K = 128
  static constexpr double kFlopsPerStage = 2.0 * 128 * 256 * 128;
};

template <bool FP4>
__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int n_stages, uint64_t budget_ns,
                                                          unsigned long long* ns_out, int* status) {
  using P = PeakCfg<FP4>;
  constexpr int kPAOff = P::kAOff, kPBOff = P::kBOff, kPSfOff = P::kSfOff, kPUsed = P::kUsed;
  constexpr int kPASlot = P::kASlot, kPBSlot = P::kBSlot, kPSfSlot = P::kSfSlot;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t done, sink;
  __shared__ uint32_t tmem_slot;
  for (int i = threadIdx.x; i < kPUsed / 4; i += blockDim.x) {
    uint32_t h = (uint32_t)i * 2654435761u + 0x9E3779B9u;
    h ^= h >> 15;
    h *= 2246822519u;
    h ^= h >> 13;
    // operand bytes: positive E4M3 codes below 0x78 (finite), or E2M1 nibble pairs without sign;
    // scale bytes 126..129
    reinterpret_cast<uint32_t*>(smem)[i] = i >= kPSfOff / 4 ? 0x7E7F8081u : (h & 0x77777777u);
  }
  if (threadIdx.x == 0) {
    mbar_init(&done, 1);
    mbar_init(&sink, (1u << 20) - 1);  // collects the per-stage commits; never waited on
    mbar_fence_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (threadIdx.x < 32) tmem_alloc(&tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  if (threadIdx.x == 0) {
    constexpr uint32_t kIdesc0 = FP4 ? mma_idesc(kMxf4E2M1, kMxf4E2M1, 128, 256, 0, 0) : mma_idesc(0, 5, 128, 256, 0, 0);
    constexpr uint32_t kSwz = FP4 ? 4 : 2, kSbo = 8 * P::kRowBytes;
    const uint64_t a0 = smem_desc(smem_addr(smem + kPAOff), 16, kSbo, kSwz);
    const uint64_t b0 = smem_desc(smem_addr(smem + kPBOff), 16, kSbo, kSwz);
    const uint64_t sf0 = smem_desc(smem_addr(smem + kPSfOff), 128, 128, 0);
    const uint32_t sft = tbase + 256;
    auto copy_sf = [&](int s) {
      const uint64_t dsc = sf0 + (uint64_t)((s * kPSfSlot) >> 4);
      const uint32_t t = sft + (uint32_t)(s * 12);
      tc_copy_sf(t, dsc);
      tc_copy_sf(t + 4, dsc + 32);
      tc_copy_sf(t + 8, dsc + 64);
    };
    copy_sf(0);
    copy_sf(1);
    const uint64_t t0 = globaltimer_ns();
    for (int g = 0; g < n_stages; ++g) {
      const int s = g % kPS;
      const uint64_t ad = a0 + (uint64_t)((s * kPASlot) >> 4), bd = b0 + (uint64_t)((s * kPBSlot) >> 4);
      const uint32_t sfa = sft + (uint32_t)(s * 12);
      if (FP4)
        (void)tc_stage2_mxf4_commit_poll(tbase, ad, bd, kIdesc0, sfa, sfa + 4, g ? 1u : 0u, &sink, &done, 1u);
      else
        (void)tc_stage4_mx_commit_poll(tbase, ad, bd, kIdesc0, sfa, sfa + 4, g ? 1u : 0u, &sink, &done, 1u);
      if (g + 2 < n_stages) copy_sf((g + 2) % kPS);
    }
    tc_commit(&done);
    if (!mbar_wait(&done, 0, budget_ns)) set_status(status, DEV_TIMEOUT);
    ns_out[blockIdx.x] = globaltimer_ns() - t0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(tbase, 512);
}

template <bool FP4>
moe_status_t measure_peak(int32_t n_stages, double* tflops) {
  using P = PeakCfg<FP4>;
  constexpr int kPSmem = P::kSmem;
  if (n_stages < 8 || n_stages > (1 << 18) || !tflops) {
    set_last_error("n_stages must be in [8, 262144] and tflops non-NULL");
    return MOE_ERR_INVALID_ARG;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    set_last_error("no CUDA device");
    return MOE_ERR_CUDA;
  }
  unsigned long long* d_ns = nullptr;
  int* d_status = nullptr;
  auto cleanup = [&]() {
    if (d_ns) cudaFree(d_ns);
    if (d_status) cudaFree(d_status);
  };
  if (cudaFuncSetAttribute(mma_peak_kernel<FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem) != cudaSuccess ||
      cudaMalloc(&d_ns, sizeof(unsigned long long) * sms) != cudaSuccess ||
      cudaMalloc(&d_status, sizeof(int)) != cudaSuccess || cudaMemset(d_status, 0, sizeof(int)) != cudaSuccess) {
    cleanup();
    set_last_error("peak measurement setup failed");
    return MOE_ERR_CUDA;
  }
  // warm-up launch, then the timed one (per-CTA globaltimer spans; the slowest CTA counts)
  mma_peak_kernel<FP4><<<sms, 128, kPSmem>>>(16, 2000000000ull, d_ns, d_status);
  mma_peak_kernel<FP4><<<sms, 128, kPSmem>>>(n_stages, 2000000000ull, d_ns, d_status);
  std::vector<unsigned long long> ns(sms);
  int status = 0;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(ns.data(), d_ns, sizeof(unsigned long long) * sms, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(&status, d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cleanup();
    set_last_error("peak measurement kernel failed");
    return MOE_ERR_CUDA;
  }
  cleanup();
  if (status) {
    set_last_error("peak measurement: device wait timed out");
    return MOE_ERR_TIMEOUT;
  }
  const double t = (double)*std::max_element(ns.begin(), ns.end()) * 1e-9;
  const double flops = P::kFlopsPerStage * (double)n_stages * sms;
  *tflops = t > 0 ? flops / t / 1e12 : 0.0;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" MOE_API moe_status_t moe_measure_mxf8f6f4_peak(int32_t n_stages, double* tflops) {
  return moe::measure_peak<false>(n_stages, tflops);
}

extern "C" MOE_API moe_status_t moe_measure_mxf4_peak(int32_t n_stages, double* tflops) {
  return moe::measure_peak<true>(n_stages, tflops);
}
