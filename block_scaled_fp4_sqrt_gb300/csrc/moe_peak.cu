// Measured peak of the block-scaled tensor-core MMA the grouped GEMMs use (tcgen05.mma
// kind::mxf8f6f4.block_scale.scale_vec::1X, E4M3 x E2M1, M = 128, N = 256, K = 32): the denominator
// of the tensor-bound roofline.  One CTA per SM issues MMAs back to back with its operands rotating
// through six shared-memory stages laid out like the GEMM's (so the tensor pipe reads fresh operands
// every stage) and the scale atoms copied into TMEM two stages ahead.  The operands are fixed
// pseudo-random finite codes; the result is discarded.
#include <algorithm>
#include <vector>

#include "moe_device.cuh"
#include "moe_testing.h"

namespace moe {

namespace {

constexpr int kPS = 6;                 // stages
constexpr int kPASlot = 4096;          // activation slot (the MMA's 128 rows read on into the next slots)
constexpr int kPBSlot = 256 * 128;     // weight slot: 256 rows x 128 padded FP4
constexpr int kPSfSlot = 3 * 512;      // scale atoms
constexpr int kPAOff = 0, kPBOff = kPS * kPASlot, kPSfOff = kPBOff + kPS * kPBSlot;
constexpr int kPUsed = kPSfOff + kPS * kPSfSlot;
constexpr int kPSmem = kPUsed + 1024;
static_assert(kPAOff + (kPS - 1) * kPASlot + 128 * 128 <= kPBOff + kPS * kPBSlot, "activation reads stay in smem");
static_assert(kPSmem <= 232448 - 64, "shared memory budget");

__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int n_stages, uint64_t budget_ns,
                                                          unsigned long long* ns_out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t done, sink;
  __shared__ uint32_t tmem_slot;
  for (int i = threadIdx.x; i < kPUsed / 4; i += blockDim.x) {
    uint32_t h = (uint32_t)i * 2654435761u + 0x9E3779B9u;
    h ^= h >> 15;
    h *= 2246822519u;
    h ^= h >> 13;
    // operand bytes: positive E4M3 codes below 0x78 (finite), any E2M1 nibble pair without sign;
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
    constexpr uint32_t kIdesc0 = mma_idesc(0, 5, 128, 256, 0, 0);
    const uint64_t a0 = smem_desc(smem_addr(smem + kPAOff), 16, 1024, 2);
    const uint64_t b0 = smem_desc(smem_addr(smem + kPBOff), 16, 1024, 2);
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
      (void)tc_stage4_mx_commit_poll(tbase, a0 + (uint64_t)((s * kPASlot) >> 4), b0 + (uint64_t)((s * kPBSlot) >> 4),
                                     kIdesc0, sft + (uint32_t)(s * 12), sft + (uint32_t)(s * 12 + 4), g ? 1u : 0u,
                                     &sink, &done, 1u);
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

}  // namespace

}  // namespace moe

extern "C" MOE_API moe_status_t moe_measure_mxf8f6f4_peak(int32_t n_stages, double* tflops) {
  using namespace moe;
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
  if (cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem) != cudaSuccess ||
      cudaMalloc(&d_ns, sizeof(unsigned long long) * sms) != cudaSuccess ||
      cudaMalloc(&d_status, sizeof(int)) != cudaSuccess || cudaMemset(d_status, 0, sizeof(int)) != cudaSuccess) {
    cleanup();
    set_last_error("peak measurement setup failed");
    return MOE_ERR_CUDA;
  }
  // warm-up launch, then the timed one (per-CTA globaltimer spans; the slowest CTA counts)
  mma_peak_kernel<<<sms, 128, kPSmem>>>(16, 2000000000ull, d_ns, d_status);
  mma_peak_kernel<<<sms, 128, kPSmem>>>(n_stages, 2000000000ull, d_ns, d_status);
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
  const double flops = 2.0 * 128 * 256 * 32 * 4 * (double)n_stages * sms;
  *tflops = t > 0 ? flops / t / 1e12 : 0.0;
  return MOE_OK;
}
