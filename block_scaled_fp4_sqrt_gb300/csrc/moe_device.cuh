// Device-side building blocks for the sm_103a MoE kernels: mbarrier / TMA / tcgen05 wrappers
// written as inline PTX, bounded waits that report a timeout instead of hanging, and the MX
// element conversions used by the activation quantisers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <float.h>

#include "moe_internal.h"

namespace moe {

// ------------------------------------------------------------------------- status reporting
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicOr(status, code);
}

// ------------------------------------------------------------------------- programmatic dependent launch
// The small kernels of the layer call pdl_trigger() on entry, so that the next kernel in the stream may
// be scheduled while they run; every kernel calls pdl_wait() after its prologue but before its first
// access to global memory, which returns once the previous kernel has completed and its writes are
// visible.  Without the launch attribute (launch_pdl) both are no-ops.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ------------------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps until the phase completes or the hint runs
// out, instead of spinning (spinning waiters steal issue slots from the MMA and TMA threads).
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most budget_ns nanoseconds (plus at
// most one suspend interval).  Returns false (and the caller reports MOE_DEV_TIMEOUT) when the
// budget runs out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_suspend(bar, parity, 200000u)) return true;
    if (globaltimer_ns() - t0 > budget_ns) return false;
  }
}

// Polling wait for the phase with the given parity: mbarrier.test_wait never suspends the thread, so it
// sees the phase complete at once.  For waiters with no other warps to steal issue slots from (the handoff
// of the accumulator in the verify-batch GEMM shape); bounded by budget_ns like mbar_wait.
__device__ __forceinline__ bool mbar_spin(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (int i = 0;; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((i & 255) == 255 && globaltimer_ns() - t0 > budget_ns) return false;
  }
}

// ------------------------------------------------------------------------- thread-block clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of every CTA of the cluster: release this CTA's prior writes, then acquire the others'.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address, in the cluster's shared window, of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Arrive on an mbarrier of another CTA of the cluster (cluster_addr from mapa_shared), releasing this
// thread's prior memory operations at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// mbar_wait for a barrier that other CTAs arrive on: acquire at cluster scope, so that what those CTAs
// released before arriving is visible afterwards.  Bounded like mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(200000u)
        : "memory");
    if (ok) return true;
    if (globaltimer_ns() - t0 > budget_ns) return false;
  }
}

// ------------------------------------------------------------------------- routing
__device__ __forceinline__ float softplus_f(float l) { return fmaxf(l, 0.f) + log1pf(expf(-fabsf(l))); }

// Warp-wide top-k of one token (the sqrt-softplus router's selection).  Lane l holds expert
// e = l + 32 i in s[i] (its score) and sel[i] (its selection key score + bias; pass -FLT_MAX where
// e >= E).  Selects the k largest keys, ties to the lower expert id, and writes the chosen ids in
// ascending order with weights route_scale * s_j / sum over the chosen s.  Ascending order comes from
// ballot prefix counts (slot i first, then lane), so nothing is sorted; the sum is lane 0's
// butterfly total, broadcast, so every weight divides by the same value.
template <int NPL>
__device__ __forceinline__ void warp_route_topk(const float (&s)[NPL], const float (&sel)[NPL], int E, int k,
                                                float route_scale, int32_t* __restrict__ ids_row,
                                                float* __restrict__ w_row) {
  const int lane = threadIdx.x & 31;
  // order-preserving 32-bit keys of the selection values (larger float -> larger key), so that one
  // round is a local scan, a warp max of the keys and a warp min of the ids holding it
  uint32_t key[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const uint32_t u = __float_as_uint(sel[i]);
    key[i] = lane + 32 * i < E ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
  }
  uint32_t taken = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t best = 0;
    int bi = NPL;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (!((taken >> i) & 1u) && lane + 32 * i < E && (bi == NPL || key[i] > best)) {
        best = key[i];
        bi = i;
      }
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, bi < NPL ? best : 0u);
    // lowest expert id among the lanes holding the maximum (a lane's own first maximum is its lowest)
    const uint32_t cand = (bi < NPL && best == m) ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu;
    const uint32_t win = __reduce_min_sync(0xFFFFFFFFu, cand);
    if ((int)(win & 31u) == lane) taken |= 1u << (win >> 5);
  }
  float ssum = 0.f;
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if ((taken >> i) & 1u) ssum += s[i];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ssum += __shfl_xor_sync(0xFFFFFFFFu, ssum, off);
  ssum = __shfl_sync(0xFFFFFFFFu, ssum, 0);
  int base = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const bool mine = (taken >> i) & 1u;
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, mine);
    if (mine) {
      const int pos = base + __popc(m & ((1u << lane) - 1u));
      ids_row[pos] = lane + 32 * i;
      w_row[pos] = route_scale * s[i] / ssum;
    }
    base += __popc(m);
  }
}

// ------------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// The CTA-pair form: this CTA's shared memory receives the tile, and the completion is counted on the
// mbarrier named by leader_bar (a shared::cluster address; the even CTA's barrier, from mapa_shared),
// which can thus track the loads of both CTAs of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y, uint32_t leader_bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(leader_bar), "l"(policy)
      : "memory");
}

// Prefetch one tile of a tensor into L2 (no shared-memory destination, no completion tracking).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
               : "memory");
}

// Prefetch a contiguous range into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ------------------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor (tcgen05 format): start address, leading / stride byte offsets
// (all >> 4), fixed version bits 46..47 = 1, swizzle mode in bits 61..63 (2 = 128-byte swizzle,
// 4 = 64-byte swizzle, 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swizzle & 7u) << 61;
  return d;
}

// Instruction descriptor of kind::mxf8f6f4 with E8M0 block scales.
// Formats: 0 = E4M3, 5 = E2M1.  M in {128}, N multiple of 16 up to 256.  sf ids pick the byte of
// the 32-bit scale word (the 32-element K block inside a 128-element group).
// kind::mxf4 (both operands E2M1, packed two per byte in shared memory, K = 64 per MMA): the E2M1
// format code of this kind is 1.
constexpr uint32_t kMxf4E2M1 = 1;

__host__ __device__ __forceinline__ constexpr uint32_t mma_idesc(uint32_t a_fmt, uint32_t b_fmt, uint32_t M,
                                                                 uint32_t N, uint32_t a_sf_id, uint32_t b_sf_id) {
  return ((b_sf_id & 3u) << 4) | ((a_fmt & 7u) << 7) | ((b_fmt & 7u) << 10) | (((N >> 3) & 63u) << 17) |
         (1u << 23) /* scale type UE8M0 */ | (((M >> 4) & 31u) << 24) | ((a_sf_id & 3u) << 29);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 128 bits from shared memory, replicated into all four 32-lane quadrants of TMEM.
__device__ __forceinline__ void tc_copy_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n}\n" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// One pipeline stage of four block-scaled MMAs (K = 4 x 32) fused with the stage's commit and a
// non-blocking test of another stage's barrier.  The test is issued first and its result is read
// only after the commit, so the barrier's latency overlaps the MMA issue instead of stalling the
// issuing thread (which would leave the tensor pipe idle: it queues only a couple of MMAs).  MMA k
// reads K columns 32k.. of the stage (descriptor address + 2k) and scale byte k (sf id k).
__device__ __forceinline__ bool tc_stage4_mx_commit_poll(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                         uint32_t idesc0, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                         uint32_t accumulate, uint64_t* commit_bar,
                                                         uint64_t* poll_bar, uint32_t poll_parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p, q, t;\n .reg .b64 a1, a2, a3, b1, b2, b3;\n .reg .b32 i1, i2, i3;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 q, [%8], %9;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " setp.eq.b32 t, 0, 0;\n"
      " add.s64 a1, %2, 2;\n add.s64 b1, %3, 2;\n"
      " add.s64 a2, %2, 4;\n add.s64 b2, %3, 4;\n"
      " add.s64 a3, %2, 6;\n add.s64 b3, %3, 6;\n"
      " or.b32 i1, %5, 0x20000010;\n or.b32 i2, %5, 0x40000020;\n or.b32 i3, %5, 0x60000030;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], %2, %3, %5, [%6], [%7], p;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], a1, b1, i1, [%6], [%7], t;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], a2, b2, i2, [%6], [%7], t;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], a3, b3, i3, [%6], [%7], t;\n"
      " tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%10];\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(ok)
      : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(accumulate), "r"(idesc0), "r"(sfa_tmem), "r"(sfb_tmem),
        "r"(smem_addr(poll_bar)), "r"(poll_parity), "r"(smem_addr(commit_bar))
      : "memory");
  return ok != 0;
}

// The MXFP4-activation variant's stage: two block-scaled MMAs of kind::mxf4 (E2M1 x E2M1, K = 64 each,
// scale_vec::2X: two E8M0 scales per row and MMA), fused with the commit and a barrier test as above.
// A stage holds K = 128 packed in 64-byte rows: MMA k reads bytes 32k.. of each row (descriptor
// address + 2k) and scale bytes 2k, 2k+1 of the 32-bit scale word (sf id 2k).
__device__ __forceinline__ bool tc_stage2_mxf4_commit_poll(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                           uint32_t idesc0, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                           uint32_t accumulate, uint64_t* commit_bar,
                                                           uint64_t* poll_bar, uint32_t poll_parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p, q, t;\n .reg .b64 a1, b1;\n .reg .b32 i1;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 q, [%8], %9;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " setp.eq.b32 t, 0, 0;\n"
      " add.s64 a1, %2, 2;\n add.s64 b1, %3, 2;\n"
      " or.b32 i1, %5, 0x40000020;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%1], %2, %3, %5, [%6], [%7], p;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%1], a1, b1, i1, [%6], [%7], t;\n"
      " tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%10];\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(ok)
      : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(accumulate), "r"(idesc0), "r"(sfa_tmem), "r"(sfb_tmem),
        "r"(smem_addr(poll_bar)), "r"(poll_parity), "r"(smem_addr(commit_bar))
      : "memory");
  return ok != 0;
}

// ---- CTA-pair (cta_group::2) forms.  The even CTA of a two-CTA cluster issues them for the pair: an
// MMA with M = 256 reads A rows 0..127 from its own shared memory and rows 128..255 from the peer's, and
// the N rows of B half from each (at the same shared-memory offsets), and writes each CTA's 128 rows of
// D into that CTA's tensor memory; a scale copy reads each CTA's own shared memory into its own tensor
// memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_copy_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Arrive on the barrier at the same offset in both CTAs of the pair once the pair's prior MMAs retire.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"((uint16_t)3)
      : "memory");
}

// The pair's form of tc_stage4_mx_commit_poll: four M = 256 block-scaled MMAs (K = 4 x 32), the stage's
// commit multicast to both CTAs' barrier, and a non-blocking test (cluster-scope acquire: the peer CTA
// arrives on these barriers) of another stage's barrier, read after the commit.
__device__ __forceinline__ bool tc_stage4_mx_pair_commit_poll(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                              uint32_t idesc0, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                              uint32_t accumulate, uint64_t* commit_bar,
                                                              uint64_t* poll_bar, uint32_t poll_parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p, q, t;\n .reg .b64 a1, a2, a3, b1, b2, b3;\n .reg .b32 i1, i2, i3;\n"
      " mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 q, [%8], %9;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " setp.eq.b32 t, 0, 0;\n"
      " add.s64 a1, %2, 2;\n add.s64 b1, %3, 2;\n"
      " add.s64 a2, %2, 4;\n add.s64 b2, %3, 4;\n"
      " add.s64 a3, %2, 6;\n add.s64 b3, %3, 6;\n"
      " or.b32 i1, %5, 0x20000010;\n or.b32 i2, %5, 0x40000020;\n or.b32 i3, %5, 0x60000030;\n"
      " tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], %2, %3, %5, [%6], [%7], p;\n"
      " tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], a1, b1, i1, [%6], [%7], t;\n"
      " tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], a2, b2, i2, [%6], [%7], t;\n"
      " tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], a3, b3, i3, [%6], [%7], t;\n"
      " tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%10], %11;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(ok)
      : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(accumulate), "r"(idesc0), "r"(sfa_tmem), "r"(sfb_tmem),
        "r"(smem_addr(poll_bar)), "r"(poll_parity), "r"(smem_addr(commit_bar)), "h"((uint16_t)3)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// Load 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------------- MX conversions
// floor(log2(a)) of a finite, positive fp32 value (normal or subnormal), from its bits.
__device__ __forceinline__ int floor_log2_f32(float a) {
  uint32_t u = __float_as_uint(a);
  int e = (int)((u >> 23) & 0xFF);
  if (e != 0) return e - 127;
  // subnormal: value = mantissa * 2^-149
  return (31 - __clz(u & 0x7FFFFF)) - 149;
}

// E8M0 block exponent for an MXFP8 (E4M3, emax 8) block with maximum magnitude amax.
__device__ __forceinline__ int mxfp8_block_exp(float amax) {
  if (!(amax > 0.0f)) return -127;
  int s = floor_log2_f32(amax) - 8;
  return s < -127 ? -127 : (s > 127 ? 127 : s);
}

// E8M0 block exponent for an MXFP4 (E2M1, emax 2) block with maximum magnitude amax.
__device__ __forceinline__ int mxfp4_block_exp(float amax) {
  if (!(amax > 0.0f)) return -127;
  int s = floor_log2_f32(amax) - 2;
  return s < -127 ? -127 : (s > 127 ? 127 : s);
}

// 2^-s as fp32 for s in [-127, 127] (2^127 is representable; 2^-127 is subnormal, built from bits).
__device__ __forceinline__ float exp2_neg_int(int s) {
  int e = 127 - s;  // biased exponent of 2^-s
  if (e >= 1) return __uint_as_float((uint32_t)e << 23);
  return __uint_as_float(1u << (22 + e));  // e in [0, -?]: only s = 127 reaches here (e = 0 -> 2^-127)
}

// ------------------------------------------------------------------------- scaled fp16 expert rows
// Block exponent s of 32 expert-row values with maximum magnitude amax: amax * 2^-s lies in [2^14, 2^15),
// inside fp16's range with its full 11 significant bits.  s stays in [-126, 127], so that 2^s and 2^-s are
// normal fp32 numbers; an all-zero block takes s = 0.
__device__ __forceinline__ int row16_block_exp(float amax) {
  if (!(amax > 0.0f)) return 0;
  const int s = floor_log2_f32(amax) - 14;
  return s < -126 ? -126 : (s > 127 ? 127 : s);
}

// The 32 products v[j] * w as fp16 times 2^-s (round to nearest even), packed in place: v[i] for i < 16 then
// holds the bits of the fp16 pair (2i, 2i + 1), element 2i in the low half, and v[16..31] is free.  The
// scale is taken from max |v| * |w| (rounding is monotonic, so this is the largest rounded product) and the
// weight folded into one multiplier w * 2^-s: scaling by a power of two commutes with rounding, so each code
// is that of the rounded product whenever nothing is subnormal.  Packing in place keeps the epilogue's
// register footprint at the 32 values.  Returns the block's scale byte s + 127.
__device__ __forceinline__ uint8_t row16_encode32(float (&v)[32], float w) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const int s = row16_block_exp(amax * fabsf(w));
  const float m = w * exp2_neg_int(s);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const __half2 h2 = __floats2half2_rn(v[2 * i] * m, v[2 * i + 1] * m);
    v[i] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&h2));
  }
  return (uint8_t)(s + 127);
}

// Packed word i of a block encoded by row16_encode32, as 16 bytes: words 4i .. 4i + 3.
__device__ __forceinline__ uint4 row16_words(const float (&v)[32], int i) {
  return make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]), __float_as_uint(v[4 * i + 2]),
                    __float_as_uint(v[4 * i + 3]));
}

// 2^(byte - 127) for a scale byte written by row16_encode32 (byte in [1, 254]).
__device__ __forceinline__ float row16_scale(uint32_t byte) { return __uint_as_float(byte << 23); }

// Round-to-nearest-even, saturating E4M3 conversion of two values (hardware cvt); lo in bits 0..7.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Round-to-nearest-even, saturating E2M1 conversion of eight values (hardware cvt); value i in bits
// 4i..4i+3, i.e. element 2j in the low nibble of byte j.
__device__ __forceinline__ uint32_t e2m1x8(float v0, float v1, float v2, float v3, float v4, float v5, float v6,
                                           float v7) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return r;
}

// One MX block of 32 values -> 16 bytes of packed E2M1 codes, each value multiplied by mul first.
__device__ __forceinline__ uint4 e2m1_block(const float (&v)[32], float mul) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = e2m1x8(v[8 * i] * mul, v[8 * i + 1] * mul, v[8 * i + 2] * mul, v[8 * i + 3] * mul, v[8 * i + 4] * mul,
                  v[8 * i + 5] * mul, v[8 * i + 6] * mul, v[8 * i + 7] * mul);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace moe
