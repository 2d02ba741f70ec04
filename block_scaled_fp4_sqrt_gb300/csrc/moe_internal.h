// Internal declarations shared by the C-ABI host code and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "moe.h"

namespace moe {

// The weighted expert rows between the down GEMM and the combine: fp16 values [rows, d] and one scale byte
// per 32 columns [rows, d / 32]; element = value * 2^(byte - 127).  The down epilogue picks each block's
// scale so that the block maximum lands in [2^14, 2^15): every element keeps fp16's 11 significant bits
// (rounding error at most 2^-11 relative) down to 2^-28 of its block maximum, whatever the weights' range.
struct ExpertRows {
  __half* val;
  uint8_t* exp;
};

// Device status bits (sticky, OR-ed into the handle's status word).
enum : int {
  DEV_BAD_EXPERT_ID = 1,   // an expert id outside [0, E) reached the permutation
  DEV_BAD_TOKEN_ID = 2,    // a token id outside [0, V) reached the hash router
  DEV_TIMEOUT = 4,         // a bounded mbarrier wait ran out
  DEV_BAD_WORK = 8,        // a work list larger than the workspace capacity
};

constexpr int kMmaM = 128;         // weight rows per MMA tile (tcgen05 M)
constexpr int kKGroup = 128;       // K elements per pipeline stage (one 128-byte swizzle row of FP8)
constexpr int kSfAtomBytes = 512;  // scale-factor atom: 128 rows x 4 K-blocks of 32
constexpr int kTileRows = 128;     // token rows per row tile (tcgen05 M) in the grouped GEMMs
constexpr int kSmallTileRows = 32; // row tiles of the verify-batch shape (short activation slots)
constexpr int kRouterDispatchMaxT = 1024;  // batches up to this size get their dispatch state from the router

// One row tile of the grouped GEMMs: rows [row0, row0 + nrows) of group `group`.
struct RowTile {
  int group;
  int row0;
  int nrows;
  int pad;
};

// Geometry of one forward call, fixed on the host from (config, T).
struct Geometry {
  int T, d, f, E, k;
  int G;            // groups: E routed + 1 shared (or E when there is no shared expert)
  int R;            // routed rows T*k
  int rows;         // R + T (shared rows follow the routed ones) or R
  int n_chunks;     // ceil(T / 32) histogram chunks
  int max_tiles;    // capacity of the row-tile list
  int bn;           // rows per tile
};

// Workspace carve-up (device pointers), see moe_workspace_layout().
struct Workspace {
  int32_t* topk_ids;    // [T, k]
  float* topk_w;        // [T, k]
  float* logits;        // [split, T, E] router partial sums
  __nv_bfloat16* w_split;  // [3, Epad, d] router weight as hi + mid + lo bf16
  int32_t* chunk_hist;  // [n_chunks, G]
  int32_t* counts;      // [G]
  int32_t* offsets;     // [G + 1]
  int32_t* tile_off;    // [G + 1] first row tile of each group
  int32_t* n_tiles;     // [1]
  RowTile* tiles;       // [max_tiles]
  int32_t* perm_tok;    // [rows]
  int32_t* inv_pos;     // [T, k]
  float* row_w;         // [rows]
  uint8_t* a_q;         // [rows, d]
  uint8_t* a_sf;        // [max_tiles, d/128, 512]
  uint8_t* h_q;         // [rows, f]
  uint8_t* h_sf;        // [max_tiles, f/128, 512]
  ExpertRows y_rows;     // [rows, d] weighted expert outputs (scaled fp16) and [rows, d / 32] scales
  int32_t* route_done;   // [1] CTA count of the small-batch router (zero between calls)
};

// Text returned by moe_last_error() on this thread.
void set_last_error(const char* msg);

// moe_forward with an optional bf16 residual stream: out = bf16(residual + layer(x)) (residual may alias out).
moe_status_t forward_impl(const moe_input_t* x, const float* router_w, const float* router_bias, moe_experts_t h,
                          moe_experts_t sh, void* out_bf16, const void* residual_bf16, moe_stream_t stream);
int experts_d_model(moe_experts_t h);
int experts_has_hash_table(moe_experts_t h);
int experts_has_resident_router(moe_experts_t h);
// Changes whenever a setter changes what the handle's launches depend on (unique over the process).
uint64_t experts_generation(moe_experts_t h);

// Launch with programmatic stream serialization: the kernel may be scheduled before the previous kernel
// in the stream has finished (it must call pdl_wait() before touching global memory, see moe_device.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Runs a set-up step once per device: kernel attributes such as the dynamic shared-memory opt-in and the
// non-portable cluster size belong to the current device, so a process that drives several GPUs must
// set them on each.  fn() returns cudaError_t; a failed step is retried on the next call.
class PerDeviceOnce {
 public:
  template <typename F>
  cudaError_t run(F&& fn) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool tracked = dev >= 0 && dev < 64;
    if (tracked && ((done_.load(std::memory_order_acquire) >> dev) & 1ull)) return cudaSuccess;
    e = fn();
    if (e == cudaSuccess && tracked) done_.fetch_or(1ull << dev, std::memory_order_acq_rel);
    return e;
  }

 private:
  std::atomic<unsigned long long> done_{0};
};

size_t workspace_layout(int max_T, int d, int f, int E, int k, Workspace* ws, void* base);

// ------------------------------------------------------------------ launchers (return cudaError_t)
constexpr int kRouterKSplitMax = 8;
int router_ksplit(int T, int E, int d);
cudaError_t launch_router_logits(const __nv_bfloat16* x, const float* w, int T, int d, int E, int ksplit,
                                 float* partial, cudaStream_t s);
// Tensor-core router: split count for T rows, padded expert count, weight split, logits partials.
int router_tc_split(int T, int E, int d);
int router_tc_epad(int E);
int router_fused_split(int T, int d);
struct DispatchOut;  // moe_dispatch_state.cuh
// The cluster router; with disp, its last CTA also writes the batch's dispatch state (done: a zeroed counter).
cudaError_t launch_router_fused(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const float* bias, int T, int E,
                                int d, int k, float route_scale, int split, int32_t* ids, float* wts, int* status,
                                uint64_t budget_ns, cudaStream_t s, int* done = nullptr,
                                const DispatchOut* disp = nullptr);
cudaError_t launch_split_router(const float* w, int E, int d, __nv_bfloat16* out, cudaStream_t s);
cudaError_t launch_router_tc(const CUtensorMap& tm_x, const CUtensorMap& tm_w, int T, int E, int d, int split,
                             float* partial, int* status, uint64_t budget_ns, cudaStream_t s);
cudaError_t launch_router_topk(const float* partial, int ksplit, const float* bias, int T, int E, int k,
                               float route_scale, int32_t* ids, float* wts, cudaStream_t s);
// Small-batch router (T <= kRouterSmallMaxT, E <= 512): fp32 logits spread over the GPU, then top-k in the
// last CTA; logits [T, E] scratch, done = a zeroed counter the kernel leaves at zero.  early_params: w and
// bias are the handle's resident copies and may be read before the programmatic-dependency wait.
// disp (optional): the last CTA also writes the dispatch state that histogram_kernel + colscan_kernel +
// groupscan_kernel would (one 32-token chunk: every chunk base is 0; at most 32 rows per group: one tile
// per non-empty group).
constexpr int kRouterSmallMaxT = 32;
struct SmallDispatch {
  int G, has_shared, bn, max_tiles;
  int32_t* chunk_hist;  // [G] (one chunk)
  int32_t* counts;      // [G]
  int32_t* offsets;     // [G + 1]
  int32_t* tile_off;    // [G + 1]
  int32_t* n_tiles;     // [1]
  RowTile* tiles;       // [max_tiles]
};
cudaError_t launch_router_small(const __nv_bfloat16* x, const float* w, const float* bias, int T, int d, int E, int k,
                                float route_scale, float* logits, int* done, int32_t* ids, float* wts,
                                int early_params, const SmallDispatch* disp, cudaStream_t s);
// The hash router; with disp, its last block also writes the batch's dispatch state (done: a zeroed counter).
cudaError_t launch_hash_route(const int32_t* tok, const int32_t* table, int V, int T, int E, int k, float route_scale,
                              int32_t* ids, float* wts, int* status, cudaStream_t s, int* done = nullptr,
                              const DispatchOut* disp = nullptr);

cudaError_t launch_histogram(const int32_t* ids, int T, int k, int E, int G, int32_t* chunk_hist, int* status,
                             cudaStream_t s);
cudaError_t launch_scan(int32_t* chunk_hist, int n_chunks, int T, int E, int G, int has_shared, int bn, int max_tiles,
                        int32_t* counts, int32_t* offsets, int32_t* tile_off, int32_t* n_tiles, RowTile* tiles,
                        int* status, cudaStream_t s, int pad_pairs = 0);
// Quantise x to MXFP8 (act_fp4: MXFP4, rows of d/2 bytes) and scatter each token row to its k routed
// rows (+ its shared row).  a_sf_atoms / a_s_rows may each be null (kernel-layout scale atoms /
// canonical [rows, d/32]).
cudaError_t launch_gather(const __nv_bfloat16* x, const int32_t* ids, const float* wts, const int32_t* chunk_hist,
                          const int32_t* offsets, const int32_t* tile_off, int T, int d, int k, int E, int G,
                          int has_shared, int bn, uint8_t* a_q, uint8_t* a_sf_atoms, uint8_t* a_s_rows,
                          int32_t* perm_tok, int32_t* inv_pos, float* row_w, int act_fp4, cudaStream_t s);
// Canonical [rows, d/32] scales -> per-tile atoms (for moe_expert_ffn on caller buffers).
cudaError_t launch_rows_sf_to_atoms(const uint8_t* a_s_rows, const RowTile* tiles, const int32_t* n_tiles, int d,
                                    int max_tiles, uint8_t* atoms, cudaStream_t s);
// Per-tile atoms -> canonical [rows, K/32] (reads back the h scales for tests).
cudaError_t launch_atoms_to_rows_sf(const uint8_t* atoms, const RowTile* tiles, const int32_t* n_tiles, int K,
                                    int max_tiles, uint8_t* rows_sf, cudaStream_t s);
// pad_pairs: every group's tile count is rounded up to an even number (the padding tile has no rows), so
// that tiles 2p and 2p + 1 belong to one group (the CTA-pair GEMM shape).
cudaError_t launch_tiles_from_offsets(const int32_t* offsets, int G, int n_rows, int bn, int max_tiles,
                                      int32_t* tile_off, int32_t* n_tiles, RowTile* tiles, int* status,
                                      cudaStream_t s, int pad_pairs = 0);

// Weight repacking at handle creation.  mode 0: gate-up rows [n, 2f, K] (gate rows 0..f-1, up rows
// f..2f-1); mode 1: down rows [n, d, K].  Packed codes [n, K/128, rows/256, 256, 64 B]: each 256-row
// slab is one output tile (mode 0: gate rows 128t.. then up rows 128t..; mode 1: rows 256t..) and one
// 128-element K group, 16 KB contiguous.  Scale atoms [n, K/128, rows/256, 2, 512] in the same order.
cudaError_t launch_pack_weights(const uint8_t* codes, int n, int rows, int K, int mode, uint8_t* packed,
                                cudaStream_t s);
cudaError_t launch_pack_weight_sf(const uint8_t* sc, int n, int rows, int K, int mode, uint8_t* atoms,
                                  cudaStream_t s);

// Tensor maps of the CTA-pair shape of the grouped GEMMs (large expert groups, MXFP8 activations).
struct PairMaps {
  CUtensorMap w, w_shared;      // weight codes with 128-row boxes (one CTA's half of a 256-row slab)
  CUtensorMap sfw, sfw_shared;  // weight scale atoms as rows of 256 B, 4-row boxes (both atoms of a slab)
  CUtensorMap sfa;              // activation (gate-up) or h (down) scale atoms, 2-row boxes (one atom)
};

// Grouped GEMMs.  act_fp4 = 0: MXFP8 activations (E4M3 rows of K bytes) x MXFP4 weights on
// kind::mxf8f6f4, weight maps of 16U4_ALIGN16B type (K = 128 elements expanded to 128-byte rows);
// act_fp4 = 1: MXFP4 activations (rows of K/2 bytes) on kind::mxf4, every map 8-bit over packed bytes
// with 64-byte rows and 64-byte swizzle.  The gate-up epilogue writes h in the same format.
cudaError_t launch_gemm_gate_up(const CUtensorMap& w_routed, const CUtensorMap& w_shared, const uint8_t* sf_routed,
                                const uint8_t* sf_shared, const CUtensorMap& act, const CUtensorMap& act_small,
                                const uint8_t* act_sf,
                                const RowTile* tiles, const int32_t* n_tiles, int max_tiles, int E, int d, int f,
                                float limit,
                                uint8_t* h_q, uint8_t* h_sf, int* status, uint64_t wait_budget_ns, int stall_loads,
                                int tile_rows, int act_fp4, int num_sms, cudaStream_t s,
                                const PairMaps* pair = nullptr);
cudaError_t launch_gemm_down(const CUtensorMap& w_routed, const CUtensorMap& w_shared, const uint8_t* sf_routed,
                             const uint8_t* sf_shared, const CUtensorMap& act, const CUtensorMap& act_small,
                             const uint8_t* act_sf,
                             const RowTile* tiles, const int32_t* n_tiles, int max_tiles, int E, int d, int f,
                             const float* row_w, ExpertRows y16, __nv_bfloat16* y_bf16, int* status,
                             uint64_t wait_budget_ns, int stall_loads, int tile_rows, int act_fp4, int num_sms,
                             cudaStream_t s,
                                const PairMaps* pair = nullptr);

// out_f32 non-NULL: the fp32 sums go there instead, without the rounding to bf16 (out is then unused).
cudaError_t launch_combine(ExpertRows y_rows, const int32_t* inv_pos, int T, int d, int k, int R, int has_shared,
                           const __nv_bfloat16* residual, __nv_bfloat16* out, cudaStream_t s,
                           float* out_f32 = nullptr);

}  // namespace moe
