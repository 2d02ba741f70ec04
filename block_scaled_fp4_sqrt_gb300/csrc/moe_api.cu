// Host side of the C ABI declared in include/moe.h: argument checks, handles, the workspace
// carve-up, TMA tensor-map encoding and the launch sequence of one layer forward.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>

#include "moe.h"
#include "moe_dispatch_state.cuh"
#include "moe_internal.h"
#include "moe_testing.h"

using namespace moe;

struct moe_experts_s {
  moe_config_t cfg;
  int n = 0;                // experts in this set
  uint8_t* w13 = nullptr;   // owned: packed gate-up codes [n, d/128, f/128, 256, 64]
  uint8_t* w2 = nullptr;    // owned: packed down codes [n, f/128, d/256, 256, 64]
  uint8_t* sf13 = nullptr;  // owned: scale atoms [n, d/128, f/128, 2, 512]
  uint8_t* sf2 = nullptr;   // owned: [n, f/128, d/256, 2, 512]
  CUtensorMap tm13;   // the same codes for kind::mxf8f6f4 (16U4_ALIGN16B, 128-byte rows in smem)
  CUtensorMap tm2;
  CUtensorMap tm13p;  // ... and for kind::mxf4 (packed 64-byte rows, 64-byte swizzle)
  CUtensorMap tm2p;
  CUtensorMap tm13h;  // kind::mxf8f6f4 codes in 128-row boxes: one CTA's half of a slab (CTA-pair GEMMs)
  CUtensorMap tm2h;
  CUtensorMap tm_sf13;  // the scale atoms as rows of 256 B, 4-row boxes (both atoms of a slab)
  CUtensorMap tm_sf2;
  int act_fp4 = 0;    // activation format: 0 = MXFP8, 1 = MXFP4 (moe_experts_set_activation_format)
  __nv_bfloat16* router_split = nullptr;  // owned: resident router weight planes (moe_experts_set_router)
  float* router_w32 = nullptr;            // owned: the resident router weights in fp32 (small batches)
  float* router_bias = nullptr;           // owned: its bias [E]
  CUtensorMap tm_router;                  // map over router_split
  const int32_t* hash_table = nullptr;
  int32_t hash_V = 0;
  void* ws_base = nullptr;
  size_t ws_bytes = 0;
  int32_t ws_max_T = 0;
  Workspace ws{};
  int* status = nullptr;  // owned: device status word
  uint64_t budget_ns = 2000000000ull;
  int num_sms = 0;
  int device = 0;
  int32_t last_T = 0;
  int32_t last_rows = 0;  // rows of the last grouped FFN (its h stays in the workspace)
  int32_t last_fwd_T = -1;     // T of the last moe_forward (its expert rows stay in the workspace), or -1
  int32_t last_fwd_shared = 0;  // whether that forward had a shared expert
  int stall_loads = 0;
  int pair_gemm = 0;  // 128-row tiles on CTA pairs (moe_testing_set_pair_gemm); one-SM kernels by default
  void* const* stage_events = nullptr;  // MOE_N_STAGES + 1 caller-owned cudaEvent_t, or null
  // Changes whenever something a recorded launch sequence depends on changes (workspace, router, hash
  // table, activation format, wait budget, test hooks, stage events): a stack's cached graph compares it.
  uint64_t generation = 0;
};

namespace {

thread_local std::string g_last_error;

// Source of handle generations: unique over the process, so a handle created at a destroyed one's
// address never repeats its generation.
std::atomic<uint64_t> g_generation{1};

void bump(moe_experts_s* h) { h->generation = g_generation.fetch_add(1, std::memory_order_relaxed); }

moe_status_t fail(moe_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

moe_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define MOE_CUDA(call, what)                       \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D K-major tensor map: inner dimension K (elements), outer `rows`, box {128, box_rows}, 128-byte swizzle.
// FP4 maps expand each 16-element chunk to 16 bytes in shared memory (the operand form of the MMA).
moe_status_t make_map(CUtensorMap* m, const void* base, bool fp4, uint64_t K, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t gdim[2] = {K, rows};
  cuuint64_t gstride[1] = {fp4 ? K / 2 : K};
  cuuint32_t box[2] = {128u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void*>(base), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MOE_OK;
}

// Packed 8-bit map for kind::mxf4 operands: rows of `row_bytes` bytes (K / 2 for MXFP4), box {64 B
// (128 E2M1 codes, one stage), box_rows}, 64-byte swizzle.
moe_status_t make_map_packed(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t gdim[2] = {row_bytes, rows};
  cuuint64_t gstride[1] = {row_bytes};
  cuuint32_t box[2] = {64u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstride, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (packed) failed (%d)", (int)r);
  return MOE_OK;
}

// Scale atoms (512 B each) viewed as rows of 256 bytes: box {256 B, box_rows}, no swizzle, so a box of 2 rows
// is one atom and a box of 4 rows two consecutive atoms, each landing contiguously in shared memory.
moe_status_t make_map_atoms(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t gdim[2] = {256u, rows};
  cuuint64_t gstride[1] = {256u};
  cuuint32_t box[2] = {256u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstride, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (scale atoms) failed (%d)", (int)r);
  return MOE_OK;
}

// bf16 K-major map: inner dimension K, outer `rows`, box {64 elements (128 B), box_rows}, 128-byte swizzle.
moe_status_t make_map_bf16(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t gdim[2] = {K, rows};
  cuuint64_t gstride[1] = {K * 2};
  cuuint32_t box[2] = {64u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (bf16) failed (%d)", (int)r);
  return MOE_OK;
}

moe_status_t check_cfg(const moe_config_t* c) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "config is NULL");
  if (c->d_model <= 0 || c->d_ff <= 0 || c->d_model % 256 || c->d_ff % 128)
    return fail(MOE_ERR_UNSUPPORTED, "d_model (%d) must be a positive multiple of 256 and d_ff (%d) of 128",
                c->d_model, c->d_ff);
  if (c->d_model > 65536 || c->d_ff > 65536) return fail(MOE_ERR_UNSUPPORTED, "d_model / d_ff above 65536");
  if (c->n_experts < 1 || c->n_experts > 1024)
    return fail(MOE_ERR_UNSUPPORTED, "n_experts (%d) must be in [1, 1024]", c->n_experts);
  if (c->top_k < 1 || c->top_k > 16 || c->top_k > c->n_experts)
    return fail(MOE_ERR_UNSUPPORTED, "top_k (%d) must be in [1, min(16, n_experts)]", c->top_k);
  if (!(c->route_scale == c->route_scale) || !(c->swiglu_limit > 0.f))
    return fail(MOE_ERR_INVALID_ARG, "route_scale must be a number and swiglu_limit positive");
  return MOE_OK;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int max_split_rows(int max_T, int E, int d) {
  // largest split * T over 1 <= T <= max_T, for the router partial sums: the split only changes with
  // ceil(T / 128), so each 128-row bucket peaks at its last T
  int best = 0;
  for (int b = 1; (b - 1) * 128 < max_T; ++b) {
    const int T = std::min(128 * b, max_T);
    best = std::max(best, router_tc_split(T, E, d) * T);
  }
  return best;
}

struct Dims {
  int rows;       // max rows incl. shared
  int G;          // max groups
  int n_chunks;
  int max_tiles;
};

Dims dims_for(int max_T, int E, int k) {
  Dims dm;
  dm.rows = max_T * (k + 1);
  dm.G = E + 1;
  dm.n_chunks = (max_T + 31) / 32;
  // the short tile shape needs the most tiles; + G more covers the padding of the CTA-pair shape, which
  // gives every group an even number of 128-row tiles
  dm.max_tiles = (dm.rows + kSmallTileRows - 1) / kSmallTileRows + 2 * dm.G;
  return dm;
}

}  // namespace

namespace moe {

void set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }

size_t workspace_layout(int max_T, int d, int f, int E, int k, Workspace* ws, void* base) {
  const Dims dm = dims_for(max_T, E, k);
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    off = align_up(off, 256);
    void* p = base ? static_cast<uint8_t*>(base) + off : nullptr;
    off += bytes;
    return p;
  };
  Workspace w{};
  w.topk_ids = (int32_t*)take((size_t)max_T * k * 4);
  w.topk_w = (float*)take((size_t)max_T * k * 4);
  w.logits = (float*)take((size_t)max_split_rows(max_T, E, d) * E * 4);
  w.w_split = (__nv_bfloat16*)take((size_t)3 * router_tc_epad(E) * d * 2);
  w.chunk_hist = (int32_t*)take((size_t)dm.n_chunks * dm.G * 4);
  w.counts = (int32_t*)take((size_t)dm.G * 4);
  w.offsets = (int32_t*)take((size_t)(dm.G + 1) * 4);
  w.tile_off = (int32_t*)take((size_t)(dm.G + 1) * 4);
  w.n_tiles = (int32_t*)take(4);
  w.tiles = (RowTile*)take((size_t)dm.max_tiles * sizeof(RowTile));
  w.perm_tok = (int32_t*)take((size_t)dm.rows * 4);
  w.inv_pos = (int32_t*)take((size_t)max_T * k * 4);
  w.row_w = (float*)take((size_t)dm.rows * 4);
  w.a_q = (uint8_t*)take((size_t)dm.rows * d);
  w.a_sf = (uint8_t*)take((size_t)dm.max_tiles * (d / 128) * kSfAtomBytes);
  w.h_q = (uint8_t*)take((size_t)dm.rows * f);
  w.h_sf = (uint8_t*)take((size_t)dm.max_tiles * (f / 128) * kSfAtomBytes);
  w.y_rows.val = (__half*)take((size_t)dm.rows * d * 2);
  w.y_rows.exp = (uint8_t*)take((size_t)dm.rows * (d / 32));
  w.route_done = (int32_t*)take(4);
  if (ws) *ws = w;
  return align_up(off, 256);
}

}  // namespace moe

extern "C" {

const char* moe_last_error(void) { return g_last_error.c_str(); }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or device";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_CHECK: return "device-side range check failed";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

size_t moe_workspace_size(const moe_config_t* cfg, int32_t max_T) {
  if (check_cfg(cfg) != MOE_OK || max_T < 1) return 0;
  return workspace_layout(max_T, cfg->d_model, cfg->d_ff, cfg->n_experts, cfg->top_k, nullptr, nullptr);
}

moe_status_t moe_experts_create(const moe_config_t* cfg, int32_t n, const uint8_t* w13_fp4, const uint8_t* w13_e8m0,
                                const uint8_t* w2_fp4, const uint8_t* w2_e8m0, moe_stream_t stream,
                                moe_experts_t* out) {
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  moe_status_t st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (n < 1 || n > 1024) return fail(MOE_ERR_INVALID_ARG, "expert count %d outside [1, 1024]", n);
  if (!w13_fp4 || !w13_e8m0 || !w2_fp4 || !w2_e8m0) return fail(MOE_ERR_INVALID_ARG, "weight pointer is NULL");
  if (!aligned(w13_fp4, 16) || !aligned(w2_fp4, 16))
    return fail(MOE_ERR_INVALID_ARG, "FP4 weight buffers must be 16-byte aligned");
  if (!aligned(w13_e8m0, 4) || !aligned(w2_e8m0, 4))
    return fail(MOE_ERR_INVALID_ARG, "scale buffers must be 4-byte aligned");
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  int major = 0, minor = 0, sms = 0;
  MOE_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "cudaDeviceGetAttribute");
  MOE_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "cudaDeviceGetAttribute");
  MOE_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3)
    return fail(MOE_ERR_UNSUPPORTED, "libmoe is built for sm_103a; device %d is sm_%d%d", dev, major, minor);
  const int d = cfg->d_model, f = cfg->d_ff;
  moe_experts_s* h = new (std::nothrow) moe_experts_s();
  if (!h) return fail(MOE_ERR_CUDA, "host allocation failed");
  h->cfg = *cfg;
  h->n = n;
  bump(h);
  h->num_sms = sms;
  h->device = dev;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t w13_bytes = (size_t)n * 2 * f * (d / 2), w2_bytes = (size_t)n * d * (f / 2);
  const size_t sf13_bytes = (size_t)n * 2 * f * (d / 32), sf2_bytes = (size_t)n * d * (f / 32);
  cudaError_t e = cudaMalloc(&h->w13, w13_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&h->w2, w2_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&h->sf13, sf13_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&h->sf2, sf2_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&h->status, sizeof(int));
  if (e == cudaSuccess) e = cudaMemsetAsync(h->status, 0, sizeof(int), s);
  if (e == cudaSuccess) e = launch_pack_weights(w13_fp4, n, 2 * f, d, 0, h->w13, s);
  if (e == cudaSuccess) e = launch_pack_weights(w2_fp4, n, d, f, 1, h->w2, s);
  if (e == cudaSuccess) e = launch_pack_weight_sf(w13_e8m0, n, 2 * f, d, 0, h->sf13, s);
  if (e == cudaSuccess) e = launch_pack_weight_sf(w2_e8m0, n, d, f, 1, h->sf2, s);
  if (e != cudaSuccess) {
    moe_experts_destroy(h);
    return cuda_fail(e, "moe_experts_create");
  }
  // packed codes as [slabs * 256 rows, 128 FP4]: one 256-row box per (output tile, K group)
  st = make_map(&h->tm13, h->w13, true, 128, (uint64_t)n * 2 * f * (d / 128), 256);
  if (st == MOE_OK) st = make_map(&h->tm2, h->w2, true, 128, (uint64_t)n * d * (f / 128), 256);
  if (st == MOE_OK) st = make_map_packed(&h->tm13p, h->w13, 64, (uint64_t)n * 2 * f * (d / 128), 256);
  if (st == MOE_OK) st = make_map_packed(&h->tm2p, h->w2, 64, (uint64_t)n * d * (f / 128), 256);
  if (st == MOE_OK) st = make_map(&h->tm13h, h->w13, true, 128, (uint64_t)n * 2 * f * (d / 128), 128);
  if (st == MOE_OK) st = make_map(&h->tm2h, h->w2, true, 128, (uint64_t)n * d * (f / 128), 128);
  if (st == MOE_OK) st = make_map_atoms(&h->tm_sf13, h->sf13, sf13_bytes / 256, 4);
  if (st == MOE_OK) st = make_map_atoms(&h->tm_sf2, h->sf2, sf2_bytes / 256, 4);
  if (st != MOE_OK) {
    moe_experts_destroy(h);
    return st;
  }
  *out = h;
  return MOE_OK;
}

void moe_experts_destroy(moe_experts_t h) {
  if (!h) return;
  if (h->w13) cudaFree(h->w13);
  if (h->w2) cudaFree(h->w2);
  if (h->sf13) cudaFree(h->sf13);
  if (h->sf2) cudaFree(h->sf2);
  if (h->status) cudaFree(h->status);
  if (h->router_split) cudaFree(h->router_split);
  if (h->router_w32) cudaFree(h->router_w32);
  if (h->router_bias) cudaFree(h->router_bias);
  delete h;
}

moe_status_t moe_experts_set_router(moe_experts_t h, const float* router_w, const float* router_bias,
                                    moe_stream_t stream) {
  if (!h) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!router_w && !router_bias) {  // drop the resident router
    MOE_CUDA(cudaStreamSynchronize(s), "stream synchronize");
    if (h->router_split) cudaFree(h->router_split);
    if (h->router_w32) cudaFree(h->router_w32);
    if (h->router_bias) cudaFree(h->router_bias);
    h->router_split = nullptr;
    h->router_w32 = nullptr;
    h->router_bias = nullptr;
    bump(h);
  return MOE_OK;
  }
  if (!router_w || !router_bias) return fail(MOE_ERR_INVALID_ARG, "router_w and router_bias go together");
  const int E = h->cfg.n_experts, d = h->cfg.d_model;
  if (E > 512) return fail(MOE_ERR_UNSUPPORTED, "the learned router supports up to 512 experts");
  if (!aligned(router_w, 16)) return fail(MOE_ERR_INVALID_ARG, "router_w must be 16-byte aligned");
  const int Epad = router_tc_epad(E);
  if (!h->router_split) {
    MOE_CUDA(cudaMalloc(&h->router_split, (size_t)3 * Epad * d * sizeof(__nv_bfloat16)), "router planes");
    cudaError_t e = cudaMalloc(&h->router_bias, (size_t)E * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&h->router_w32, (size_t)E * d * sizeof(float));
    if (e != cudaSuccess) {
      cudaFree(h->router_split);
      if (h->router_bias) cudaFree(h->router_bias);
      h->router_split = nullptr;
      h->router_bias = nullptr;
      return cuda_fail(e, "router bias / fp32 copy");
    }
    const moe_status_t st = make_map_bf16(&h->tm_router, h->router_split, 64, (uint64_t)3 * Epad * (d / 64), 256);
    if (st != MOE_OK) {  // leave the handle without a resident router
      cudaFree(h->router_split);
      cudaFree(h->router_w32);
      cudaFree(h->router_bias);
      h->router_split = nullptr;
      h->router_w32 = nullptr;
      h->router_bias = nullptr;
      return st;
    }
  }
  MOE_CUDA(launch_split_router(router_w, E, d, h->router_split, s), "router weight split");
  MOE_CUDA(cudaMemcpyAsync(h->router_w32, router_w, (size_t)E * d * sizeof(float), cudaMemcpyDeviceToDevice, s),
           "router weight copy");
  MOE_CUDA(cudaMemcpyAsync(h->router_bias, router_bias, (size_t)E * sizeof(float), cudaMemcpyDeviceToDevice, s),
           "router bias copy");
  bump(h);
  return MOE_OK;
}

moe_status_t moe_experts_set_hash_table(moe_experts_t h, const int32_t* table, int32_t V) {
  if (!h) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
  if (table && V < 1) return fail(MOE_ERR_INVALID_ARG, "hash table needs V >= 1");
  h->hash_table = table;
  h->hash_V = table ? V : 0;
  bump(h);
  return MOE_OK;
}

moe_status_t moe_set_workspace(moe_experts_t h, void* ws, size_t bytes, int32_t max_T) {
  if (!h) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
  if (!ws || max_T < 1) return fail(MOE_ERR_INVALID_ARG, "workspace pointer NULL or max_T < 1");
  if (!aligned(ws, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const size_t need = workspace_layout(max_T, h->cfg.d_model, h->cfg.d_ff, h->cfg.n_experts, h->cfg.top_k, nullptr,
                                       nullptr);
  if (bytes < need) return fail(MOE_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed for max_T %d", bytes, need, max_T);
  workspace_layout(max_T, h->cfg.d_model, h->cfg.d_ff, h->cfg.n_experts, h->cfg.top_k, &h->ws, ws);
  // the small-batch router's CTA count starts at zero (and every call leaves it there)
  MOE_CUDA(cudaMemset(h->ws.route_done, 0, sizeof(int32_t)), "router counter");
  h->ws_base = ws;
  h->ws_bytes = bytes;
  h->ws_max_T = max_T;
  bump(h);
  return MOE_OK;
}

moe_status_t moe_experts_set_activation_format(moe_experts_t h, int32_t format) {
  if (!h) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
  if (format != MOE_ACT_MXFP8 && format != MOE_ACT_MXFP4) return fail(MOE_ERR_INVALID_ARG, "unknown activation format");
  h->act_fp4 = format == MOE_ACT_MXFP4 ? 1 : 0;
  bump(h);
  return MOE_OK;
}

moe_status_t moe_set_wait_budget(moe_experts_t h, uint64_t budget_ns) {
  if (!h || budget_ns == 0) return fail(MOE_ERR_INVALID_ARG, "handle NULL or zero budget");
  h->budget_ns = budget_ns;
  bump(h);
  return MOE_OK;
}

static moe_status_t check_input(const moe_experts_s* h, const moe_input_t* x) {
  if (!h) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
  if (!x) return fail(MOE_ERR_INVALID_ARG, "input is NULL");
  if (x->T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d is negative", x->T);
  if (x->T > 0 && !x->x_bf16) return fail(MOE_ERR_INVALID_ARG, "x is NULL");
  if (x->x_bf16 && !aligned(x->x_bf16, 16)) return fail(MOE_ERR_INVALID_ARG, "x must be 16-byte aligned");
  if (!h->ws_base) return fail(MOE_ERR_WORKSPACE, "no workspace attached (moe_set_workspace)");
  if (x->T > h->ws_max_T) return fail(MOE_ERR_WORKSPACE, "T = %d above the workspace's max_T = %d", x->T, h->ws_max_T);
  return MOE_OK;
}

// disp: the small-batch router (learned routing, T <= kRouterSmallMaxT) writes the dispatch state;
// dout: the cluster router (learned, up to 256 experts) or the hash router writes it (T <= kRouterDispatchMaxT).
static moe_status_t route_into(moe_experts_s* h, const moe_input_t* x, const float* router_w, const float* router_bias,
                               int32_t* ids, float* wts, cudaStream_t s, const SmallDispatch* disp = nullptr,
                               const DispatchOut* dout = nullptr) {
  const int T = x->T, E = h->cfg.n_experts, k = h->cfg.top_k, d = h->cfg.d_model;
  if (h->hash_table) {
    if (router_w || router_bias) return fail(MOE_ERR_INVALID_ARG, "hash layer: router_w and router_bias must be NULL");
    if (!x->token_ids) return fail(MOE_ERR_INVALID_ARG, "hash layer: token_ids is NULL");
    if (T == 0) return MOE_OK;
    MOE_CUDA(launch_hash_route(x->token_ids, h->hash_table, h->hash_V, T, E, k, h->cfg.route_scale, ids, wts, h->status,
                               s, h->ws.route_done, dout),
             "hash route");
    return MOE_OK;
  }
  // router_w = router_bias = NULL: the handle's resident router (moe_experts_set_router), split once
  const bool resident = !router_w && !router_bias && h->router_split;
  if (!resident && (!router_w || !router_bias))
    return fail(MOE_ERR_INVALID_ARG, "router_w / router_bias is NULL and the handle has no resident router");
  if (x->token_ids) return fail(MOE_ERR_INVALID_ARG, "token_ids given but no hash table is set");
  if (E > 512) return fail(MOE_ERR_UNSUPPORTED, "the learned router supports up to 512 experts");
  if (!resident && !aligned(router_w, 16)) return fail(MOE_ERR_INVALID_ARG, "router_w must be 16-byte aligned");
  if (T == 0) return MOE_OK;
  if (T <= kRouterSmallMaxT) {  // small batches: fp32 logits over the whole GPU and top-k, one kernel
    MOE_CUDA(launch_router_small(static_cast<const __nv_bfloat16*>(x->x_bf16), resident ? h->router_w32 : router_w,
                                 resident ? h->router_bias : router_bias, T, d, E, k, h->cfg.route_scale, h->ws.logits,
                                 h->ws.route_done, ids, wts, resident ? 1 : 0, disp, s),
             "router");
    return MOE_OK;
  }
  CUtensorMap tm_x, tm_w;
  const int Epad = router_tc_epad(E);
  moe_status_t st = make_map_bf16(&tm_x, x->x_bf16, (uint64_t)d, (uint64_t)T, 128);
  if (st != MOE_OK) return st;
  if (resident) {
    tm_w = h->tm_router;
    router_bias = h->router_bias;
  } else {
    // the split planes are tile-contiguous [256 x 64] blocks: viewed as a [3 * Epad * d / 64, 64] matrix
    st = make_map_bf16(&tm_w, h->ws.w_split, 64, (uint64_t)3 * Epad * (d / 64), 256);
    if (st != MOE_OK) return st;
    MOE_CUDA(launch_split_router(router_w, E, d, h->ws.w_split, s), "router weight split");
  }
  if (E <= 256) {  // logits, split-K reduction and top-k in one cluster kernel
    MOE_CUDA(launch_router_fused(tm_x, tm_w, router_bias, T, E, d, k, h->cfg.route_scale, router_fused_split(T, d), ids,
                                 wts, h->status, h->budget_ns, s, h->ws.route_done, dout),
             "router");
    return MOE_OK;
  }
  const int split = router_tc_split(T, E, d);
  MOE_CUDA(launch_router_tc(tm_x, tm_w, T, E, d, split, h->ws.logits, h->status, h->budget_ns, s), "router logits");
  MOE_CUDA(launch_router_topk(h->ws.logits, split, router_bias, T, E, k, h->cfg.route_scale, ids, wts, s),
           "router top-k");
  return MOE_OK;
}

moe_status_t moe_route(moe_experts_t h, const moe_input_t* x, const float* router_w, const float* router_bias,
                       int32_t* topk_ids, float* topk_w, moe_stream_t stream) {
  moe_status_t st = check_input(h, x);
  if (st != MOE_OK) return st;
  if (x->T > 0 && (!topk_ids || !topk_w)) return fail(MOE_ERR_INVALID_ARG, "topk_ids / topk_w is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = route_into(h, x, router_w, router_bias, topk_ids, topk_w, s);
  if (st == MOE_OK) h->last_T = x->T;
  return st;
}

moe_status_t moe_permute(moe_experts_t h, const moe_input_t* x, const int32_t* topk_ids, int32_t* counts,
                         int32_t* offsets, int32_t* perm_tok, int32_t* inv_pos, uint8_t* a_q, uint8_t* a_s,
                         moe_stream_t stream) {
  moe_status_t st = check_input(h, x);
  if (st != MOE_OK) return st;
  if (!counts || !offsets || !perm_tok || !inv_pos) return fail(MOE_ERR_INVALID_ARG, "an output pointer is NULL");
  if (x->T > 0 && !topk_ids) return fail(MOE_ERR_INVALID_ARG, "topk_ids is NULL");
  if ((a_q && !aligned(a_q, 16)) || (a_s && !aligned(a_s, 4)))
    return fail(MOE_ERR_INVALID_ARG, "a_q must be 16-byte and a_s 4-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int T = x->T, E = h->cfg.n_experts, k = h->cfg.top_k, d = h->cfg.d_model;
  const Dims dm = dims_for(h->ws_max_T, E, k);
  const int n_chunks = (T + 31) / 32;
  if (T == 0) {
    MOE_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s), "memset");
    MOE_CUDA(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s), "memset");
    return MOE_OK;
  }
  MOE_CUDA(launch_histogram(topk_ids, T, k, E, E, h->ws.chunk_hist, h->status, s), "histogram");
  MOE_CUDA(launch_scan(h->ws.chunk_hist, n_chunks, T, E, E, 0, kTileRows, dm.max_tiles, counts, offsets,
                       h->ws.tile_off, h->ws.n_tiles, h->ws.tiles, h->status, s),
           "scan");
  uint8_t* q = a_q ? a_q : h->ws.a_q;
  MOE_CUDA(launch_gather(static_cast<const __nv_bfloat16*>(x->x_bf16), topk_ids, nullptr, h->ws.chunk_hist, offsets,
                         h->ws.tile_off, T, d, k, E, E, 0, kTileRows, q, nullptr, a_s, perm_tok, inv_pos, nullptr,
                         h->act_fp4, s),
           "gather");
  return MOE_OK;
}

static void mark_stage(const moe_experts_s* h, int i, cudaStream_t s) {
  if (h->stage_events) cudaEventRecord(static_cast<cudaEvent_t>(h->stage_events[i]), s);
}

// Row-tile height for a call: verify batches (at most ~16 rows per expert on average) use 32-row tiles,
// whose short activation slots leave room for a deeper pipeline; larger batches use 128-row tiles.
static int tile_rows_for(int rows, int groups) {
  return rows <= 16 * groups ? kSmallTileRows : kTileRows;
}

// 128-row tiles of MXFP8 activations run on CTA pairs when the handle asks for it (moe_testing_set_pair_gemm).
static bool use_pairs(const moe_experts_s* h, int tile_rows) {
  return tile_rows == kTileRows && !h->act_fp4 && h->pair_gemm;
}

// pair: the work list pads every group to an even number of 128-row tiles; run both GEMMs on CTA pairs.
static moe_status_t run_ffn(moe_experts_s* h, moe_experts_s* sh, int rows, int E_groups_shared_index,
                            const uint8_t* a_q, const uint8_t* a_sf_atoms, const float* row_w, ExpertRows y16,
                            __nv_bfloat16* y_bf16, int max_tiles, int tile_rows, bool timed, cudaStream_t s,
                            bool pair = false) {
  const int d = h->cfg.d_model, f = h->cfg.d_ff;
  const int fp4 = h->act_fp4;
  CUtensorMap tm_a, tm_a32, tm_h, tm_h32;
  moe_status_t st;
  if (fp4) {  // MXFP4 rows of d / 2 and f / 2 bytes
    st = make_map_packed(&tm_a, a_q, (uint64_t)d / 2, (uint64_t)rows, kTileRows);
    if (st == MOE_OK) st = make_map_packed(&tm_a32, a_q, (uint64_t)d / 2, (uint64_t)rows, 32);
    if (st == MOE_OK) st = make_map_packed(&tm_h, h->ws.h_q, (uint64_t)f / 2, (uint64_t)rows, kTileRows);
    if (st == MOE_OK) st = make_map_packed(&tm_h32, h->ws.h_q, (uint64_t)f / 2, (uint64_t)rows, 32);
  } else {
    st = make_map(&tm_a, a_q, false, (uint64_t)d, (uint64_t)rows, kTileRows);
    if (st == MOE_OK) st = make_map(&tm_a32, a_q, false, (uint64_t)d, (uint64_t)rows, 32);
    if (st == MOE_OK) st = make_map(&tm_h, h->ws.h_q, false, (uint64_t)f, (uint64_t)rows, kTileRows);
    if (st == MOE_OK) st = make_map(&tm_h32, h->ws.h_q, false, (uint64_t)f, (uint64_t)rows, 32);
  }
  if (st != MOE_OK) return st;
  const moe_experts_s* shx = sh ? sh : h;
  pair = pair && !fp4 && tile_rows == kTileRows;
  PairMaps pm13, pm2;
  if (pair) {
    pm13.w = h->tm13h;
    pm13.w_shared = shx->tm13h;
    pm13.sfw = h->tm_sf13;
    pm13.sfw_shared = shx->tm_sf13;
    pm2.w = h->tm2h;
    pm2.w_shared = shx->tm2h;
    pm2.sfw = h->tm_sf2;
    pm2.sfw_shared = shx->tm_sf2;
    st = make_map_atoms(&pm13.sfa, a_sf_atoms, (uint64_t)max_tiles * (d / 128) * 2, 2);
    if (st == MOE_OK) st = make_map_atoms(&pm2.sfa, h->ws.h_sf, (uint64_t)max_tiles * (f / 128) * 2, 2);
    if (st != MOE_OK) return st;
  }
  MOE_CUDA(launch_gemm_gate_up(fp4 ? h->tm13p : h->tm13, fp4 ? shx->tm13p : shx->tm13, h->sf13, shx->sf13, tm_a, tm_a32,
                               a_sf_atoms, h->ws.tiles, h->ws.n_tiles, max_tiles, E_groups_shared_index, d, f,
                               h->cfg.swiglu_limit, h->ws.h_q, h->ws.h_sf, h->status, h->budget_ns, h->stall_loads,
                               tile_rows, fp4, h->num_sms, s, pair ? &pm13 : nullptr),
           "gate-up GEMM");
  if (timed) mark_stage(h, 3, s);
  MOE_CUDA(launch_gemm_down(fp4 ? h->tm2p : h->tm2, fp4 ? shx->tm2p : shx->tm2, h->sf2, shx->sf2, tm_h, tm_h32,
                            h->ws.h_sf, h->ws.tiles, h->ws.n_tiles, max_tiles, E_groups_shared_index, d, f, row_w, y16,
                            y_bf16, h->status, h->budget_ns, h->stall_loads, tile_rows, fp4, h->num_sms, s,
                            pair ? &pm2 : nullptr),
           "down GEMM");
  return MOE_OK;
}

moe_status_t moe_expert_ffn(moe_experts_t h, int32_t n_rows, const int32_t* offsets, const uint8_t* a_q,
                            const uint8_t* a_s, const float* row_w, void* y_bf16, moe_stream_t stream) {
  if (!h) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
  if (n_rows < 0) return fail(MOE_ERR_INVALID_ARG, "n_rows is negative");
  if (!h->ws_base) return fail(MOE_ERR_WORKSPACE, "no workspace attached (moe_set_workspace)");
  const Dims dm = dims_for(h->ws_max_T, h->cfg.n_experts, h->cfg.top_k);
  if (n_rows > dm.rows) return fail(MOE_ERR_WORKSPACE, "n_rows = %d above the workspace capacity %d", n_rows, dm.rows);
  if (h->n + 1 > dm.G) return fail(MOE_ERR_WORKSPACE, "expert set larger than the workspace's group capacity");
  if (n_rows == 0) return MOE_OK;
  if (!a_q || !a_s || !y_bf16) return fail(MOE_ERR_INVALID_ARG, "a_q / a_s / y is NULL");
  if (!aligned(a_q, 16) || !aligned(a_s, 4) || !aligned(y_bf16, 16))
    return fail(MOE_ERR_INVALID_ARG, "a_q and y must be 16-byte aligned, a_s 4-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int groups = offsets ? h->n : 1;
  const int bn = tile_rows_for(n_rows, groups);
  const bool pair = use_pairs(h, bn);
  MOE_CUDA(launch_tiles_from_offsets(offsets, groups, n_rows, bn, dm.max_tiles, h->ws.tile_off,
                                     h->ws.n_tiles, h->ws.tiles, h->status, s, pair ? 1 : 0),
           "tile list");
  MOE_CUDA(launch_rows_sf_to_atoms(a_s, h->ws.tiles, h->ws.n_tiles, h->cfg.d_model, dm.max_tiles, h->ws.a_sf, s),
           "scale atoms");
  h->last_rows = n_rows;
  return run_ffn(h, nullptr, n_rows, h->n, a_q, h->ws.a_sf, row_w, ExpertRows{nullptr, nullptr},
                 static_cast<__nv_bfloat16*>(y_bf16), dm.max_tiles, bn, false, s, pair);
}

moe_status_t moe_set_stage_events(moe_experts_t h, void* const* events, int32_t n) {
  if (!h) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
  if (events && n < MOE_N_STAGES + 1) return fail(MOE_ERR_INVALID_ARG, "need %d events", MOE_N_STAGES + 1);
  if (events)
    for (int i = 0; i <= MOE_N_STAGES; ++i)
      if (!events[i]) return fail(MOE_ERR_INVALID_ARG, "event %d is NULL", i);
  h->stage_events = events;
  bump(h);
  return MOE_OK;
}

moe_status_t moe_forward(const moe_input_t* x, const float* router_w, const float* router_bias, moe_experts_t h,
                         moe_experts_t sh, void* out_bf16, moe_stream_t stream) {
  return moe::forward_impl(x, router_w, router_bias, h, sh, out_bf16, nullptr, stream);
}

}  // extern "C"

namespace moe {

moe_status_t forward_impl(const moe_input_t* x, const float* router_w, const float* router_bias, moe_experts_t h,
                          moe_experts_t sh, void* out_bf16, const void* residual_bf16, moe_stream_t stream) {
  moe_status_t st = check_input(h, x);
  if (st != MOE_OK) return st;
  if (h->n != h->cfg.n_experts) return fail(MOE_ERR_INVALID_ARG, "routed set must hold cfg.n_experts experts");
  if (sh) {
    if (sh->n != 1) return fail(MOE_ERR_INVALID_ARG, "shared set must hold exactly one expert");
    if (sh->cfg.d_model != h->cfg.d_model || sh->cfg.d_ff != h->cfg.d_ff)
      return fail(MOE_ERR_INVALID_ARG, "shared expert shape differs from the routed experts");
    if (sh->act_fp4 != h->act_fp4)
      return fail(MOE_ERR_INVALID_ARG, "shared and routed experts use different activation formats");
  }
  if (x->T > 0 && !out_bf16) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
  if (out_bf16 && !aligned(out_bf16, 16)) return fail(MOE_ERR_INVALID_ARG, "out must be 16-byte aligned");
  if (residual_bf16 && !aligned(residual_bf16, 16)) return fail(MOE_ERR_INVALID_ARG, "residual must be 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int T = x->T, E = h->cfg.n_experts, k = h->cfg.top_k, d = h->cfg.d_model;
  const int has_shared = sh ? 1 : 0;
  const int G = E + has_shared;
  const int R = T * k;
  const int rows = R + (has_shared ? T : 0);
  const Dims dm = dims_for(h->ws_max_T, E, k);
  const int n_chunks = (T + 31) / 32;
  const int bn = tile_rows_for(R, E);
  // learned routing of a small batch: the small-batch router's last CTA also writes the dispatch state
  const bool small_dispatch = !h->hash_table && T >= 1 && T <= kRouterSmallMaxT && bn >= kRouterSmallMaxT;
  // the small-batch router's dispatch writes one tile per group: no pair padding, so one-SM GEMMs there
  const bool pair = !small_dispatch && use_pairs(h, bn);
  // batches up to kRouterDispatchMaxT rows: the cluster router's (or the hash router's) last CTA writes it
  const bool big_dispatch = !small_dispatch && T >= 1 && T <= kRouterDispatchMaxT &&
                            (h->hash_table ? dispatch_state_smem_ints(G, T) * 4 <= 48 * 1024 : E <= 256);
  const bool router_dispatch = small_dispatch || big_dispatch;
  SmallDispatch sd{G, has_shared, bn, dm.max_tiles, h->ws.chunk_hist, h->ws.counts, h->ws.offsets, h->ws.tile_off,
                   h->ws.n_tiles, h->ws.tiles};
  DispatchOut dout{G, has_shared, bn, dm.max_tiles, pair ? 1 : 0, h->ws.chunk_hist, h->ws.counts, h->ws.offsets,
                   h->ws.tile_off, h->ws.n_tiles, h->ws.tiles};
  mark_stage(h, 0, s);
  st = route_into(h, x, router_w, router_bias, h->ws.topk_ids, h->ws.topk_w, s, small_dispatch ? &sd : nullptr,
                  big_dispatch ? &dout : nullptr);
  if (st != MOE_OK) return st;
  h->last_T = T;
  h->last_fwd_T = -1;
  mark_stage(h, 1, s);
  if (T == 0) {
    for (int i = 2; i <= MOE_N_STAGES; ++i) mark_stage(h, i, s);
    return MOE_OK;
  }
  if (!router_dispatch) {
    MOE_CUDA(launch_histogram(h->ws.topk_ids, T, k, E, G, h->ws.chunk_hist, h->status, s), "histogram");
    MOE_CUDA(launch_scan(h->ws.chunk_hist, n_chunks, T, E, G, has_shared, bn, dm.max_tiles, h->ws.counts,
                         h->ws.offsets, h->ws.tile_off, h->ws.n_tiles, h->ws.tiles, h->status, s, pair ? 1 : 0),
             "scan");
  }
  MOE_CUDA(launch_gather(static_cast<const __nv_bfloat16*>(x->x_bf16), h->ws.topk_ids, h->ws.topk_w, h->ws.chunk_hist,
                         h->ws.offsets, h->ws.tile_off, T, d, k, E, G, has_shared, bn, h->ws.a_q, h->ws.a_sf,
                         nullptr, h->ws.perm_tok, h->ws.inv_pos, h->ws.row_w, h->act_fp4, s),
           "gather");
  mark_stage(h, 2, s);
  st = run_ffn(h, sh, rows, E, h->ws.a_q, h->ws.a_sf, h->ws.row_w, h->ws.y_rows, nullptr, dm.max_tiles, bn, true, s,
               pair);
  if (st != MOE_OK) return st;
  h->last_rows = rows;
  mark_stage(h, 4, s);
  MOE_CUDA(launch_combine(h->ws.y_rows, h->ws.inv_pos, T, d, k, R, has_shared,
                          static_cast<const __nv_bfloat16*>(residual_bf16), static_cast<__nv_bfloat16*>(out_bf16), s),
           "combine");
  mark_stage(h, 5, s);
  h->last_fwd_T = T;
  h->last_fwd_shared = has_shared;
  return MOE_OK;
}

int experts_d_model(moe_experts_t h) { return h ? h->cfg.d_model : 0; }

int experts_has_hash_table(moe_experts_t h) { return h && h->hash_table ? 1 : 0; }

int experts_has_resident_router(moe_experts_t h) { return h && h->router_split ? 1 : 0; }

uint64_t experts_generation(moe_experts_t h) { return h ? h->generation : 0; }

}  // namespace moe

extern "C" {

moe_status_t moe_get_routing(moe_experts_t h, const int32_t** ids, const float** w, int32_t* T) {
  if (!h || !ids || !w || !T) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  if (!h->ws_base) return fail(MOE_ERR_WORKSPACE, "no workspace attached");
  *ids = h->ws.topk_ids;
  *w = h->ws.topk_w;
  *T = h->last_T;
  return MOE_OK;
}

moe_status_t moe_testing_read_h(moe_experts_t h, uint8_t* h_q, uint8_t* h_s, int32_t* n_rows, moe_stream_t stream) {
  if (!h || !n_rows) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  if (!h->ws_base) return fail(MOE_ERR_WORKSPACE, "no workspace attached");
  *n_rows = h->last_rows;
  if (h->last_rows == 0 || (!h_q && !h_s)) return MOE_OK;  // a query of the row count
  if (!h_q || !h_s || !aligned(h_s, 4)) return fail(MOE_ERR_INVALID_ARG, "h_q / h_s NULL or h_s not 4-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int f = h->cfg.d_ff;
  const Dims dm = dims_for(h->ws_max_T, h->cfg.n_experts, h->cfg.top_k);
  const size_t row_bytes = h->act_fp4 ? (size_t)f / 2 : (size_t)f;
  MOE_CUDA(cudaMemcpyAsync(h_q, h->ws.h_q, row_bytes * h->last_rows, cudaMemcpyDeviceToDevice, s), "h codes");
  MOE_CUDA(launch_atoms_to_rows_sf(h->ws.h_sf, h->ws.tiles, h->ws.n_tiles, f, dm.max_tiles, h_s, s), "h scales");
  return MOE_OK;
}

moe_status_t moe_testing_read_y32(moe_experts_t h, float* y32, int32_t* T, moe_stream_t stream) {
  if (!h || !T) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  if (!h->ws_base) return fail(MOE_ERR_WORKSPACE, "no workspace attached");
  if (h->last_fwd_T < 0) return fail(MOE_ERR_INVALID_ARG, "no moe_forward on this handle since its last other call");
  *T = h->last_fwd_T;
  if (h->last_fwd_T == 0 || !y32) return MOE_OK;  // a query of the row count
  if (!aligned(y32, 16)) return fail(MOE_ERR_INVALID_ARG, "y32 must be 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int Tl = h->last_fwd_T, k = h->cfg.top_k;
  MOE_CUDA(launch_combine(h->ws.y_rows, h->ws.inv_pos, Tl, h->cfg.d_model, k, Tl * k, h->last_fwd_shared, nullptr,
                          nullptr, s, y32),
           "fp32 combine");
  return MOE_OK;
}

moe_status_t moe_testing_set_pair_gemm(moe_experts_t h, int32_t enable) {
  if (!h) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
  h->pair_gemm = enable ? 1 : 0;
  bump(h);
  return MOE_OK;
}

moe_status_t moe_testing_stall_loads(moe_experts_t h, int32_t enable) {
  if (!h) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
  h->stall_loads = enable ? 1 : 0;
  bump(h);
  return MOE_OK;
}

moe_status_t moe_check(moe_experts_t h, moe_stream_t stream) {
  if (!h) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MOE_CUDA(cudaStreamSynchronize(s), "stream synchronize");
  int v = 0;
  MOE_CUDA(cudaMemcpy(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost), "status read");
  if (v == 0) return MOE_OK;
  MOE_CUDA(cudaMemset(h->status, 0, sizeof(int)), "status clear");
  if (v & DEV_TIMEOUT) return fail(MOE_ERR_TIMEOUT, "a device wait expired (status 0x%x)", v);
  return fail(MOE_ERR_DEVICE_CHECK, "device range check failed (status 0x%x)", v);
}

}  // extern "C"
