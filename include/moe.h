/*
 * moe.h -- C ABI of libmoe, the GB300 (sm_103a) forward pass of a DeepSeek-V4-Flash-style
 * Mixture-of-Experts layer over a speculative-decode verify batch.
 *
 * The layer (DeepSeek-V4-Flash pages):
 *   - "sqrt-softplus MoE routing with hash layers" (TensorSharp DeepSeek V4 Flash page, section
 *     "How TensorSharp runs it"), top-k = 6 of 256 routed experts plus one always-on shared expert,
 *     route_scale = 1.5, swiglu_limit = 10 (FaStar model card, "Speeds, Sizes, Times" and "Model
 *     Architecture and Objective");
 *   - expert weights in MXFP4: E2M1 values with one E8M0 scale per 32 (model card "Preprocessing";
 *     TensorSharp page, "Getting a drafter"), gate / up / down = w1 / w3 / w2 (ds4 issue, "Loader
 *     spec -- mtp.* tensor map");
 *   - gate -> top-6 -> dispatch -> routed + shared expert FFNs -> combine (pypto page, "MoE and
 *     output stages"), the weighted sum being the moe_scatter_add epilogue (TensorSharp page, "DSpark
 *     and MoE CPU offload together").
 * Activations enter the expert GEMMs as MXFP8 (E4M3, one E8M0 scale per 32 along the reduction
 * dimension), as do the SwiGLU outputs before the down projection (MXFP4 in the variant that
 * moe_experts_set_activation_format selects).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers unless stated otherwise; row-major; the caller owns
 *     them.  bf16 tensors are passed as void*.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream).  The
 *     returned status covers host-side argument checks and launch errors only.  Conditions found on
 *     the device (an out-of-range expert or token id, a bounded wait that ran out) are recorded in a
 *     sticky per-handle status word and reported by moe_check().
 *   - No per-call path allocates device memory: moe_experts_create (its copy of the weights) and
 *     moe_experts_set_router (its resident router) allocate once at set-up; per-call scratch lives in a
 *     caller-provided workspace (moe_workspace_size / moe_set_workspace).
 *   - Shapes: d_model a multiple of 256, d_ff of 128; n_experts in [1, 1024]; top_k in [1, min(16,
 *     n_experts)]; n_experts <= 512 for the learned router (hash routing has no such limit).
 *   - Nothing is thread-safe per handle: calls on one handle must be ordered by the caller (one
 *     stream, or explicit events).  Two handles may be used concurrently.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, wrong mode */
  MOE_ERR_UNSUPPORTED = 2, /* shape outside the supported set, or the GPU is not sm_103 */
  MOE_ERR_WORKSPACE = 3,   /* workspace missing or smaller than the call needs */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed (text in moe_last_error()) */
  MOE_ERR_DEVICE_CHECK = 5, /* moe_check: a device-side range check failed */
  MOE_ERR_TIMEOUT = 6      /* moe_check: a bounded device wait expired */
} moe_status_t;

typedef struct {
  int32_t d_model;    /* hidden size d (4096 in the pages' model), a multiple of 256 */
  int32_t d_ff;       /* expert FFN width f (2048) */
  int32_t n_experts;  /* routed experts E (256); 1 for a shared-expert handle */
  int32_t top_k;      /* experts per token k (6) */
  float route_scale;  /* routed weights sum to this (1.5) */
  float swiglu_limit; /* SwiGLU clamp L (10): h = silu(min(gate, L)) * clamp(up, -L, L) */
} moe_config_t;

typedef struct moe_experts_s* moe_experts_t;

/* One batch of token rows. */
typedef struct {
  const void* x_bf16;       /* [T, d_model] bf16, 16-byte aligned */
  int32_t T;                /* rows (tokens) in the batch, >= 0 */
  const int32_t* token_ids; /* [T] token ids, hash-routed layers only (else NULL) */
} moe_input_t;

/*
 * Create an expert set of `n` experts in the canonical MXFP4 layout:
 *   w13_fp4 [n, 2*d_ff, d_model/2]  gate rows 0..d_ff-1 (w1) then up rows d_ff..2*d_ff-1 (w3); element
 *                                    2i of a row is the low nibble of byte i; E2M1 code = sign bit 3,
 *                                    exponent bits 2..1, mantissa bit 0;
 *   w13_e8m0 [n, 2*d_ff, d_model/32] one E8M0 scale byte (2^(b-127)) per 32 consecutive elements;
 *   w2_fp4  [n, d_model, d_ff/2], w2_e8m0 [n, d_model, d_ff/32]  the down projection (w2).
 * The handle copies codes and scales into its own device buffers in a tile-contiguous order (every
 * 16 KB block the GEMMs stream is contiguous in HBM); the copy is enqueued on `stream`, so the
 * inputs may be released once `stream` has passed this call.  Code buffers 16-byte aligned, scale
 * buffers 4-byte aligned.  A routed set uses n = cfg->n_experts; a shared expert is a set with n = 1.
 * Errors: MOE_ERR_INVALID_ARG (null / misaligned / n < 1), MOE_ERR_UNSUPPORTED (shape or GPU),
 * MOE_ERR_CUDA.  *out is NULL on error.
 * Passages: the expert FFN runs as a fused dequantisation + GEMM over the MXFP4 payload, 13.4 MB per
 * expert (FaStar README, "Features" and "Expert virtual memory"); the experts are FP4 with one E8M0
 * scale per 32 weights (model card, "Preprocessing" and its glossary; TensorSharp page, "Getting a
 * drafter"); a layer holds experts.{0..255}.{w1,w2,w3} and shared_experts.{w1,w2,w3} (ds4 issue,
 * "Resolved questions").
 */
MOE_API moe_status_t moe_experts_create(const moe_config_t* cfg, int32_t n, const uint8_t* w13_fp4, const uint8_t* w13_e8m0,
                                const uint8_t* w2_fp4, const uint8_t* w2_e8m0, moe_stream_t stream,
                                moe_experts_t* out);

/*
 * Turn a routed set into a hash-routed layer: table [V, top_k] int32 (device, borrowed) maps a
 * token id to its experts ("hash routing over the first 3 layers", model card "Speeds, Sizes,
 * Times"; the .fst.tid2eid sidecar).  Routing weights are route_scale / top_k.  Pass table = NULL to
 * return to learned routing.  Token ids outside [0, V) or table entries outside [0, n_experts) are
 * reported by moe_check (MOE_ERR_DEVICE_CHECK) and replaced by valid ids.
 */
MOE_API moe_status_t moe_experts_set_hash_table(moe_experts_t experts, const int32_t* table, int32_t V);

/*
 * Activation format of an expert set (default MOE_ACT_MXFP8).  MOE_ACT_MXFP8: x and the SwiGLU output
 * h are quantised to MXFP8 (E4M3 codes, one E8M0 scale per 32 along the reduction dimension) and the
 * grouped GEMMs run tcgen05 kind::mxf8f6f4 (E4M3 x E2M1).  MOE_ACT_MXFP4: x and h are quantised to
 * MXFP4 with the weights' own rule (E2M1 codes packed two per byte, element 2i in the low nibble of
 * byte i; scale exponent floor(log2(amax)) - 2; round to nearest even, saturating at +-6) and the
 * GEMMs run kind::mxf4 (E2M1 x E2M1): twice the tensor-core rate at a coarser activation precision.
 * This is the MXFP4-activation prefill variant; the pages quantise only the weights to MXFP4 (model
 * card "Preprocessing"; TensorSharp page "Getting a drafter").  It changes the layouts of moe_permute's
 * a_q output and moe_expert_ffn's a_q input to [rows, d_model/2] packed codes.  In moe_forward the
 * routed set and the shared expert must use the same format.  Takes effect on later calls.
 * Errors: MOE_ERR_INVALID_ARG (NULL handle, unknown format).
 */
#define MOE_ACT_MXFP8 0
#define MOE_ACT_MXFP4 1
MOE_API moe_status_t moe_experts_set_activation_format(moe_experts_t experts, int32_t format);

/*
 * Make the learned router resident on a routed set: router_w fp32 [E, d_model] (16-byte aligned) and
 * router_bias fp32 [E], both device buffers, are converted once into the form the router kernels read
 * (three bf16 planes whose sum is router_w exactly, in the tile order of the tensor-core router, plus an
 * fp32 copy for batches of up to 32 rows), into memory the handle allocates and owns
 * (6 * E_pad * d_model + 4 * E * d_model + 4 * E bytes; E_pad = E rounded up to 256).
 * The copy is enqueued on `stream`; the inputs may be released once `stream` has passed the call.  Later
 * moe_route / moe_forward calls (and stack layers) with router_w = router_bias = NULL use it and skip
 * the per-call conversion; calls that pass router weights still use those.  Calling it again replaces
 * the contents; router_w = router_bias = NULL frees it (after synchronising `stream`).  A hash table, when
 * set, takes precedence.  Errors: MOE_ERR_INVALID_ARG (NULL handle, one of the two NULL, misaligned),
 * MOE_ERR_UNSUPPORTED (E > 512), MOE_ERR_CUDA.
 */
MOE_API moe_status_t moe_experts_set_router(moe_experts_t experts, const float* router_w, const float* router_bias,
                                            moe_stream_t stream);

/* Bytes of workspace a routed set needs for batches of up to max_T rows (with a shared expert). */
MOE_API size_t moe_workspace_size(const moe_config_t* cfg, int32_t max_T);

/* Attach caller-owned device workspace (256-byte aligned) sized for up to max_T rows. */
MOE_API moe_status_t moe_set_workspace(moe_experts_t experts, void* workspace, size_t bytes, int32_t max_T);

/*
 * Router.  Learned: logits l = x . router_w^T in fp32 (router_w fp32 [E, d_model]), score
 * s = sqrt(softplus(l)), the top_k experts by s + router_bias (fp32 [E]; ties to the lower id),
 * weights route_scale * s_j / sum of the selected s (the bias steers selection only).
 * Hash layer (a table is set): router_w and router_bias must be NULL, x->token_ids non-NULL.
 * Learned layer with router_w = router_bias = NULL: the handle's resident router (moe_experts_set_router).
 * Outputs: topk_ids int32 [T, top_k] ascending per row, topk_w fp32 [T, top_k].
 * Uses the workspace.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_WORKSPACE, MOE_ERR_CUDA.
 * Passages: routed experts chosen by sqrt-softplus routing, with hash routing on hash layers
 * (TensorSharp page, "How TensorSharp runs it"); top-6 of 256, route_scale 1.5, hash routing over the
 * first layers (model card, "Speeds, Sizes, Times"); the router is ffn.gate.weight with ffn.gate.bias
 * (ds4 issue, "Resolved questions").  The bias steering selection only, the normalisation over the
 * selected scores and the ascending id order are readings of those passages.
 */
MOE_API moe_status_t moe_route(moe_experts_t experts, const moe_input_t* x, const float* router_w, const float* router_bias,
                       int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/*
 * Token -> expert permutation and MXFP8 activation quantisation (the dispatch step).
 * Inputs: x, topk_ids [T, top_k] (each row's ids distinct).  Outputs (R = T * top_k):
 *   counts [E]       rows per expert;      offsets [E+1]  exclusive prefix sums (offsets[E] = R);
 *   perm_tok [R]     token of each row, rows expert-major with tokens ascending inside an expert;
 *   inv_pos [T, top_k]  row of (t, topk_ids[t, j]);
 *   a_q [R, d_model] E4M3 codes of x[perm_tok[r]] (round-to-nearest-even, saturating at +-448),
 *   a_s [R, d_model/32] E8M0 bytes, exponent floor(log2(amax of the 32-block)) - 8 (0 for a zero block).
 * a_q / a_s may be NULL (not written).  Uses the workspace.  Ids outside [0, E) are reported by
 * moe_check and treated as expert 0.  With MOE_ACT_MXFP4 set on the handle a_q is [R, d_model/2]
 * packed E2M1 codes and the a_s exponent is floor(log2(amax)) - 2.
 * Passage: the gate's top-6 routing feeds a dispatch to the routed expert FFNs and a combine back
 * (pypto page, "MoE and output stages"), here one GPU's permutation instead of an EP collective.  The
 * MXFP8 element rules (E4M3 round-to-nearest-even, saturating; E8M0 = floor(log2 amax) - 8) are the OCP
 * MX ones the layer contract names; the pages' own kernels quantise activations per token to INT8.
 */
MOE_API moe_status_t moe_permute(moe_experts_t experts, const moe_input_t* x, const int32_t* topk_ids, int32_t* counts,
                         int32_t* offsets, int32_t* perm_tok, int32_t* inv_pos, uint8_t* a_q, uint8_t* a_s,
                         moe_stream_t stream);

/*
 * Grouped expert FFN over n_rows MXFP8 rows a_q [n_rows, d_model] / a_s [n_rows, d_model/32]
 * (the layout moe_permute writes): row r belongs to expert g when offsets[g] <= r < offsets[g+1]
 * (offsets int32 [n+1] of the handle's n experts, offsets[0] = 0, offsets[n] = n_rows; NULL = every
 * row uses expert 0).  y[r] = row_w[r] * W2_g . q8(silu(min(W1_g a_r, L)) * clamp(W3_g a_r, -L, L)),
 * with q8 the MXFP8 quantisation along d_ff; row_w fp32 [n_rows] or NULL (= 1); y bf16
 * [n_rows, d_model].  Uses the workspace of the handle (n_rows <= max_T * (top_k + 1)).  With
 * MOE_ACT_MXFP4 set on the handle a_q is [n_rows, d_model/2] packed E2M1 codes and h is quantised to
 * MXFP4 instead (q8 becomes q4).
 * Passages: the expert FFN is a fused dequantisation + GEMM (FaStar README, "Features"); the linear
 * layers end in a SiLU-times-up op with clamp (SiLUMulClamp, TensorSharp page, "How TensorSharp runs it")
 * with swiglu_limit = 10 (model card, "Model Architecture and Objective"); w1 = gate, w3 = up, w2 =
 * down (ds4 issue, "Resolved questions").
 */
MOE_API moe_status_t moe_expert_ffn(moe_experts_t experts, int32_t n_rows, const int32_t* offsets, const uint8_t* a_q,
                            const uint8_t* a_s, const float* row_w, void* y_bf16, moe_stream_t stream);

/*
 * The whole layer: out[t] = sum_j w_tj * FFN_{e_tj}(x_t) + FFN_shared(x_t), bf16 [T, d_model]
 * (each weighted row kept as fp16 with a power-of-two scale per 32 columns, the rows summed in fp32 in
 * slot order, one rounding to bf16).  `shared` may be NULL (no shared expert).  Routing as in
 * moe_route (hash layers: router_w = router_bias = NULL).  The routing of the last call stays in
 * the workspace (moe_get_routing).  Everything stays on the device: the call never waits for the
 * GPU and copies nothing to or from the host.
 * Passages: gate -> top-6 -> dispatch -> routed and shared expert FFNs -> combine (pypto page, "MoE and
 * output stages"; 64 requests x 8 verify rows = 512 rows per step, its "Deployment configuration"); the
 * combine is a weighted-sum scatter epilogue after the expert FFNs (moe_scatter_add, TensorSharp page,
 * "DSpark and MoE CPU offload together" and "Fitting the model"); one always-on shared expert (model
 * card, "Speeds, Sizes, Times").
 */
MOE_API moe_status_t moe_forward(const moe_input_t* x, const float* router_w, const float* router_bias,
                         moe_experts_t experts, moe_experts_t shared, void* out_bf16, moe_stream_t stream);

/* Device pointers to the routing of the last moe_route / moe_forward on this handle (valid until
 * the next call): ids int32 [T, top_k], weights fp32 [T, top_k]. */
MOE_API moe_status_t moe_get_routing(moe_experts_t experts, const int32_t** topk_ids, const float** topk_w, int32_t* T);

/*
 * Stage timing (the per-stage timing the TensorSharp page exposes as TS_DSV4_PERF = 2).  events holds
 * n >= MOE_N_STAGES + 1 cudaEvent_t handles created by the caller; every later moe_forward on this
 * handle records events[i] on its stream before stage i and events[MOE_N_STAGES] after the last one.
 * Stages: 0 route, 1 dispatch (histogram, scan, quantise + gather), 2 gate-up GEMM, 3 down GEMM,
 * 4 combine.  The handle keeps the pointer array (not a copy) until it is replaced; events = NULL
 * switches the recording off.
 */
#define MOE_N_STAGES 5
MOE_API moe_status_t moe_set_stage_events(moe_experts_t experts, void* const* events, int32_t n);

/* Synchronise `stream`, then return and clear the handle's sticky device status:
 * MOE_OK, MOE_ERR_DEVICE_CHECK (range check) or MOE_ERR_TIMEOUT (bounded wait expired). */
MOE_API moe_status_t moe_check(moe_experts_t experts, moe_stream_t stream);

/* Upper bound, in nanoseconds, of every device-side wait (default 2 s). */
MOE_API moe_status_t moe_set_wait_budget(moe_experts_t experts, uint64_t budget_ns);

/*
 * Learned router that allocates nothing -- for callers that can't call cudaMalloc: plug-ins whose host
 * framework owns all device memory, and latency-critical paths that must not enter an allocator (an
 * allocation may synchronise the device or take a lock).  It needs no expert handle and no workspace.
 * (The pages have no counterpart; it is the same router as moe_route.)
 * Computes exactly what moe_route computes for a learned (not hash) layer: cfg gives d_model,
 * n_experts (<= 512), top_k and route_scale; x, router_w, router_bias, topk_ids, topk_w as there.
 * Its split-K partial sums live in one fixed 4 MiB array of library device memory (1,048,576 fp32),
 * which every GPU that loads the library holds until the process exits; batches with
 * T * n_experts > 1,048,576 (T > 4096 at 256 experts) are rejected with MOE_ERR_WORKSPACE.
 * Every call looks up that array's device address in the current context (so the address follows a
 * context that was destroyed and recreated); the first call on a device also loads the library's
 * device code there, so make that first call before any stream capture.  All calls share the array
 * and it keeps the last call's
 * contents (every call overwrites what it reads), so calls that overlap on the GPU -- on different
 * streams, or from several host threads -- race: order them.
 */
MOE_API moe_status_t moe_route_noalloc(const moe_config_t* cfg, const moe_input_t* x, const float* router_w,
                                       const float* router_bias, int32_t* topk_ids, float* topk_w,
                                       moe_stream_t stream);

/*
 * A stack of MoE layers run back to back on one stream.  It is the MoE part of a whole model in the
 * decode / verify regime: the model card's "Model Architecture and Objective" gives 43 layers, the first
 * ones hash-routed.  Every layer's experts stay resident in HBM.
 *
 * Layer l reads the bf16 residual stream x_l and writes x_{l+1} = bf16(x_l + moe_forward_l(x_l)).  The
 * residual enters the combine's fixed-order fp32 sum first, then the routed rows, then the shared row.
 *
 * moe_stack_layer_t (one layer)
 *   experts      required; its hash table (moe_experts_set_hash_table) makes the layer hash-routed.
 *   shared       may be NULL.
 *   router_w     NULL on hash layers; on the others required unless the handle has a resident router
 *                (moe_experts_set_router), which NULL selects.
 *   router_bias  likewise.
 * The stack keeps these pointers; the caller owns the handles and buffers and keeps them alive.  Every
 * layer handle needs a workspace (moe_set_workspace).  Layers may share one workspace: they run one after
 * the other on the same stream.
 *
 * moe_stack_create
 *   Validates the layers (same d_model; router weights exactly on the non-hash layers).
 *   use_graph != 0: moe_stack_forward records all layers' launches once into a CUDA graph and replays it.
 *   Returns MOE_ERR_INVALID_ARG on bad layers.
 *
 * moe_stack_forward
 *   x           bf16 [T, d] (its token_ids serve the hash layers).
 *   out         bf16 [T, d]: receives x_L.
 *   scratch     bf16 [T, d]: intermediate x_l; needed when there is more than one layer.
 *   x, out and scratch must be distinct and 16-byte aligned.
 *   Without graph mode: enqueues L moe_forward-equivalent launch sequences on the stream.
 *   With graph mode:
 *     - On the first call, or when x, token_ids, out, scratch or T differ from the captured ones, or when
 *       a setter (moe_set_workspace, moe_experts_set_router, moe_experts_set_hash_table,
 *       moe_experts_set_activation_format, moe_set_wait_budget, moe_set_stage_events) has been called on
 *       one of the layers' handles since the capture, it runs the layers once directly on a private
 *       stream, captures them into a graph there, and synchronises.  The call returns with the result
 *       already in out.
 *     - Otherwise it launches the cached graph on the stream.
 *   Device-side status is reported per layer handle by moe_check.  Host-side validation and CUDA errors
 *   are returned.
 */
typedef struct moe_stack_s* moe_stack_t;
typedef struct {
  moe_experts_t experts;
  moe_experts_t shared;
  const float* router_w;
  const float* router_bias;
} moe_stack_layer_t;

MOE_API moe_status_t moe_stack_create(const moe_stack_layer_t* layers, int32_t n_layers, int32_t use_graph,
                                      moe_stack_t* out);
MOE_API moe_status_t moe_stack_forward(moe_stack_t stack, const moe_input_t* x, void* out_bf16, void* scratch_bf16,
                                       moe_stream_t stream);
MOE_API void moe_stack_destroy(moe_stack_t stack);

/*
 * Checkpoint ingest: an array of 17-byte MXFP4 blocks -> the canonical codes and scales of
 * moe_experts_create.  Each block is one E8M0 scale byte followed by 16 bytes holding 32 E2M1 codes
 * (sign bit 3).  The format comes from the model card's "Conversion to the .fst container" (17-byte
 * blocks, 1 e8m0 scale + the FP4 codes).  The TensorSharp page's "Getting a drafter" says the checkpoint
 * is GGUF's MXFP4 layout up to nibble order, so the caller names the order:
 *   MOE_MX_NIBBLES_PAIRED  byte i holds elements 2i (low nibble) and 2i+1 (high nibble): canonical.
 *   MOE_MX_NIBBLES_SPLIT   byte i holds elements i (low nibble) and i+16 (high nibble).
 * A [rows x K] matrix stored as rows * K/32 blocks, row-major, becomes:
 *   codes   [rows][K/2], element 2i in the low nibble of byte i;
 *   scales  [rows][K/32].
 * blocks is device memory of 17 * n_blocks bytes; codes (16 * n_blocks) and scales (n_blocks) are
 * caller-owned device memory.  Asynchronous on the stream.  Returns MOE_ERR_INVALID_ARG for a NULL
 * buffer, a negative count or an unknown order; n_blocks = 0 does nothing.
 */
enum { MOE_MX_NIBBLES_PAIRED = 0, MOE_MX_NIBBLES_SPLIT = 1 };
MOE_API moe_status_t moe_mx_blocks_unpack(const uint8_t* blocks, int64_t n_blocks, int32_t nibble_order,
                                          uint8_t* codes, uint8_t* scales, moe_stream_t stream);

MOE_API void moe_experts_destroy(moe_experts_t experts);
MOE_API const char* moe_status_string(moe_status_t status);
/* Text of the last host-side error on this thread ("" if none). */
MOE_API const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
