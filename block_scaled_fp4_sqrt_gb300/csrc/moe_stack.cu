// A stack of MoE layers run back to back on one stream: the MoE part of a whole DeepSeek-V4-Flash-style
// model in the decode / verify regime (43 layers, the first ones hash-routed: model card, "Model
// Architecture and Objective"; every layer's 256 routed + 1 shared experts resident in HBM, which the
// 13.4 MB-per-expert payload of the FaStar README, "Expert virtual memory", puts at 148 GB).
//
// Layer l reads the bf16 residual stream x_l and writes x_{l+1} = bf16(x_l + MoE_l(x_l)): the combine
// kernel adds the residual in its fixed-order fp32 sum, so the stream costs no extra pass.  Buffers
// ping-pong between the caller's output and scratch so that the last layer writes the output.
//
// With graph mode on, the first call (and any call whose pointers or batch size differ from the
// captured ones, or after a setter changed a layer handle) records every layer's launches on a private
// stream into one CUDA graph; later calls replay it on the caller's stream, which removes the host work
// of L x 9 launches and their tensor-map encodes.  The captured kernels read the buffers named at
// capture time, whose contents may change freely between calls.  A handle setter (a new workspace,
// router, hash table, activation format, wait budget, stage events) changes the handle's generation,
// which is part of the graph's key, so a replay never reaches a buffer the handle no longer uses.
#include <vector>

#include "moe_internal.h"

struct moe_stack_s {
  std::vector<moe_stack_layer_t> layers;
  int d_model = 0;
  int use_graph = 0;
  cudaStream_t capture = nullptr;
  cudaGraphExec_t exec = nullptr;
  // what the cached graph was captured with
  const void* key_x = nullptr;
  const int32_t* key_tok = nullptr;
  void* key_out = nullptr;
  void* key_scratch = nullptr;
  int32_t key_T = -1;
  std::vector<uint64_t> key_gen;  // generations of every layer's routed and shared handles
};

namespace {

moe_status_t stack_fail(moe_status_t st, const char* msg) {
  moe::set_last_error(msg);
  return st;
}

// Enqueue every layer on stream s.
moe_status_t run_layers(moe_stack_s* st, const moe_input_t* x, void* out, void* scratch, cudaStream_t s) {
  const int L = (int)st->layers.size();
  const void* in = x->x_bf16;
  for (int l = 0; l < L; ++l) {
    void* dst = ((L - 1 - l) % 2 == 0) ? out : scratch;
    const moe_stack_layer_t& ly = st->layers[(size_t)l];
    moe_input_t xi{in, x->T, moe::experts_has_hash_table(ly.experts) ? x->token_ids : nullptr};
    const moe_status_t r = moe::forward_impl(&xi, ly.router_w, ly.router_bias, ly.experts, ly.shared, dst, in,
                                             reinterpret_cast<moe_stream_t>(s));
    if (r != MOE_OK) return r;
    in = dst;
  }
  return MOE_OK;
}

std::vector<uint64_t> generations(const moe_stack_s* st) {
  std::vector<uint64_t> g;
  g.reserve(2 * st->layers.size());
  for (const moe_stack_layer_t& ly : st->layers) {
    g.push_back(moe::experts_generation(ly.experts));
    g.push_back(moe::experts_generation(ly.shared));
  }
  return g;
}

}  // namespace

extern "C" {

moe_status_t moe_stack_create(const moe_stack_layer_t* layers, int32_t n_layers, int32_t use_graph,
                              moe_stack_t* out) {
  if (!out) return stack_fail(MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!layers || n_layers < 1) return stack_fail(MOE_ERR_INVALID_ARG, "need at least one layer");
  const int d = moe::experts_d_model(layers[0].experts);
  for (int l = 0; l < n_layers; ++l) {
    if (!layers[l].experts) return stack_fail(MOE_ERR_INVALID_ARG, "a layer has no routed expert handle");
    if (moe::experts_d_model(layers[l].experts) != d)
      return stack_fail(MOE_ERR_INVALID_ARG, "layers differ in d_model");
    if (layers[l].shared && moe::experts_d_model(layers[l].shared) != d)
      return stack_fail(MOE_ERR_INVALID_ARG, "a shared expert differs in d_model");
    const bool hashed = moe::experts_has_hash_table(layers[l].experts) != 0;
    const bool given = layers[l].router_w != nullptr;
    if (hashed ? given : !(given || moe::experts_has_resident_router(layers[l].experts)))
      return stack_fail(MOE_ERR_INVALID_ARG,
                        "a layer needs either a hash table or router weights (given, or resident), not both");
  }
  moe_stack_s* st = new moe_stack_s();
  st->layers.assign(layers, layers + n_layers);
  st->d_model = d;
  st->use_graph = use_graph ? 1 : 0;
  *out = st;
  return MOE_OK;
}

moe_status_t moe_stack_forward(moe_stack_t st, const moe_input_t* x, void* out_bf16, void* scratch_bf16,
                               moe_stream_t stream) {
  if (!st || !x) return stack_fail(MOE_ERR_INVALID_ARG, "stack or input is NULL");
  if (x->T < 0) return stack_fail(MOE_ERR_INVALID_ARG, "T is negative");
  if (x->T == 0) return MOE_OK;
  if (!x->x_bf16 || !out_bf16) return stack_fail(MOE_ERR_INVALID_ARG, "x or out is NULL");
  if (st->layers.size() > 1 && !scratch_bf16)
    return stack_fail(MOE_ERR_INVALID_ARG, "a stack of more than one layer needs a scratch buffer");
  if (out_bf16 == x->x_bf16 || (scratch_bf16 && (scratch_bf16 == x->x_bf16 || scratch_bf16 == out_bf16)))
    return stack_fail(MOE_ERR_INVALID_ARG, "x, out and scratch must be distinct buffers");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!st->use_graph) return run_layers(st, x, out_bf16, scratch_bf16, s);

  std::vector<uint64_t> gen = generations(st);
  const bool hit = st->exec && st->key_x == x->x_bf16 && st->key_tok == x->token_ids && st->key_out == out_bf16 &&
                   st->key_scratch == scratch_bf16 && st->key_T == x->T && st->key_gen == gen;
  if (!hit) {
    if (!st->capture && cudaStreamCreateWithFlags(&st->capture, cudaStreamNonBlocking) != cudaSuccess)
      return stack_fail(MOE_ERR_CUDA, "could not create the capture stream");
    // one direct pass first: it initialises the kernels' one-time attributes outside the capture and
    // leaves the same results the graph will produce
    if (cudaStreamSynchronize(s) != cudaSuccess) return stack_fail(MOE_ERR_CUDA, "stream synchronise failed");
    moe_status_t r = run_layers(st, x, out_bf16, scratch_bf16, st->capture);
    if (r != MOE_OK) return r;
    if (cudaStreamBeginCapture(st->capture, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
      return stack_fail(MOE_ERR_CUDA, "could not begin the graph capture");
    r = run_layers(st, x, out_bf16, scratch_bf16, st->capture);
    cudaGraph_t graph = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(st->capture, &graph);
    if (r != MOE_OK) {
      if (graph) cudaGraphDestroy(graph);
      return r;
    }
    if (ce != cudaSuccess || !graph) return stack_fail(MOE_ERR_CUDA, "graph capture failed");
    cudaGraphExec_t exec = nullptr;
    const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ie != cudaSuccess) return stack_fail(MOE_ERR_CUDA, "graph instantiation failed");
    if (st->exec) cudaGraphExecDestroy(st->exec);
    st->exec = exec;
    st->key_x = x->x_bf16;
    st->key_tok = x->token_ids;
    st->key_out = out_bf16;
    st->key_scratch = scratch_bf16;
    st->key_T = x->T;
    st->key_gen = std::move(gen);
    // the direct pass ran on the capture stream: order the caller's stream after it
    if (cudaStreamSynchronize(st->capture) != cudaSuccess) return stack_fail(MOE_ERR_CUDA, "capture stream failed");
    return MOE_OK;
  }
  if (cudaGraphLaunch(st->exec, s) != cudaSuccess) return stack_fail(MOE_ERR_CUDA, "graph launch failed");
  return MOE_OK;
}

void moe_stack_destroy(moe_stack_t st) {
  if (!st) return;
  if (st->exec) cudaGraphExecDestroy(st->exec);
  if (st->capture) cudaStreamDestroy(st->capture);
  delete st;
}

}  // extern "C"
