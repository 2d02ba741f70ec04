"""moe_stack_forward: layers run back to back on the bf16 residual stream x_{l+1} = bf16(x_l + y_l).

Each layer is checked against the oracle on the GPU's own input to that layer (a prefix of the stack):
expert ids bit for bit, and x_{l+1} within the layer tolerance plus one bf16 rounding of x_l + y_l.
The graph mode must reproduce the direct launches bit for bit, follow new input contents on replay,
and re-capture when the batch size changes.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

from gpu_support import TOL_MAX_RMS, TOL_MEAN_REL, bf16_to_f64, device, x_to_device

pytestmark = pytest.mark.gpu

T = 16
HASH = synth.Workload("stack_hash", T, 256, 128, 8, 2, hash_vocab=100)
LEARNED = synth.Workload("stack_learned", T, 256, 128, 8, 2)
SEEDS = [100, 101, 102, 103]


@pytest.fixture(scope="module")
def stack_layers():
    import __graft_entry__ as g
    g.build_cuda()
    from block_scaled_fp4_sqrt_gb300 import MoELayer
    inputs = [synth.gen_layer(HASH if i == 0 else LEARNED, s) for i, s in enumerate(SEEDS)]
    layers = [MoELayer.from_host(inp, device=device(), max_T=T) for inp in inputs]
    yield inputs, layers
    for ly in layers:
        ly.close()


def _stack(layers, use_graph=False):
    from block_scaled_fp4_sqrt_gb300 import MoEStack
    return MoEStack(layers, max_T=T, use_graph=use_graph)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def test_stack_matches_the_oracle_layer_by_layer(stack_layers):
    inputs, layers = stack_layers
    x0 = synth.gen_x(7, T, 256)
    tok = torch.from_numpy(inputs[0].token_ids).to(device())
    x_l = x0
    for l in range(len(layers)):
        st = _stack(layers[: l + 1])
        out = st.forward(x_to_device(x0), token_ids=tok)
        torch.cuda.synchronize()
        st.check()
        x_next = _bits(out)
        inp = inputs[l]
        ids_gpu = layers[l].last_topk_ids().cpu().numpy()
        if inp.hash_table is not None:
            ids_ref, wts_ref = oracle.hash_route(inp.token_ids, inp.hash_table, 2, 1.5)
        else:
            ids_ref, wts_ref, margin = oracle.route(x_l, inp.router_w, inp.router_bias, 2, 1.5)
            assert margin.min() > 1e-5, f"layer {l}: a top-k gap of {margin.min():.2e} is too close to call"
        assert np.array_equal(ids_gpu, ids_ref), f"layer {l}: expert ids differ"
        y_ref = oracle.layer(x_l, ids_ref, wts_ref, inp.experts, inp.shared, 10.0)
        xl = bf16_to_f64(torch.from_numpy(x_l.view(np.int16)).view(torch.bfloat16))
        want = xl + y_ref
        got = bf16_to_f64(torch.from_numpy(x_next.view(np.int16)).view(torch.bfloat16))
        rms = float(np.sqrt(np.mean(y_ref ** 2)))
        err = np.abs(got - want)
        assert np.all(err <= TOL_MAX_RMS * rms + 2.0 ** -8 * np.abs(want)), f"layer {l}: max error {err.max():.3e}"
        assert err.sum() <= TOL_MEAN_REL * np.abs(y_ref).sum() + 2.0 ** -8 * np.abs(want).sum(), f"layer {l}"
        st.close()
        x_l = x_next


def test_graph_replay_matches_direct_launches(stack_layers):
    inputs, layers = stack_layers
    tok = torch.from_numpy(inputs[0].token_ids).to(device())
    xa = x_to_device(synth.gen_x(7, T, 256))
    xb = x_to_device(synth.gen_x(8, T, 256))
    direct, graph = _stack(layers), _stack(layers, use_graph=True)
    try:
        ref_a = direct.forward(xa, token_ids=tok).clone()
        ref_b = direct.forward(xb, token_ids=tok).clone()
        ref_h = direct.forward(xa[:8], token_ids=tok[:8]).clone()
        x = xa.clone()
        out = torch.empty_like(x)
        graph.forward(x, token_ids=tok, out=out)  # capture
        torch.cuda.synchronize()
        assert torch.equal(out, ref_a)
        x.copy_(xb)  # same buffers, new contents: a replay
        graph.forward(x, token_ids=tok, out=out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_b)
        x.copy_(xa)
        graph.forward(x, token_ids=tok, out=out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_a)
        out8 = torch.empty((8, 256), dtype=torch.bfloat16, device=device())
        graph.forward(x[:8], token_ids=tok[:8], out=out8)  # another batch size: a new capture
        torch.cuda.synchronize()
        assert torch.equal(out8, ref_h)
        graph.check()
    finally:
        direct.close()
        graph.close()


def test_stack_rejects_aliased_buffers(stack_layers):
    from block_scaled_fp4_sqrt_gb300 import MoEError
    inputs, layers = stack_layers
    st = _stack(layers)
    try:
        x = x_to_device(synth.gen_x(7, T, 256))
        tok = torch.from_numpy(inputs[0].token_ids).to(device())
        with pytest.raises(MoEError):
            st.forward(x, token_ids=tok, out=x)
    finally:
        st.close()


def test_stack_with_resident_routers(stack_layers):
    """Learned layers whose router is resident on the handle (moe_experts_set_router): the same output
    as the stack that passes router weights, directly and replayed from a graph."""
    from block_scaled_fp4_sqrt_gb300 import moe_experts_set_router
    inputs, layers = stack_layers
    tok = torch.from_numpy(inputs[0].token_ids).to(device())
    x = x_to_device(synth.gen_x(9, T, 256))
    ref_st = _stack(layers)
    ref = ref_st.forward(x, token_ids=tok).clone()
    ref_st.close()
    learned = [ly for ly in layers if ly.hash_table is None]
    try:
        for ly in learned:
            moe_experts_set_router(ly.h, ly.router_w, ly.router_bias)
            ly.resident_router = True
        for use_graph in (False, True):
            st = _stack(layers, use_graph=use_graph)
            out = torch.empty_like(x)
            st.forward(x, token_ids=tok, out=out)
            st.forward(x, token_ids=tok, out=out)
            torch.cuda.synchronize()
            st.check()
            assert torch.equal(out, ref)
            st.close()
    finally:
        for ly in learned:
            ly.resident_router = False
            moe_experts_set_router(ly.h, None, None)


def test_graph_recaptures_after_a_handle_setter(stack_layers):
    """A cached graph bakes in each layer's workspace.  After moe_set_workspace moves every layer to a new
    buffer and the old one is freed (filled with garbage first, so stale reads would show), the next call
    must capture again and still reproduce the direct launches bit for bit."""
    from block_scaled_fp4_sqrt_gb300 import moe_set_workspace, moe_workspace_size
    inputs, layers = stack_layers
    tok = torch.from_numpy(inputs[0].token_ids).to(device())
    x = x_to_device(synth.gen_x(11, T, 256))
    direct, graph = _stack(layers), _stack(layers, use_graph=True)
    try:
        ref = direct.forward(x, token_ids=tok).clone()
        out = torch.empty_like(x)
        graph.forward(x, token_ids=tok, out=out)  # capture
        graph.forward(x, token_ids=tok, out=out)  # replay
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        old = graph.workspaces[0]
        new = torch.empty(moe_workspace_size(layers[0].cfg, T), dtype=torch.uint8, device=device())
        for ly in layers:
            moe_set_workspace(ly.h, new, T)
        graph.workspaces = [new]
        old.fill_(0xA5)  # whatever the graph would read from the old buffer is now garbage
        torch.cuda.synchronize()
        del old
        out.zero_()
        graph.forward(x, token_ids=tok, out=out)  # the handles changed: a new capture
        graph.forward(x, token_ids=tok, out=out)  # and its replay
        torch.cuda.synchronize()
        graph.check()
        assert torch.equal(out, ref)
    finally:
        direct.close()
        graph.close()
