"""The tiled router (E > 32) splits H across blocks and adds the splits'
partial logits in a fixed order. The split count is a function of H and E
alone, so

  * a token's top-k and gates must not depend on how many other tokens are in
    the call (a batch of 300 and its first 77 tokens route those 77 tokens
    identically, bit for bit), and
  * moe_route_static, which routes from its own built-in scratch, must give
    the same bits as moe_forward for these shapes too.

The shapes make the router split: H=384 gives 12 chunks per half at E=128 (6
splits) and 24 at E=256 (8 splits)."""
import ctypes

import pytest
import torch

import moe_inputs as mi
import mixture_experts_layer_sigmoid_gb300 as moe

pytestmark = pytest.mark.gpu

SHAPES = {
    "e128_softmax_zipf": mi.scaled(mi.WORKLOADS["qwen3_235b"], T=300, H=384, E=128, F=128),
    "e256_sigmoid_bias": mi.scaled(mi.WORKLOADS["deepseek_v3"], T=300, H=384, E=256, F=128, Fs=0),
}


def _inputs(w):
    return {k: (None if v is None else v.cuda()) for k, v in mi.make_inputs(w, with_grad_out=False).items()}


def _route(layer, g, T):
    _, out = layer.forward(g["x"][:T].contiguous(), g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"], routing=True)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_routing_of_a_token_does_not_depend_on_the_batch(name):
    w = SHAPES[name]
    g = _inputs(w)
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score)
    full = _route(layer, g, w.T)
    part = _route(layer, g, 77)
    assert torch.equal(part["topk_idx"], full["topk_idx"][:77])
    assert torch.equal(part["gates"], full["gates"][:77])


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_route_static_matches_forward_when_the_router_splits_h(name):
    w = SHAPES[name]
    g = _inputs(w)
    lib = moe.load_library()
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score)
    ref = _route(layer, g, w.T)
    out = dict(topk_idx=torch.full((w.T, w.k), -7, dtype=torch.int32, device="cuda"),
               gates=torch.full((w.T, w.k), float("nan"), device="cuda"),
               counts=torch.full((w.E,), -7, dtype=torch.int32, device="cuda"),
               offsets=torch.full((w.E + 1,), -7, dtype=torch.int32, device="cuda"),
               row_of=torch.full((w.T, w.k), -7, dtype=torch.int32, device="cuda"))
    p = lambda t: None if t is None else t.data_ptr()
    st = lib.moe_route_static(layer.plan, w.T, p(g["x"]), p(g["Wr"]), p(g["b"]), p(out["topk_idx"]),
                              p(out["gates"]), p(out["counts"]), p(out["offsets"]), p(out["row_of"]),
                              torch.cuda.current_stream().cuda_stream)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    torch.cuda.synchronize()
    for key in ("topk_idx", "counts", "offsets", "row_of"):
        assert torch.equal(out[key], ref[key]), key
    assert torch.equal(out["gates"], ref["gates"])


@pytest.mark.parametrize("E,router_kernels", [(8, 1), (128, 2)])
def test_stage_times_count_every_kernel_of_a_stage(E, router_kernels):
    """moe_stage_times reports kernel launches per stage, not calls: the router
    weight gradient is two kernels (tile partial sums, then their per-expert
    sums) and the router is two when it splits H (E > 32), one otherwise."""
    w = mi.scaled(mi.WORKLOADS["qwen3_235b"], T=300, H=384, E=E, k=2, F=128)
    g = {k: (None if v is None else v.cuda()) for k, v in mi.make_inputs(w).items()}
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score, stage_timing=True)
    layer.forward(g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"])
    layer.backward(g["dY"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    st = layer.stage_times()
    assert st["router"][0] == router_kernels
    assert st["router_wgrad"][0] == 2
    for name in ("scan", "index", "permute", "fc1_swiglu", "fc2", "combine", "fc1_wgrad"):
        assert st[name][0] == 1, name
