"""moe_route_static: routing for callers that cannot allocate device memory.

Some callers cannot give this library a workspace: their device memory is
owned by a framework pool or by a budget fixed at start-up, or they run in
loops that must not call cudaMalloc. moe_route_static routes tokens using a
scratch array built into the library instead. This test calls it through the
C ABI twice in a row, on two different inputs, and checks each result
against the routing outputs of the existing entry point, moe_forward (same
kernels, so the integers and the gates must agree exactly). It also checks
that a token count beyond the built-in scratch is refused before launch.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

import moe_inputs as mi
import mixture_experts_layer_sigmoid_gb300 as moe

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else t.data_ptr()


@pytest.mark.parametrize("dtype", [mi.FP32, mi.BF16, mi.FP8_BLOCK])
def test_route_static_matches_forward_on_two_calls_in_a_row(dtype):
    """fp32 activations route through the fp32 router; the bf16 and the
    blockwise-FP8 layers both route from bf16 activations."""
    lib = moe.load_library()
    base = mi.scaled(mi.WORKLOADS["qwen3_235b"], T=520, H=384, E=32, F=384, dtype=dtype)
    cases = [base, mi.scaled(base, T=333, seed=base.seed + 7)]
    layer = moe.MoELayer(base.H, base.E, base.F, base.k, base.T, score=base.score, dtype=dtype)
    stream = torch.cuda.current_stream().cuda_stream
    for w in cases:
        g = {k: (None if v is None else v.cuda()) for k, v in mi.make_inputs(w, with_grad_out=False).items()}
        _, ref = layer.forward(g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"], routing=True)
        out = dict(topk_idx=torch.full((w.T, w.k), -7, dtype=torch.int32, device="cuda"),
                   gates=torch.full((w.T, w.k), float("nan"), device="cuda"),
                   counts=torch.full((w.E,), -7, dtype=torch.int32, device="cuda"),
                   offsets=torch.full((w.E + 1,), -7, dtype=torch.int32, device="cuda"),
                   row_of=torch.full((w.T, w.k), -7, dtype=torch.int32, device="cuda"))
        st = lib.moe_route_static(layer.plan, w.T, _p(g["x"]), _p(g["Wr"]), _p(g["b"]),
                                  _p(out["topk_idx"]), _p(out["gates"]), _p(out["counts"]),
                                  _p(out["offsets"]), _p(out["row_of"]), stream)
        assert st == moe.MOE_OK, moe.moe_status_string(st)
        torch.cuda.synchronize()
        for name in ("topk_idx", "counts", "offsets", "row_of"):
            assert torch.equal(out[name], ref[name]), name
        torch.testing.assert_close(out["gates"], ref["gates"], rtol=0, atol=0)


def test_route_static_refuses_token_counts_beyond_its_scratch():
    lib = moe.load_library()
    layer = moe.MoELayer(256, 256, 256, 8, 40000, score=moe.MOE_SCORE_SIGMOID)
    buf = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    st = lib.moe_route_static(layer.plan, 40000, p, p, None, p, p, p, p, p, None)
    assert st == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    st = lib.moe_route_static(layer.plan, 2000, p, p, None, p, p, p, p, None, None)
    assert st == moe.MOE_ERR_INVALID_ARG
