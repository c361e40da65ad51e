"""Parity of the CUDA layer (through its C ABI) with the fp64 oracle, on
seeded inputs small enough for the oracle to finish in seconds but spanning
several 128-row tiles, ragged expert segments, both score functions, the
shared expert, skewed routing, empty experts and the degenerate cases
(one expert; k = E)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from harness import full_parity, run_gpu, check_routing, oracle_layer, compare_all

pytestmark = pytest.mark.gpu

W = mi.WORKLOADS
CASES = {
    "tiny_fp32": W["tiny_fp32"],
    "mixtral_small": mi.scaled(W["mixtral_8x7b"], T=333, H=256, F=512),
    "deepseek_small": mi.scaled(W["deepseek_v3"], T=260, H=256, E=16, F=256, Fs=256),
    "qwen_small_ragged_n": mi.scaled(W["qwen3_235b"], T=520, H=384, E=32, F=384),
    "fp32_sigmoid_shared": mi.scaled(W["deepseek_v3"], T=100, H=128, E=4, k=2, F=128, Fs=128,
                                     dtype=mi.FP32),
    "single_expert_top1": mi.scaled(W["mixtral_8x7b"], T=150, H=128, E=1, k=1, F=256),
    "k_equals_E": mi.scaled(W["mixtral_8x7b"], T=100, H=128, E=4, k=4, F=128),
    "softmax_bias_k3": mi.scaled(W["qwen3_235b"], T=400, H=256, E=12, k=3, F=256),
    "rows_in_cta_pairs": mi.scaled(W["mixtral_8x7b"], T=1100, H=256, E=4, k=2, F=256),
    # CTA pairs over the experts of two or more tiles (an odd last tile beside
    # a ghost) plus single CTAs over the one-tile experts: expert tile counts
    # 1, 2, 3, 5, 7 (Zipf) and 1-4 with an exactly full 128-row segment
    # (sigmoid, bias, shared expert)
    "pairs_and_one_tile_experts_zipf": mi.scaled(W["qwen3_235b"], T=1300, H=256, E=8, k=2, F=256),
    "deepseek_pairs_and_one_tile_experts": mi.scaled(W["deepseek_v3"], T=1040, H=256, E=16, k=4,
                                                     F=256, Fs=128),
    "qwen_e128_tiled_router": mi.scaled(W["qwen3_235b"], T=700, H=256, E=128, F=128),
    "deepseek_e256_sigmoid_shared": mi.scaled(W["deepseek_v3"], T=512, H=256, E=256, F=128, Fs=128),
    # tiled router for E > 32: E not a multiple of 4 (Wr rows copied in 4-byte
    # pieces), E/32 rounded up to 2 and 4 experts per lane, a ragged last
    # router block (T = 257), and fp32 activations through the same kernel
    "e37_router_unaligned_rows": mi.scaled(W["qwen3_235b"], T=300, H=256, E=37, k=3, F=128),
    "e100_router_ragged_block": mi.scaled(W["deepseek_v3"], T=257, H=384, E=100, k=6, F=128, Fs=0),
    "fp32_e42_router": mi.scaled(W["qwen3_235b"], T=97, H=128, E=42, k=2, F=128, dtype=mi.FP32),
    # degenerate sizes: one token (one router block, one padded row per expert)
    "one_token": mi.scaled(W["mixtral_8x7b"], T=1, H=128, E=4, k=2, F=128),
    "one_token_fp32_shared": mi.scaled(W["deepseek_v3"], T=1, H=128, E=8, k=3, F=128, Fs=128,
                                       dtype=mi.FP32),
}


@pytest.mark.parametrize("name", list(CASES))
def test_layer_matches_oracle(name):
    rep, _ = full_parity(CASES[name])
    print(name, rep)


# Memory-efficient permutation: the same layer with the routing weights
# folded into the expert activations must meet the same bounds.
FOLD_CASES = ["tiny_fp32", "mixtral_small", "deepseek_small", "qwen_small_ragged_n",
              "fp32_sigmoid_shared", "rows_in_cta_pairs", "deepseek_e256_sigmoid_shared",
              "deepseek_pairs_and_one_tile_experts"]


@pytest.mark.parametrize("name", FOLD_CASES)
def test_folded_gates_match_oracle(name):
    rep, _ = full_parity(CASES[name], fold=True)
    print(name, "folded", rep)


# Capacity-limited dropping: (case, capacity factor, folded gates); every case
# drops assignments of its busiest experts. The Zipf-biased Qwen-shaped case is
# routed so unevenly (one expert gets 487 of 520 tokens) that a factor of 1
# drops 37% of all slots; the max/rms bound is relative to the rms of the
# reference, which shrinks with every dropped expert output while the bf16
# rounding of the kept ones does not, so that case uses a factor of 2 (14%);
# the CTA-pair and DeepSeek-shaped cases drop a few assignments (13 and 7), the
# Zipf case with one-tile experts 237 of the hottest expert's 887.
CAPACITY_CASES = [("mixtral_small", 0.6, False), ("qwen_small_ragged_n", 2.0, False),
                  ("fp32_sigmoid_shared", 0.75, False), ("rows_in_cta_pairs", 1.0, False),
                  ("deepseek_small", 1.5, True), ("mixtral_small", 0.6, True),
                  ("pairs_and_one_tile_experts_zipf", 2.0, False)]


@pytest.mark.parametrize("name,cf,fold", CAPACITY_CASES)
def test_capacity_dropping_matches_oracle(name, cf, fold):
    import oracle
    w = CASES[name]
    rep, gpu = full_parity(w, fold=fold, capacity_factor=cf)
    C = oracle.capacity(w.T, w.k, w.E, cf)
    assert int(gpu["counts"].max()) > C, "case drops nothing"
    print(name, cf, "fold" if fold else "", rep)


@pytest.mark.parametrize("name", ["tiny_fp32", "mixtral_small", "qwen_e128_tiled_router",
                                  "deepseek_e256_sigmoid_shared"])
def test_router_replay_matches_oracle(name):
    """Router replay: the given experts are used for every token; scores and
    gates come from the logits over that set."""
    import oracle
    w = CASES[name]
    inp = mi.make_inputs(w)
    rng = np.random.default_rng(7)
    replay = np.stack([rng.choice(w.E, w.k, replace=False) for _ in range(w.T)]).astype(np.int32)
    gpu, _ = run_gpu(w, inp, replay=replay)
    assert np.array_equal(gpu["topk_idx"].numpy(), replay)
    x, Wr, b = (None if inp[n] is None else inp[n].float().numpy().astype(np.float64) for n in ("x", "Wr", "b"))
    r = oracle.route(x, Wr, b, w.k, w.score, replay_topk=replay, replay_mask=np.ones(w.T, bool))
    assert np.array_equal(r["topk"], replay)
    np.testing.assert_allclose(gpu["gates"].numpy(), r["gates"], rtol=1e-4, atol=1e-6)
    ref = oracle_layer(w, inp, r)
    print(name, compare_all(w, inp, r, gpu, ref))


def test_router_replay_out_of_range_is_reported():
    import mixture_experts_layer_sigmoid_gb300 as moe
    w = CASES["mixtral_small"]
    inp = mi.make_inputs(w)
    replay = np.zeros((w.T, w.k), np.int32)
    replay[:, 1] = 1
    replay[5, 0] = w.E                         # outside [0, E)
    g = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score, dtype=w.dtype)
    layer.forward(g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"],
                  replay_topk=torch.as_tensor(replay).cuda())
    torch.cuda.synchronize()
    assert layer.status(w.T) == moe.MOE_ERR_INVALID_ARG


def test_folded_gates_shrink_saved_buffer():
    import mixture_experts_layer_sigmoid_gb300 as moe
    w = CASES["deepseek_small"]
    a = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score, Fs=w.Fs)
    b = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score, Fs=w.Fs, fold_gates=True)
    sa, _ = moe.moe_workspace_size(a.plan, w.T)
    sb, _ = moe.moe_workspace_size(b.plan, w.T)
    rp = -(-(w.T * w.k + w.E * 127) // 128) * 128     # row capacity of the permuted buffers
    assert sa - sb >= 2 * rp * (w.F + w.H) - 2 * 256, (sa, sb)


def test_empty_experts_get_zero_gradients():
    w = mi.scaled(W["mixtral_8x7b"], T=200, H=256, E=8, k=2, F=256)
    inp = mi.make_inputs(w)
    b = torch.zeros(8)
    b[[1, 4]] = -30.0                       # experts 1 and 4 receive no token
    inp["b"] = b
    gpu, _ = run_gpu(w, inp)
    assert gpu["counts"][1] == 0 and gpu["counts"][4] == 0
    r, _ = check_routing(w, inp, gpu)
    ref = oracle_layer(w, inp, r)
    for e in (1, 4):
        for n in ("dW_gate", "dW_up", "dW_down"):
            assert torch.count_nonzero(gpu[n][e]) == 0
    compare_all(w, inp, r, gpu, ref)


# (case, folded gates) for the determinism and CUDA-graph tests: bf16 with a
# shared expert, fp32, the blockwise-FP8 layer, and the folded order
REPEAT_CASES = [("deepseek_small", False), ("fp32_sigmoid_shared", False), ("fp8_small", False),
                ("deepseek_small", True), ("fp8_small", True)]
FP8_SMALL = mi.scaled(W["qwen3_235b_fp8"], T=600, H=256, E=8, k=4, F=256)


def _case(name):
    return FP8_SMALL if name == "fp8_small" else CASES[name]


@pytest.mark.parametrize("name,fold", REPEAT_CASES)
def test_deterministic_bitwise(name, fold):
    w = _case(name)
    inp = mi.make_inputs(w)
    a, layer = run_gpu(w, inp, fold=fold)
    b, _ = run_gpu(w, inp, layer=layer)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_bad_call_arguments_are_rejected_before_launch():
    import ctypes
    import mixture_experts_layer_sigmoid_gb300 as moe
    w = CASES["mixtral_small"]
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T)
    lib = moe.load_library()
    saved, ws = layer.buffers(w.T)
    x = torch.zeros(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    args = moe.moe_fwd_args_t(x=x.data_ptr(), Wr=x.data_ptr(), W_gate=x.data_ptr(), W_up=x.data_ptr(),
                              W_down=x.data_ptr(), y=x.data_ptr())
    st = lib.moe_forward(layer.plan, w.T, ctypes.byref(args), saved.data_ptr(), 16, ws.data_ptr(),
                         ws.numel(), None)
    assert st == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    st = lib.moe_forward(layer.plan, w.T + 1, ctypes.byref(args), saved.data_ptr(), saved.numel(),
                         ws.data_ptr(), ws.numel(), None)
    assert st == moe.MOE_ERR_INVALID_ARG
    args.x = x.data_ptr() + 2
    st = lib.moe_forward(layer.plan, w.T, ctypes.byref(args), saved.data_ptr(), saved.numel(),
                         ws.data_ptr(), ws.numel(), None)
    assert st == moe.MOE_ERR_MISALIGNED
    args.x = x.data_ptr()
    args.Ws_gate = x.data_ptr()            # shared weights on a layer without a shared expert
    st = lib.moe_forward(layer.plan, w.T, ctypes.byref(args), saved.data_ptr(), saved.numel(),
                         ws.data_ptr(), ws.numel(), None)
    assert st == moe.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("name,fold", REPEAT_CASES)
def test_forward_backward_capture_in_a_cuda_graph(name, fold):
    """A call enqueues kernels only (no host synchronisation, no allocation),
    so forward + backward can be captured once and replayed; the replay
    reproduces the eager results bit for bit."""
    import mixture_experts_layer_sigmoid_gb300 as moe
    w = _case(name)
    inp = mi.make_inputs(w)
    g = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score, dtype=w.dtype, Fs=w.Fs, fold_gates=fold)
    args = (g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"], g["Wsg"], g["Wsu"], g["Wsd"])
    y = torch.empty_like(g["x"])
    grads = None
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.forward(*args, y=y)
        grads = layer.backward(g["dY"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], g["Wsg"],
                               g["Wsu"], g["Wsd"])
    torch.cuda.synchronize()
    eager = {"y": y.clone(), **{k: v.clone() for k, v in grads.items()}}
    for t in [y, *grads.values()]:
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        layer.forward(*args, y=y)
        layer.backward(g["dY"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], g["Wsg"], g["Wsu"],
                       g["Wsd"], grads=grads)
    graph.replay()
    torch.cuda.synchronize()
    assert layer.status(w.T) == 0
    assert torch.equal(y, eager["y"])
    for k, v in grads.items():
        assert torch.equal(v, eager[k]), k


def test_update_bias_matches_oracle():
    import oracle
    import mixture_experts_layer_sigmoid_gb300 as moe
    rng = np.random.default_rng(3)
    for E in (1, 8, 37, 256):
        counts = rng.integers(0, 500, E).astype(np.int32)
        if E == 8:
            counts[:] = 40                         # balanced: no change
        b = rng.standard_normal(E).astype(np.float32)
        c_d = torch.as_tensor(counts).cuda()
        b_d = torch.as_tensor(b).cuda()
        moe.moe_update_bias(E, c_d.data_ptr(), 0.01, b_d.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert np.array_equal(b_d.cpu().numpy(), oracle.update_bias(b, counts, 0.01)), E
