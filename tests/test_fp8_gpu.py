"""Blockwise-FP8 layer (MOE_FP8_BLOCK) on the GPU against the fp64 oracle.

The quantiser the layer uses must give the oracle's E4M3 bytes and fp32
scales bit for bit on the same bf16 input, in all four block layouts. The
whole layer (forward and backward) must match the oracle's FP8 layer within
the FP8 bounds on every output and gradient: relative L2 <= 4e-2 and
max |error| <= 1.5e-1 * rms(ref); weight gradients also within 4e-2 relative
L2 over every expert's block ("Scalable Training of Mixture-of-Experts
Models with Megatron Core", §5, blockwise FP8)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import mixture_experts_layer_sigmoid_gb300 as moe
from harness import TIE_REL, rel_errors, to_np, upload, write_report

pytestmark = pytest.mark.gpu


def _quant(x, mode, with_t=False):
    R, C = x.shape
    dev = x.device
    codes = torch.empty((R, C), dtype=torch.uint8, device=dev)
    codes_t = torch.empty((C, R), dtype=torch.uint8, device=dev)
    if mode == moe.MOE_Q_ROWS:
        sc = torch.empty((R, C // 128), device=dev)
        sct = torch.empty((C // 128, R // 128), device=dev) if with_t else None
    elif mode == moe.MOE_Q_TILES:
        sc, sct = torch.empty((R // 128, C // 128), device=dev), torch.empty((C // 128, R // 128), device=dev)
    elif mode == moe.MOE_Q_COLS_T:
        sc, sct = None, torch.empty((C, R // 128), device=dev)
    else:
        sc, sct = None, torch.empty((C // 128, R // 128), device=dev)
    p = lambda t: None if t is None else t.data_ptr()
    moe.moe_fp8_quantize(R, C, mode, x.data_ptr(), codes.data_ptr(), p(sc), codes_t.data_ptr(), p(sct),
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), None if sc is None else sc.cpu().numpy(), codes_t.cpu().numpy(), \
        None if sct is None else sct.cpu().numpy()


def test_quantisers_match_oracle_bit_for_bit():
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(384, 512, generator=g) * torch.logspace(-3, 2, 512)).to(torch.bfloat16)
    x[0:128, 0:128] = 0                      # an all-zero block (scale 1)
    x[200, 300] = 3.0e4                      # a large outlier
    xf = x.float().numpy()
    xd = x.cuda()
    c, s, _, _ = _quant(xd, moe.MOE_Q_ROWS)
    oc, os_ = oracle.fp8_quantize(xf, oracle.FP8_ROWS)
    assert np.array_equal(c, oc) and np.array_equal(s, os_)
    c, s, ct, st = _quant(xd, moe.MOE_Q_TILES)
    oc, os_ = oracle.fp8_quantize(xf, oracle.FP8_TILES)
    assert np.array_equal(c, oc) and np.array_equal(s, os_)
    oct_, ost = oracle.fp8_quantize(np.ascontiguousarray(xf.T), oracle.FP8_TILES)
    assert np.array_equal(ct, oct_) and np.array_equal(st, ost)
    _, _, ct, st = _quant(xd, moe.MOE_Q_COLS_T)
    oc, os_ = oracle.fp8_quantize(xf, oracle.FP8_COLS)
    assert np.array_equal(ct, oc.T) and np.array_equal(st, os_.T)
    _, _, ct, st = _quant(xd, moe.MOE_Q_TILES_T)
    assert np.array_equal(ct, oct_) and np.array_equal(st, ost)
    # one pass: 1x128 row codes and the transpose's 128x128-block codes
    c, s, ct, st = _quant(xd, moe.MOE_Q_ROWS, with_t=True)
    oc, os_ = oracle.fp8_quantize(xf, oracle.FP8_ROWS)
    assert np.array_equal(c, oc) and np.array_equal(s, os_)
    assert np.array_equal(ct, oct_) and np.array_equal(st, ost)


FP8_CASES = {
    "qwen_fp8_small": mi.scaled(mi.WORKLOADS["qwen3_235b_fp8"], T=600, H=256, E=8, k=4, F=256),
    "qwen_fp8_ragged": mi.scaled(mi.WORKLOADS["qwen3_235b_fp8"], T=450, H=384, E=16, k=8, F=384),
    # T*k >= 512*E: many row tiles per expert (odd tile counts), N = F = 384
    # ends in a half column tile
    "qwen_fp8_many_rows_per_expert": mi.scaled(mi.WORKLOADS["qwen3_235b_fp8"], T=1100, H=256, E=4, k=2,
                                               F=384),
}


@pytest.mark.parametrize("name", list(FP8_CASES))
def test_fp8_layer_matches_oracle(name):
    _fp8_parity(name, False)


@pytest.mark.parametrize("name", ["qwen_fp8_small", "qwen_fp8_many_rows_per_expert"])
def test_fp8_folded_gates_match_oracle(name):
    """Memory-efficient permutation on the FP8 layer: g h is quantised for
    fc2 instead of h; the same deviation bounds hold."""
    _fp8_parity(name, True)


def _fp8_parity(name, fold):
    print(name, fp8_layer_parity(FP8_CASES[name], fold))


# Capacity-limited dropping in both FP8 recipes: a dropped assignment never
# reaches its expert, so the quantisation blocks of the weight-gradient
# operands (128 or 32 rows along the tokens) hold the kept rows and zeros.
FP8_CAPACITY_CASES = [("qwen_fp8_small", mi.FP8_BLOCK, 1.0, False),
                      ("qwen_fp8_many_rows_per_expert", mi.FP8_BLOCK, 0.8, True),
                      ("qwen_fp8_small", mi.MXFP8, 1.0, False),
                      ("qwen_fp8_many_rows_per_expert", mi.MXFP8, 0.8, True),
                      ("qwen_fp8_ragged", mi.MXFP8, 1.5, False)]


@pytest.mark.parametrize("name,dtype,cf,fold", FP8_CAPACITY_CASES)
def test_fp8_capacity_dropping_matches_oracle(name, dtype, cf, fold):
    print(name, dtype, cf, fold, fp8_layer_parity(mi.scaled(FP8_CASES[name], dtype=dtype), fold, cf))


def fp8_layer_parity(w, fold=False, capacity_factor=0.0):
    """The FP8 layer on workload w (blockwise or MXFP8, by w.dtype) against
    the oracle's FP8 layer in the same recipe (bounds in the module
    docstring); with capacity_factor > 0 the oracle drops the same
    assignments (capacity_keep). Returns the error report."""
    inp = mi.make_inputs(w)
    g = upload(inp)
    mx = w.dtype == mi.MXFP8
    nv = w.dtype == mi.NVFP4
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score,
                         dtype=moe.MOE_NVFP4 if nv else moe.MOE_MXFP8 if mx else moe.MOE_FP8_BLOCK,
                         fold_gates=fold, capacity_factor=capacity_factor, Fs=w.Fs)
    ws = (g["Wsg"], g["Wsu"], g["Wsd"])
    y, rt = layer.forward(g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"], *ws, routing=True)
    gr = layer.backward(g["dY"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], *ws)
    torch.cuda.synchronize()
    assert layer.status(w.T) == 0
    d = {k: to_np(v) for k, v in inp.items()}
    r = oracle.route(d["x"], d["Wr"], d["b"], w.k, w.score)
    gt = rt["topk_idx"].cpu().numpy()
    tie = (r["gap_set"] < TIE_REL) | (r["gap_order"] < TIE_REL)
    mism = np.any(gt != r["topk"], axis=1)
    assert not np.any(mism & ~tie)
    if mism.any():
        r = oracle.route(d["x"], d["Wr"], d["b"], w.k, w.score, replay_topk=gt, replay_mask=mism)
    keep = None
    if capacity_factor > 0:
        C = oracle.capacity(w.T, w.k, w.E, capacity_factor)
        keep = oracle.capacity_keep(r["topk"], w.E, C)
        assert (keep == 0).any(), "case drops nothing"
    ref = oracle.layer_fp8(d["x"], d["Wr"], d["Wg"], d["Wu"], d["Wd"], r["topk"], r["gates"],
                           r["scores"], w.score, d["dY"], Wsg=d.get("Wsg"), Wsu=d.get("Wsu"),
                           Wsd=d.get("Wsd"), fold=fold,
                           recipe=oracle.RECIPE_NV if nv else oracle.RECIPE_MX if mx else oracle.RECIPE_BLOCK,
                           keep=keep)
    rep = {}

    def check(gname, got, want):
        rl2, mr = rel_errors(got, want)
        if nv:
            # NVFP4: an intermediate's E2M1 code one step off (a one-ulp bf16
            # difference on a rounding boundary) shifts a row of the output
            # (bounds in test_nv_gpu's docstring)
            rms = np.sqrt(np.mean(np.square(want))) if want.size else 0.0
            far = float(np.mean(np.abs(got - want) > 1.5e-1 * rms)) if rms > 0 else 0.0
            rep[gname] = (rl2, mr, far)
            assert rl2 <= 4e-2 and far <= 1e-3 and mr <= 1.0, (gname, rl2, mr, far)
        else:
            rep[gname] = (rl2, mr)
            assert rl2 <= 4e-2 and mr <= 1.5e-1, (gname, rl2, mr)

    for gname, oname in (("y", "y"), ("dX", "dX")):
        check(gname, to_np(y if gname == "y" else gr[gname]), ref[oname])
    shared = (("dWs_gate", "dWsg"), ("dWs_up", "dWsu"), ("dWs_down", "dWsd")) if w.Fs else ()
    for gname, oname in (("dWr", "dWr"), ("dW_gate", "dWg"), ("dW_up", "dWu"), ("dW_down", "dWd")) + shared:
        got = to_np(gr[gname])
        want = ref[oname]
        check(gname, got, want)
        blocks = zip(got.T, want.T) if gname == "dWr" else zip(got, want)
        for gb, wb in blocks:
            nw = np.linalg.norm(wb)
            if nw == 0:
                assert np.all(gb == 0)
            else:
                assert np.linalg.norm(gb - wb) / nw <= 4e-2, gname
    write_report(f"{w.name} T{w.T} H{w.H} E{w.E} k{w.k} F{w.F} {'nvfp4' if nv else 'mxfp8' if mx else 'fp8'}"
                 + (" fold" if fold else "") + (f" capacity {capacity_factor}" if capacity_factor else ""),
                 rep)
    return rep


@pytest.mark.parametrize("fold,dtype", [(False, mi.FP8_BLOCK), (True, mi.FP8_BLOCK), (False, mi.MXFP8)])
def test_fp8_weight_cache_gives_identical_results(fold, dtype):
    """Weights quantised once by moe_quantize_weights and passed as the
    weight cache (the bf16 weights not passed at all) give the same bits as
    the layer quantising them inside every forward; for the blockwise recipe
    the cache holds the oracle's 128x128-block codes."""
    w = mi.scaled(FP8_CASES["qwen_fp8_ragged"], dtype=dtype)
    g = upload(mi.make_inputs(w))
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score,
                         dtype=moe.MOE_MXFP8 if dtype == mi.MXFP8 else moe.MOE_FP8_BLOCK, fold_gates=fold)
    y0 = layer.forward(g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"])
    gr0 = layer.backward(g["dY"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    ref = {"y": y0.clone(), **{k: v.clone() for k, v in gr0.items()}}
    cache = layer.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    like = (g["Wg"], g["Wu"], g["Wd"])
    for _ in range(2):                         # the cache is reused across steps
        y1 = layer.forward(g["x"], g["Wr"], g["b"], None, None, None, weight_cache=cache)
        gr1 = layer.backward(g["dY"], g["x"], g["Wr"], None, None, None, weight_cache=cache, like=like)
        torch.cuda.synchronize()
        assert layer.status(w.T) == 0
        assert torch.equal(y1, ref["y"])
        for k, v in gr1.items():
            assert torch.equal(v, ref[k]), k
    if dtype == mi.MXFP8:
        return
    # the cache's first block: W_gate codes of expert 0 and their scales
    oc, os_ = oracle.fp8_quantize(g["Wg"][0].float().cpu().numpy(), oracle.FP8_TILES)
    n = w.H * w.F
    assert np.array_equal(cache[:n].cpu().numpy().reshape(w.H, w.F), oc)
    # scales follow the codes of all experts, 256-byte aligned
    off = -(-(w.E * n) // 256) * 256
    sc = cache[off:off + 4 * os_.size].cpu().view(torch.float32).numpy().reshape(os_.shape)
    assert np.array_equal(sc, os_)


def test_weight_cache_is_refused_outside_fp8():
    w = mi.scaled(FP8_CASES["qwen_fp8_small"], dtype=mi.BF16)
    g = upload(mi.make_inputs(w))
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score)
    assert moe.moe_weight_cache_size(layer.plan) == 0
    with pytest.raises(moe.MoEError) as e:
        layer.quantize_weights(g["Wg"], g["Wu"], g["Wd"], cache=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoEError) as e:
        layer.forward(g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"],
                      weight_cache=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
