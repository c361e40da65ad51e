"""Parity at the full layer sizes (Mixtral-8x7B-, DeepSeek-V3- and
Qwen3-235B-shaped expert layers), in the launch configuration bench.py times.

The whole layer runs on the GPU; the fp64 oracle then checks
  - routing for every token (top-k bit-exact except near-ties, counts,
    padded offsets and the full permutation),
  - y and dX rows of sampled tokens (first, last, hottest-expert and tied
    tokens), computed one by one by the oracle's per-token form,
  - sampled entries of the expert weight gradients (hottest and coldest
    non-empty expert, and the shared expert), each within the forward-error
    bound of the bf16 arithmetic.
dWr needs every routed token's expert outputs, so at these sizes it is
covered by the mid-size tests only.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from harness import TIE_REL, WGRAD_BOUND_SLACK, _expert_wgrad_bounds, rel_errors, to_np

pytestmark = pytest.mark.gpu

CONFIGS = ["mixtral_8x7b", "deepseek_v3", "qwen3_235b"]


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name", CONFIGS)
def test_full_size_layer(name):
    from mixture_experts_layer_sigmoid_gb300 import MoELayer
    w = mi.WORKLOADS[name]
    g = mi.make_inputs(w, "cuda")
    layer = MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score, dtype=w.dtype, Fs=w.Fs)
    y, rt = layer.forward(g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"], g["Wsg"], g["Wsu"],
                          g["Wsd"], routing=True)
    gr = layer.backward(g["dY"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], g["Wsg"], g["Wsu"],
                        g["Wsd"])
    torch.cuda.synchronize()
    assert layer.status(w.T) == 0

    # ---- routing of every token
    x = to_np(g["x"])
    dY = to_np(g["dY"])
    Wr = to_np(g["Wr"])
    b = to_np(g["b"])
    r = oracle.route(x, Wr, b, w.k, w.score)
    gt = rt["topk_idx"].cpu().numpy()
    tie = (r["gap_set"] < TIE_REL) | (r["gap_order"] < TIE_REL)
    mism = np.any(gt != r["topk"], axis=1)
    assert not np.any(mism & ~tie), f"top-k differs on non-tie tokens {np.nonzero(mism & ~tie)[0][:5]}"
    for t in np.nonzero(mism)[0]:
        s = r["scores"][t]
        kth = np.sort(s)[::-1][w.k - 1]
        assert np.all(s[gt[t]] >= kth * (1 - 2 * TIE_REL)), f"token {t}: invalid tied choice"
    if mism.any():
        r = oracle.route(x, Wr, b, w.k, w.score, replay_topk=gt, replay_mask=mism)
    d = oracle.dispatch(r["topk"], w.E)
    counts = d["counts"]
    assert np.array_equal(rt["counts"].cpu().numpy(), counts)
    poff = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    assert np.array_equal(rt["offsets"].cpu().numpy(), poff)
    e_of = r["topk"].astype(np.int64)
    mapped = rt["row_of"].cpu().numpy().astype(np.int64) - poff[e_of] + d["offsets"][e_of]
    assert np.array_equal(mapped, d["row_of"])
    np.testing.assert_allclose(rt["gates"].cpu().numpy(), r["gates"], rtol=1e-4, atol=1e-6)
    print(f"{name}: near-tie tokens {int(tie.sum())}, GPU chose differently on {int(mism.sum())}")

    # ---- sampled rows of y and dX
    hot = int(np.argmax(counts))
    nonempty = np.nonzero(counts)[0]
    cold = int(nonempty[np.argmin(counts[nonempty])])
    toks = {0, w.T - 1, int(np.nonzero((r["topk"] == hot).any(1))[0][0]),
            int(np.nonzero((r["topk"] == cold).any(1))[0][0])}
    toks |= set(np.nonzero(tie)[0][:2].tolist())
    toks = np.array(sorted(toks))
    need = sorted(set(r["topk"][toks].ravel().tolist()) | {hot, cold})
    W = oracle.ExpertWeights(w.E, {e: _bits(g["Wg"][e]) for e in need},
                             {e: _bits(g["Wu"][e]) for e in need},
                             {e: _bits(g["Wd"][e]) for e in need},
                             *(None if g[n] is None else _bits(g[n]) for n in ("Wsg", "Wsu", "Wsd")))
    tr = oracle.token_rows(x[toks], dY[toks], Wr, W, r["topk"][toks], r["gates"][toks],
                           r["scores"][toks], w.score)
    for nm, got in (("y", to_np(y)[toks]), ("dX", to_np(gr["dX"])[toks])):
        rl2, mr = rel_errors(got, tr[nm])
        assert rl2 <= 1e-2 and mr <= 4e-2, f"{nm} rows: rel L2 {rl2:.3e}, max/rms {mr:.3e}"

    # ---- sampled weight-gradient entries, with their error bounds
    rng = np.random.default_rng(0)
    ents = []
    for e in (hot, cold):
        fs = rng.choice(w.F, 3, replace=False)
        hs = rng.choice(w.H, 3, replace=False)
        ents += [("dWg", e, int(h), int(f)) for h, f in zip(hs, fs)]
        ents += [("dWu", e, int(h), int(f)) for h, f in zip(hs, fs)]
        ents += [("dWd", e, int(f), int(h)) for h, f in zip(hs, fs)]
    if w.Fs:
        fs = rng.choice(w.Fs, 3, replace=False)
        hs = rng.choice(w.H, 3, replace=False)
        ents += [(n, 0, int(h), int(f)) for n in ("dWsg", "dWsu") for h, f in zip(hs, fs)]
        ents += [("dWsd", 0, int(f), int(h)) for h, f in zip(hs, fs)]
    ref = oracle.dw_entries(x, dY, W, r["topk"], r["gates"], ents)
    gpu_name = dict(dWg="dW_gate", dWu="dW_up", dWd="dW_down", dWsg="dWs_gate", dWsu="dWs_up",
                    dWsd="dWs_down")
    for (n, e, i, j), want in zip(ents, ref):
        t = gr[gpu_name[n]]
        got = float((t[i, j] if n.startswith("dWs") else t[e, i, j]).item())
        f = i if n in ("dWd", "dWsd") else j
        if n.startswith("dWs"):
            rows = np.arange(w.T)
            gate = np.ones((w.T, 1))
            Wg_, Wu_, Wd_ = (to_np(g[m]) for m in ("Wsg", "Wsu", "Wsd"))
        else:
            rows, slots = np.nonzero(r["topk"] == e)
            gate = r["gates"][rows, slots][:, None]
            Wg_, Wu_, Wd_ = to_np(g["Wg"][e]), to_np(g["Wu"][e]), to_np(g["Wd"][e])
        bg, bu, bd, _ = _expert_wgrad_bounds(x[rows], Wg_[:, [f]], Wu_[:, [f]], Wd_[[f], :], gate,
                                             dY[rows], dYp_rounded=not n.startswith("dWs"))
        bound = {"dWg": bg, "dWu": bu, "dWd": bd, "dWsg": bg, "dWsu": bu, "dWsd": bd}[n]
        bnd = bound[0, j] if n in ("dWd", "dWsd") else bound[i, 0]
        assert abs(got - want) <= WGRAD_BOUND_SLACK * bnd, (n, e, i, j, got, want, bnd)


def test_full_size_fp8_layer():
    """Qwen3-shaped layer in blockwise FP8: routing bit-exact, the layer's
    weight quantiser bit-exact against the oracle on sampled experts, and
    sampled output rows within the E4M3 deviation scale of the exact layer
    (an output passes through up to ~6 successive E4M3 roundings of 3.6% rms
    each: at most 9% relative, as pinned on the oracle's FP8 layer)."""
    import mixture_experts_layer_sigmoid_gb300 as moe
    w = mi.WORKLOADS["qwen3_235b_fp8"]
    g = mi.make_inputs(w, "cuda")
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score, dtype=moe.MOE_FP8_BLOCK)
    y, rt = layer.forward(g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"], routing=True)
    gr = layer.backward(g["dY"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    assert layer.status(w.T) == 0
    assert torch.isfinite(y).all() and torch.isfinite(gr["dX"]).all()
    x, dY, Wr, b = to_np(g["x"]), to_np(g["dY"]), to_np(g["Wr"]), to_np(g["b"])
    r = oracle.route(x, Wr, b, w.k, w.score)
    gt = rt["topk_idx"].cpu().numpy()
    tie = (r["gap_set"] < TIE_REL) | (r["gap_order"] < TIE_REL)
    mism = np.any(gt != r["topk"], axis=1)
    assert not np.any(mism & ~tie)
    if mism.any():
        r = oracle.route(x, Wr, b, w.k, w.score, replay_topk=gt, replay_mask=mism)
    counts = np.bincount(r["topk"].ravel(), minlength=w.E)
    assert np.array_equal(rt["counts"].cpu().numpy(), counts)
    hot = int(np.argmax(counts))
    # the weight quantiser on two experts' full-size blocks
    for e in (0, hot):
        W = g["Wg"][e].contiguous()
        R, C = W.shape
        codes = torch.empty((R, C), dtype=torch.uint8, device="cuda")
        codes_t = torch.empty((C, R), dtype=torch.uint8, device="cuda")
        sc = torch.empty((R // 128, C // 128), device="cuda")
        sct = torch.empty((C // 128, R // 128), device="cuda")
        moe.moe_fp8_quantize(R, C, moe.MOE_Q_TILES, W.data_ptr(), codes.data_ptr(), sc.data_ptr(),
                             codes_t.data_ptr(), sct.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        oc, os_ = oracle.fp8_quantize(W.float().cpu().numpy(), oracle.FP8_TILES)
        assert np.array_equal(codes.cpu().numpy(), oc) and np.array_equal(sc.cpu().numpy(), os_)
        assert np.array_equal(codes_t.cpu().numpy(), oc.T)
    # sampled rows against the exact layer
    toks = np.array(sorted({0, w.T - 1, int(np.nonzero((r["topk"] == hot).any(1))[0][0]), 777}))
    need = sorted(set(r["topk"][toks].ravel().tolist()))
    Wx = oracle.ExpertWeights(w.E, {e: _bits(g["Wg"][e]) for e in need},
                              {e: _bits(g["Wu"][e]) for e in need},
                              {e: _bits(g["Wd"][e]) for e in need})
    tr = oracle.token_rows(x[toks], dY[toks], Wr, Wx, r["topk"][toks], r["gates"][toks],
                           r["scores"][toks], w.score)
    for nm, got in (("y", to_np(y)[toks]), ("dX", to_np(gr["dX"])[toks])):
        rl2, _ = rel_errors(got, tr[nm])
        assert 0.0 < rl2 < 0.09, (nm, rl2)
