"""Parity at the full layer sizes (Mixtral-8x7B-, DeepSeek-V3- and
Qwen3-235B-shaped expert layers), in the launch configuration bench.py times.

The whole layer runs on the GPU; the fp64 oracle then checks
  - routing for every token (top-k bit-exact except near-ties, counts,
    padded offsets and the full permutation),
  - y and dX rows of sampled tokens (first, last, hottest-expert and tied
    tokens), computed one by one by the oracle's per-token form,
  - sampled entries of the expert weight gradients (hottest and coldest
    non-empty expert, and the shared expert): all but at most one must be
    the bf16 rounding of the bf16 rounding-chain emulation's sum
    (tests/bf16_chain.py) up to fp32 summation error, and every one within
    its deviation envelope; the pair (rel L2, max|err| / rms) against the
    exact fp64 entries is reported, with rms taken over the whole GPU tensor.
dWr needs every routed token's expert outputs, so at these sizes it is
covered by the mid-size tests only.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import bf16_chain as bc
from harness import TIE_REL, rel_errors, to_np, write_report

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
    rms = {n: float(gr[m].float().pow(2).mean().sqrt().item()) for n, m in gpu_name.items() if m in gr}
    errs = {}
    worst, misses = 0.0, 0
    for (n, e, i, j), want in zip(ents, ref):
        t = gr[gpu_name[n]]
        got = float((t[i, j] if n.startswith("dWs") else t[e, i, j]).item())
        f = i if n in ("dWd", "dWsd") else j
        shared = n.startswith("dWs")
        if shared:
            rows = np.arange(w.T)
            gate = np.ones(w.T)
            Wg_, Wu_, Wd_ = (to_np(g[m]) for m in ("Wsg", "Wsu", "Wsd"))
        else:
            rows, slots = np.nonzero(r["topk"] == e)
            gate = r["gates"][rows, slots]
            Wg_, Wu_, Wd_ = to_np(g["Wg"][e]), to_np(g["Wu"][e]), to_np(g["Wd"][e])
        c = bc.expert_chain(x[rows], Wg_[:, [f]], Wu_[:, [f]], Wd_[[f], :], gate, dY[rows],
                            scale_dy=not shared)
        key = n.replace("dWs", "dW")
        at = (0, j) if key == "dWd" else (i, 0)
        tight, env = bc.entry_check(got, c, key, *at)
        misses += tight > 1.0
        worst = max(worst, env)
        assert env <= 1.0, (n, e, i, j, got, want, float(c[key][at]))
        errs.setdefault(n, []).append((got, want))
    # a sample of 18-27 entries: at most one may miss the tight rounding bound
    assert misses <= 1, f"{misses} sampled entries are not the bf16 rounding of the emulated sum"
    report = {"tight_misses": int(misses), "worst_envelope_ratio": float(worst)}
    for n, pairs in errs.items():
        got_, want_ = np.array(pairs).T
        report[gpu_name[n] + "_sampled"] = (float(np.linalg.norm(got_ - want_) / np.linalg.norm(want_)),
                                            float(np.abs(got_ - want_).max() / rms[n]))
    print(name, report)
    write_report(f"{name} full size, sampled weight-gradient entries", report)


def _full_size_fp8_case(wl, dtype, recipe, check_weight_quantiser):
    """A Qwen3-shaped FP8 layer at full size: routing bit-exact, the layer's
    weight quantiser bit-exact against the oracle on sampled experts, and
    sampled y and dX rows within the FP8 bounds (relative L2 <= 4e-2,
    max|err| <= 1.5e-1 rms) of the oracle's FP8 layer in the same recipe."""
    import mixture_experts_layer_sigmoid_gb300 as moe
    w = mi.WORKLOADS[wl]
    g = mi.make_inputs(w, "cuda")
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score, dtype=dtype, Fs=w.Fs)
    ws = (g["Wsg"], g["Wsu"], g["Wsd"])
    y, rt = layer.forward(g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"], *ws, routing=True)
    gr = layer.backward(g["dY"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], *ws)
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
    for e in (0, hot):
        check_weight_quantiser(g["Wg"][e].contiguous())
    # sampled rows against the oracle's FP8 layer run on those tokens alone:
    # y and dX of a token depend only on its own row (row blocks of its
    # activations and gradients, weight blocks of its experts and of the
    # shared expert), and dz only on its selected experts' scores, so the
    # layer restricted to the sampled tokens and the experts they select
    # (renumbered) gives their rows exactly
    toks = np.array(sorted({0, w.T - 1, int(np.nonzero((r["topk"] == hot).any(1))[0][0])}))
    need = sorted(set(r["topk"][toks].ravel().tolist()))
    renum = np.full(w.E, -1, np.int32)
    renum[need] = np.arange(len(need), dtype=np.int32)
    topk_s = renum[r["topk"][toks]]
    stack = lambda n: np.stack([to_np(g[n][e]) for e in need])
    q = oracle.layer_fp8(x[toks], Wr[:, need], stack("Wg"), stack("Wu"), stack("Wd"), topk_s,
                         r["gates"][toks], r["scores"][toks][:, need], w.score, dY[toks],
                         Wsg=to_np(g["Wsg"]), Wsu=to_np(g["Wsu"]), Wsd=to_np(g["Wsd"]), recipe=recipe)
    report = {}
    for nm, got in (("y", to_np(y)[toks]), ("dX", to_np(gr["dX"])[toks])):
        rl2, mr = rel_errors(got, q[nm])
        report[nm + "_rows"] = (rl2, mr)
        assert rl2 <= 4e-2 and mr <= 1.5e-1, (nm, rl2, mr)
    print(wl, report)
    write_report(f"{wl} full size, sampled token rows", report)


def test_full_size_fp8_layer():
    """Blockwise FP8 (1x128 / 128x128 fp32 scales)."""
    import mixture_experts_layer_sigmoid_gb300 as moe

    def check(W):
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

    _full_size_fp8_case("qwen3_235b_fp8", moe.MOE_FP8_BLOCK, oracle.RECIPE_BLOCK, check)


def test_full_size_mxfp8_layer():
    """MXFP8 (1x32 blocks, UE8M0 scales): the weight quantiser checked in
    both block directions (1x32 along each row, 32x1 down each column)."""
    import mixture_experts_layer_sigmoid_gb300 as moe
    from test_mx_gpu import _atoms_to_scales, _mxq

    def check(W):
        R, C = W.shape
        q, sq, qc, sc = _mxq(W, rows=True, cols=1)
        Wf = W.float().cpu().numpy()
        oc_r, os_r = oracle.mx_quantize(Wf, oracle.MX_ROWS)
        oc_c, os_c = oracle.mx_quantize(Wf, oracle.MX_COLS)
        assert np.array_equal(q, oc_r) and np.array_equal(_atoms_to_scales(sq, R, C), os_r)
        assert np.array_equal(qc, oc_c.T) and np.array_equal(_atoms_to_scales(sc, C, R), os_c.T)

    _full_size_fp8_case("qwen3_235b_mxfp8", moe.MOE_MXFP8, oracle.RECIPE_MX, check)


def test_full_size_deepseek_mxfp8_layer():
    """The DeepSeek-V3 shape in MXFP8, with its shared expert (a dense group
    of the 8192 token rows through the same engine)."""
    import mixture_experts_layer_sigmoid_gb300 as moe
    from test_mx_gpu import _atoms_to_scales, _mxq

    def check(W):
        R, C = W.shape
        q, sq, _, _ = _mxq(W, rows=True, cols=None)
        oc_r, os_r = oracle.mx_quantize(W.float().cpu().numpy(), oracle.MX_ROWS)
        assert np.array_equal(q, oc_r) and np.array_equal(_atoms_to_scales(sq, R, C), os_r)

    _full_size_fp8_case("deepseek_v3_mxfp8", moe.MOE_MXFP8, oracle.RECIPE_MX, check)


def _full_size_nv_case(wl):
    """NVFP4 at full size. A token's rows no longer depend on its own values
    alone (each expert tensor's fp32 scale comes from the expert's whole
    segment), so the oracle checks what it can compute exactly: the weight
    quantiser bit for bit on sampled experts in both orientations, and the
    weight gradients of the coldest non-empty expert -- every token routed
    to it is given to the oracle's NVFP4 layer, so that expert's segment
    (its tensors and tensor scales) is complete -- within the NVFP4 bounds
    of test_nv_gpu; sampled y and dX rows are checked against the exact
    layer's rows within the E2M1 error scale (rel L2 < 0.4, the bound the
    oracle's own NVFP4 layer meets against the exact one)."""
    import mixture_experts_layer_sigmoid_gb300 as moe
    from test_nv_gpu import _atoms_to_scales, _nvq, _unpack
    w = mi.WORKLOADS[wl]
    g = mi.make_inputs(w, "cuda")
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score, dtype=moe.MOE_NVFP4, Fs=w.Fs)
    ws = (g["Wsg"], g["Wsu"], g["Wsd"])
    y, rt = layer.forward(g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"], *ws, routing=True)
    gr = layer.backward(g["dY"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], *ws)
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
    nonempty = np.nonzero(counts)[0]
    cold = int(nonempty[np.argmin(counts[nonempty])])
    for e in (0, hot):
        W = g["Wg"][e].contiguous()
        R, C = W.shape
        amax, q, sq, qt, st = _nvq(W)
        Wf = W.float().cpu().numpy()
        oc_r, os_r, _ = oracle.nv_quantize(Wf, oracle.NV_ROWS)
        oc_c, os_c, _ = oracle.nv_quantize(Wf, oracle.NV_COLS)
        assert amax == np.abs(Wf).max()
        assert np.array_equal(_unpack(q, R, C), oc_r) and np.array_equal(_atoms_to_scales(sq, R, C), os_r)
        assert np.array_equal(_unpack(qt, C, R), oc_c.T) and np.array_equal(_atoms_to_scales(st, C, R), os_c.T)
    # the coldest expert's weight gradients, its whole segment in the oracle
    toks = np.nonzero((r["topk"] == cold).any(1))[0]
    need = sorted(set(r["topk"][toks].ravel().tolist()))
    renum = np.full(w.E, -1, np.int32)
    renum[need] = np.arange(len(need), dtype=np.int32)
    stack = lambda n: np.stack([to_np(g[n][e]) for e in need])
    q = oracle.layer_fp8(x[toks], Wr[:, need], stack("Wg"), stack("Wu"), stack("Wd"), renum[r["topk"][toks]],
                         r["gates"][toks], r["scores"][toks][:, need], w.score, dY[toks],
                         recipe=oracle.RECIPE_NV)
    report = {"cold_expert_rows": int(counts[cold])}
    for gname, oname in (("dW_gate", "dWg"), ("dW_up", "dWu"), ("dW_down", "dWd")):
        got = to_np(gr[gname][cold])
        want = q[oname][renum[cold]]
        rl2, mr = rel_errors(got, want)
        rms = np.sqrt(np.mean(np.square(want)))
        far = float(np.mean(np.abs(got - want) > 1.5e-1 * rms))
        report[gname + "_cold"] = (rl2, mr, far)
        assert rl2 <= 4e-2 and far <= 1e-3 and mr <= 1.0, (gname, rl2, mr, far)
    # sampled rows against the exact layer, within the E2M1 error scale
    rows = np.array(sorted({0, w.T - 1, int(toks[0])}))
    needr = sorted(set(r["topk"][rows].ravel().tolist()))
    We = oracle.ExpertWeights(w.E, {e: _bits(g["Wg"][e]) for e in needr},
                              {e: _bits(g["Wu"][e]) for e in needr},
                              {e: _bits(g["Wd"][e]) for e in needr},
                              *(None if g[n] is None else _bits(g[n]) for n in ("Wsg", "Wsu", "Wsd")))
    tr = oracle.token_rows(x[rows], dY[rows], Wr, We, r["topk"][rows], r["gates"][rows], r["scores"][rows],
                           w.score)
    for nm, got in (("y", to_np(y)[rows]), ("dX", to_np(gr["dX"])[rows])):
        rl2, mr = rel_errors(got, tr[nm])
        report[nm + "_rows_vs_exact"] = (rl2, mr)
        assert 0.02 < rl2 < 0.4, (nm, rl2)
    print(wl, report)
    write_report(f"{wl} full size", report)


def test_full_size_nvfp4_layer():
    _full_size_nv_case("qwen3_235b_nvfp4")


def test_full_size_deepseek_nvfp4_layer():
    _full_size_nv_case("deepseek_v3_nvfp4")
