"""Parity harness: run the CUDA layer through its C ABI and the fp64 oracle
on the same seeded inputs, and compare.

Comparison rules (from the layer's definition; the oracle cites "Scalable
Training of Mixture-of-Experts Models with Megatron Core", §2):
  - top-k indices, per-expert counts, padded offsets and the permutation are
    compared bit for bit, except "near-tie" tokens whose oracle scores at the
    selection boundary (k-th vs (k+1)-th) or inside the selection order differ
    by less than 1e-5 relative. For those, any of the tied answers is correct:
    the GPU's choice is checked to be one of them and the oracle then uses
    that choice (router replay) so downstream tensors compare like with like;
  - floating-point tensors: relative L2 error and max |error| / rms(reference)
    within the bounds of the dtype (bf16: 1e-2 and 4e-2; fp32: 1e-4 and 1e-3).
"""
from __future__ import annotations

import numpy as np
import torch

import moe_inputs as mi
import oracle

TIE_REL = 1e-5
BOUNDS = {mi.BF16: (1e-2, 4e-2), mi.FP32: (1e-4, 1e-3)}


def to_np(t):
    return None if t is None else t.detach().cpu().double().numpy()


def rel_errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = got - ref
    nref = np.linalg.norm(ref)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    rel_l2 = np.linalg.norm(diff) / nref if nref > 0 else np.linalg.norm(diff)
    max_rel = np.max(np.abs(diff)) / rms if rms > 0 else np.max(np.abs(diff), initial=0.0)
    return float(rel_l2), float(max_rel)


def assert_close(name, got, ref, dtype):
    l2b, mab = BOUNDS[dtype]
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    rl2, mr = rel_errors(got, ref)
    assert rl2 <= l2b and mr <= mab, f"{name}: rel L2 {rl2:.3e} (<= {l2b}), max/rms {mr:.3e} (<= {mab})"
    return rl2, mr


def upload(inp, device="cuda"):
    return {k: (None if v is None else v.to(device)) for k, v in inp.items()}


def run_gpu(w: mi.Workload, inp, layer=None, backward=True):
    """Forward (+ backward) through the C ABI; returns host copies."""
    from mixture_experts_layer_sigmoid_gb300 import MoELayer
    g = upload(inp)
    if layer is None:
        layer = MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score, dtype=w.dtype, Fs=w.Fs)
    y, r = layer.forward(g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"], g["Wsg"], g["Wsu"],
                         g["Wsd"], routing=True)
    out = dict(y=y, **r)
    if backward:
        out.update(layer.backward(g["dY"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], g["Wsg"],
                                  g["Wsu"], g["Wsd"]))
    torch.cuda.synchronize()
    st = layer.status(w.T)
    assert st == 0, f"device status {st}"
    return {k: v.cpu() for k, v in out.items()}, layer


def check_routing(w, inp, gpu):
    """Bit-exact routing check; returns (oracle route dict with replay, n_ties)."""
    x = to_np(inp["x"])
    Wr = to_np(inp["Wr"])
    b = to_np(inp["b"])
    r = oracle.route(x, Wr, b, w.k, w.score)
    g_topk = gpu["topk_idx"].numpy()
    tie = (r["gap_set"] < TIE_REL) | (r["gap_order"] < TIE_REL)
    mismatch = np.any(g_topk != r["topk"], axis=1)
    bad = mismatch & ~tie
    assert not np.any(bad), f"top-k differs on {int(bad.sum())} non-tie tokens, e.g. {np.nonzero(bad)[0][:5]}"
    # tied tokens: the GPU's selection must be one of the tied answers
    for t in np.nonzero(mismatch)[0]:
        s = r["scores"][t]
        sel = g_topk[t]
        assert len(set(sel.tolist())) == w.k
        kth = np.sort(s)[::-1][w.k - 1]
        assert np.all(s[sel] >= kth * (1 - 2 * TIE_REL) - 1e-300), f"token {t}: invalid tied choice"
        assert np.all(np.diff(s[sel]) <= np.abs(s[sel][:-1]) * 2 * TIE_REL), f"token {t}: bad order"
    if np.any(mismatch):
        r = oracle.route(x, Wr, b, w.k, w.score, replay_topk=g_topk, replay_mask=mismatch)
    assert np.array_equal(g_topk, r["topk"])
    d = oracle.dispatch(r["topk"], w.E)
    assert np.array_equal(gpu["counts"].numpy(), d["counts"])
    pc = (d["counts"] + 127) // 128 * 128
    poff = np.concatenate([[0], np.cumsum(pc)]).astype(np.int64)
    assert np.array_equal(gpu["offsets"].numpy(), poff)
    g_row = gpu["row_of"].numpy().astype(np.int64)
    e = r["topk"].astype(np.int64)
    mapped = g_row - poff[e] + d["offsets"][e]
    assert np.array_equal(mapped, d["row_of"])
    return r, int(tie.sum())


def oracle_layer(w, inp, r, backward=True):
    args = {k: to_np(inp[k]) for k in ("x", "Wg", "Wu", "Wd", "Wsg", "Wsu", "Wsd")}
    y = oracle.forward(args["x"], args["Wg"], args["Wu"], args["Wd"], r["topk"], r["gates"],
                       args["Wsg"], args["Wsu"], args["Wsd"])
    out = dict(y=y)
    if backward:
        g = oracle.backward(args["x"], to_np(inp["Wr"]), args["Wg"], args["Wu"], args["Wd"],
                            r["topk"], r["gates"], r["scores"], to_np(inp["dY"]), w.score,
                            args["Wsg"], args["Wsu"], args["Wsd"])
        out.update(g)
    return out


GRAD_NAMES = [("dX", "dX"), ("dWr", "dWr"), ("dW_gate", "dWg"), ("dW_up", "dWu"),
              ("dW_down", "dWd"), ("dWs_gate", "dWsg"), ("dWs_up", "dWsu"), ("dWs_down", "dWsd")]


def full_parity(w: mi.Workload, backward=True):
    inp = mi.make_inputs(w, "cpu", with_grad_out=backward)
    gpu, layer = run_gpu(w, inp, backward=backward)
    r, nties = check_routing(w, inp, gpu)
    np.testing.assert_allclose(gpu["gates"].numpy(), r["gates"], rtol=1e-4, atol=1e-6)
    ref = oracle_layer(w, inp, r, backward)
    report = {"near_ties": nties}
    report["y"] = assert_close("y", to_np(gpu["y"]), ref["y"], w.dtype)
    if backward:
        for gname, oname in GRAD_NAMES:
            if oname in ref:
                report[gname] = assert_close(gname, to_np(gpu[gname]), ref[oname], w.dtype)
    return report, gpu
