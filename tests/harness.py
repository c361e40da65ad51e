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
  - every floating-point tensor is reported with the pair (relative L2 error,
    max |error| / rms(reference)) against the exact fp64 oracle, and y and dX
    must meet the bounds of the dtype (bf16: 1e-2 and 4e-2; fp32: 1e-4 and
    1e-3), as must every fp32-layer gradient;
  - the bf16 router weight gradient dWr must meet relative L2 <= 1e-2, and
    max |error| <= 4e-2 rms(ref) unless its bf16 emulation (gate gradients
    from the stored bf16 expert outputs) itself exceeds that, in which case
    the GPU may not exceed the emulation's by more than 10%; against the
    emulation its relative L2 error must stay below 1e-3;
  - bf16 expert weight gradients (dW_gate, dW_up, dW_down and the shared
    expert's) must meet relative L2 <= 1e-2 over the whole tensor and over
    each expert's block, and max |error| <= 4e-2 rms(ref) wherever bf16
    storage of the layer's intermediates allows it. Where it does not --
    tests/bf16_chain.py emulates that storage exactly, and on heavy-tailed
    gradients its own max error exceeds 4e-2 rms (tests/test_bf16_chain.py)
    -- the GPU's max error may not exceed the emulation's by more than 10%.
    In addition at least 98% of the elements must be the bf16 rounding of the
    emulated sum up to fp32 summation error, and every element within the
    envelope of two moved terms (bf16_chain.rounding_check).
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import moe_inputs as mi
import oracle
import bf16_chain as bc

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


MAX_FLOOR_MARGIN = 1.10      # GPU max error vs the bf16-storage floor, where that floor exceeds 4e-2
DWR_EMU_REL_L2 = 1e-3        # dWr against its bf16 emulation (fp32 sums, rare one-ulp operand moves)


def _floor_check(name, mr, floor):
    assert mr <= max(4e-2, MAX_FLOOR_MARGIN * floor), (
        f"{name}: max/rms {mr:.3e} above 4e-2 and above {MAX_FLOOR_MARGIN} x the bf16-storage "
        f"floor {floor:.3e}")


def assert_wgrad(name, got, ref, wg):
    """bf16 expert weight gradient against the fp64 oracle and the bf16
    rounding-chain emulation wg (bf16_chain.WGrad)."""
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    rl2, mr = rel_errors(got, ref)
    assert rl2 <= 1e-2, f"{name}: rel L2 {rl2:.3e} > 1e-2"
    blocks = [(got, ref)] if ref.ndim == 2 else list(zip(got, ref))
    for e, (g_, r_) in enumerate(blocks):
        nr = np.linalg.norm(r_)
        if nr == 0:
            assert np.all(g_ == 0), f"{name}[{e}]: expert without tokens has a nonzero gradient"
            continue
        assert np.linalg.norm(g_ - r_) / nr <= 1e-2, f"{name}[{e}]: block rel L2 > 1e-2"
    _, floor = rel_errors(bc.rn_bf16(wg.S), ref)
    _floor_check(name, mr, floor)
    short = name.replace("dW_gate", "dWg").replace("dW_up", "dWu").replace("dW_down", "dWd") \
        .replace("dWs_gate", "dWsg").replace("dWs_up", "dWsu").replace("dWs_down", "dWsd")
    ratio, miss, worst = bc.rounding_check(got, wg, short)
    assert miss <= bc.TIGHT_MISS_FRAC, (f"{name}: {100 * miss:.2f}% of the elements are not the bf16 "
                                        f"rounding of the emulated sum (at most "
                                        f"{100 * bc.TIGHT_MISS_FRAC}% may be)")
    assert worst <= 1.0, f"{name}: an element is outside its deviation envelope (ratio {worst:.3f})"
    exact = float(np.mean(got == bc.rn_bf16(wg.S)))
    return dict(rel_l2=rl2, max_rms=mr, floor_max_rms=floor, exact_frac=exact,
                tight_miss_frac=miss, worst_envelope_ratio=worst)


def assert_dwr_bf16(got, ref, emu):
    """Router weight gradient of the bf16 layer (fp32 output): the contract
    pair against the oracle (max error against the bf16-storage floor where
    that exceeds 4e-2), and relative L2 against its bf16 emulation."""
    assert np.all(np.isfinite(got)), "dWr: non-finite values"
    rl2, mr = rel_errors(got, ref)
    assert rl2 <= 1e-2, f"dWr: rel L2 {rl2:.3e} > 1e-2"
    _, floor = rel_errors(emu, ref)
    _floor_check("dWr", mr, floor)
    emu_l2 = float(np.linalg.norm(got - emu) / np.linalg.norm(ref)) if np.linalg.norm(ref) > 0 else 0.0
    assert emu_l2 <= DWR_EMU_REL_L2, f"dWr: rel L2 against the bf16 emulation {emu_l2:.3e}"
    return dict(rel_l2=rl2, max_rms=mr, floor_max_rms=floor, emu_rel_l2=emu_l2)


def upload(inp, device="cuda"):
    return {k: (None if v is None else v.to(device)) for k, v in inp.items()}


def run_gpu(w: mi.Workload, inp, layer=None, backward=True, fold=False, capacity_factor=0.0,
            replay=None):
    """Forward (+ backward) through the C ABI; returns host copies. fold:
    memory-efficient permutation (routing weights folded into h);
    capacity_factor: capacity-limited dropping; replay: T×k experts to route
    to (router replay)."""
    from mixture_experts_layer_sigmoid_gb300 import MoELayer
    g = upload(inp)
    if layer is None:
        layer = MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score, dtype=w.dtype, Fs=w.Fs,
                         fold_gates=fold, capacity_factor=capacity_factor)
    rep = None if replay is None else torch.as_tensor(replay, dtype=torch.int32).cuda()
    y, r = layer.forward(g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"], g["Wsg"], g["Wsu"],
                         g["Wsd"], routing=True, replay_topk=rep)
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
                       args["Wsg"], args["Wsu"], args["Wsd"], keep=r.get("keep"))
    out = dict(y=y)
    if backward:
        g = oracle.backward(args["x"], to_np(inp["Wr"]), args["Wg"], args["Wu"], args["Wd"],
                            r["topk"], r["gates"], r["scores"], to_np(inp["dY"]), w.score,
                            args["Wsg"], args["Wsu"], args["Wsd"], keep=r.get("keep"))
        out.update(g)
    return out


GRAD_NAMES = [("dX", "dX"), ("dWr", "dWr"), ("dW_gate", "dWg"), ("dW_up", "dWu"),
              ("dW_down", "dWd"), ("dWs_gate", "dWsg"), ("dWs_up", "dWsu"), ("dWs_down", "dWsd")]
EXPERT_WGRADS = {"dWg", "dWu", "dWd", "dWsg", "dWsu", "dWsd"}


def compare_all(w, inp, r, gpu, ref, backward=True, fold=False):
    """Compare every output and gradient with the rules of this module.
    Returns, per tensor, the contract's pair (relative L2, max|err|/rms) against
    the fp64 oracle (plus, for bf16 expert weight gradients, the bf16-storage
    floor of the second and the rounding-consistency figures)."""
    report = {"y": assert_close("y", to_np(gpu["y"]), ref["y"], w.dtype)}
    if not backward:
        return report
    chain = dwr = None
    if w.dtype == mi.BF16:
        d = {k: to_np(inp[k]) for k in ("x", "Wg", "Wu", "Wd", "Wsg", "Wsu", "Wsd", "dY")}
        chain = bc.layer_wgrads(d["x"], d["Wg"], d["Wu"], d["Wd"], r["topk"], r["gates"], d["dY"],
                                d["Wsg"], d["Wsu"], d["Wsd"], fold=fold, keep=r.get("keep"))
        sel = np.take_along_axis(r["scores"], r["topk"].astype(np.int64), 1)
        dwr = bc.layer_dwr(d["x"], d["Wg"], d["Wu"], d["Wd"], r["topk"], r["gates"], sel, d["dY"],
                           w.score, w.E, fold=fold, keep=r.get("keep"))[0]
    for gname, oname in GRAD_NAMES:
        if oname not in ref:
            continue
        got = to_np(gpu[gname])
        if chain is not None and oname in EXPERT_WGRADS:
            report[gname] = assert_wgrad(gname, got, ref[oname], chain[oname])
        elif dwr is not None and oname == "dWr":
            report[gname] = assert_dwr_bf16(got, ref[oname], dwr)
        else:
            report[gname] = assert_close(gname, got, ref[oname], w.dtype)
    return report


def write_report(case, report):
    """Append one case's parity figures to the JSON-lines file named by the
    MOE_PARITY_REPORT environment variable (no-op when it is unset)."""
    path = os.environ.get("MOE_PARITY_REPORT")
    if not path:
        return
    def conv(v):
        if isinstance(v, dict):
            return {k: conv(x) for k, x in v.items()}
        if isinstance(v, (tuple, list)):
            return [conv(x) for x in v]
        return float(v) if isinstance(v, (float, np.floating)) else v
    with open(path, "a") as f:
        f.write(json.dumps({"case": case, **conv(report)}) + "\n")


def full_parity(w: mi.Workload, backward=True, fold=False, capacity_factor=0.0):
    inp = mi.make_inputs(w, "cpu", with_grad_out=backward)
    gpu, layer = run_gpu(w, inp, backward=backward, fold=fold, capacity_factor=capacity_factor)
    r, nties = check_routing(w, inp, gpu)
    if capacity_factor > 0:
        C = oracle.capacity(w.T, w.k, w.E, capacity_factor)
        r["keep"] = oracle.capacity_keep(r["topk"], w.E, C)
    np.testing.assert_allclose(gpu["gates"].numpy(), r["gates"], rtol=1e-4, atol=1e-6)
    ref = oracle_layer(w, inp, r, backward)
    report = compare_all(w, inp, r, gpu, ref, backward, fold=fold)
    report["near_ties"] = nties
    dt = {mi.FP32: "fp32", mi.BF16: "bf16", mi.FP8_BLOCK: "fp8"}[w.dtype]
    write_report(f"{w.name} T{w.T} H{w.H} E{w.E} k{w.k} F{w.F} Fs{w.Fs} {dt}"
                 + (" fold" if fold else "") + (f" cf{capacity_factor}" if capacity_factor else ""),
                 report)
    return report, gpu
