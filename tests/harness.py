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
    within the bounds of the dtype (bf16: 1e-2 and 4e-2; fp32: 1e-4 and 1e-3);
  - bf16 weight gradients (dW_gate, dW_up, dW_down, the shared expert's, and
    the router's dWr, whose expert columns are sums over each expert's
    tokens): relative L2 <= 1e-2 over the whole tensor AND over each
    expert's block, and every element within the first-order forward-error
    bound of the bf16/fp32 arithmetic that produces it (wgrad_bounds). The
    max |error| / rms criterion is not used for them: each entry is a sum over
    the expert's rows of products of bf16-rounded MMA operands, the entries
    are heavy-tailed (max/rms up to ~15 with skewed routing), and rounding
    alone then exceeds 4e-2 * rms at the largest entries for any bf16-operand
    implementation.
"""
from __future__ import annotations

import numpy as np
import torch

import moe_inputs as mi
import oracle

TIE_REL = 1e-5
BOUNDS = {mi.BF16: (1e-2, 4e-2), mi.FP32: (1e-4, 1e-3)}
WGRAD_BOUND_SLACK = 1.5      # headroom over the first-order bound (second-order terms)
BF16_U = 2.0 ** -8           # bf16 unit roundoff
FP32_U = 2.0 ** -24          # fp32 unit roundoff, per accumulated term (worst case)


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


def _sig(a):
    return 1.0 / (1.0 + np.exp(-a))


def _expert_wgrad_bounds(X, Wg, Wu, Wd, g, dY, dYp_rounded=True):
    """First-order worst-case |error| bounds of the bf16 path's weight
    gradients of one expert (rows X with gates g and output gradients dY).

    Each stage's error bound is carried forward: a, u (fp32 sums over H,
    rounded to bf16), h = silu(a) u (bf16), dYp = g dY (bf16), dh = dYp Wd^T
    (fp32 sum over H), dA = dh u silu'(a) and dU = dh silu(a) (bf16); then
    the wgrad sums over the M rows (fp32) and the bf16 output rounding."""
    U, V = BF16_U, FP32_U
    M, H = X.shape
    a = X @ Wg
    uu = X @ Wu
    s = _sig(a)
    silu = a * s
    d1 = s * (1 + a * (1 - s))
    d2 = s * (1 - s) * (2 + a * (1 - 2 * s))
    aX = np.abs(X)
    a_err = U * np.abs(a) + H * V * (aX @ np.abs(Wg))
    u_err = U * np.abs(uu) + H * V * (aX @ np.abs(Wu))
    h = silu * uu
    h_err = U * np.abs(h) + np.abs(d1 * uu) * a_err + np.abs(silu) * u_err
    dYp = g * dY
    dYp_err = U * np.abs(dYp) if dYp_rounded else np.zeros_like(dYp)
    dh = dYp @ Wd.T
    dh_err = (U + H * V) * (np.abs(dYp) @ np.abs(Wd).T)
    dU = dh * silu
    dU_err = U * np.abs(dU) + np.abs(silu) * dh_err + np.abs(dh * d1) * a_err
    dA = dh * uu * d1
    dA_err = (U * np.abs(dA) + np.abs(uu * d1) * dh_err + np.abs(dh * d1) * u_err
              + np.abs(dh * uu * d2) * a_err)
    mv = M * V
    bd = (h_err.T @ np.abs(dYp) + np.abs(h).T @ dYp_err + mv * (np.abs(h).T @ np.abs(dYp))
          + U * np.abs(h.T @ dYp))
    bg = aX.T @ dA_err + mv * (aX.T @ np.abs(dA)) + U * np.abs(X.T @ dA)
    bu = aX.T @ dU_err + mv * (aX.T @ np.abs(dU)) + U * np.abs(X.T @ dU)
    # gate gradient dg = <dY, Yp> with Yp = h Wd (fp32 sum over F, bf16 output)
    F = Wd.shape[0]
    yp = h @ Wd
    yp_err = h_err @ np.abs(Wd) + F * V * (np.abs(h) @ np.abs(Wd)) + U * np.abs(yp)
    dg_err = (np.abs(dY) * yp_err).sum(1) + H * V * (np.abs(dY) * np.abs(yp)).sum(1)
    return bg, bu, bd, dg_err


def wgrad_bounds(w, inp, r):
    """Elementwise error bounds for every weight gradient of the bf16 path:
    the experts' (stacked E×…), the shared expert's and the router's dWr.

    dWr[h][e] = sum over e's tokens of x[t][h] dz[t][e]; dz is linear in the
    gate gradients dg = <dY, Yp>, whose error comes from the bf16 expert
    output Yp (h rounding, fp32 sum over F, bf16 output) and the fp32 sum
    over H; the dz formula's coefficients carry it to dz."""
    U, V = BF16_U, FP32_U
    x, dY = to_np(inp["x"]), to_np(inp["dY"])
    Wg, Wu, Wd = to_np(inp["Wg"]), to_np(inp["Wu"]), to_np(inp["Wd"])
    out = {n: np.zeros_like(v) for n, v in (("dWg", Wg), ("dWu", Wu), ("dWd", Wd))}
    dg_err = np.zeros_like(r["gates"])
    for e in range(w.E):
        toks, slots = np.nonzero(r["topk"] == e)
        if len(toks) == 0:
            continue
        out["dWg"][e], out["dWu"][e], out["dWd"][e], dg_err[toks, slots] = _expert_wgrad_bounds(
            x[toks], Wg[e], Wu[e], Wd[e], r["gates"][toks, slots][:, None], dY[toks])
    if w.Fs:
        out["dWsg"], out["dWsu"], out["dWsd"], _ = _expert_wgrad_bounds(
            x, to_np(inp["Wsg"]), to_np(inp["Wsu"]), to_np(inp["Wsd"]), np.ones((w.T, 1)), dY,
            dYp_rounded=False)
    g = r["gates"]
    spread = dg_err + (g * dg_err).sum(1, keepdims=True)
    if w.score == mi.SOFTMAX:
        dz_err = g * spread
    else:
        s = np.take_along_axis(r["scores"], r["topk"].astype(np.int64), 1)
        dz_err = s * (1 - s) / s.sum(1, keepdims=True) * spread
    # magnitude of dz itself, for the fp32 accumulation term of the router wgrad
    dz_mag = np.zeros_like(g)
    ref_dg = r.get("dg")
    if ref_dg is not None:
        spread_m = np.abs(ref_dg) + (g * np.abs(ref_dg)).sum(1, keepdims=True)
        dz_mag = g * spread_m if w.score == mi.SOFTMAX else s * (1 - s) / s.sum(1, keepdims=True) * spread_m
    dz_err_dense = np.zeros((w.T, w.E))
    dz_mag_dense = np.zeros((w.T, w.E))
    np.put_along_axis(dz_err_dense, r["topk"].astype(np.int64), dz_err, 1)
    np.put_along_axis(dz_mag_dense, r["topk"].astype(np.int64), dz_mag, 1)
    counts = np.bincount(r["topk"].ravel(), minlength=w.E)
    ax = np.abs(x)
    out["dWr"] = ax.T @ dz_err_dense + counts[None, :] * V * (ax.T @ dz_mag_dense)
    return out


def assert_wgrad(name, got, ref, bound):
    """bf16 weight gradient: rel L2 (whole and per expert block) + elementwise bound."""
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
    ratio = np.abs(got - ref) / (WGRAD_BOUND_SLACK * bound + 1e-30)
    worst = float(ratio.max())
    assert worst <= 1.0, (f"{name}: |error| above the bf16 forward-error bound "
                          f"(worst ratio {worst:.3f} at {np.unravel_index(ratio.argmax(), ratio.shape)})")
    return rl2, mr, worst


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
COLUMN_BLOCKS = {"dWr"}      # one block per expert column


def compare_all(w, inp, r, gpu, ref, backward=True):
    """Compare every output and gradient with the rules of this module."""
    report = {"y": assert_close("y", to_np(gpu["y"]), ref["y"], w.dtype)}
    if not backward:
        return report
    bounds = wgrad_bounds(w, inp, dict(r, dg=ref.get("dg"))) if w.dtype == mi.BF16 else None
    for gname, oname in GRAD_NAMES:
        if oname not in ref:
            continue
        got = to_np(gpu[gname])
        if bounds is not None and oname in EXPERT_WGRADS:
            report[gname] = assert_wgrad(gname, got, ref[oname], bounds[oname])
        elif bounds is not None and oname in COLUMN_BLOCKS:
            report[gname] = assert_wgrad(gname, got.T, ref[oname].T, bounds[oname].T)
        else:
            report[gname] = assert_close(gname, got, ref[oname], w.dtype)
    return report


def full_parity(w: mi.Workload, backward=True, fold=False, capacity_factor=0.0):
    inp = mi.make_inputs(w, "cpu", with_grad_out=backward)
    gpu, layer = run_gpu(w, inp, backward=backward, fold=fold, capacity_factor=capacity_factor)
    r, nties = check_routing(w, inp, gpu)
    if capacity_factor > 0:
        C = oracle.capacity(w.T, w.k, w.E, capacity_factor)
        r["keep"] = oracle.capacity_keep(r["topk"], w.E, C)
    np.testing.assert_allclose(gpu["gates"].numpy(), r["gates"], rtol=1e-4, atol=1e-6)
    ref = oracle_layer(w, inp, r, backward)
    report = compare_all(w, inp, r, gpu, ref, backward)
    report["near_ties"] = nties
    return report, gpu
