"""The bf16 layer's rounding chain, emulated in numpy (test infrastructure).

The bf16 workloads store the layer's activations and gradients in bf16 and
accumulate every sum in fp32 ("Scalable Training of Mixture-of-Experts Models
with Megatron Core", §5 Selective precision: FP32 is kept for the router and
accumulation, lower precision for the rest). This module follows the same
formulas as the fp64 oracle (SwiGLU expert FFN, gate-weighted combine, chain
rule of L = sum(dY * y)) but rounds every stored intermediate to bf16 at the
points where a bf16 implementation must store it:

  forward   a, u = x Wg, x Wu (sums kept exact, then stored: RN(a), RN(u));
            h = RN(silu(a) u) from the unrounded sums (memory-efficient order:
            h' = RN(g silu(a) u)); Yp = RN(h Wd)
  backward  dYp = RN(g dY) (memory-efficient order: dY itself);
            dh = dYp Wd^T; dA = RN(dh u silu'(a)), dU = RN(dh silu(a)) from the
            STORED RN(a), RN(u); the weight gradients h^T dYp, x^T dA, x^T dU
            before their final bf16 rounding.

Sums are taken in fp64 here, so the only differences from an exact bf16-
storage implementation with fp32 accumulation are that implementation's fp32
summation errors (about 2^-24 sqrt(K) relative), and the rare one-ulp
difference in a stored intermediate that they cause.

It serves two purposes. A CPU test shows with it that the maximum-error bound
max|err| <= 4e-2 rms(ref) cannot be met against the exact fp64 layer by any
implementation that stores these intermediates in bf16, on heavy-tailed
weight gradients (the bound measures bf16 storage, not the kernels). The GPU
parity tests use it as a second, much tighter reference for the expert weight
gradients: nearly every GPU element must be the bf16 rounding of the emulated
sum up to fp32 summation error, and every element within a derived envelope
(rounding_check).

With rounding switched off (``rnd=None``) every function reduces to the fp64
oracle's definitions; tests/test_bf16_chain.py pins that equality.
"""
from __future__ import annotations

import numpy as np

BF16_HALF_ULP_REL = 2.0 ** -8   # max relative rounding error of RN to bf16 (half ulp / value)


def rn_bf16(v):
    """Round fp64 values to bf16 the way an fp32 kernel does: RN to fp32,
    then round-to-nearest-even on the upper 16 bits."""
    f = np.asarray(v, np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    finite = (u & 0x7F800000) != 0x7F800000
    r = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    r = np.where(finite, r, u).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def ulp_bf16(v):
    """Spacing of bf16 values at |v| (the ulp of the binade holding v; for 0
    the smallest normal spacing)."""
    m, e = np.frexp(np.abs(np.asarray(v, np.float64)))   # |v| = m 2^e, m in [0.5, 1)
    ulp = np.ldexp(1.0, e - 8)
    return np.where(m == 0, np.ldexp(1.0, -133), ulp)


def _sig(a):
    return 1.0 / (1.0 + np.exp(-a))


def expert_chain(X, Wg, Wu, Wd, g, dY, fold=False, scale_dy=True, rnd=rn_bf16):
    """One expert (or the shared expert) of the bf16 layer.

    X: M x H rows routed to the expert (exact bf16 values), Wg, Wu: H x Fc,
    Wd: Fc x H (Fc = any subset of the FFN columns, e.g. one sampled column),
    g: M routing weights, dY: M x H output gradients of the rows' tokens.
    fold: memory-efficient order (g folded into h). scale_dy: the routed
    experts scale dY by g before fc2's data gradient; the shared expert is
    added unweighted (scale_dy False, g = 1). rnd: rounding of stored values
    (None = exact).

    Returns dict: Yp (M x H, stored), dg (M), dWg, dWu (H x Fc), dWd (Fc x H)
    before their output rounding, and the per-element magnitudes the GPU
    comparison needs (sqrt of the sums of squared terms, and the sums of
    absolute terms, of each weight-gradient entry)."""
    R = (lambda v: v) if rnd is None else rnd
    g = np.asarray(g, np.float64).reshape(-1, 1)
    a = X @ Wg
    u = X @ Wu
    h = a * _sig(a) * u
    A, U = R(a), R(u)
    Hh = R(g * h) if fold else R(h)
    Yp = R(Hh @ Wd)
    dYp = dY if fold else (R(g * dY) if scale_dy else dY)
    dh = dYp @ Wd.T
    s = _sig(A)
    silu = A * s
    dsilu = s * (1.0 + A * (1.0 - s))
    if fold:
        hr = silu * U
        dg = (dh * hr).sum(1)
        dh = g * dh
        Hw = R(g * hr)            # g h recomputed from the stored a, u for fc2's wgrad
    else:
        dg = (dY * Yp).sum(1)
        Hw = Hh
    dA = R(dh * U * dsilu)
    dU = R(dh * silu)
    out = dict(Yp=Yp, dg=dg, dWg=X.T @ dA, dWu=X.T @ dU, dWd=Hw.T @ dYp)
    aX = np.abs(X)
    out["l1_dWg"] = aX.T @ np.abs(dA)
    out["l1_dWu"] = aX.T @ np.abs(dU)
    out["l1_dWd"] = np.abs(Hw).T @ np.abs(dYp)
    out["M"] = X.shape[0]
    if rnd is not None:
        # How far a stored operand of an fp32 implementation can sit from the
        # emulation's: one bf16 ulp (its fp32 value was within fp32 error of a
        # rounding midpoint) plus what the upstream fp32 sums and one-ulp
        # differences of upstream stored values move it (first order).
        H = X.shape[1]
        acc_a = H * 2.0 ** -24 * (aX @ np.abs(Wg))
        acc_u = H * 2.0 ** -24 * (aX @ np.abs(Wu))
        env_A = ulp_bf16(A) + acc_a
        env_U = ulp_bf16(U) + acc_u
        pd = np.abs(dYp) @ np.abs(Wd).T
        env_dh = H * 2.0 ** -24 * pd
        if fold:
            env_dh = np.abs(g) * env_dh
        elif scale_dy:
            # one stored dYp value of the row one ulp away
            env_dh = env_dh + 2.0 ** -7 * np.sqrt((dYp * dYp) @ (Wd * Wd).T)
        d2 = s * (1.0 - s) * (2.0 + A * (1.0 - 2.0 * s))          # silu''(A)
        out["env_dA"] = (ulp_bf16(dA) + np.abs(U * dsilu) * env_dh + np.abs(dh * dsilu) * env_U
                         + np.abs(dh * U * d2) * env_A)
        out["env_dU"] = ulp_bf16(dU) + np.abs(silu) * env_dh + np.abs(dh * dsilu) * env_A
        dsilu_a = _sig(a) * (1.0 + a * (1.0 - _sig(a)))
        if fold:
            env_H = ulp_bf16(Hw) + np.abs(g) * (np.abs(dsilu * U) * env_A + np.abs(silu) * env_U)
        else:
            env_H = ulp_bf16(Hw) + np.abs(dsilu_a * u) * acc_a + np.abs(a * _sig(a)) * acc_u
        out["env_H"] = env_H
        out["env_dYp"] = ulp_bf16(dYp) if (scale_dy and not fold) else np.zeros_like(dYp)
        out["ops"] = dict(X=X, dA=dA, dU=dU, Hw=Hw, dYp=dYp)
    return out


def layer_wgrads(x, Wg, Wu, Wd, topk, gates, dY, Wsg=None, Wsu=None, Wsd=None, fold=False,
                 keep=None, rnd=rn_bf16):
    """Expert weight gradients of the whole bf16 layer, before output rounding.

    Rows of expert e are its tokens in token order (slots with keep == 0,
    dropped by capacity, are left out, as the layer computes nothing for
    them). Returns dict name -> (value, l2, l1, rows) with name in dWg, dWu,
    dWd (E x ...) and, with a shared expert, dWsg, dWsu, dWsd."""
    topk = np.asarray(topk)
    E = Wg.shape[0]
    res = {n: WGrad(np.zeros_like(W), np.zeros_like(W), [None] * E) for n, W in (("dWg", Wg), ("dWu", Wu), ("dWd", Wd))}
    for e in range(E):
        sel = topk == e
        if keep is not None:
            sel &= np.asarray(keep, bool)
        toks, slots = np.nonzero(sel)
        if len(toks) == 0:
            continue
        c = expert_chain(x[toks], Wg[e], Wu[e], Wd[e], gates[toks, slots], dY[toks], fold=fold,
                         rnd=rnd)
        for n in ("dWg", "dWu", "dWd"):
            res[n].S[e], res[n].l1[e], res[n].chains[e] = c[n], c["l1_" + n], c
    if Wsg is not None:
        c = expert_chain(x, Wsg, Wsu, Wsd, np.ones(x.shape[0]), dY, scale_dy=False, rnd=rnd)
        for n, s in (("dWg", "dWsg"), ("dWu", "dWsu"), ("dWd", "dWsd")):
            res[s] = WGrad(c[n], c["l1_" + n], [c])
    return res


class WGrad:
    """Emulated weight gradient: S = the sums before output rounding (E x ...
    or one matrix), l1 = sums of |terms|, chains = the expert_chain result of
    each block (None for an expert without rows)."""

    def __init__(self, S, l1, chains):
        self.S, self.l1, self.chains = S, l1, chains


def router_dz(dg, gates, sel_scores, score):
    """Router logit gradient of the selected slots from the gate gradients
    (the chain rule through the gate renormalisation): softmax scores give
    dz_j = g_j (dg_j - sum_i g_i dg_i); sigmoid scores s give
    dz_j = s_j (1 - s_j) (dg_j - sum_i g_i dg_i) / sum_i s_i."""
    spread = dg - (gates * dg).sum(1, keepdims=True)
    if score == 0:
        return gates * spread
    return sel_scores * (1.0 - sel_scores) * spread / sel_scores.sum(1, keepdims=True)


def layer_dwr(x, Wg, Wu, Wd, topk, gates, sel_scores, dY, score, E, fold=False, keep=None,
              rnd=rn_bf16):
    """Router weight gradient dWr = x^T dz (H x E) with the gate gradients of
    the bf16 layer: dg = <dY, Yp> from the stored bf16 expert outputs (memory-
    efficient order: dg = <dY Wd^T, h> from the stored a, u). Dropped slots
    (keep == 0) have dg = 0. Also returns the per-entry sqrt of the sums of
    squared terms and the sums of absolute terms."""
    topk = np.asarray(topk)
    T, k = topk.shape
    dg = np.zeros((T, k))
    for e in range(E):
        sel = topk == e
        if keep is not None:
            sel &= np.asarray(keep, bool)
        toks, slots = np.nonzero(sel)
        if len(toks) == 0:
            continue
        c = expert_chain(x[toks], Wg[e], Wu[e], Wd[e], gates[toks, slots], dY[toks], fold=fold, rnd=rnd)
        dg[toks, slots] = c["dg"]
    dz = router_dz(dg, gates, sel_scores, score)
    dzd = np.zeros((T, E))
    np.put_along_axis(dzd, topk.astype(np.int64), dz, 1)
    return x.T @ dzd, np.sqrt((x * x).T @ (dzd * dzd)), np.abs(x).T @ np.abs(dzd)


# Rounding consistency of a GPU weight-gradient element with the emulated sum
# S (before output rounding). An implementation with fp32 sums stores
# RN_bf16(S + d): d is its fp32 accumulation error over the K rows (at most
# K 2^-24 sum|terms|, the classical bound for recursive summation) plus the
# terms whose stored operands differ from the emulation's. Such differences
# are rare (an operand's fp32 value must fall within fp32 error of a bf16
# rounding midpoint: observed for about one stored value in 10^4), so:
#   - for most elements |gpu - S| <= half a bf16 ulp at S + K 2^-24 sum|terms|
#     ("tight"); at most TIGHT_MISS_FRAC of the elements may miss it;
#   - every element must satisfy it after adding MAX_MOVED_TERMS times the
#     largest deviation one term can take (|x| times the envelope of its
#     operand's deviation, expert_chain's env_*).
TIGHT_MISS_FRAC = 0.02
MAX_MOVED_TERMS = 2.0

_TERMS = {"dWg": ("X", "dA", "env_dA"), "dWu": ("X", "dU", "env_dU")}


def _max_term_move(name, c, i, j):
    """Largest move of one term of entry (i, j) of block `name` of chain c."""
    o = c["ops"]
    if name in _TERMS:
        xa, _, env = _TERMS[name]
        return np.max(np.abs(o[xa][:, i]) * c[env][:, j])
    # dWd[f, h] = sum over rows of Hw[:, f] dYp[:, h]
    return np.max(np.abs(o["dYp"][:, j]) * c["env_H"][:, i] + np.abs(o["Hw"][:, i]) * c["env_dYp"][:, j])


def rounding_check(got, wg, name):
    """Returns (tight ratio per element, fraction missing it, worst ratio of
    the per-element bound over the missing elements) for GPU values `got`
    against the emulation wg (a WGrad of the same shape)."""
    got = np.asarray(got, np.float64)
    stacked = got.ndim == 3
    K = np.array([0 if c is None else c["M"] for c in wg.chains], np.float64)
    Kb = K[:, None, None] if stacked else K[0]
    tight = 0.5 * ulp_bf16(wg.S) + Kb * 2.0 ** -24 * wg.l1
    dev = np.abs(got - wg.S)
    ratio = dev / np.where(tight > 0, tight, 1e-300)
    miss = np.argwhere(ratio > 1.0)
    worst = 0.0
    base = name[:2] + name[3:] if name.startswith("dWs") else name     # dWsg -> dWg
    for idx in miss:
        e, i, j = (idx if stacked else (0, *idx))
        c = wg.chains[e]
        allow = tight[tuple(idx)] + MAX_MOVED_TERMS * _max_term_move(base, c, i, j)
        worst = max(worst, dev[tuple(idx)] / allow)
    return ratio, len(miss) / got.size, worst


def entry_check(got, c, name, i, j):
    """(tight ratio, per-element-bound ratio) of one GPU entry against an
    expert_chain result c (possibly computed on a subset of the columns; i, j
    index c's block)."""
    S = c[name][i, j]
    tight = 0.5 * ulp_bf16(S) + c["M"] * 2.0 ** -24 * c["l1_" + name][i, j]
    dev = abs(float(got) - S)
    allow = tight + MAX_MOVED_TERMS * _max_term_move(name, c, i, j)
    return dev / tight, dev / allow
