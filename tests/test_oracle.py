"""Pins of the fp64 oracle and of the input generator (CPU only).

Each check ties the oracle to something other than itself: a published test
vector, brute force over all candidate answers, a closed form computed a
different way, an invariant of the layer, or central finite differences of
the loss. The layer's stages are those of "Scalable Training of
Mixture-of-Experts Models with Megatron Core", §2 (Route, Dispatch, Expert
Computation, Combine).
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ generator
def test_splitmix64_published_vector():
    vals = [int(l) for l in open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt"))
            if l.strip() and not l.startswith("#")]
    assert [mi.splitmix64_py(1234567, c) for c in range(5)] == vals
    got = mi.splitmix64_t(1234567, torch.arange(5)).tolist()
    assert [v & mi.MASK64 for v in got] == vals


def test_generator_torch_matches_python_and_moments():
    key = mi.tensor_key(7, 3)
    idx = [0, 1, 2, 3, 1000, 1001, 123457]
    t = mi.normal_t(key, 0, 123458, "cpu")
    for i in idx:
        assert t[i].item() == pytest.approx(mi.normal_py(key, i), rel=1e-13, abs=1e-13)
    big = mi.normal_t(key, 0, 1 << 18, "cpu")
    assert abs(big.mean().item()) < 0.01
    assert abs(big.var().item() - 1.0) < 0.01
    # slices regenerate independently
    s = mi.normal_t(key, 5000, 100, "cpu")
    assert torch.equal(s, t[5000:5100])


def test_generator_permutation_and_zipf_bias():
    w = mi.scaled(mi.WORKLOADS["qwen3_235b"], E=16)
    b = mi.make_bias(w).double()
    ranks = torch.round(torch.exp(-b / 1.5)).long()
    assert sorted(ranks.tolist()) == list(range(1, 17))


# --------------------------------------------------------------------- helpers
def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _silu(a):
    return a / (1.0 + np.exp(-a))


def _swiglu_dense(x, Wg, Wu, Wd):
    return (_silu(x @ Wg) * (x @ Wu)) @ Wd


def _layer(T=24, H=16, E=6, k=2, F=12, Fs=0, score=oracle.SOFTMAX, bias=False, seed=0):
    p = dict(x=_rand((T, H), seed), Wr=_rand((H, E), seed + 1, 0.4),
             b=_rand(E, seed + 2, 0.5) if bias else None,
             Wg=_rand((E, H, F), seed + 3, H ** -0.5), Wu=_rand((E, H, F), seed + 4, H ** -0.5),
             Wd=_rand((E, F, H), seed + 5, F ** -0.5), dY=_rand((T, H), seed + 6))
    if Fs:
        p.update(Wsg=_rand((H, Fs), seed + 7, H ** -0.5), Wsu=_rand((H, Fs), seed + 8, H ** -0.5),
                 Wsd=_rand((Fs, H), seed + 9, Fs ** -0.5))
    else:
        p.update(Wsg=None, Wsu=None, Wsd=None)
    p.update(k=k, score=score)
    return p


def _route(p):
    return oracle.route(p["x"], p["Wr"], p["b"], p["k"], p["score"])


def _fwd(p, r):
    return oracle.forward(p["x"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                          p["Wsg"], p["Wsu"], p["Wsd"])


# ---------------------------------------------------------------------- route
@pytest.mark.parametrize("score", [oracle.SOFTMAX, oracle.SIGMOID])
@pytest.mark.parametrize("E,k", [(4, 1), (6, 2), (8, 3), (5, 5)])
def test_topk_brute_force(score, E, k):
    p = _layer(T=40, E=E, k=k, score=score, bias=True, seed=E * 10 + k)
    r = _route(p)
    z = p["x"] @ p["Wr"] + p["b"]
    np.testing.assert_allclose(r["logits"], z, rtol=1e-12, atol=1e-12)
    for t in range(40):
        s = r["scores"][t]
        best = max(itertools.combinations(range(E), k), key=lambda S: sum(s[list(S)]))
        assert sorted(r["topk"][t]) == sorted(best)
        order = np.lexsort((np.arange(E), -s))[:k]          # score desc, index asc
        assert list(r["topk"][t]) == list(order)


def test_topk_equal_scores_take_lower_index():
    H, E = 4, 6
    x = np.ones((1, H))
    Wr = np.zeros((H, E))
    Wr[:, [1, 3, 4]] = 1.0          # experts 1, 3, 4 tie for the top
    r = oracle.route(x, Wr, None, 2, oracle.SOFTMAX)
    assert list(r["topk"][0]) == [1, 3]
    assert r["gap_order"][0] == 0.0 and r["gap_set"][0] == 0.0
    r = oracle.route(x, Wr, None, 3, oracle.SIGMOID)
    assert list(r["topk"][0]) == [1, 3, 4]
    assert r["gap_set"][0] > 0.1


@pytest.mark.parametrize("k", [1, 2, 4])
def test_gates_closed_forms(k):
    p = _layer(T=50, E=8, k=k, bias=True, seed=3)
    r = _route(p)
    z = r["logits"]
    np.testing.assert_allclose(r["gates"].sum(1), 1.0, rtol=0, atol=1e-14)
    # softmax over all E, renormalised over S == softmax over the selected logits
    zs = np.take_along_axis(z, r["topk"].astype(np.int64), 1)
    ref = np.exp(zs - zs.max(1, keepdims=True))
    ref /= ref.sum(1, keepdims=True)
    np.testing.assert_allclose(r["gates"], ref, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(r["scores"].sum(1), 1.0, atol=1e-14)
    if k == 1:
        assert np.all(r["gates"] == 1.0)
    p["score"] = oracle.SIGMOID
    r = _route(p)
    s = 1.0 / (1.0 + np.exp(-z))
    ss = np.take_along_axis(s, r["topk"].astype(np.int64), 1)
    np.testing.assert_allclose(r["gates"], ss / ss.sum(1, keepdims=True), rtol=1e-13)


def test_route_replay_uses_given_selection():
    p = _layer(T=10, E=6, k=2, seed=5)
    r = _route(p)
    alt = r["topk"].copy()
    alt[3] = alt[3][::-1]
    alt[7] = [5, 0] if list(alt[7]) != [5, 0] else [4, 1]
    mask = np.zeros(10, np.uint8)
    mask[[3, 7]] = 1
    r2 = oracle.route(p["x"], p["Wr"], None, 2, oracle.SOFTMAX, alt, mask)
    assert np.array_equal(r2["topk"], alt)
    s = r2["scores"][7][alt[7]]
    np.testing.assert_allclose(r2["gates"][7], s / s.sum(), rtol=1e-14)
    np.testing.assert_array_equal(r2["gates"][0], r["gates"][0])


# ------------------------------------------------------------------- dispatch
def test_dispatch_invariants_and_permutation_identity():
    p = _layer(T=64, E=8, k=3, bias=True, seed=11)
    r = _route(p)
    d = oracle.dispatch(r["topk"], 8)
    T, k = r["topk"].shape
    assert d["counts"].sum() == T * k
    assert np.array_equal(d["counts"], np.bincount(r["topk"].ravel(), minlength=8))
    assert d["offsets"][0] == 0 and np.array_equal(np.diff(d["offsets"]), d["counts"])
    assert sorted(d["row_of"].ravel()) == list(range(T * k))          # bijection
    assert np.array_equal(d["slot_of"][d["row_of"].ravel()], np.arange(T * k))
    for e in range(8):
        seg = d["slot_of"][d["offsets"][e]:d["offsets"][e + 1]]
        toks = seg // k
        assert np.all(np.diff(toks) > 0)                                # token ascending
        assert np.all(r["topk"].ravel()[seg] == e)
    Xp = p["x"][d["slot_of"] // k]                                      # permute
    back = Xp[d["row_of"]]                                              # unpermute
    for j in range(k):
        assert np.array_equal(back[:, j, :], p["x"])


# -------------------------------------------------------------------- forward
def test_single_expert_top1_is_dense_swiglu():
    p = _layer(T=20, H=16, E=1, k=1, F=24, seed=2)
    r = _route(p)
    y = _fwd(p, r)
    ref = _swiglu_dense(p["x"], p["Wg"][0], p["Wu"][0], p["Wd"][0])
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("score", [oracle.SOFTMAX, oracle.SIGMOID])
def test_identical_experts_give_dense_ffn_for_any_routing(score):
    p = _layer(T=30, E=5, k=3, score=score, bias=True, seed=4)
    for key in ("Wg", "Wu", "Wd"):
        p[key] = np.repeat(p[key][:1], 5, axis=0)
    y = _fwd(p, _route(p))
    ref = _swiglu_dense(p["x"], p["Wg"][0], p["Wu"][0], p["Wd"][0])
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_expert_rows_shared_expert_and_linearity():
    p = _layer(T=18, E=4, k=2, Fs=10, seed=6)
    r = _route(p)
    y, Yp = oracle.forward(p["x"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                           p["Wsg"], p["Wsu"], p["Wsd"], want_Yp=True)
    d = oracle.dispatch(r["topk"], 4)
    for row in range(18 * 2):
        t, j = divmod(int(d["slot_of"][row]), 2)
        e = r["topk"][t, j]
        ref = _swiglu_dense(p["x"][t:t + 1], p["Wg"][e], p["Wu"][e], p["Wd"][e])[0]
        np.testing.assert_allclose(Yp[row], ref, rtol=1e-12, atol=1e-13)
    y0 = oracle.forward(p["x"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"])
    np.testing.assert_allclose(y - y0, _swiglu_dense(p["x"], p["Wsg"], p["Wsu"], p["Wsd"]),
                               rtol=1e-12, atol=1e-12)
    y2 = oracle.forward(p["x"], p["Wg"], p["Wu"], 2.0 * p["Wd"], r["topk"], r["gates"])
    np.testing.assert_allclose(y2, 2.0 * y0, rtol=1e-14, atol=1e-14)


# ------------------------------------------------------------------- backward
def _loss(p):
    r = _route(p)
    return float((p["dY"] * _fwd(p, r)).sum()), r["topk"]


@pytest.mark.parametrize("score,bias,Fs", [(oracle.SOFTMAX, False, 0), (oracle.SIGMOID, True, 6),
                                           (oracle.SOFTMAX, True, 5)])
def test_backward_finite_differences(score, bias, Fs):
    p = _layer(T=10, H=8, E=5, k=2, F=6, Fs=Fs, score=score, bias=bias, seed=21)
    r = _route(p)
    g = oracle.backward(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                        r["scores"], p["dY"], score, p["Wsg"], p["Wsu"], p["Wsd"])
    names = [("x", "dX"), ("Wr", "dWr"), ("Wg", "dWg"), ("Wu", "dWu"), ("Wd", "dWd")]
    if Fs:
        names += [("Wsg", "dWsg"), ("Wsu", "dWsu"), ("Wsd", "dWsd")]
    rng = np.random.default_rng(0)
    eps = 1e-6
    checked = 0
    for pn, gn in names:
        flat = p[pn].reshape(-1)
        for idx in rng.choice(flat.size, size=min(flat.size, 12), replace=False):
            old = flat[idx]
            flat[idx] = old + eps
            lp, tp = _loss(p)
            flat[idx] = old - eps
            lm, tm = _loss(p)
            flat[idx] = old
            if not (np.array_equal(tp, r["topk"]) and np.array_equal(tm, r["topk"])):
                continue                    # the perturbation changed the routing
            fd = (lp - lm) / (2 * eps)
            an = g[gn].reshape(-1)[idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (gn, idx, fd, an)
            checked += 1
    assert checked >= 40


def test_backward_expert_without_tokens_has_zero_gradient():
    p = _layer(T=12, E=4, k=1, bias=False, seed=8)
    p["b"] = np.array([0.0, 0.0, -40.0, 0.0])      # expert 2 never chosen
    r = _route(p)
    assert not np.any(r["topk"] == 2)
    g = oracle.backward(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                        r["scores"], p["dY"], oracle.SOFTMAX)
    for n in ("dWg", "dWu", "dWd"):
        assert np.all(g[n][2] == 0.0)
    assert np.all(g["dWr"] == 0.0)                  # k = 1: gates are all 1


def test_softmax_router_gradient_rows_sum_to_zero():
    p = _layer(T=30, E=6, k=3, seed=9)
    r = _route(p)
    g = oracle.backward(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                        r["scores"], p["dY"], oracle.SOFTMAX)
    np.testing.assert_allclose(g["dWr"].sum(1), 0.0, atol=1e-12)


# ------------------------------------------------------------ sampled forms
def _bf16_bits(a):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16), t.double().numpy()


@pytest.mark.parametrize("storage", ["f32", "bf16"])
def test_sampled_rows_and_entries_match_full_oracle(storage):
    p = _layer(T=16, H=8, E=4, k=2, F=6, Fs=4, score=oracle.SIGMOID, bias=True, seed=31)
    conv = {}
    for n in ("Wg", "Wu", "Wd", "Wsg", "Wsu", "Wsd"):
        if storage == "bf16":
            conv[n], p[n] = _bf16_bits(p[n])
        else:
            p[n] = p[n].astype(np.float32).astype(np.float64)
            conv[n] = p[n].astype(np.float32)
    r = _route(p)
    g = oracle.backward(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                        r["scores"], p["dY"], oracle.SIGMOID, p["Wsg"], p["Wsu"], p["Wsd"])
    y = _fwd(p, r)
    W = oracle.ExpertWeights(4, {e: conv["Wg"][e] for e in range(4)},
                             {e: conv["Wu"][e] for e in range(4)},
                             {e: conv["Wd"][e] for e in range(4)},
                             conv["Wsg"], conv["Wsu"], conv["Wsd"])
    toks = np.array([0, 5, 9, 15])
    tr = oracle.token_rows(p["x"][toks], p["dY"][toks], p["Wr"], W, r["topk"][toks],
                           r["gates"][toks], r["scores"][toks], oracle.SIGMOID)
    np.testing.assert_allclose(tr["y"], y[toks], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(tr["dX"], g["dX"][toks], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(tr["dg"], g["dg"][toks], rtol=1e-12, atol=1e-13)
    ents = [("dWg", 1, 3, 2), ("dWu", 3, 7, 5), ("dWd", 0, 5, 1), ("dWd", 2, 0, 7),
            ("dWsg", 0, 2, 3), ("dWsu", 0, 7, 0), ("dWsd", 0, 3, 6)]
    out = oracle.dw_entries(p["x"], p["dY"], W, r["topk"], r["gates"], ents)
    for (n, e, i, j), v in zip(ents, out):
        ref = g[n][i, j] if n.startswith("dWs") else g[n][e, i, j]
        assert v == pytest.approx(ref, rel=1e-12, abs=1e-13)


# ------------------------------------------------- capacity-limited dropping
def test_capacity_keep_rule_brute_force():
    """Kept assignments of each expert are exactly its C earliest tokens."""
    p = _layer(T=60, E=5, k=2, bias=True, seed=31)
    r = _route(p)
    for C in (0, 3, 17, 60):
        keep = oracle.capacity_keep(r["topk"], 5, C)
        for e in range(5):
            toks = sorted(int(t) for t, j in zip(*np.nonzero(r["topk"] == e)))
            kept = sorted(int(t) for t, j in zip(*np.nonzero((r["topk"] == e) & (keep == 1))))
            assert kept == toks[:C]
    assert oracle.capacity(T=4096, k=2, E=8, factor=1.25) == 1280
    assert oracle.capacity(T=10, k=3, E=4, factor=1.0) == 8      # ceil(7.5)


def test_capacity_above_max_load_is_dropless():
    p = _layer(T=30, E=4, k=2, Fs=5, bias=True, seed=32)
    r = _route(p)
    keep = oracle.capacity_keep(r["topk"], 4, 60)
    assert keep.all()
    y0 = _fwd(p, r)
    y1 = oracle.forward(p["x"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"], p["Wsg"],
                        p["Wsu"], p["Wsd"], keep=keep)
    assert np.array_equal(y0, y1)
    g0 = oracle.backward(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                         r["scores"], p["dY"], p["score"], p["Wsg"], p["Wsu"], p["Wsd"])
    g1 = oracle.backward(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                         r["scores"], p["dY"], p["score"], p["Wsg"], p["Wsu"], p["Wsd"], keep=keep)
    for n in g0:
        assert np.array_equal(g0[n], g1[n]), n


def test_capacity_dropped_top1_token_gets_only_the_shared_expert():
    p = _layer(T=20, E=3, k=1, Fs=4, seed=33)
    r = _route(p)
    keep = oracle.capacity_keep(r["topk"], 3, 2)
    assert (keep == 0).any()
    y = oracle.forward(p["x"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"], p["Wsg"],
                       p["Wsu"], p["Wsd"], keep=keep)
    shared = _swiglu_dense(p["x"], p["Wsg"], p["Wsu"], p["Wsd"])
    dropped = keep[:, 0] == 0
    np.testing.assert_allclose(y[dropped], shared[dropped], rtol=1e-12, atol=1e-12)
    e0 = r["topk"][~dropped, 0]
    ref = np.stack([_swiglu_dense(p["x"][[t]], p["Wg"][e], p["Wu"][e], p["Wd"][e])[0]
                    for t, e in zip(np.nonzero(~dropped)[0], e0)]) + shared[~dropped]
    np.testing.assert_allclose(y[~dropped], ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("score", [oracle.SOFTMAX, oracle.SIGMOID])
def test_capacity_backward_finite_differences(score):
    """Gradients with dropped slots (routing and drops held fixed) against
    central differences of the dropping forward."""
    p = _layer(T=16, H=8, E=3, k=2, F=6, Fs=4, score=score, bias=True, seed=34)
    r = _route(p)
    C = 7
    keep = oracle.capacity_keep(r["topk"], 3, C)
    assert (keep == 0).sum() >= 3
    g = oracle.backward(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                        r["scores"], p["dY"], score, p["Wsg"], p["Wsu"], p["Wsd"], keep=keep)
    assert np.all(g["dg"][keep == 0] == 0.0)

    def loss():
        rr = _route(p)
        kk = oracle.capacity_keep(rr["topk"], 3, C)
        y = oracle.forward(p["x"], p["Wg"], p["Wu"], p["Wd"], rr["topk"], rr["gates"], p["Wsg"],
                           p["Wsu"], p["Wsd"], keep=kk)
        return float((p["dY"] * y).sum()), rr["topk"]

    rng = np.random.default_rng(1)
    eps, checked = 1e-6, 0
    for pn, gn in [("x", "dX"), ("Wr", "dWr"), ("Wg", "dWg"), ("Wu", "dWu"), ("Wd", "dWd"),
                   ("Wsd", "dWsd")]:
        flat = p[pn].reshape(-1)
        for idx in rng.choice(flat.size, size=min(flat.size, 12), replace=False):
            old = flat[idx]
            flat[idx] = old + eps
            lp, tp = loss()
            flat[idx] = old - eps
            lm, tm = loss()
            flat[idx] = old
            if not (np.array_equal(tp, r["topk"]) and np.array_equal(tm, r["topk"])):
                continue
            an = g[gn].reshape(-1)[idx]
            assert abs((lp - lm) / (2 * eps) - an) <= 1e-6 * max(1.0, abs(an)), (gn, idx)
            checked += 1
    assert checked >= 40


# ------------------------------------------ auxiliary-loss-free bias update
def test_update_bias_moves_load_towards_the_mean():
    counts = np.array([10, 2, 6, 6, 0, 12], np.int32)        # mean 6
    b = np.array([0.5, -0.25, 0.0, 1.0, 0.0, -1.0], np.float32)
    nb = oracle.update_bias(b, counts, 0.125)
    np.testing.assert_array_equal(nb, np.array([0.375, -0.125, 0.0, 1.0, 0.125, -1.125], np.float32))
    # a balanced load leaves the bias unchanged; the step sizes are +-rate or 0
    assert np.array_equal(oracle.update_bias(b, np.full(6, 7, np.int32), 0.3), b)
    d = oracle.update_bias(np.zeros(6, np.float32), counts, 1.0)
    assert set(d.tolist()) <= {-1.0, 0.0, 1.0}


def test_update_bias_mean_is_compared_exactly():
    # mean 10/3: no expert is at the mean; a float mean could misclassify
    counts = np.array([3, 3, 4], np.int32)
    nb = oracle.update_bias(np.zeros(3, np.float32), counts, 1.0)
    np.testing.assert_array_equal(nb, np.array([1.0, 1.0, -1.0], np.float32))
