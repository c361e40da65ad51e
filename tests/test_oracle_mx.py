"""Pins of the oracle's MXFP8 pieces (CPU only).

MXFP8 ("Scalable Training of Mixture-of-Experts Models with Megatron Core",
§5 Platform-specific recipes: the default FP8 recipe on Blackwell, 1x32
granularity): each block of 32 values along a GEMM's contraction dimension
shares a power-of-two scale 2^e (an UE8M0 byte e + 127) and each value is
stored as the E4M3 code of v / 2^e. Reading of the scale: the smallest e
with amax <= 448 2^e (no value saturates), in [-127, 127]; all-zero blocks
take e = -127.

Pins: the exponent rule by brute force over every positive finite bf16 value
(and random fp32 values), the codes against PyTorch's float8_e4m3fn
conversion (an independent E4M3 implementation), block locality, and the
whole MXFP8 layer against an independent numpy layer with PyTorch's codec
(several experts, ragged segments) and against the exact layer within the
E4M3 error scale.
"""
import numpy as np
import pytest
import torch

import oracle


def _e_brute(amax):
    """Smallest e in [-127, 127] with amax <= 448 2^e (exact power-of-two
    arithmetic in fp64)."""
    if amax == 0:
        return -127
    e = -127
    while e < 127 and amax > np.ldexp(448.0, e):
        e += 1
    return e


def test_mx_exponent_every_bf16_value():
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32)         # positive finite bf16
    vals = (bits << 16).view(np.float32)
    got = np.array([oracle.mx_exponent(v) for v in vals])
    # vectorised brute force: e = smallest with amax <= 448 2^e
    e = np.full(len(vals), -127)
    for cand in range(-127, 128):
        fits = vals.astype(np.float64) <= np.ldexp(448.0, cand)
        e = np.where((e == -127) & ~(vals.astype(np.float64) <= np.ldexp(448.0, -127)) & fits, cand, e)
    assert np.array_equal(got, e)
    for v in (1e-40, 1.0, 448.0, 448.0 * (1 + 2 ** -7), 896.0, 3.0e38, 0.0):
        assert oracle.mx_exponent(np.float32(v)) == _e_brute(float(np.float32(v))), v
    assert oracle.mx_exponent(448.0) == 0 and oracle.mx_exponent(449.0) == 1
    assert oracle.mx_exponent(0.875) == -9 and oracle.mx_exponent(0.876) == -8


def _torch_codes(v, e):
    f = np.ldexp(v.astype(np.float64), -e.astype(np.int64)).astype(np.float32)
    assert np.all(np.abs(f) <= 448.0)
    return torch.from_numpy(np.ascontiguousarray(f)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("mode", [oracle.MX_ROWS, oracle.MX_COLS])
def test_mx_codes_match_torch_e4m3(mode):
    rng = np.random.default_rng(3)
    M, K = 100, 192                                   # 100 rows: a ragged last 32-row block
    X = (rng.standard_normal((M, K)) * 10.0 ** rng.uniform(-6, 4, (M, 1))).astype(np.float32)
    X[:, :32] = 0                                     # all-zero blocks
    X[7, 40] = 3.0e4
    codes, sc = oracle.mx_quantize(X, mode)
    if mode == oracle.MX_ROWS:
        amax = np.abs(X).reshape(M, K // 32, 32).max(2)
        e = np.vectorize(_e_brute)(amax.astype(np.float64))
        assert np.array_equal(sc, (e + 127).astype(np.uint8))
        want = _torch_codes(X, np.repeat(e, 32, axis=1))
    else:
        pad = np.zeros((-M % 32, K), np.float32)
        amax = np.abs(np.vstack([X, pad])).reshape(-1, 32, K).max(1)
        e = np.vectorize(_e_brute)(amax.astype(np.float64))
        assert np.array_equal(sc, (e + 127).astype(np.uint8))
        want = _torch_codes(X, np.repeat(e, 32, axis=0)[:M])
    assert np.array_equal(codes, want)
    # each block's largest magnitude lands within a factor two below 448
    dq = oracle.e4m3_decode(codes)
    big = np.abs(dq).reshape(M, K // 32, 32).max(2) if mode == oracle.MX_ROWS else None
    if big is not None:
        nz = amax > 0
        assert np.all(big[nz] > 224.0 * (1 - 2 ** -3)) and np.all(big[nz] <= 448.0)


def test_mx_blocks_are_local():
    rng = np.random.default_rng(4)
    X = rng.standard_normal((64, 128)).astype(np.float32)
    c0, _ = oracle.mx_quantize(X, oracle.MX_ROWS)
    X2 = X.copy()
    X2[5, 40] *= 100
    c2, _ = oracle.mx_quantize(X2, oracle.MX_ROWS)
    ch = np.argwhere(c2 != c0)
    assert np.all(ch[:, 0] == 5) and np.all((ch[:, 1] >= 32) & (ch[:, 1] < 64))
    c0, _ = oracle.mx_quantize(X, oracle.MX_COLS)
    c2, _ = oracle.mx_quantize(X2, oracle.MX_COLS)
    ch = np.argwhere(c2 != c0)
    assert np.all(ch[:, 1] == 40) and np.all(ch[:, 0] < 32)


# ---- an independent MXFP8 layer: numpy, rows gathered per expert, torch's codec
def _mx(X, axis):
    """Quantise-dequantise along `axis` (1: 1x32 within rows; 0: 32-row blocks
    per column counted from row 0)."""
    X = np.asarray(X, np.float64)
    if axis == 0:
        return _mx(X.T, 1).T
    M, K = X.shape
    pad = -K % 32
    Xp = np.hstack([X, np.zeros((M, pad))]).reshape(M, -1, 32)
    amax = np.abs(Xp.astype(np.float32)).max(2).astype(np.float64)
    e = np.vectorize(_e_brute)(amax)[:, :, None]
    f = np.ldexp(Xp.astype(np.float32).astype(np.float64), -e).astype(np.float32)
    q = torch.from_numpy(np.ascontiguousarray(f)).to(torch.float8_e4m3fn).double().numpy()
    return np.ldexp(q, e).reshape(M, -1)[:, :K]


def _layer(T, H, E, k, F, seed):
    rng = np.random.default_rng(seed)
    return dict(x=rng.standard_normal((T, H)), Wr=rng.standard_normal((H, E)) * 0.1,
                Wg=rng.standard_normal((E, H, F)) * H ** -0.5, Wu=rng.standard_normal((E, H, F)) * H ** -0.5,
                Wd=rng.standard_normal((E, F, H)) * F ** -0.5, dY=rng.standard_normal((T, H)))


@pytest.mark.parametrize("fold,drop", [(False, False), (True, False), (False, True), (True, True)])
def test_mx_layer_matches_independent_mx_swiglu(fold, drop):
    """drop: capacity 100 per expert; the expert's segment (and its 32-row
    blocks) is its first 100 assignments, the dropped slots get dg = 0."""
    T, H, E, k, F = 333, 256, 3, 2, 256
    p = _layer(T, H, E, k, F, seed=23)
    b = np.array([0.8, 0.0, -0.9])
    r = oracle.route(p["x"], p["Wr"], b, k, oracle.SOFTMAX)
    counts = np.bincount(r["topk"].ravel(), minlength=E)
    assert np.all(counts % 32 != 0)                   # every segment ends in a partial block
    keep = oracle.capacity_keep(r["topk"], E, 100) if drop else np.ones_like(r["topk"], np.uint8)
    if drop:
        assert np.all(counts > 100)
    q = oracle.layer_fp8(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                         r["scores"], oracle.SOFTMAX, p["dY"], fold=fold, recipe=oracle.RECIPE_MX,
                         keep=keep if drop else None)
    if drop:
        assert np.all(q["dg"][keep == 0] == 0) and np.all(q["dg"][keep == 1] != 0)
    bf = lambda v: torch.from_numpy(np.ascontiguousarray(v)).to(torch.bfloat16).double().numpy()
    y = np.zeros((T, H))
    ref = {n: np.zeros_like(p[w]) for n, w in (("dWg", "Wg"), ("dWu", "Wu"), ("dWd", "Wd"))}
    for e in range(E):
        toks, slots = np.nonzero((r["topk"] == e) & (keep == 1))
        g = r["gates"][toks, slots][:, None]
        X = p["x"][toks]
        Wg_f, Wu_f, Wd_f = _mx(p["Wg"][e], 0), _mx(p["Wu"][e], 0), _mx(p["Wd"][e], 0)
        Wg_b, Wu_b, Wd_b = _mx(p["Wg"][e], 1), _mx(p["Wu"][e], 1), _mx(p["Wd"][e], 1)
        xq = _mx(X, 1)
        a32, u32 = xq @ Wg_f, xq @ Wu_f
        h32 = a32 / (1 + np.exp(-a32)) * u32
        h = bf(g * h32) if fold else bf(h32)
        a, u = bf(a32), bf(u32)
        Yp = bf(_mx(h, 1) @ Wd_f)
        y[toks] += Yp if fold else g * Yp
        dYp = bf(p["dY"][toks]) if fold else bf(g * p["dY"][toks])
        dh = _mx(dYp, 1) @ Wd_b.T
        sg = 1 / (1 + np.exp(-a))
        if fold:
            dh = g * dh
            h = bf(g * (a * sg * u))
        dA = bf(dh * u * sg * (1 + a * (1 - sg)))
        dU = bf(dh * a * sg)
        ref["dWd"][e] = _mx(h, 0).T @ _mx(dYp, 0)
        ref["dWg"][e] = _mx(X, 0).T @ _mx(dA, 0)
        ref["dWu"][e] = _mx(X, 0).T @ _mx(dU, 0)
        dX_e = _mx(dA, 1) @ Wg_b.T + _mx(dU, 1) @ Wu_b.T
        ref.setdefault("dXp", []).append((toks, dX_e))
    ref["y"] = y
    for n in ("y", "dWg", "dWu", "dWd"):
        v = ref[n]
        close = np.isclose(q[n], v, rtol=1e-9, atol=1e-9 * np.abs(v).max())
        assert close.mean() > 0.999, (n, close.mean())
        assert np.linalg.norm(q[n] - v) / np.linalg.norm(v) < 1e-3, n


@pytest.mark.parametrize("fold", [False, True])
def test_mx_layer_tracks_the_exact_layer(fold):
    """Each E4M3 rounding of an MX block perturbs a value by at most 2^-4
    relative (a bit more for values far below their block's maximum, which
    fall into E4M3's coarser subnormal steps); an output passes through up
    to ~6 roundings, so it stays within ~9% rms of the exact layer."""
    p = _layer(T=150, H=256, E=4, k=2, F=256, seed=5)
    r = oracle.route(p["x"], p["Wr"], None, 2, oracle.SOFTMAX)
    q = oracle.layer_fp8(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                         r["scores"], oracle.SOFTMAX, p["dY"], fold=fold, recipe=oracle.RECIPE_MX)
    y = oracle.forward(p["x"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"])
    g = oracle.backward(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"], r["scores"],
                        p["dY"], oracle.SOFTMAX)
    g["y"] = y
    qb = oracle.layer_fp8(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                          r["scores"], oracle.SOFTMAX, p["dY"], fold=fold, recipe=oracle.RECIPE_BLOCK)
    for n in q:
        if n == "dg":
            continue
        rel = np.linalg.norm(q[n] - g[n]) / np.linalg.norm(g[n])
        assert 0.005 < rel < 0.09, (n, rel)
        # a different recipe: not the blockwise layer's numbers
        assert np.linalg.norm(q[n] - qb[n]) > 1e-6 * np.linalg.norm(qb[n]), n
