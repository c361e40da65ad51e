"""Pins of the oracle's NVFP4 pieces (CPU only).

NVFP4 ("Scalable Training of Mixture-of-Experts Models with Megatron Core",
§5 Platform-specific recipes: NVFP4 for Blackwell; §5 Kernel and shape
optimization: grouped quantisation ahead of the grouped NVFP4 GEMMs). The
pages give no parameters; the reading is the format itself: E2M1 values,
16-value blocks along K with unsigned E4M3 scales, one fp32 scale
S = 2688 / amax per tensor (one expert's operand of one grouped GEMM; the
fc1 weights [Wg | Wu] and their output gradients [dA | dU] one tensor each).

Pins: the E2M1 code table against the format's bit fields; the encoder by
brute-force nearest search with ties to the even code; the block scales and
codes against an independent numpy implementation that uses PyTorch's E4M3
conversion; the tensor scale's effect (largest block at scale 448); block
locality; and the whole NVFP4 layer against an independent numpy layer
(several experts, segments that end in partial 16-row blocks, folded gates,
capacity drops) and against the exact layer within the E2M1 error scale.
"""
import numpy as np
import pytest
import torch

import oracle


def _e2m1_from_bits(c):
    """Value of a 4-bit E2M1 code from its fields: sign, 2-bit exponent with
    bias 1, 1-bit mantissa; exponent 0 is subnormal (0.m x 2^0)."""
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    v = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + 0.5 * m)
    return -v if s else v


_GRID = np.array([_e2m1_from_bits(c) for c in range(8)])


def _e2m1_brute(f):
    """Nearest E2M1 code of an fp32 value (ties to the code whose mantissa bit
    is 0), saturating at 6, with the value's sign bit (-0 included)."""
    m = min(abs(float(f)), 6.0)                        # saturation
    d = np.abs(_GRID - m)
    best = np.flatnonzero(d == d.min())
    c = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
    return c | (8 if np.signbit(f) else 0)


def test_e2m1_decode_is_the_format():
    got = oracle.e2m1_decode(np.arange(16))
    want = np.array([_e2m1_from_bits(c) for c in range(16)])
    assert np.array_equal(got, want)
    assert list(got[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_encode_is_nearest_ties_to_even():
    mids = (_GRID[1:] + _GRID[:-1]) / 2                # every tie
    rng = np.random.default_rng(1)
    vals = np.concatenate([_GRID, mids, mids + 1e-6, mids - 1e-6, rng.uniform(-9, 9, 2000),
                           [6.0001, 7.0, 1e30, 1e-30, 0.0]]).astype(np.float32)
    vals = np.concatenate([vals, -vals])
    assert np.signbit(vals[-1])                          # -0.0 is among them
    got = oracle.e2m1_encode(vals)
    want = np.array([_e2m1_brute(v) for v in vals], np.uint8)
    assert np.array_equal(got, want)
    # the ties: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    assert list(oracle.e2m1_decode(oracle.e2m1_encode(mids))) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def _e4m3_torch(f32):
    t = torch.from_numpy(np.ascontiguousarray(f32, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy(), t.float().numpy()


def _nv_numpy(X, by_row, amax=None):
    """Independent NVFP4 quantisation of X as one tensor (or of the tensor
    whose largest magnitude is `amax`): codes, scale bytes and the
    dequantised values; fp32 arithmetic step by step in numpy."""
    X = np.asarray(X, np.float32)
    if not by_row:
        c, sb, dq = _nv_numpy(X.T, True, amax)
        return c.T, sb.T, dq.T
    M, K = X.shape
    pad = -K % 16
    Xp = np.hstack([X, np.zeros((M, pad), np.float32)]).reshape(M, -1, 16)
    am = np.float32(np.abs(X).max() if amax is None else amax)
    S = np.float32(2688.0) / am if am > 0 else np.float32(1.0)
    a = np.abs(Xp).max(2)
    sf = (a * S).astype(np.float32) / np.float32(6.0)
    assert np.all(sf <= 448.0 * (1 + 2 ** -20))
    sb, s = _e4m3_torch(sf)
    with np.errstate(divide="ignore"):
        r = np.where(s > 0, S / np.where(s > 0, s, 1).astype(np.float32), 0).astype(np.float32)
    v = (Xp * r[:, :, None]).astype(np.float32)
    codes = np.vectorize(_e2m1_brute, otypes=[np.uint8])(v)
    codes = np.where(s[:, :, None] > 0, codes, 0).astype(np.uint8)
    vals = np.array([_e2m1_from_bits(c) for c in range(16)])[codes]
    dq = vals * s.astype(np.float64)[:, :, None] / np.float64(S)
    return codes.reshape(M, -1)[:, :K], sb, dq.reshape(M, -1)[:, :K]


@pytest.mark.parametrize("mode", [oracle.NV_ROWS, oracle.NV_COLS])
def test_nv_quantize_matches_independent_numpy(mode):
    rng = np.random.default_rng(7)
    M, K = 72, 96                                   # 72 rows: a ragged last 16-row block
    X = (rng.standard_normal((M, K)) * 10.0 ** rng.uniform(-5, 2, (M, 1))).astype(np.float32)
    X[:16, :16] = 0                                 # an all-zero block in both modes
    X[3, 50] = -250.0                               # the tensor maximum
    X[9, 5] = 1e-38                                 # a value far below its block's maximum
    codes, sc, S = oracle.nv_quantize(X, mode)
    assert S == np.float32(2688.0) / np.float32(250.0)
    c2, s2, _ = _nv_numpy(X, mode == oracle.NV_ROWS)
    assert np.array_equal(codes, c2)
    assert np.array_equal(sc, s2)
    # the block holding the tensor maximum gets the largest E4M3 scale and code -6
    blk = (3, 50 // 16) if mode == oracle.NV_ROWS else (0, 50)
    assert sc[blk] == 0x7E and codes[3, 50] == 0xF
    # all-zero tensor: S = 1 and zero codes and scales
    z, zs, S0 = oracle.nv_quantize(np.zeros((16, 32), np.float32), mode)
    assert S0 == 1.0 and not z.any() and not zs.any()


def test_nv_dequantised_error_is_within_half_a_step():
    """|v - q s / S| <= half the E2M1 step at |v| (relative to the block's
    scale s / S), plus the saturation allowance of the rounded E4M3 scale."""
    rng = np.random.default_rng(9)
    X = rng.standard_normal((64, 128)).astype(np.float32)
    codes, sc, S = oracle.nv_quantize(X, oracle.NV_ROWS)
    s = oracle.e4m3_decode(sc)                                     # [64][8]
    dq = oracle.e2m1_decode(codes) * np.repeat(s, 16, axis=1) / np.float64(S)
    unit = np.repeat(s, 16, axis=1) / np.float64(S)                # value of code 1.0
    # step of the E2M1 grid at the quantised magnitude: 0.5 below 2, 1 to 4, 2 above
    m = np.abs(X) / unit
    step = np.where(m < 2, 0.5, np.where(m < 4, 1.0, 2.0)) * unit
    sat = np.maximum(np.abs(X) - 6 * unit, 0)
    assert np.all(np.abs(X - dq) <= step / 2 + sat + 1e-12)


def test_nv_blocks_are_local():
    rng = np.random.default_rng(4)
    X = rng.standard_normal((64, 128)).astype(np.float32)
    X[0, 0] = 50.0                                  # the tensor maximum stays put
    c0, s0, _ = oracle.nv_quantize(X, oracle.NV_ROWS)
    X2 = X.copy()
    X2[5, 40] *= 8
    c2, s2, _ = oracle.nv_quantize(X2, oracle.NV_ROWS)
    ch = np.argwhere(c2 != c0)
    assert len(ch) and np.all(ch[:, 0] == 5) and np.all((ch[:, 1] >= 32) & (ch[:, 1] < 48))
    assert np.array_equal(np.argwhere(s2 != s0), [[5, 2]])
    c0, _, _ = oracle.nv_quantize(X, oracle.NV_COLS)
    c2, _, _ = oracle.nv_quantize(X2, oracle.NV_COLS)
    ch = np.argwhere(c2 != c0)
    assert len(ch) and np.all(ch[:, 1] == 40) and np.all(ch[:, 0] < 16)


# ---- an independent NVFP4 layer: numpy, rows gathered per expert
def _nv(X, axis, amax):
    """Dequantised NVFP4 of X along `axis` (1: 1x16 within rows; 0: 16-row
    blocks per column counted from row 0) in the tensor of maximum amax."""
    return _nv_numpy(X, axis == 1, amax)[2]


def _layer(T, H, E, k, F, seed):
    rng = np.random.default_rng(seed)
    return dict(x=rng.standard_normal((T, H)), Wr=rng.standard_normal((H, E)) * 0.1,
                Wg=rng.standard_normal((E, H, F)) * H ** -0.5, Wu=rng.standard_normal((E, H, F)) * H ** -0.5,
                Wd=rng.standard_normal((E, F, H)) * F ** -0.5, dY=rng.standard_normal((T, H)))


def _bf(v):
    return torch.from_numpy(np.ascontiguousarray(v)).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("fold,drop", [(False, False), (True, False), (False, True), (True, True)])
def test_nv_layer_matches_independent_nv_swiglu(fold, drop):
    """drop: capacity 100 per expert; the expert's segment (its 16-row blocks
    and its tensor scales) holds its first 100 assignments alone."""
    T, H, E, k, F = 333, 256, 3, 2, 256
    p = _layer(T, H, E, k, F, seed=23)
    for n in ("x", "Wg", "Wu", "Wd", "dY"):
        p[n] = _bf(p[n])                                # bf16 inputs, as the layer takes them
    b = np.array([0.8, 0.0, -0.9])
    r = oracle.route(p["x"], p["Wr"], b, k, oracle.SOFTMAX)
    counts = np.bincount(r["topk"].ravel(), minlength=E)
    assert np.all(counts % 16 != 0)                     # every segment ends in a partial block
    keep = oracle.capacity_keep(r["topk"], E, 100) if drop else np.ones_like(r["topk"], np.uint8)
    if drop:
        assert np.all(counts > 100)
    q = oracle.layer_fp8(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                         r["scores"], oracle.SOFTMAX, p["dY"], fold=fold, recipe=oracle.RECIPE_NV,
                         keep=keep if drop else None)
    if drop:
        assert np.all(q["dg"][keep == 0] == 0) and np.all(q["dg"][keep == 1] != 0)
    am = lambda *ms: max(np.abs(np.asarray(m, np.float32)).max() for m in ms)
    y = np.zeros((T, H))
    ref = {n: np.zeros_like(p[w]) for n, w in (("dWg", "Wg"), ("dWu", "Wu"), ("dWd", "Wd"))}
    for e in range(E):
        toks, slots = np.nonzero((r["topk"] == e) & (keep == 1))
        g = r["gates"][toks, slots][:, None]
        X = p["x"][toks]
        aw1, awd = am(p["Wg"][e], p["Wu"][e]), am(p["Wd"][e])
        Wg_f, Wu_f, Wd_f = _nv(p["Wg"][e], 0, aw1), _nv(p["Wu"][e], 0, aw1), _nv(p["Wd"][e], 0, awd)
        Wg_b, Wu_b, Wd_b = _nv(p["Wg"][e], 1, aw1), _nv(p["Wu"][e], 1, aw1), _nv(p["Wd"][e], 1, awd)
        xq = _nv(X, 1, am(X))
        a32, u32 = xq @ Wg_f, xq @ Wu_f
        h32 = a32 / (1 + np.exp(-a32)) * u32
        h = _bf(g * h32) if fold else _bf(h32)
        a, u = _bf(a32), _bf(u32)
        Yp = _bf(_nv(h, 1, am(h)) @ Wd_f)
        y[toks] += Yp if fold else g * Yp
        dYp = _bf(p["dY"][toks]) if fold else _bf(g * p["dY"][toks])
        dh = _nv(dYp, 1, am(dYp)) @ Wd_b.T
        sg = 1 / (1 + np.exp(-a))
        if fold:
            dh = g * dh
            h = _bf(g * (a * sg * u))
        dA = _bf(dh * u * sg * (1 + a * (1 - sg)))
        dU = _bf(dh * a * sg)
        adu = am(dA, dU)
        ref["dWd"][e] = _nv(h, 0, am(h)).T @ _nv(dYp, 0, am(dYp))
        ref["dWg"][e] = _nv(X, 0, am(X)).T @ _nv(dA, 0, adu)
        ref["dWu"][e] = _nv(X, 0, am(X)).T @ _nv(dU, 0, adu)
    ref["y"] = y
    for n in ("y", "dWg", "dWu", "dWd"):
        v = ref[n]
        close = np.isclose(q[n], v, rtol=1e-9, atol=1e-9 * np.abs(v).max())
        assert close.mean() > 0.999, (n, close.mean())
        assert np.linalg.norm(q[n] - v) / np.linalg.norm(v) < 1e-3, n


@pytest.mark.parametrize("fold", [False, True])
def test_nv_layer_tracks_the_exact_layer(fold):
    """An E2M1 rounding perturbs a value by up to a sixth of its block's
    largest magnitude (half the grid step 2 at the top of the range, relative
    to 6), and the E4M3 block scale adds up to 2^-4 relative; for Gaussian
    blocks of 16 the rms perturbation is about 12-15% of a value, a GEMM of
    two quantised operands ~0.2, and an output passes through up to three
    such GEMMs: 0.2-0.3 rms from the exact layer on these inputs (within
    0.4), well apart from it, and about 3.5x the MXFP8 layer's distance."""
    p = _layer(T=150, H=256, E=4, k=2, F=256, seed=5)
    r = oracle.route(p["x"], p["Wr"], None, 2, oracle.SOFTMAX)
    q = oracle.layer_fp8(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                         r["scores"], oracle.SOFTMAX, p["dY"], fold=fold, recipe=oracle.RECIPE_NV)
    y = oracle.forward(p["x"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"])
    g = oracle.backward(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"], r["scores"],
                        p["dY"], oracle.SOFTMAX)
    g["y"] = y
    qm = oracle.layer_fp8(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                          r["scores"], oracle.SOFTMAX, p["dY"], fold=fold, recipe=oracle.RECIPE_MX)
    for n in q:
        if n == "dg":
            continue
        rel = np.linalg.norm(q[n] - g[n]) / np.linalg.norm(g[n])
        rel_mx = np.linalg.norm(qm[n] - g[n]) / np.linalg.norm(g[n])
        assert 0.03 < rel < 0.4, (n, rel)
        assert rel > 2 * rel_mx, (n, rel, rel_mx)       # coarser than MXFP8


def test_nv_tensor_scale_is_per_expert_and_scale_free():
    """Scaling one expert's Wd by 4 leaves its E4M3 block scales and E2M1 codes
    unchanged (its tensor scale absorbs the power of two: every step of the
    recipe commutes with it), so that expert's rows of y are exactly 4x, and
    -- each expert being its own tensor -- every other row is unchanged bit
    for bit. A tensor scale shared across experts would move the other
    experts' codes once expert 0 holds the largest weight."""
    T, H, E, k, F = 96, 128, 3, 1, 128
    p = _layer(T, H, E, k, F, seed=31)
    for n in ("x", "Wg", "Wu", "Wd"):
        p[n] = _bf(p[n])
    r = oracle.route(p["x"], p["Wr"], None, k, oracle.SOFTMAX)
    run = lambda Wd: oracle.layer_fp8(p["x"], p["Wr"], p["Wg"], p["Wu"], Wd, r["topk"], r["gates"],
                                      r["scores"], oracle.SOFTMAX, recipe=oracle.RECIPE_NV)["y"]
    y0 = run(p["Wd"])
    Wd = p["Wd"].copy()
    Wd[0] *= 4.0
    assert np.abs(Wd[0]).max() > np.abs(p["Wd"][1:]).max()     # expert 0 now holds the largest weight
    y1 = run(Wd)
    mine = r["topk"][:, 0] == 0
    assert mine.any() and (~mine).any()
    assert np.array_equal(y1[mine], 4.0 * y0[mine])
    assert np.array_equal(y1[~mine], y0[~mine])
