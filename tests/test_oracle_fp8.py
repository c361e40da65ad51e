"""Pins of the oracle's blockwise-FP8 (E4M3) pieces (CPU only).

E4M3 is pinned to PyTorch's float8_e4m3fn conversion (an independent
implementation of the same OCP format) on every code and on random, tie and
out-of-range values; the block quantiser to its exactness and locality
properties; the FP8 layer to the exact layer within the E4M3 error scale
("Scalable Training of Mixture-of-Experts Models with Megatron Core", §5,
blockwise FP8: 1x128 activation/gradient tiles, 128x128 weight blocks).
"""
import numpy as np
import pytest
import torch

import oracle


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2        # 0x7F, 0xFF
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_torch_and_saturates():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(20000) * 10 ** rng.uniform(-4, 2.5, 20000),
                           rng.uniform(-448, 448, 5000)]).astype(np.float32)
    grid = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))           # 0 .. 448
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)               # exact ties
    vals = np.concatenate([vals, mids, -mids, grid.astype(np.float32)])
    vals = vals[np.abs(vals) <= 448.0]          # torch's cast gives NaN beyond the range
    ours = oracle.e4m3_encode(vals)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    big = np.array([448.0, 449.0, 480.0, 1e4, 1e30, -500.0], np.float32)
    assert list(oracle.e4m3_encode(big)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def test_e4m3_encode_every_bf16_value_matches_torch():
    """Every finite bf16 value within the E4M3 range, both signs."""
    bits = np.arange(0x0000, 0x7F80, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    vals = vals[vals <= 448.0]
    vals = np.concatenate([vals, -vals])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(vals), ref)


@pytest.mark.parametrize("mode", [oracle.FP8_ROWS, oracle.FP8_TILES, oracle.FP8_COLS])
def test_block_quantiser_exactness_and_locality(mode):
    rng = np.random.default_rng(1)
    X = (rng.standard_normal((300, 256)) * 3).astype(np.float32)
    codes, scales = oracle.fp8_quantize(X, mode)
    dq = oracle.e4m3_decode(codes)
    if mode == oracle.FP8_ROWS:
        s = np.repeat(scales, 128, axis=1)
        amax = np.abs(X).reshape(300, 2, 128).max(2)
    elif mode == oracle.FP8_TILES:
        s = np.repeat(np.repeat(scales, 128, 0), 128, 1)[:300, :256]
        amax = np.array([[np.abs(X[r:r + 128, c:c + 128]).max() for c in range(0, 256, 128)]
                         for r in range(0, 300, 128)])
    else:
        s = np.repeat(scales, 128, 0)[:300]
        amax = np.array([np.abs(X[r:r + 128]).max(0) for r in range(0, 300, 128)])
    np.testing.assert_array_equal(scales, (amax / np.float32(448)).astype(np.float32))
    deq = dq * s
    # every value within half an E4M3 step of itself (relative 2^-4, or 2^-10 * s near 0)
    err = np.abs(deq - X)
    assert np.all(err <= np.maximum(np.abs(X) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 1e-6))
    assert np.sum(np.abs(dq) == 448.0) >= scales.size        # each block's amax maps to 448
    # locality: changing one element moves only its own block
    X2 = X.copy()
    X2[5, 7] *= 50
    c2, s2 = oracle.fp8_quantize(X2, mode)
    changed = np.argwhere(c2 != codes)
    if mode == oracle.FP8_ROWS:
        assert np.all(changed[:, 0] == 5) and np.all(changed[:, 1] < 128)
    elif mode == oracle.FP8_TILES:
        assert np.all(changed[:, 0] < 128) and np.all(changed[:, 1] < 128)
    else:
        assert np.all(changed[:, 1] == 7) and np.all(changed[:, 0] < 128)
    # exactness: representable values with a power-of-two block maximum round-trip
    Y = (oracle.e4m3_decode(rng.integers(0, 0x7E, (128, 128)).astype(np.uint8)) * 2.0 ** -3)
    Y[0, 0] = 448.0 * 2.0 ** -3
    cy, sy = oracle.fp8_quantize(Y.astype(np.float32), oracle.FP8_TILES)
    assert sy[0, 0] == 2.0 ** -3
    assert np.array_equal(oracle.e4m3_decode(cy) * 2.0 ** -3, Y)


def _layer(T, H, E, k, F, Fs, score, seed):
    rng = np.random.default_rng(seed)
    p = dict(x=rng.standard_normal((T, H)), Wr=rng.standard_normal((H, E)) * 0.1,
             Wg=rng.standard_normal((E, H, F)) * H ** -0.5, Wu=rng.standard_normal((E, H, F)) * H ** -0.5,
             Wd=rng.standard_normal((E, F, H)) * F ** -0.5, dY=rng.standard_normal((T, H)))
    if Fs:
        p.update(Wsg=rng.standard_normal((H, Fs)) * H ** -0.5, Wsu=rng.standard_normal((H, Fs)) * H ** -0.5,
                 Wsd=rng.standard_normal((Fs, H)) * Fs ** -0.5)
    else:
        p.update(Wsg=None, Wsu=None, Wsd=None)
    return p


@pytest.mark.parametrize("score,Fs,fold", [(oracle.SOFTMAX, 0, False), (oracle.SIGMOID, 128, False),
                                           (oracle.SOFTMAX, 0, True), (oracle.SIGMOID, 128, True)])
def test_fp8_layer_tracks_the_exact_layer(score, Fs, fold):
    """Both rounding orders (routing weight applied after fc2, or folded into
    h before it) stay within the E4M3 deviation scale of the exact layer."""
    p = _layer(T=150, H=256, E=4, k=2, F=256, Fs=Fs, score=score, seed=3)
    r = oracle.route(p["x"], p["Wr"], None, 2, score)
    q = oracle.layer_fp8(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                         r["scores"], score, p["dY"], p["Wsg"], p["Wsu"], p["Wsd"], fold=fold)
    y = oracle.forward(p["x"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"], p["Wsg"], p["Wsu"], p["Wsd"])
    g = oracle.backward(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"], r["scores"],
                        p["dY"], score, p["Wsg"], p["Wsu"], p["Wsd"])
    g["y"] = y
    # each E4M3 rounding perturbs a value by at most 2^-4 relative (2^-4/sqrt(3)
    # = 3.6% rms); an output depends on up to ~6 successive roundings, so its
    # deviation from the exact layer is sqrt(6) x 3.6% = 9% rms at most
    for n in q:
        if n == "dg":
            continue
        rel = np.linalg.norm(q[n] - g[n]) / np.linalg.norm(g[n])
        assert 0.005 < rel < 0.09, (n, rel)


# ---- an independent FP8 SwiGLU for one expert, codec = torch's float8_e4m3fn
def _cast(v, s):
    f = np.clip((v.astype(np.float32) / np.float32(s)).astype(np.float32), -448, 448)
    return torch.from_numpy(np.ascontiguousarray(f)).to(torch.float8_e4m3fn).double().numpy() * float(s)


def _q_rows(X):
    out = np.empty_like(X)
    for r in range(X.shape[0]):
        for c in range(0, X.shape[1], 128):
            v = X[r, c:c + 128]
            a = np.float32(np.abs(v.astype(np.float32)).max())
            out[r, c:c + 128] = _cast(v, np.float32(a / np.float32(448)) if a else np.float32(1))
    return out


def _q_cols(X):
    return _q_rows(X.T).T if X.shape[0] % 128 == 0 else None


def _q_tiles(X):
    out = np.empty_like(X)
    for r in range(0, X.shape[0], 128):
        for c in range(0, X.shape[1], 128):
            v = X[r:r + 128, c:c + 128]
            a = np.float32(np.abs(v.astype(np.float32)).max())
            out[r:r + 128, c:c + 128] = _cast(v, np.float32(a / np.float32(448)) if a else np.float32(1))
    return out


def test_fp8_single_expert_matches_independent_fp8_swiglu():
    T, H, F = 256, 256, 384
    p = _layer(T=T, H=H, E=1, k=1, F=F, Fs=0, score=oracle.SOFTMAX, seed=7)
    r = oracle.route(p["x"], p["Wr"], None, 1, oracle.SOFTMAX)
    q = oracle.layer_fp8(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                         r["scores"], oracle.SOFTMAX, p["dY"])
    x, dY = p["x"], p["dY"]
    bf = lambda v: torch.from_numpy(np.ascontiguousarray(v)).to(torch.bfloat16).double().numpy()
    Wg, Wu, Wd = _q_tiles(p["Wg"][0]), _q_tiles(p["Wu"][0]), _q_tiles(p["Wd"][0])
    xq = _q_rows(x)
    a32, u32 = xq @ Wg, xq @ Wu
    h = bf(a32 / (1 + np.exp(-a32)) * u32)
    a, u = bf(a32), bf(u32)
    sg = 1 / (1 + np.exp(-a))
    y = bf(_q_rows(h) @ Wd)
    dY = bf(dY)                                 # gate 1: the stored output gradient is bf16
    dh = _q_rows(dY) @ Wd.T
    dA = bf(dh * u * sg * (1 + a * (1 - sg)))
    dU = bf(dh * a * sg)
    ref = dict(y=y, dWd=(_q_cols(h).T @ _q_tiles(dY))[None],
               dX=_q_rows(dA) @ Wg.T + _q_rows(dU) @ Wu.T,
               dWg=(_q_cols(x).T @ _q_tiles(dA))[None], dWu=(_q_cols(x).T @ _q_tiles(dU))[None])
    for n, v in ref.items():
        # both sides round the same fp64 values to bf16; an fp64 summation-order
        # difference can move a value across a bf16 (or E4M3) rounding boundary,
        # so compare in aggregate and require exact agreement almost everywhere
        close = np.isclose(q[n], v, rtol=1e-9, atol=1e-9 * np.abs(v).max())
        assert close.mean() > 0.999, (n, close.mean())
        assert np.linalg.norm(q[n] - v) / np.linalg.norm(v) < 1e-3, n


def _q_cols_segment(X):
    """Per column over 128-row blocks counted from the segment's first row
    (the last block may be shorter)."""
    out = np.empty_like(X)
    for r in range(0, X.shape[0], 128):
        for c in range(X.shape[1]):
            v = X[r:r + 128, c]
            a = np.float32(np.abs(v.astype(np.float32)).max())
            out[r:r + 128, c] = _cast(v, np.float32(a / np.float32(448)) if a else np.float32(1))
    return out


@pytest.mark.parametrize("fold,drop", [(False, False), (True, False), (False, True), (True, True)])
def test_fp8_multi_expert_matches_independent_fp8_swiglu(fold, drop):
    """Several experts with ragged segments (more than one 128-token block,
    the last one partial): the weight-gradient operands are quantised per
    expert segment, in 128-token blocks counted from the segment's first row.
    An independent FP8 layer (torch's E4M3 codec, rows gathered per expert
    with numpy) must give the oracle's y and weight gradients. drop: capacity
    130 per expert, so each expert's segment is its first 130 assignments
    (a dropped assignment never reaches the expert) and the dropped slots get
    dg = 0."""
    T, H, E, k, F = 333, 256, 3, 2, 256
    p = _layer(T=T, H=H, E=E, k=k, F=F, Fs=0, score=oracle.SOFTMAX, seed=21)
    b = np.array([0.8, 0.0, -0.9])                    # uneven loads: all segments ragged
    r = oracle.route(p["x"], p["Wr"], b, k, oracle.SOFTMAX)
    counts = np.bincount(r["topk"].ravel(), minlength=E)
    assert np.all(counts > 128) and np.all(counts % 128 != 0) and len(set(counts)) == E
    keep = oracle.capacity_keep(r["topk"], E, 130) if drop else np.ones_like(r["topk"], np.uint8)
    if drop:
        assert np.all(counts > 130) and (keep == 0).sum() == counts.sum() - 3 * 130
    q = oracle.layer_fp8(p["x"], p["Wr"], p["Wg"], p["Wu"], p["Wd"], r["topk"], r["gates"],
                         r["scores"], oracle.SOFTMAX, p["dY"], fold=fold,
                         keep=keep if drop else None)
    if drop:
        assert np.all(q["dg"][keep == 0] == 0) and np.all(q["dg"][keep == 1] != 0)
    bf = lambda v: torch.from_numpy(np.ascontiguousarray(v)).to(torch.bfloat16).double().numpy()
    y = np.zeros((T, H))
    ref = {n: np.zeros_like(p[w]) for n, w in (("dWg", "Wg"), ("dWu", "Wu"), ("dWd", "Wd"))}
    for e in range(E):
        toks, slots = np.nonzero((r["topk"] == e) & (keep == 1))   # the expert's rows, token order
        g = r["gates"][toks, slots][:, None]
        X = p["x"][toks]
        Wg, Wu, Wd = _q_tiles(p["Wg"][e]), _q_tiles(p["Wu"][e]), _q_tiles(p["Wd"][e])
        xq = _q_rows(X)
        a32, u32 = xq @ Wg, xq @ Wu
        h32 = a32 / (1 + np.exp(-a32)) * u32
        h = bf(g * h32) if fold else bf(h32)
        a, u = bf(a32), bf(u32)
        Yp = bf(_q_rows(h) @ Wd)
        y[toks] += Yp if fold else g * Yp
        dYp = bf(p["dY"][toks]) if fold else bf(g * p["dY"][toks])   # stored bf16
        dh = _q_rows(dYp) @ Wd.T
        sg = 1 / (1 + np.exp(-a))
        if fold:
            hr = a * sg * u
            dh = g * dh
            h = bf(g * hr)
        dA = bf(dh * u * sg * (1 + a * (1 - sg)))
        dU = bf(dh * a * sg)
        ref["dWd"][e] = _q_cols_segment(h).T @ _q_tiles(dYp)
        ref["dWg"][e] = _q_cols_segment(X).T @ _q_tiles(dA)
        ref["dWu"][e] = _q_cols_segment(X).T @ _q_tiles(dU)
    ref["y"] = y
    for n, v in ref.items():
        close = np.isclose(q[n], v, rtol=1e-9, atol=1e-9 * np.abs(v).max())
        assert close.mean() > 0.999, (n, close.mean())
        assert np.linalg.norm(q[n] - v) / np.linalg.norm(v) < 1e-3, n
    if drop:
        return
    # a block origin at a multiple of 128 of the whole permuted buffer, instead
    # of each segment's first row, gives visibly different weight gradients
    e = 1
    toks, slots = np.nonzero(r["topk"] == e)
    off = counts[0]                                   # segment start in an unpadded buffer
    X = p["x"][toks]
    shifted = np.concatenate([np.zeros(((off % 128), H)), X])
    wrong = _q_cols_segment(shifted)[off % 128:]
    assert np.linalg.norm(wrong - _q_cols_segment(X)) > 1e-3 * np.linalg.norm(X)
