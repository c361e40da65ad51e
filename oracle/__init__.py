"""fp64 CPU oracle of one Mixture-of-Experts layer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The product path never does: it shares no code
with the oracle.

The arithmetic lives in ``oracle.c`` (plain C loops in fp64, OpenMP over
independent rows); this module compiles it with gcc on first use and wraps
it with numpy arrays. What each function computes, with citations to
"Scalable Training of Mixture-of-Experts Models with Megatron Core", is
stated in ``oracle.c``.

Parity status: every function is pinned by tests/test_oracle.py (brute
force, closed forms, invariants and finite differences); none is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

SOFTMAX, SIGMOID = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = ctypes.CDLL(_LIB)
    return _lib


_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def _d(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _i(a):
    return None if a is None else a.ctypes.data_as(_ip)


def _u8(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte))


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def route(x, Wr, b, k, score, replay_topk=None, replay_mask=None):
    """Route: logits, scores, top-k, gates and the near-tie gaps.

    Returns dict(logits T×E, scores T×E, topk T×k int32, gates T×k,
    gap_set T, gap_order T)."""
    lib = _load()
    x, Wr, b = _f64(x), _f64(Wr), _f64(b)
    T, H = x.shape
    E = Wr.shape[1]
    out = dict(logits=np.empty((T, E)), scores=np.empty((T, E)),
               topk=np.empty((T, k), np.int32), gates=np.empty((T, k)),
               gap_set=np.empty(T), gap_order=np.empty(T))
    rt = _i32(replay_topk)
    rm = None if replay_mask is None else np.ascontiguousarray(replay_mask, dtype=np.uint8)
    rc = lib.oracle_route(T, H, E, k, score, _d(x), _d(Wr), _d(b), _i(rt),
                          None if rm is None else rm.ctypes.data_as(ctypes.c_void_p),
                          _d(out["logits"]), _d(out["scores"]), _i(out["topk"]),
                          _d(out["gates"]), _d(out["gap_set"]), _d(out["gap_order"]))
    if rc:
        raise ValueError("oracle_route: bad arguments")
    return out


def capacity_keep(topk, E, C):
    """Capacity-limited dropping ("Scalable Training of Mixture-of-Experts
    Models with Megatron Core", §7 Load Balancing; the pages give no rule for
    which assignments an expert drops): expert e keeps the first C of its
    assignments in token order and drops the rest. Returns the T×k mask of
    kept slots (uint8)."""
    topk = np.asarray(topk)
    T, k = topk.shape
    keep = np.zeros((T, k), np.uint8)
    seen = np.zeros(E, np.int64)
    for t in range(T):
        for j in range(k):
            e = int(topk[t, j])
            if seen[e] < C:
                keep[t, j] = 1
            seen[e] += 1
    return keep


def update_bias(b, counts, rate):
    """Auxiliary-loss-free load balancing ("Scalable Training of
    Mixture-of-Experts Models with Megatron Core", §7 Load Balancing, no rule
    printed): b_e + rate * sign(mean(counts) - counts_e), sign(0) = 0, in
    fp32 as the bias is stored."""
    counts = np.asarray(counts, np.int64)
    d = counts.sum() - len(counts) * counts          # E * (mean - c_e), exact
    return (np.asarray(b, np.float32) + np.float32(rate) * np.sign(d).astype(np.float32)).astype(np.float32)


def capacity(T, k, E, factor):
    """Rows an expert computes: ceil(factor * T * k / E)."""
    return int(np.ceil(np.float64(np.float32(factor)) * T * k / E))


def dispatch(topk, E):
    """Dispatch: counts E, offsets E+1, row_of T×k, slot_of R (int32)."""
    lib = _load()
    topk = _i32(topk)
    T, k = topk.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    row_of = np.empty((T, k), np.int32)
    slot_of = np.empty(T * k, np.int32)
    if lib.oracle_dispatch(T, E, k, _i(topk), _i(counts), _i(offsets), _i(row_of), _i(slot_of)):
        raise ValueError("oracle_dispatch: bad arguments")
    return dict(counts=counts, offsets=offsets, row_of=row_of, slot_of=slot_of)


def forward(x, Wg, Wu, Wd, topk, gates, Wsg=None, Wsu=None, Wsd=None, want_Yp=False, keep=None):
    """Layer output y (T×H) for a given routing; optionally Yp (R×H). keep:
    optional T×k mask of the slots not dropped (capacity_keep)."""
    lib = _load()
    x, Wg, Wu, Wd = _f64(x), _f64(Wg), _f64(Wu), _f64(Wd)
    Wsg, Wsu, Wsd = _f64(Wsg), _f64(Wsu), _f64(Wsd)
    topk, gates = _i32(topk), _f64(gates)
    keep = None if keep is None else np.ascontiguousarray(keep, np.uint8)
    T, H = x.shape
    E, _, F = Wg.shape
    k = topk.shape[1]
    Fs = 0 if Wsg is None else Wsg.shape[1]
    y = np.empty((T, H))
    Yp = np.empty((T * k, H)) if want_Yp else None
    if lib.oracle_forward(T, H, E, k, F, Fs, _d(x), _d(Wg), _d(Wu), _d(Wd),
                          _d(Wsg), _d(Wsu), _d(Wsd), _i(topk), _d(gates), _d(y), _d(Yp),
                          _u8(keep)):
        raise ValueError("oracle_forward: bad arguments")
    return (y, Yp) if want_Yp else y


def backward(x, Wr, Wg, Wu, Wd, topk, gates, scores, dY, score,
             Wsg=None, Wsu=None, Wsd=None, keep=None):
    """All gradients of L = sum(dY * y) with the routing (and, with keep, the
    dropped slots) held fixed."""
    lib = _load()
    x, Wr, Wg, Wu, Wd = _f64(x), _f64(Wr), _f64(Wg), _f64(Wu), _f64(Wd)
    Wsg, Wsu, Wsd = _f64(Wsg), _f64(Wsu), _f64(Wsd)
    topk, gates, scores, dY = _i32(topk), _f64(gates), _f64(scores), _f64(dY)
    keep = None if keep is None else np.ascontiguousarray(keep, np.uint8)
    T, H = x.shape
    E, _, F = Wg.shape
    k = topk.shape[1]
    Fs = 0 if Wsg is None else Wsg.shape[1]
    g = dict(dX=np.empty((T, H)), dWr=np.empty((H, E)), dWg=np.empty((E, H, F)),
             dWu=np.empty((E, H, F)), dWd=np.empty((E, F, H)), dg=np.empty((T, k)))
    if Fs:
        g.update(dWsg=np.empty((H, Fs)), dWsu=np.empty((H, Fs)), dWsd=np.empty((Fs, H)))
    rc = lib.oracle_backward(T, H, E, k, F, Fs, score, _d(x), _d(Wr), _d(Wg), _d(Wu), _d(Wd),
                             _d(Wsg), _d(Wsu), _d(Wsd), _i(topk), _d(gates), _d(scores), _d(dY),
                             _d(g["dX"]), _d(g["dWr"]), _d(g["dWg"]), _d(g["dWu"]), _d(g["dWd"]),
                             _d(g.get("dWsg")), _d(g.get("dWsu")), _d(g.get("dWsd")), _d(g["dg"]),
                             _u8(keep))
    if rc:
        raise ValueError("oracle_backward: bad arguments")
    return g


# ------------------------------------------------------------ large layers
def _storage(a):
    """(contiguous array, wtype) for float32 or bfloat16-bits weights."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, 0
    if a.dtype == np.uint16:
        return a, 1
    raise TypeError("weights must be float32 or bfloat16 bits (uint16)")


class ExpertWeights:
    """Per-expert weight blocks in storage format (float32 or bf16 bits).

    ``Wg``, ``Wu``, ``Wd`` map expert index -> array (H×F, H×F, F×H); experts
    not present are not touched by the computation that uses this object."""

    def __init__(self, E, Wg, Wu, Wd, Wsg=None, Wsu=None, Wsd=None):
        self.E = E
        self._keep = []
        self.wtype = None
        self.pg = (ctypes.c_void_p * E)()
        self.pu = (ctypes.c_void_p * E)()
        self.pd = (ctypes.c_void_p * E)()
        for e in Wg:
            for arr, tab in ((Wg[e], self.pg), (Wu[e], self.pu), (Wd[e], self.pd)):
                a, wt = _storage(arr)
                self.wtype = wt if self.wtype is None else self.wtype
                if wt != self.wtype:
                    raise TypeError("mixed weight storage types")
                self._keep.append(a)
                tab[e] = a.ctypes.data
        self.shared = []
        for arr in (Wsg, Wsu, Wsd):
            if arr is None:
                self.shared.append(None)
                continue
            a, wt = _storage(arr)
            self._keep.append(a)
            self.shared.append(a.ctypes.data)
        self.F = next(iter(Wg.values())).shape[1] if Wg else 0
        self.Fs = 0 if Wsg is None else Wsg.shape[1]
        if self.wtype is None:
            self.wtype = 0


def token_rows(xs, dYs, Wr, W: ExpertWeights, topk, gates, scores, score):
    """y, dX and dg rows of selected tokens (same definitions, per token)."""
    lib = _load()
    xs, dYs, Wr = _f64(xs), _f64(dYs), _f64(Wr)
    topk, gates, scores = _i32(topk), _f64(gates), _f64(scores)
    n, H = xs.shape
    k = topk.shape[1]
    y, dX, dg = np.empty((n, H)), np.empty((n, H)), np.empty((n, k))
    sg, su, sd = W.shared
    rc = lib.oracle_token_rows(n, H, W.E, k, W.F, W.Fs, score, W.wtype, _d(xs), _d(dYs), _d(Wr),
                               W.pg, W.pu, W.pd, ctypes.c_void_p(sg), ctypes.c_void_p(su),
                               ctypes.c_void_p(sd), _i(topk), _d(gates), _d(scores),
                               _d(y), _d(dX), _d(dg))
    if rc:
        raise ValueError("oracle_token_rows: bad arguments or missing expert weights")
    return dict(y=y, dX=dX, dg=dg)


DW_KIND = dict(dWg=0, dWu=1, dWd=2, dWsg=3, dWsu=4, dWsd=5)


def dw_entries(x, dY, W: ExpertWeights, topk, gates, entries):
    """Weight-gradient entries; ``entries`` = list of (name, e, i, j)."""
    lib = _load()
    x, dY = _f64(x), _f64(dY)
    topk, gates = _i32(topk), _f64(gates)
    T, H = x.shape
    k = topk.shape[1]
    n = len(entries)
    which = np.array([DW_KIND[q[0]] for q in entries], np.int32)
    ee = np.array([q[1] for q in entries], np.int32)
    ii = np.array([q[2] for q in entries], np.int32)
    jj = np.array([q[3] for q in entries], np.int32)
    out = np.empty(n)
    sg, su, sd = W.shared
    rc = lib.oracle_dw_entries(T, H, W.E, k, max(W.F, 1), W.Fs, W.wtype, _d(x), _d(dY),
                               W.pg, W.pu, W.pd, ctypes.c_void_p(sg), ctypes.c_void_p(su),
                               ctypes.c_void_p(sd), _i(topk), _d(gates), n, _i(which), _i(ee),
                               _i(ii), _i(jj), _d(out))
    if rc:
        raise ValueError("oracle_dw_entries: bad arguments or missing expert weights")
    return out


# ------------------------------------------------------------ blockwise FP8
def e4m3_decode(codes):
    """fp64 values of E4M3 codes (OCP format definition)."""
    lib = _load()
    lib.oracle_e4m3_decode.restype = ctypes.c_double
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_ubyte]
    return np.array([lib.oracle_e4m3_decode(int(c)) for c in np.asarray(codes).ravel()]).reshape(np.shape(codes))


def e4m3_encode(values):
    """E4M3 codes of fp32 values (round to nearest even, saturating)."""
    lib = _load()
    lib.oracle_e4m3_encode.restype = ctypes.c_ubyte
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    v = np.asarray(values, np.float32)
    return np.array([lib.oracle_e4m3_encode(float(f)) for f in v.ravel()], np.uint8).reshape(v.shape)


FP8_ROWS, FP8_TILES, FP8_COLS = 0, 1, 2


def fp8_quantize(X, mode):
    """(codes, scales) of an fp32 matrix: mode FP8_ROWS (1x128 along rows),
    FP8_TILES (128x128), FP8_COLS (per column over 128-row blocks)."""
    lib = _load()
    X = np.ascontiguousarray(X, np.float32)
    M, K = X.shape
    codes = np.empty((M, K), np.uint8)
    if mode == FP8_ROWS:
        scales = np.empty((M, K // 128), np.float32)
    elif mode == FP8_TILES:
        scales = np.empty(((M + 127) // 128, (K + 127) // 128), np.float32)
    else:
        scales = np.empty(((M + 127) // 128, K), np.float32)
    rc = lib.oracle_fp8_quantize(M, K, mode, X.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                 codes.ctypes.data_as(ctypes.c_void_p),
                                 scales.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    if rc:
        raise ValueError("oracle_fp8_quantize: bad arguments")
    return codes, scales


MX_ROWS, MX_COLS = 0, 1


def mx_exponent(amax):
    """MXFP8 block exponent e (scale 2^e, UE8M0 byte e + 127) of a block
    maximum: the smallest e with amax <= 448 2^e, in [-127, 127]."""
    lib = _load()
    lib.oracle_mx_exponent.restype = ctypes.c_int
    lib.oracle_mx_exponent.argtypes = [ctypes.c_float]
    return int(lib.oracle_mx_exponent(float(amax)))


def mx_quantize(X, mode):
    """(codes, UE8M0 scale bytes) of an fp32 matrix in MXFP8: mode MX_ROWS
    (1x32 along rows, scales M x K/32) or MX_COLS (per column over 32-row
    blocks, scales ceil(M/32) x K)."""
    lib = _load()
    X = np.ascontiguousarray(X, np.float32)
    M, K = X.shape
    codes = np.empty((M, K), np.uint8)
    scales = np.empty((M, K // 32) if mode == MX_ROWS else ((M + 31) // 32, K), np.uint8)
    rc = lib.oracle_mx_quantize(M, K, mode, X.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                codes.ctypes.data_as(ctypes.c_void_p), scales.ctypes.data_as(ctypes.c_void_p))
    if rc:
        raise ValueError("oracle_mx_quantize: bad arguments")
    return codes, scales


NV_ROWS, NV_COLS = 0, 1


def e2m1_decode(codes):
    """fp64 values of 4-bit E2M1 codes (format definition)."""
    lib = _load()
    lib.oracle_e2m1_decode.restype = ctypes.c_double
    lib.oracle_e2m1_decode.argtypes = [ctypes.c_ubyte]
    return np.array([lib.oracle_e2m1_decode(int(c)) for c in np.asarray(codes).ravel()]).reshape(np.shape(codes))


def e2m1_encode(values):
    """E2M1 codes of fp32 values (nearest, ties to the even code, saturating)."""
    lib = _load()
    lib.oracle_e2m1_encode.restype = ctypes.c_ubyte
    lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
    v = np.asarray(values, np.float32)
    return np.array([lib.oracle_e2m1_encode(float(f)) for f in v.ravel()], np.uint8).reshape(v.shape)


def nv_tensor_scale(amax):
    """NVFP4 per-tensor fp32 scale S = 2688 / amax (1 for an all-zero tensor)."""
    lib = _load()
    lib.oracle_nv_tensor_scale.restype = ctypes.c_float
    lib.oracle_nv_tensor_scale.argtypes = [ctypes.c_float]
    return np.float32(lib.oracle_nv_tensor_scale(float(amax)))


def nv_quantize(X, mode):
    """(codes, E4M3 scale bytes, tensor scale S) of an fp32 matrix as one
    NVFP4 tensor: mode NV_ROWS (1x16 along rows, scales M x K/16) or NV_COLS
    (per column over 16-row blocks, scales ceil(M/16) x K). Codes are one
    4-bit code per byte."""
    lib = _load()
    X = np.ascontiguousarray(X, np.float32)
    M, K = X.shape
    codes = np.empty((M, K), np.uint8)
    scales = np.empty((M, K // 16) if mode == NV_ROWS else ((M + 15) // 16, K), np.uint8)
    S = ctypes.c_float(0.0)
    rc = lib.oracle_nv_quantize(M, K, mode, X.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                codes.ctypes.data_as(ctypes.c_void_p), scales.ctypes.data_as(ctypes.c_void_p),
                                ctypes.byref(S))
    if rc:
        raise ValueError("oracle_nv_quantize: bad arguments")
    return codes, scales, np.float32(S.value)


RECIPE_BLOCK, RECIPE_MX, RECIPE_NV = 0, 1, 2


def layer_fp8(x, Wr, Wg, Wu, Wd, topk, gates, scores, score, dY=None, Wsg=None, Wsu=None,
              Wsd=None, fold=False, recipe=RECIPE_BLOCK, keep=None):
    """FP8 layer: y, and when dY is given every gradient. recipe: RECIPE_BLOCK
    (blockwise FP8, fp32 block scales), RECIPE_MX (MXFP8, 1x32 blocks with
    power-of-two scales) or RECIPE_NV (NVFP4: E2M1 values, 1x16 blocks with
    E4M3 scales, one fp32 scale per expert operand). fold: the memory-efficient permutation's order
    (routing weight folded into h before fc2), with its rounding points.
    keep: optional T x k mask of the slots that are not dropped
    (capacity_keep); a dropped assignment never reaches its expert, so the
    expert's segment, and every quantisation block counted along it, holds
    its kept rows alone; its dg is 0."""
    lib = _load()
    x, Wr, Wg, Wu, Wd = _f64(x), _f64(Wr), _f64(Wg), _f64(Wu), _f64(Wd)
    Wsg, Wsu, Wsd = _f64(Wsg), _f64(Wsu), _f64(Wsd)
    topk, gates, scores, dY = _i32(topk), _f64(gates), _f64(scores), _f64(dY)
    T, H = x.shape
    E, _, F = Wg.shape
    k = topk.shape[1]
    Fs = 0 if Wsg is None else Wsg.shape[1]
    out = dict(y=np.empty((T, H)))
    if dY is not None:
        out.update(dX=np.empty((T, H)), dWr=np.empty((H, E)), dWg=np.empty((E, H, F)),
                   dWu=np.empty((E, H, F)), dWd=np.empty((E, F, H)), dg=np.empty((T, k)))
        if Fs:
            out.update(dWsg=np.empty((H, Fs)), dWsu=np.empty((H, Fs)), dWsd=np.empty((Fs, H)))
    rc = lib.oracle_layer_fp8(T, H, E, k, F, Fs, score, _d(x), _d(Wr), _d(Wg), _d(Wu), _d(Wd),
                              _d(Wsg), _d(Wsu), _d(Wsd), _i(topk), _d(gates), _d(scores), _d(dY),
                              _d(out["y"]), _d(out.get("dX")), _d(out.get("dWr")),
                              _d(out.get("dWg")), _d(out.get("dWu")), _d(out.get("dWd")),
                              _d(out.get("dWsg")), _d(out.get("dWsu")), _d(out.get("dWsd")),
                              _d(out.get("dg")), 1 if fold else 0, int(recipe),
                              _u8(None if keep is None else np.ascontiguousarray(keep, np.uint8)))
    if rc:
        raise ValueError("oracle_layer_fp8: bad arguments")
    return out
