"""Single-GPU Mixture-of-Experts layer for GB300 (sm_103a): Python binding.

A thin ctypes binding of the C ABI declared in ``include/moe.h``. Every step
of the layer (router, top-k, dispatch tables, permute, grouped GEMMs with
fused SwiGLU, combine, and the whole backward) runs in the hand-written CUDA
kernels of ``libmoe_gb300.so``. PyTorch is only used here to allocate device
memory and to supply the current CUDA stream; there is no CPU or PyTorch
fallback: if the library is missing, importing the layer raises.

The layer follows "Scalable Training of Mixture-of-Experts Models with
Megatron Core", §2 (Route, Dispatch, Expert Computation, Combine).
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_MISALIGNED = 3
MOE_ERR_WORKSPACE_TOO_SMALL = 4
MOE_ERR_CUDA = 5
MOE_ERR_DEVICE_TIMEOUT = 6
MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1
MOE_FP32, MOE_BF16, MOE_FP8_BLOCK, MOE_MXFP8, MOE_NVFP4 = 0, 1, 2, 3, 4
MOE_FLAG_STAGE_TIMING = 1
MOE_FLAG_FOLD_GATES = 2

# Names the library exports (include/moe.h).
EXPORTS = ("moe_plan_create", "moe_plan_destroy", "moe_workspace_size", "moe_forward",
           "moe_backward", "moe_read_status", "moe_status_string", "moe_stage_times",
           "moe_route_static", "moe_fp8_quantize", "moe_diag_wait_timeout", "moe_update_bias",
           "moe_weight_cache_size", "moe_quantize_weights", "moe_mx_quantize", "moe_nv_quantize",
           "moe_abi_version")
MOE_Q_ROWS, MOE_Q_TILES, MOE_Q_COLS_T, MOE_Q_TILES_T = 0, 1, 2, 3


class moe_config_t(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("E", ctypes.c_int), ("F", ctypes.c_int), ("Fs", ctypes.c_int),
                ("top_k", ctypes.c_int), ("T_max", ctypes.c_int), ("score", ctypes.c_int),
                ("dtype", ctypes.c_int), ("flags", ctypes.c_uint), ("capacity_factor", ctypes.c_float)]


_vp = ctypes.c_void_p


class moe_fwd_args_t(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("x", "Wr", "b", "W_gate", "W_up", "W_down", "Ws_gate", "Ws_up",
                                   "Ws_down", "y", "topk_idx", "gates", "counts", "offsets",
                                   "row_of", "replay_topk", "weight_cache")]


class moe_bwd_args_t(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("dY", "x", "Wr", "W_gate", "W_up", "W_down", "Ws_gate", "Ws_up",
                                   "Ws_down", "dX", "dWr", "dW_gate", "dW_up", "dW_down", "dWs_gate",
                                   "dWs_up", "dWs_down", "weight_cache")]


class moe_stage_time_t(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 24), ("launches", ctypes.c_int), ("total_ms", ctypes.c_float)]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {moe_status_string(status)} (status {status})")


_lib = None


def load_library() -> ctypes.CDLL:
    """Load libmoe_gb300.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(build it with mixture_experts_layer_sigmoid_gb300._build.build())")
        lib = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER
        lib.moe_plan_create.argtypes = [P(moe_config_t), ctypes.c_int, P(_vp)]
        lib.moe_plan_destroy.argtypes = [_vp]
        lib.moe_workspace_size.argtypes = [_vp, ctypes.c_int, P(ctypes.c_size_t), P(ctypes.c_size_t)]
        lib.moe_forward.argtypes = [_vp, ctypes.c_int, P(moe_fwd_args_t), _vp, ctypes.c_size_t, _vp,
                                    ctypes.c_size_t, _vp]
        lib.moe_backward.argtypes = [_vp, ctypes.c_int, P(moe_bwd_args_t), _vp, ctypes.c_size_t, _vp,
                                     ctypes.c_size_t, _vp]
        lib.moe_read_status.argtypes = [_vp, _vp, _vp]
        lib.moe_status_string.argtypes = [ctypes.c_int]
        lib.moe_status_string.restype = ctypes.c_char_p
        lib.moe_stage_times.argtypes = [_vp, P(moe_stage_time_t), ctypes.c_int, P(ctypes.c_int)]
        lib.moe_route_static.argtypes = [_vp, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
        lib.moe_fp8_quantize.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp,
                                         _vp, _vp]
        lib.moe_diag_wait_timeout.argtypes = [_vp, _vp]
        lib.moe_update_bias.argtypes = [ctypes.c_int, _vp, ctypes.c_float, _vp, _vp]
        lib.moe_weight_cache_size.argtypes = [_vp, P(ctypes.c_size_t)]
        lib.moe_quantize_weights.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
        lib.moe_mx_quantize.argtypes = [ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp]
        lib.moe_nv_quantize.argtypes = [ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
        lib.moe_abi_version.argtypes = []
        for n in EXPORTS:
            if n not in ("moe_status_string", "moe_abi_version"):
                getattr(lib, n).restype = ctypes.c_int
        _lib = lib
    return _lib


# ------------------------------------------------------- C ABI, same names
def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(status).decode()


def moe_abi_version() -> int:
    return load_library().moe_abi_version()


def moe_plan_create(cfg: moe_config_t, device: int) -> int:
    plan = _vp()
    st = load_library().moe_plan_create(ctypes.byref(cfg), device, ctypes.byref(plan))
    if st != MOE_OK:
        raise MoEError(st, "moe_plan_create")
    return plan.value


def moe_plan_destroy(plan: int) -> None:
    load_library().moe_plan_destroy(plan)


def moe_workspace_size(plan: int, T: int):
    s, w = ctypes.c_size_t(), ctypes.c_size_t()
    st = load_library().moe_workspace_size(plan, T, ctypes.byref(s), ctypes.byref(w))
    if st != MOE_OK:
        raise MoEError(st, "moe_workspace_size")
    return s.value, w.value


def moe_forward(plan: int, T: int, args: moe_fwd_args_t, saved: int, saved_bytes: int, ws: int,
                ws_bytes: int, stream: int) -> None:
    st = load_library().moe_forward(plan, T, ctypes.byref(args), saved, saved_bytes, ws, ws_bytes,
                                    stream)
    if st != MOE_OK:
        raise MoEError(st, "moe_forward")


def moe_backward(plan: int, T: int, args: moe_bwd_args_t, saved: int, saved_bytes: int, ws: int,
                 ws_bytes: int, stream: int) -> None:
    st = load_library().moe_backward(plan, T, ctypes.byref(args), saved, saved_bytes, ws, ws_bytes,
                                     stream)
    if st != MOE_OK:
        raise MoEError(st, "moe_backward")


def moe_read_status(plan: int, ws: int, stream: int) -> int:
    return load_library().moe_read_status(plan, ws, stream)


def moe_stage_times(plan: int):
    """{stage: (launches, total_ms)} since the previous call (timing plans)."""
    cap = 64
    buf = (moe_stage_time_t * cap)()
    n = ctypes.c_int()
    st = load_library().moe_stage_times(plan, buf, cap, ctypes.byref(n))
    if st != MOE_OK:
        raise MoEError(st, "moe_stage_times")
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(min(n.value, cap))}


def moe_fp8_quantize(rows: int, cols: int, mode: int, x: int, codes: int, scales: int, codes_t: int,
                     scales_t: int, stream: int) -> None:
    st = load_library().moe_fp8_quantize(rows, cols, mode, x, codes, scales, codes_t, scales_t, stream)
    if st != MOE_OK:
        raise MoEError(st, "moe_fp8_quantize")


def moe_weight_cache_size(plan: int) -> int:
    n = ctypes.c_size_t()
    st = load_library().moe_weight_cache_size(plan, ctypes.byref(n))
    if st != MOE_OK:
        raise MoEError(st, "moe_weight_cache_size")
    return n.value


def moe_quantize_weights(plan: int, W_gate: int, W_up: int, W_down: int, cache: int, cache_bytes: int,
                         stream: int) -> None:
    st = load_library().moe_quantize_weights(plan, W_gate, W_up, W_down, cache, cache_bytes, stream)
    if st != MOE_OK:
        raise MoEError(st, "moe_quantize_weights")


def moe_mx_quantize(rows: int, cols: int, x: int, codes: int, scales: int, codes_c: int, scales_c: int,
                    col_transposed: int, stream: int) -> None:
    st = load_library().moe_mx_quantize(rows, cols, x, codes, scales, codes_c, scales_c, col_transposed, stream)
    if st != MOE_OK:
        raise MoEError(st, "moe_mx_quantize")


def moe_nv_quantize(rows: int, cols: int, x: int, amax: int, codes: int, scales: int, codes_t: int,
                    scales_t: int, stream: int) -> None:
    st = load_library().moe_nv_quantize(rows, cols, x, amax, codes, scales, codes_t, scales_t, stream)
    if st != MOE_OK:
        raise MoEError(st, "moe_nv_quantize")


def moe_update_bias(E: int, counts: int, rate: float, b: int, stream: int) -> None:
    """Auxiliary-loss-free bias update: b_e += rate * sign(mean count - count_e)."""
    st = load_library().moe_update_bias(E, counts, rate, b, stream)
    if st != MOE_OK:
        raise MoEError(st, "moe_update_bias")


# ------------------------------------------------- torch-allocated wrapper
def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


class MoELayer:
    """One MoE layer on one GPU; torch allocates ``saved`` and the workspace.

    Weights are passed per call (they are inputs of the C ABI). Layouts are
    those of include/moe.h: x T×H, Wr H×E fp32, b E fp32, W_gate/W_up E×H×F,
    W_down E×F×H, shared expert H×Fs, H×Fs, Fs×H.

    ``fold_gates`` selects the memory-efficient permutation (MOE_FLAG_FOLD_GATES):
    the routing weights are folded into the expert activations, and the saved
    buffer keeps neither h nor the permuted expert outputs. ``capacity_factor``
    > 0 enables capacity-limited dropping (earliest tokens kept per expert)."""

    def __init__(self, H, E, F, top_k, T_max, score=MOE_SCORE_SOFTMAX, dtype=MOE_BF16, Fs=0,
                 device=0, stage_timing=False, fold_gates=False, capacity_factor=0.0):
        import torch
        self.torch = torch
        flags = (MOE_FLAG_STAGE_TIMING if stage_timing else 0) | (MOE_FLAG_FOLD_GATES if fold_gates else 0)
        self.cfg = moe_config_t(H=H, E=E, F=F, Fs=Fs, top_k=top_k, T_max=T_max, score=score,
                                dtype=dtype, flags=flags, capacity_factor=capacity_factor)
        self.device = torch.device("cuda", device)
        self.plan = moe_plan_create(self.cfg, device)
        self._bufs: Dict[int, tuple] = {}
        self.act_dtype = torch.float32 if dtype == MOE_FP32 else torch.bfloat16

    def __del__(self):
        try:
            moe_plan_destroy(self.plan)
        except Exception:
            pass

    def buffers(self, T):
        if T not in self._bufs:
            sb, wb = moe_workspace_size(self.plan, T)
            t = self.torch
            self._bufs[T] = (t.empty(sb, dtype=t.uint8, device=self.device),
                             t.empty(wb, dtype=t.uint8, device=self.device))
        return self._bufs[T]

    def stream(self) -> int:
        return self.torch.cuda.current_stream(self.device).cuda_stream

    def quantize_weights(self, W_gate, W_up, W_down, cache=None):
        """Quantised-expert plans (FP8_BLOCK, MXFP8, NVFP4): the weight cache
        (a uint8 device tensor) holding the codes and scales of the expert
        weights (NVFP4: also each expert's tensor maxima); pass it as
        weight_cache to forward and backward."""
        t = self.torch
        n = moe_weight_cache_size(self.plan)
        if cache is None:
            cache = t.empty(n, dtype=t.uint8, device=self.device)
        moe_quantize_weights(self.plan, W_gate.data_ptr(), W_up.data_ptr(), W_down.data_ptr(),
                             cache.data_ptr(), cache.numel(), self.stream())
        return cache

    def forward(self, x, Wr, b, W_gate, W_up, W_down, Ws_gate=None, Ws_up=None, Ws_down=None,
                routing: bool = False, y=None, replay_topk=None, weight_cache=None):
        """replay_topk: optional T×k int32 device tensor of experts to route to
        (router replay) instead of the top-k selection. weight_cache: FP8
        plans, from quantize_weights (W_gate, W_up, W_down may then be None)."""
        t = self.torch
        T = x.shape[0]
        saved, ws = self.buffers(T)
        y = t.empty_like(x) if y is None else y
        out = {}
        if routing:
            k, E = self.cfg.top_k, self.cfg.E
            out = dict(topk_idx=t.empty((T, k), dtype=t.int32, device=x.device),
                       gates=t.empty((T, k), dtype=t.float32, device=x.device),
                       counts=t.empty(E, dtype=t.int32, device=x.device),
                       offsets=t.empty(E + 1, dtype=t.int32, device=x.device),
                       row_of=t.empty((T, k), dtype=t.int32, device=x.device))
        a = moe_fwd_args_t(x=_ptr(x), Wr=_ptr(Wr), b=_ptr(b), W_gate=_ptr(W_gate), W_up=_ptr(W_up),
                           W_down=_ptr(W_down), Ws_gate=_ptr(Ws_gate), Ws_up=_ptr(Ws_up),
                           Ws_down=_ptr(Ws_down), y=_ptr(y), topk_idx=_ptr(out.get("topk_idx")),
                           gates=_ptr(out.get("gates")), counts=_ptr(out.get("counts")),
                           offsets=_ptr(out.get("offsets")), row_of=_ptr(out.get("row_of")),
                           replay_topk=_ptr(replay_topk), weight_cache=_ptr(weight_cache))
        moe_forward(self.plan, T, a, saved.data_ptr(), saved.numel(), ws.data_ptr(), ws.numel(),
                    self.stream())
        return (y, out) if routing else y

    def backward(self, dY, x, Wr, W_gate, W_up, W_down, Ws_gate=None, Ws_up=None, Ws_down=None,
                 grads=None, weight_cache=None, like=None):
        """weight_cache: the cache given to the forward (FP8 plans). like:
        (W_gate, W_up, W_down)-shaped templates for the gradients when the
        weights themselves are not passed."""
        t = self.torch
        T = x.shape[0]
        saved, ws = self.buffers(T)
        if grads is None:
            lg, lu, ld = like if like is not None else (W_gate, W_up, W_down)
            grads = dict(dX=t.empty_like(x), dWr=t.empty_like(Wr), dW_gate=t.empty_like(lg),
                         dW_up=t.empty_like(lu), dW_down=t.empty_like(ld))
            if Ws_gate is not None:
                grads.update(dWs_gate=t.empty_like(Ws_gate), dWs_up=t.empty_like(Ws_up),
                             dWs_down=t.empty_like(Ws_down))
        g = grads
        a = moe_bwd_args_t(dY=_ptr(dY), x=_ptr(x), Wr=_ptr(Wr), W_gate=_ptr(W_gate), W_up=_ptr(W_up),
                           W_down=_ptr(W_down), Ws_gate=_ptr(Ws_gate), Ws_up=_ptr(Ws_up),
                           Ws_down=_ptr(Ws_down), dX=_ptr(g["dX"]), dWr=_ptr(g["dWr"]),
                           dW_gate=_ptr(g["dW_gate"]), dW_up=_ptr(g["dW_up"]),
                           dW_down=_ptr(g["dW_down"]), dWs_gate=_ptr(g.get("dWs_gate")),
                           dWs_up=_ptr(g.get("dWs_up")), dWs_down=_ptr(g.get("dWs_down")),
                           weight_cache=_ptr(weight_cache))
        moe_backward(self.plan, T, a, saved.data_ptr(), saved.numel(), ws.data_ptr(), ws.numel(),
                     self.stream())
        return grads

    def stage_times(self):
        return moe_stage_times(self.plan)

    def status(self, T) -> int:
        _, ws = self.buffers(T)
        return moe_read_status(self.plan, ws.data_ptr(), self.stream())
