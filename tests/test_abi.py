"""The C ABI library: it loads, exports every entry point include/moe.h
declares, and validates arguments before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_sigmoid_gb300 as moe
from mixture_experts_layer_sigmoid_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return moe.load_library()


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_bound_names():
    assert declared_entry_points() == sorted(moe.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), name
    assert moe.moe_abi_version() == 3


def test_status_strings(lib):
    for code in range(7):
        assert moe.moe_status_string(code) not in ("", "unknown status")
    assert moe.moe_status_string(99) == "unknown status"


def _cfg(**kw):
    base = dict(H=256, E=8, F=512, Fs=0, top_k=2, T_max=1024, score=0, dtype=1, flags=0)
    base.update(kw)
    return moe.moe_config_t(**base)


@pytest.mark.parametrize("bad", [dict(H=100), dict(H=0), dict(F=200), dict(Fs=64), dict(E=0),
                                 dict(E=257), dict(top_k=0), dict(top_k=9), dict(top_k=9, E=16),
                                 dict(E=2, top_k=3), dict(T_max=0), dict(score=2), dict(dtype=7),
                                 dict(flags=4), dict(flags=8), dict(capacity_factor=-1.0),
                                 dict(capacity_factor=float("nan")), dict(capacity_factor=float("inf"))])
def test_plan_create_rejects_bad_configs(lib, bad):
    plan = ctypes.c_void_p()
    st = lib.moe_plan_create(ctypes.byref(_cfg(**bad)), 0, ctypes.byref(plan))
    assert st == moe.MOE_ERR_INVALID_ARG
    assert plan.value is None


@pytest.mark.parametrize("dtype", [2, 3])
def test_fp8_with_capacity_dropping_passes_validation(lib, dtype):
    """Both FP8 recipes accept capacity-limited dropping: the config is valid
    (a plan on a GPU; without one, only the device query fails)."""
    plan = ctypes.c_void_p()
    st = lib.moe_plan_create(ctypes.byref(_cfg(dtype=dtype, capacity_factor=1.0)), 0, ctypes.byref(plan))
    # (UNSUPPORTED only for a device that is not sm_103)
    assert st in (moe.MOE_OK, moe.MOE_ERR_CUDA) or (st == moe.MOE_ERR_UNSUPPORTED and not _has_sm103())
    if st == moe.MOE_OK:
        assert lib.moe_plan_destroy(plan) == moe.MOE_OK


def _has_sm103():
    try:
        import torch
        return torch.cuda.is_available() and torch.cuda.get_device_capability(0) == (10, 3)
    except Exception:
        return False


def test_blockwise_fp8_with_shared_expert_is_reported_unsupported(lib):
    plan = ctypes.c_void_p()
    assert lib.moe_plan_create(ctypes.byref(_cfg(dtype=2, Fs=256)), 0,
                               ctypes.byref(plan)) == moe.MOE_ERR_UNSUPPORTED


def test_mxfp8_with_shared_expert_passes_validation(lib):
    plan = ctypes.c_void_p()
    st = lib.moe_plan_create(ctypes.byref(_cfg(dtype=3, Fs=256)), 0, ctypes.byref(plan))
    assert st in (moe.MOE_OK, moe.MOE_ERR_CUDA) or (st == moe.MOE_ERR_UNSUPPORTED and not _has_sm103())
    if st == moe.MOE_OK:
        assert lib.moe_plan_destroy(plan) == moe.MOE_OK


def test_nvfp4_needs_256_multiples(lib):
    """NVFP4 data GEMMs take 256-value k blocks: H, F and Fs must be
    multiples of 256 (UNSUPPORTED otherwise, before any device work)."""
    for bad in (dict(H=384), dict(F=384), dict(Fs=128)):
        plan = ctypes.c_void_p()
        assert lib.moe_plan_create(ctypes.byref(_cfg(dtype=4, **bad)), 0,
                                   ctypes.byref(plan)) == moe.MOE_ERR_UNSUPPORTED
        assert plan.value is None
    plan = ctypes.c_void_p()
    st = lib.moe_plan_create(ctypes.byref(_cfg(dtype=4, Fs=256, capacity_factor=1.0)), 0, ctypes.byref(plan))
    assert st in (moe.MOE_OK, moe.MOE_ERR_CUDA) or (st == moe.MOE_ERR_UNSUPPORTED and not _has_sm103())
    if st == moe.MOE_OK:
        assert lib.moe_plan_destroy(plan) == moe.MOE_OK


def test_nv_quantize_validates_arguments(lib):
    buf = ctypes.create_string_buffer(64)
    p = ctypes.cast(buf, ctypes.c_void_p)
    q = lambda *a: lib.moe_nv_quantize(*a, None)
    assert q(100, 128, p, p, p, p, None, None) == moe.MOE_ERR_INVALID_ARG   # rows % 128
    assert q(128, 128, None, p, p, p, None, None) == moe.MOE_ERR_INVALID_ARG  # no input
    assert q(128, 128, p, None, p, p, None, None) == moe.MOE_ERR_INVALID_ARG  # no amax
    assert q(128, 128, p, p, p, None, None, None) == moe.MOE_ERR_INVALID_ARG  # codes without scales
    assert q(128, 128, p, p, None, None, None, None) == moe.MOE_ERR_INVALID_ARG  # no output


def test_null_arguments(lib):
    assert lib.moe_plan_create(None, 0, None) == moe.MOE_ERR_INVALID_ARG
    s, w = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.moe_workspace_size(None, 16, ctypes.byref(s), ctypes.byref(w)) == moe.MOE_ERR_INVALID_ARG
    args = moe.moe_fwd_args_t()
    assert lib.moe_forward(None, 16, ctypes.byref(args), None, 0, None, 0, None) == moe.MOE_ERR_INVALID_ARG
    bargs = moe.moe_bwd_args_t()
    assert lib.moe_backward(None, 16, ctypes.byref(bargs), None, 0, None, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_read_status(None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_plan_destroy(None) == moe.MOE_OK
    n = ctypes.c_size_t()
    assert lib.moe_weight_cache_size(None, ctypes.byref(n)) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_weights(None, None, None, None, None, 0, None) == moe.MOE_ERR_INVALID_ARG


def test_valid_config_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    plan = ctypes.c_void_p()
    st = lib.moe_plan_create(ctypes.byref(_cfg()), 0, ctypes.byref(plan))
    assert st in (moe.MOE_ERR_CUDA, moe.MOE_ERR_INVALID_ARG)
    assert plan.value is None


def test_update_bias_rejects_bad_arguments(lib):
    buf = ctypes.c_void_p(16)        # never dereferenced: rejected before any launch
    for E, counts, rate, b in ((0, buf, 0.1, buf), (257, buf, 0.1, buf), (8, None, 0.1, buf),
                               (8, buf, 0.1, None), (8, buf, float("nan"), buf),
                               (8, buf, float("inf"), buf)):
        assert lib.moe_update_bias(E, counts, rate, b, None) == moe.MOE_ERR_INVALID_ARG
