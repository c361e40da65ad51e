"""Failure detection on the device without faulting the GPU: the bounded
mbarrier wait every pipelined kernel uses runs out on a barrier that nothing
signals, reports MOE_ERR_DEVICE_TIMEOUT through the workspace status word,
and the context stays usable for a normal layer call afterwards."""
import time

import pytest
import torch

import moe_inputs as mi
import mixture_experts_layer_sigmoid_gb300 as moe
from harness import run_gpu

pytestmark = pytest.mark.gpu


def test_stalled_wait_reports_timeout_and_device_stays_usable():
    w = mi.scaled(mi.WORKLOADS["mixtral_8x7b"], T=200, H=256, E=4, k=2, F=256)
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T)
    _, ws = layer.buffers(w.T)
    lib = moe.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.time()
    assert lib.moe_diag_wait_timeout(ws.data_ptr(), stream) == moe.MOE_OK
    st = moe.moe_read_status(layer.plan, ws.data_ptr(), stream)
    elapsed = time.time() - t0
    assert st == moe.MOE_ERR_DEVICE_TIMEOUT, moe.moe_status_string(st)
    assert 1.0 < elapsed < 30.0
    # the context is intact: a full forward + backward still runs clean
    out, _ = run_gpu(w, mi.make_inputs(w), layer=layer)
    assert torch.isfinite(out["y"]).all()
