"""Guard bands and unwritten outputs, in place of a memory checker (the
device sanitizer is not available on this GPU pool).

Every buffer the layer writes through the C ABI -- y, dX and the weight
gradients, the saved buffer and the workspace -- is a view into a larger
allocation with a canary band of 4 KiB on each side, and the outputs start
NaN-filled. After forward and backward every output element must have been
written (finite) and every band must still hold its canary bytes (nothing
written past a buffer). The layer overwrites its gradients and writes zeros
for experts that receive no tokens, so an all-finite gradient also shows
that empty experts are handled ("Scalable Training of Mixture-of-Experts
Models with Megatron Core", §2: dropless routing gives experts ragged,
possibly empty, token counts)."""
import pytest
import torch

import moe_inputs as mi
import mixture_experts_layer_sigmoid_gb300 as moe
from harness import upload

pytestmark = pytest.mark.gpu

GUARD = 4096
CANARY = 0xA5

W = mi.WORKLOADS
CASES = {
    "bf16_ragged": mi.scaled(W["mixtral_8x7b"], T=333, H=256, E=8, k=2, F=384),
    "bf16_sigmoid_shared": mi.scaled(W["deepseek_v3"], T=260, H=256, E=16, F=256, Fs=256),
    # Zipf-biased routing over 64 experts: several experts get no tokens
    "bf16_zipf_empty_experts": mi.scaled(W["qwen3_235b"], T=130, H=256, E=64, k=2, F=256),
    "fp32_shared": mi.scaled(W["deepseek_v3"], T=100, H=128, E=4, k=2, F=128, Fs=128, dtype=mi.FP32),
    "fp8_ragged": mi.scaled(W["qwen3_235b_fp8"], T=450, H=384, E=16, k=8, F=384),
}


class Carved:
    """A byte range with canary bands on both sides."""

    def __init__(self, nbytes, dev):
        self.n = nbytes
        self.buf = torch.full((GUARD + nbytes + GUARD,), CANARY, dtype=torch.uint8, device=dev)

    def view(self, shape=None, dtype=torch.uint8):
        v = self.buf[GUARD:GUARD + self.n]
        return v if shape is None else v.view(dtype).view(shape)

    def bands_intact(self):
        return bool((self.buf[:GUARD] == CANARY).all()) and bool((self.buf[GUARD + self.n:] == CANARY).all())


def carve_like(t):
    c = Carved(t.numel() * t.element_size(), t.device)
    v = c.view(t.shape, t.dtype)
    v.fill_(float("nan"))
    return c, v


@pytest.mark.parametrize("fold", [False, True])
@pytest.mark.parametrize("name", list(CASES))
def test_outputs_fully_written_and_nothing_written_past_a_buffer(name, fold):
    w = CASES[name]
    inp = mi.make_inputs(w, "cpu", with_grad_out=True)
    g = upload(inp)
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score, dtype=w.dtype, Fs=w.Fs, fold_gates=fold)
    sb, wb = moe.moe_workspace_size(layer.plan, w.T)
    saved, ws = Carved(sb, "cuda"), Carved(wb, "cuda")
    layer._bufs[w.T] = (saved.view(), ws.view())
    cy, y = carve_like(g["x"])
    _, route = layer.forward(g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"], g["Wsg"], g["Wsu"],
                             g["Wsd"], y=y, routing=True)
    carved = {"y": (cy, y)}
    grads = {}
    for key, like in [("dX", g["x"]), ("dWr", g["Wr"]), ("dW_gate", g["Wg"]), ("dW_up", g["Wu"]),
                      ("dW_down", g["Wd"])] + ([("dWs_gate", g["Wsg"]), ("dWs_up", g["Wsu"]),
                                                ("dWs_down", g["Wsd"])] if w.Fs else []):
        c, v = carve_like(like)
        carved[key] = (c, v)
        grads[key] = v
    layer.backward(g["dY"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], g["Wsg"], g["Wsu"], g["Wsd"],
                   grads=grads)
    torch.cuda.synchronize()
    assert layer.status(w.T) == 0
    for key, (c, v) in carved.items():
        assert bool(torch.isfinite(v.float()).all()), f"{key}: elements left unwritten"
        assert c.bands_intact(), f"{key}: written past the buffer"
    assert saved.bands_intact(), "saved buffer: written past its end or before its start"
    assert ws.bands_intact(), "workspace: written past its end or before its start"
    # experts with no tokens: each of their weight-gradient entries is an exact zero
    empty = (route["counts"] == 0).nonzero().flatten().tolist()
    if name == "bf16_zipf_empty_experts":
        assert len(empty) > 0
    for key in ("dW_gate", "dW_up", "dW_down"):
        for e in empty:
            assert bool((grads[key][e] == 0).all()), f"{key}[{e}] of an empty expert"
