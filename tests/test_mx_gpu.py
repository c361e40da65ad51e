"""MXFP8 layer (MOE_MXFP8) on the GPU against the oracle's MXFP8 layer.

"Scalable Training of Mixture-of-Experts Models with Megatron Core", §5
Platform-specific recipes: MXFP8 with 1x32 granularity, the default FP8
recipe on Blackwell. The quantiser the layer uses must give the oracle's
E4M3 codes and UE8M0 scales bit for bit, in every orientation the layer
uses (blocks along rows; blocks down columns, transposed or in place), with
the scales in the layout the GEMMs copy into tensor memory. The whole layer,
forward and backward, must match the oracle's MXFP8 layer within the FP8
bounds: relative L2 <= 4e-2 and max |error| <= 1.5e-1 rms(ref) on every
output and gradient."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import mixture_experts_layer_sigmoid_gb300 as moe
from test_fp8_gpu import fp8_layer_parity

pytestmark = pytest.mark.gpu


def _atoms_to_scales(atoms, n, K):
    """Scale bytes [n][K/32] of an operand [n][K] from its 512-byte atoms."""
    a = atoms.reshape(n // 128, K // 128, 512)
    m = np.arange(128)
    j = np.arange(4)
    idx = (16 * (m % 32) + 4 * (m // 32))[:, None] + j[None, :]          # [128][4]
    out = a[:, :, idx]                                                    # [n/128][K/128][128][4]
    return out.transpose(0, 2, 1, 3).reshape(n, K // 32)


def _mxq(x, rows=True, cols=None):
    R, C = x.shape
    dev = x.device
    q = torch.empty((R, C), dtype=torch.uint8, device=dev) if rows else None
    sq = torch.empty(R * C // 32, dtype=torch.uint8, device=dev) if rows else None
    qc = None
    if cols is not None:
        qc = torch.empty((C, R) if cols == 1 else (R, C), dtype=torch.uint8, device=dev)
    sc = torch.empty(R * C // 32, dtype=torch.uint8, device=dev) if cols is not None else None
    p = lambda t: None if t is None else t.data_ptr()
    moe.moe_mx_quantize(R, C, x.data_ptr(), p(q), p(sq), p(qc), p(sc), 1 if cols == 1 else 0,
                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    n = lambda t: None if t is None else t.cpu().numpy()
    return n(q), n(sq), n(qc), n(sc)


def test_mx_quantiser_matches_oracle_bit_for_bit():
    g = torch.Generator().manual_seed(6)
    x = (torch.randn(384, 512, generator=g) * torch.logspace(-4, 3, 512)).to(torch.bfloat16)
    x[0:32, 0:32] = 0                        # an all-zero block
    x[200, 300] = 3.0e4
    x[5, 7] = 1e-38                          # a tiny value next to normal ones
    xf = x.float().numpy()
    xd = x.cuda()
    R, C = xf.shape
    oc_r, os_r = oracle.mx_quantize(xf, oracle.MX_ROWS)
    oc_c, os_c = oracle.mx_quantize(xf, oracle.MX_COLS)
    q, sq, qc, sc = _mxq(xd, rows=True, cols=1)
    assert np.array_equal(q, oc_r)
    assert np.array_equal(_atoms_to_scales(sq, R, C), os_r)
    assert np.array_equal(qc, oc_c.T)
    assert np.array_equal(_atoms_to_scales(sc, C, R), os_c.T)
    q, sq, qc, sc = _mxq(xd, rows=False, cols=0)
    assert q is None and np.array_equal(qc, oc_c)
    assert np.array_equal(_atoms_to_scales(sc, C, R), os_c.T)


MX_CASES = {
    "single_expert": mi.scaled(mi.WORKLOADS["qwen3_235b_mxfp8"], T=256, H=256, E=1, k=1, F=256),
    "mx_small": mi.scaled(mi.WORKLOADS["qwen3_235b_mxfp8"], T=600, H=256, E=8, k=4, F=256),
    "mx_ragged": mi.scaled(mi.WORKLOADS["qwen3_235b_mxfp8"], T=450, H=384, E=16, k=8, F=384),
    "mx_many_rows_per_expert": mi.scaled(mi.WORKLOADS["qwen3_235b_mxfp8"], T=1100, H=256, E=4, k=2,
                                         F=384),
    "mx_sigmoid_e64": mi.scaled(mi.WORKLOADS["deepseek_v3"], T=300, H=256, E=64, k=6, F=128, Fs=0,
                                dtype=mi.MXFP8),
    # DeepSeek-shaped with the shared expert: a dense group of T = 300 rows
    # (codes padded to 384; CTA pairs with a ghost half; Fs != F)
    "mx_deepseek_shared": mi.scaled(mi.WORKLOADS["deepseek_v3"], T=300, H=256, E=16, k=4, F=256,
                                    Fs=384, dtype=mi.MXFP8),
    # one dense tile of 100 rows (single CTAs)
    "mx_shared_one_tile": mi.scaled(mi.WORKLOADS["deepseek_v3"], T=100, H=256, E=8, k=2, F=128,
                                    Fs=256, dtype=mi.MXFP8),
}


@pytest.mark.parametrize("name", list(MX_CASES))
def test_mx_layer_matches_oracle(name):
    print(name, fp8_layer_parity(MX_CASES[name], False))


@pytest.mark.parametrize("name", ["mx_small", "mx_many_rows_per_expert", "mx_deepseek_shared"])
def test_mx_folded_gates_match_oracle(name):
    print(name, "folded", fp8_layer_parity(MX_CASES[name], True))


def test_mx_shared_expert_with_capacity_dropping_matches_oracle():
    print("mx_deepseek_shared capacity", fp8_layer_parity(MX_CASES["mx_deepseek_shared"], False, 1.0))


def test_mx_layer_is_deterministic_and_graph_capturable():
    w = MX_CASES["mx_ragged"]
    g = {k: (None if v is None else v.cuda()) for k, v in mi.make_inputs(w).items()}
    layer = moe.MoELayer(w.H, w.E, w.F, w.k, w.T, score=w.score, dtype=moe.MOE_MXFP8)
    args = (g["x"], g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"])
    y = torch.empty_like(g["x"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.forward(*args, y=y)
        grads = layer.backward(g["dY"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    eager = {"y": y.clone(), **{k: v.clone() for k, v in grads.items()}}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        layer.forward(*args, y=y)
        layer.backward(g["dY"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], grads=grads)
    for t in [y, *grads.values()]:
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert layer.status(w.T) == 0
    assert torch.equal(y, eager["y"])
    for k, v in grads.items():
        assert torch.equal(v, eager[k]), k
