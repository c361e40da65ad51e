"""Exact score ties on the GPU: duplicated router columns give two experts
bit-identical logits (and scores) for every token. The layer's reading of
top-k -- equal scores go to the lower expert index, slots in descending
score -- must then decide the selection and the slot order bit for bit, on
both router kernels (E <= 32, and the tiled, H-split router for E > 32) and
both score functions."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from harness import TIE_REL, run_gpu, to_np

pytestmark = pytest.mark.gpu

# (workload, (source, duplicate) column pairs)
CASES = {
    "softmax_e8": (mi.scaled(mi.WORKLOADS["mixtral_8x7b"], T=700, H=256, E=8, k=2, F=128),
                   [(1, 5), (2, 3)]),
    "sigmoid_e64_tiled": (mi.scaled(mi.WORKLOADS["deepseek_v3"], T=600, H=512, E=64, k=6, F=128, Fs=0),
                          [(0, 63), (7, 8), (20, 40), (21, 41)]),
    # Zipf-biased: the pairs are drawn from the most favoured experts (below)
    "softmax_e128_bias": (mi.scaled(mi.WORKLOADS["qwen3_235b"], T=400, H=256, E=128, k=8, F=128),
                          None),
}


@pytest.mark.parametrize("name", list(CASES))
def test_exact_ties_go_to_the_lower_expert_index(name):
    w, pairs = CASES[name]
    inp = mi.make_inputs(w, "cpu", with_grad_out=False)
    if pairs is None:
        order = torch.argsort(inp["b"], descending=True).tolist()
        pairs = [tuple(sorted((order[0], order[3]))), tuple(sorted((order[1], order[6])))]
    Wr = inp["Wr"].clone()
    for src, dup in pairs:
        Wr[:, dup] = Wr[:, src]
    inp["Wr"] = Wr
    if inp["b"] is not None:
        b = inp["b"].clone()
        for src, dup in pairs:
            b[dup] = b[src]
        inp["b"] = b
    gpu, _ = run_gpu(w, inp, backward=False)
    g_topk = gpu["topk_idx"].numpy()
    r = oracle.route(to_np(inp["x"]), to_np(Wr), to_np(inp["b"]), w.k, w.score)
    s = r["scores"]
    for src, dup in pairs:
        assert np.array_equal(s[:, src], s[:, dup])
    # tokens whose near-ties (relative gap < 1e-5 among the top k+1 scores)
    # are all exact ties: the answer is unique under the lower-index rule
    srt = -np.sort(-s, axis=1)[:, : w.k + 1]
    gaps = (srt[:, :-1] - srt[:, 1:]) / np.abs(srt[:, :-1])
    near = gaps < TIE_REL
    inexact = np.any(near & (gaps > 0), axis=1)
    exact = np.any(gaps == 0, axis=1) & ~inexact
    assert exact.sum() >= 20, f"too few exactly tied tokens ({exact.sum()})"
    decided = ~inexact
    assert np.array_equal(g_topk[decided], r["topk"][decided]), \
        f"{int(np.sum(np.any(g_topk[decided] != r['topk'][decided], 1)))} decided tokens differ"
    # the rule itself, on the GPU's answer: a duplicate is never chosen without
    # its source, and never ahead of it
    for src, dup in pairs:
        for t in np.nonzero((g_topk == dup).any(1) & decided)[0]:
            row = list(g_topk[t])
            assert src in row and row.index(src) < row.index(dup), (t, row)
    # gates of tied experts are bit-identical
    gg = gpu["gates"].numpy()
    for t in np.nonzero(exact)[0]:
        row = list(g_topk[t])
        for src, dup in pairs:
            if src in row and dup in row:
                assert gg[t, row.index(src)] == gg[t, row.index(dup)]
