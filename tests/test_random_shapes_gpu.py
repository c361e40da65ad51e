"""Parity against the oracle on seeded, randomly drawn small layer shapes.

The hand-picked cases cover each kernel's special paths; these draws cover
their combinations: expert counts from 1 to 256 (every router kernel and
its 4- and 16-byte weight staging), top-k from 1 to 8, token counts that are
not multiples of the 32-token router block or the 128-row tile, softmax or
sigmoid scores with or without a per-expert bias, a shared expert, and the
bf16, fp32 and blockwise-FP8 layers ("Scalable Training of Mixture-of-
Experts Models with Megatron Core", §2 and §5). Each case runs the full
parity comparison of tests/harness.py (bit-exact routing except near-ties,
bounds on every output and gradient), or the FP8 layer's comparison with the
oracle's FP8 layer."""
import numpy as np
import pytest

import moe_inputs as mi
from harness import full_parity

pytestmark = pytest.mark.gpu


def _draw(i):
    rng = np.random.default_rng(1000 + i)
    dtype = [mi.BF16, mi.BF16, mi.FP32, mi.FP8_BLOCK][i % 4]
    E = int(rng.choice([1, 2, 5, 8, 13, 24, 32, 33, 47, 64, 96, 127, 128, 160, 256]))
    k = int(rng.integers(1, min(8, E) + 1))
    H = int(rng.choice([128, 256, 384]))
    F = int(rng.choice([128, 256, 384]))
    T = int(rng.integers(1, 520))
    score = int(rng.integers(0, 2))
    Fs = int(rng.choice([0, 128])) if dtype != mi.FP8_BLOCK else 0
    bias = str(rng.choice(["none", "normal", "zipf"]))
    return mi.Workload(name=f"random{i}", T=T, H=H, E=E, k=k, F=F, Fs=Fs, score=score, dtype=dtype,
                       bias=bias, seed=5000 + i)


@pytest.mark.parametrize("i", range(16))
def test_random_shape_matches_oracle(i):
    w = _draw(i)
    if w.dtype == mi.FP8_BLOCK:
        from test_fp8_gpu import fp8_layer_parity
        rep = fp8_layer_parity(w)
    else:
        rep, _ = full_parity(w)
    print(w, rep)
