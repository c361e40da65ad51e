"""Seeded synthetic inputs for one Mixture-of-Experts layer.

This module is shared by the tests, the benchmark and the smoke check. It
holds the workload shapes and a counter-based random generator, and nothing
of the layer's arithmetic (no routing, no expert FFN, no gradients).

Generator: element ``c`` of the stream with key ``K`` is the ``c``-th output of
SplitMix64 seeded with ``K`` (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; the finaliser constants are
Vigna's). Uniforms take the top 53 bits, ``(v >> 11) + 0.5`` times ``2**-53``,
so they lie in the open interval (0, 1). Normals come from the Box-Muller
transform on consecutive pairs of uniforms. Every value depends only on
(seed, tensor id, flat index), so any slice of a tensor can be regenerated
on its own, on the host or on a CUDA device, with identical integer
arithmetic.

The shapes stand in for the expert layers of the models that "Scalable
Training of Mixture-of-Experts Models with Megatron Core" evaluates (§8,
Performance Evaluation: DeepSeek-V3 and Qwen3-235B; §9, Expert Parallelism:
Mixtral-8x7B). No dataset is read.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

GOLDEN = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1


def _s64(v: int) -> int:
    """Two's-complement int64 view of a uint64 constant."""
    v &= MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


# ---------------------------------------------------------------- pure Python
def splitmix64_py(key: int, c: int) -> int:
    """c-th output (0-based) of SplitMix64 seeded with ``key``; exact ints."""
    z = (key + (c + 1) * GOLDEN) & MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def uniform_py(key: int, c: int) -> float:
    return ((splitmix64_py(key, c) >> 11) + 0.5) * 2.0 ** -53


def normal_py(key: int, i: int) -> float:
    u1 = uniform_py(key, 2 * (i // 2))
    u2 = uniform_py(key, 2 * (i // 2) + 1)
    r = math.sqrt(-2.0 * math.log(u1))
    return r * (math.cos(2 * math.pi * u2) if i % 2 == 0 else math.sin(2 * math.pi * u2))


def tensor_key(seed: int, tensor_id: int) -> int:
    """Stream key of one tensor: output ``tensor_id`` of the stream ``seed``."""
    return splitmix64_py(seed & MASK64, tensor_id)


# ---------------------------------------------------------------- torch (any device)
def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 holding uint64 bits."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def splitmix64_t(key: int, c: torch.Tensor) -> torch.Tensor:
    """Vectorised :func:`splitmix64_py`; ``c`` is int64, result int64 bits."""
    z = c + 1
    z = z * _s64(GOLDEN) + _s64(key)
    z = (z ^ _lsr(z, 30)) * _s64(MIX1)
    z = (z ^ _lsr(z, 27)) * _s64(MIX2)
    return z ^ _lsr(z, 31)


def uniform_t(key: int, c: torch.Tensor) -> torch.Tensor:
    top = _lsr(splitmix64_t(key, c), 11)
    return (top.to(torch.float64) + 0.5) * (2.0 ** -53)


def normal_t(key: int, start: int, count: int, device) -> torch.Tensor:
    """Normals ``start .. start+count-1`` of the stream ``key`` in float64."""
    i = torch.arange(start, start + count, dtype=torch.int64, device=device)
    pair = i // 2
    u1 = uniform_t(key, 2 * pair)
    u2 = uniform_t(key, 2 * pair + 1)
    r = torch.sqrt(-2.0 * torch.log(u1))
    ang = (2.0 * math.pi) * u2
    return torch.where(i % 2 == 0, r * torch.cos(ang), r * torch.sin(ang))


def normal_tensor(seed: int, tensor_id: int, shape, std: float, dtype: torch.dtype,
                  device="cpu", chunk: int = 1 << 26) -> torch.Tensor:
    """A tensor of N(0, std**2) values, rounded once (RNE) to ``dtype``."""
    key = tensor_key(seed, tensor_id)
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=dtype, device=device)
    for s0 in range(0, n, chunk):
        cnt = min(chunk, n - s0)
        out[s0:s0 + cnt] = (normal_t(key, s0, cnt, device) * std).to(dtype)
    return out.view(*shape)


def permutation(seed: int, tensor_id: int, n: int) -> torch.Tensor:
    """A seeded permutation of 0..n-1: indices sorted by their uniform draw."""
    key = tensor_key(seed, tensor_id)
    u = uniform_t(key, torch.arange(n, dtype=torch.int64))
    return torch.argsort(u, stable=True)


# ---------------------------------------------------------------- workloads
SOFTMAX, SIGMOID = 0, 1
FP32, BF16, FP8_BLOCK, MXFP8, NVFP4 = 0, 1, 2, 3, 4

# tensor ids within one seed
TID = dict(x=1, Wr=2, b=3, Wg=4, Wu=5, Wd=6, Wsg=7, Wsu=8, Wsd=9, dY=10, perm=11)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    F: int
    Fs: int = 0            # shared-expert width, 0 = none
    score: int = SOFTMAX
    dtype: int = BF16
    bias: str = "none"     # "none" | "normal" (b ~ N(0, 0.5)) | "zipf" (1.5 ln(1/rank))
    seed: int = 0

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == FP32 else torch.bfloat16

    @property
    def R(self) -> int:
        return self.T * self.k

    def flops_fwd_bwd(self) -> float:
        """Algorithmic FLOPs of one forward + backward pass (2 per MAC).

        Expert GEMMs: 6HF per routed row forward (fc1 gate, fc1 up, fc2) and
        twice that backward (dgrad + wgrad); the shared expert the same per
        token; the router GEMM 2THE forward and the sparse router backward
        4TkH. Zero padding rows and elementwise work are not counted."""
        ex = 18.0 * self.H * self.F * self.R + 18.0 * self.H * self.Fs * self.T
        return ex + 2.0 * self.T * self.H * self.E + 4.0 * self.T * self.k * self.H


WORKLOADS: Dict[str, Workload] = {
    # the five layer shapes
    "tiny_fp32": Workload("tiny_fp32", T=256, H=128, E=4, k=2, F=256, dtype=FP32, seed=0),
    "mixtral_8x7b": Workload("mixtral_8x7b", T=4096, H=4096, E=8, k=2, F=14336, seed=1000),
    "deepseek_v3": Workload("deepseek_v3", T=8192, H=7168, E=256, k=8, F=2048, Fs=2048,
                            score=SIGMOID, bias="normal", seed=2000),
    "qwen3_235b": Workload("qwen3_235b", T=16384, H=4096, E=128, k=8, F=1536, bias="zipf",
                           seed=3000),
    "qwen3_235b_fp8": Workload("qwen3_235b_fp8", T=16384, H=4096, E=128, k=8, F=1536,
                               dtype=FP8_BLOCK, bias="zipf", seed=4000),
    # the same shape in the MXFP8 recipe (1x32 blocks, power-of-two scales)
    "qwen3_235b_mxfp8": Workload("qwen3_235b_mxfp8", T=16384, H=4096, E=128, k=8, F=1536,
                                 dtype=MXFP8, bias="zipf", seed=4000),
    # the DeepSeek-V3 shape (with its shared expert) in the MXFP8 recipe, on
    # the bf16 workload's inputs
    "deepseek_v3_mxfp8": Workload("deepseek_v3_mxfp8", T=8192, H=7168, E=256, k=8, F=2048, Fs=2048,
                                  score=SIGMOID, dtype=MXFP8, bias="normal", seed=2000),
    # the same two shapes in the NVFP4 recipe (E2M1 values, 1x16 blocks with
    # E4M3 scales, one fp32 scale per expert tensor)
    "qwen3_235b_nvfp4": Workload("qwen3_235b_nvfp4", T=16384, H=4096, E=128, k=8, F=1536,
                                 dtype=NVFP4, bias="zipf", seed=4000),
    "deepseek_v3_nvfp4": Workload("deepseek_v3_nvfp4", T=8192, H=7168, E=256, k=8, F=2048, Fs=2048,
                                  score=SIGMOID, dtype=NVFP4, bias="normal", seed=2000),
}


def scaled(w: Workload, **kw) -> Workload:
    """A smaller workload of the same family (same score, bias and dtype)."""
    return dataclasses.replace(w, **kw)


def router_std(H: int) -> float:
    """Router weight std: variance 0.02 at H=128, scaled by fan-in 128/H."""
    return math.sqrt(0.02 * 128.0 / H)


def make_bias(w: Workload) -> Optional[torch.Tensor]:
    if w.bias == "none":
        return None
    if w.bias == "normal":
        return normal_tensor(w.seed, TID["b"], (w.E,), math.sqrt(0.5), torch.float32)
    if w.bias == "zipf":
        perm = permutation(w.seed, TID["perm"], w.E)
        rank = torch.empty(w.E, dtype=torch.float64)
        rank[perm] = torch.arange(1, w.E + 1, dtype=torch.float64)
        return (1.5 * torch.log(1.0 / rank)).to(torch.float32)
    raise ValueError(w.bias)


def make_inputs(w: Workload, device="cpu", with_grad_out: bool = True) -> Dict[str, torch.Tensor]:
    """All inputs of one forward + backward in their storage dtypes.

    Layouts (row-major): x T×H; Wr H×E fp32; b E fp32; Wg, Wu E×H×F;
    Wd E×F×H; Wsg, Wsu H×Fs; Wsd Fs×H; dY T×H."""
    dt = w.torch_dtype if w.dtype not in (FP8_BLOCK, MXFP8, NVFP4) else torch.bfloat16
    g = {}
    g["x"] = normal_tensor(w.seed, TID["x"], (w.T, w.H), 1.0, dt, device)
    g["Wr"] = normal_tensor(w.seed, TID["Wr"], (w.H, w.E), router_std(w.H), torch.float32, device)
    b = make_bias(w)
    g["b"] = None if b is None else b.to(device)
    g["Wg"] = normal_tensor(w.seed, TID["Wg"], (w.E, w.H, w.F), 1.0 / math.sqrt(w.H), dt, device)
    g["Wu"] = normal_tensor(w.seed, TID["Wu"], (w.E, w.H, w.F), 1.0 / math.sqrt(w.H), dt, device)
    g["Wd"] = normal_tensor(w.seed, TID["Wd"], (w.E, w.F, w.H), 1.0 / math.sqrt(w.F), dt, device)
    if w.Fs:
        g["Wsg"] = normal_tensor(w.seed, TID["Wsg"], (w.H, w.Fs), 1.0 / math.sqrt(w.H), dt, device)
        g["Wsu"] = normal_tensor(w.seed, TID["Wsu"], (w.H, w.Fs), 1.0 / math.sqrt(w.H), dt, device)
        g["Wsd"] = normal_tensor(w.seed, TID["Wsd"], (w.Fs, w.H), 1.0 / math.sqrt(w.Fs), dt, device)
    else:
        g["Wsg"] = g["Wsu"] = g["Wsd"] = None
    if with_grad_out:
        g["dY"] = normal_tensor(w.seed, TID["dY"], (w.T, w.H), 1.0, dt, device)
    return g
