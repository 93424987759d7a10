"""Seeded synthetic inputs, shared by the tests, the bench and the smoke check.

This module holds no logsumexp arithmetic: only seeded random draws and the
named workload recipes, so that the CUDA path and the oracle can be fed the
very same values.  A generator on a given device is deterministic for a given
seed; values drawn on CPU and on CUDA differ, so a caller that needs the same
tensor on both sides draws it once and copies it.

Distribution notation: ``N(mu, var)`` names the variance, so N(0, 4) has
standard deviation 2 and N(0, 0.1) has standard deviation sqrt(0.1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, mean: float = 0.0, var: float = 1.0, device="cpu") -> torch.Tensor:
    """fp32 draws from N(mean, var)."""
    t = torch.randn(tuple(shape), generator=generator(seed, device), dtype=torch.float32,
                    device=device)
    std = math.sqrt(var)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t


def uniform(shape, seed: int, lo: float, hi: float, device="cpu") -> torch.Tensor:
    """fp32 draws from U[lo, hi)."""
    t = torch.rand(tuple(shape), generator=generator(seed, device), dtype=torch.float32,
                   device=device)
    return t.mul_(hi - lo).add_(lo)


def bernoulli_mask(shape, seed: int, p: float, device="cpu") -> torch.Tensor:
    """bool mask, each entry True with probability p."""
    u = torch.rand(tuple(shape), generator=generator(seed, device), dtype=torch.float32,
                   device=device)
    return u < p


@dataclass(frozen=True)
class Workload:
    """A named workload: what is computed, on which shape, from which recipe."""
    name: str
    op: str                      # "lse_dim0" | "log_softmax" | "gn_act_lse" | "softmax" |
                                 # "log_softmax_dim0" | "group_norm" | "gn_act_residual" |
                                 # "conv_gn_act_lse"
    shape: tuple
    recipe: str
    params: dict = field(default_factory=dict)

    @property
    def numel(self) -> int:
        return math.prod(self.shape)


# The five workloads of the hot path.  Shapes follow the pages' problems: the
# logsumexp-over-dim-0 task (R,B,D)=(4,10,32); the LogSoftmax task (4096, 393216);
# the Conv2d/GroupNorm/Tanh/HardSwish/residual/LogSumExp task, whose conv output
# is [128, 64, 126, 126] (3x3 valid conv of a 128x128 input), G=16, eps=1e-5.
WORKLOADS = {
    "lse_dim0_4x10x32": Workload(
        "lse_dim0_4x10x32", "lse_dim0", (4, 10, 32),
        "x ~ N(0,1), seed 1", {"seed": 1}),
    "log_softmax_256x4096": Workload(
        "log_softmax_256x4096", "log_softmax", (256, 4096),
        "x ~ N(0,4) (std 2), seed 2; each entry set to -inf with probability 0.01 "
        "(mask seed 102); no row is entirely -inf", {"seed": 2, "mask_seed": 102, "p_ninf": 0.01}),
    "lse_dim0_32x8192x4096": Workload(
        "lse_dim0_32x8192x4096", "lse_dim0", (32, 8192, 4096),
        "x ~ U[-20,20), seed 3", {"seed": 3}),
    "log_softmax_4096x393216": Workload(
        "log_softmax_4096x393216", "log_softmax", (4096, 393216),
        "x ~ N(0,1), seed 4", {"seed": 4}),
    "gn_act_lse_128x64x126x126": Workload(
        "gn_act_lse_128x64x126x126", "gn_act_lse", (128, 64, 126, 126),
        "y ~ N(0,1) seed 5 (stand-in for the 3x3 conv output); gamma ~ U[0.5,1.5) seed 105; "
        "beta ~ N(0,0.1) seed 205; G=16, eps=1e-5",
        {"seed": 5, "gamma_seed": 105, "beta_seed": 205, "G": 16, "eps": 1e-5}),
}

# The operations beside the hot path, each on the shape and recipe of the
# hot-path workload it sits next to: softmax on the LogSoftmax rows,
# log_softmax over dim 0 of the (R, B, D) tensor, and GroupNorm alone and the
# chain without its lse on the conv output.
for _name, _op, _like in (
        ("softmax_4096x393216", "softmax", "log_softmax_4096x393216"),
        ("log_softmax_dim0_32x8192x4096", "log_softmax_dim0", "lse_dim0_32x8192x4096"),
        ("group_norm_128x64x126x126", "group_norm", "gn_act_lse_128x64x126x126"),
        ("gn_act_residual_128x64x126x126", "gn_act_residual", "gn_act_lse_128x64x126x126")):
    _w = WORKLOADS[_like]
    WORKLOADS[_name] = Workload(_name, _op, _w.shape, _w.recipe, dict(_w.params, like=_like))

# The chain from its convolution's input: x [128, 8, 128, 128] through Conv2d(8 -> 64, 3 x 3,
# valid, bias) to the y of the chain above.  The weights are drawn like a freshly
# initialised layer (uniform within +-1/sqrt(fan_in), fan_in = 8 * 3 * 3).
WORKLOADS["conv_gn_act_lse_128x8x128x128"] = Workload(
    "conv_gn_act_lse_128x8x128x128", "conv_gn_act_lse", (128, 8, 128, 128),
    "x ~ N(0,1) seed 6; w [64,8,3,3] and bias [64] ~ U[-1/sqrt(72), 1/sqrt(72)) seeds 106, 206; "
    "gamma ~ U[0.5,1.5) seed 105; beta ~ N(0,0.1) seed 205; G=16, eps=1e-5",
    {"seed": 6, "w_seed": 106, "bias_seed": 206, "gamma_seed": 105, "beta_seed": 205, "Cout": 64,
     "G": 16, "eps": 1e-5})


def make_inputs(w: Workload | str, device="cpu", shape=None):
    """Draw the inputs of a workload (optionally at another shape, same recipe).

    Returns a dict of tensors: {"x"} for lse_dim0 / log_softmax,
    {"y", "gamma", "beta"} for gn_act_lse."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    shape = tuple(shape) if shape is not None else w.shape
    p = w.params
    base = p.get("like", w.name.split("@")[0])
    if base == "lse_dim0_4x10x32":
        return {"x": normal(shape, p["seed"], device=device)}
    if base == "log_softmax_256x4096":
        x = normal(shape, p["seed"], var=4.0, device=device)
        mask = bernoulli_mask(shape, p["mask_seed"], p["p_ninf"], device=device)
        x.masked_fill_(mask, float("-inf"))
        if x.ndim == 2 and x.shape[1] > 0:
            all_ninf = torch.isneginf(x).all(dim=1)
            if bool(all_ninf.any()):
                raise RuntimeError("recipe produced an all -inf row; pick another seed")
        return {"x": x}
    if base == "lse_dim0_32x8192x4096":
        return {"x": uniform(shape, p["seed"], -20.0, 20.0, device=device)}
    if base == "log_softmax_4096x393216":
        return {"x": normal(shape, p["seed"], device=device)}
    if base == "conv_gn_act_lse_128x8x128x128":
        Cin, Cout = shape[1], p["Cout"]
        bound = 1.0 / math.sqrt(Cin * 9)
        return {
            "x": normal(shape, p["seed"], device=device),
            "w": uniform((Cout, Cin, 3, 3), p["w_seed"], -bound, bound, device=device),
            "bias": uniform((Cout,), p["bias_seed"], -bound, bound, device=device),
            "gamma": uniform((Cout,), p["gamma_seed"], 0.5, 1.5, device=device),
            "beta": normal((Cout,), p["beta_seed"], var=0.1, device=device),
        }
    if base == "gn_act_lse_128x64x126x126":
        C = shape[1]
        return {
            "y": normal(shape, p["seed"], device=device),
            "gamma": uniform((C,), p["gamma_seed"], 0.5, 1.5, device=device),
            "beta": normal((C,), p["beta_seed"], var=0.1, device=device),
        }
    raise KeyError(w.name)
