"""Seeded synthetic inputs for the MoE expert layer.

This module only draws random numbers and names workload shapes; it holds none of the
layer's arithmetic.  Both the CUDA path's tests/benchmark and the CPU oracle take their
inputs from here.

Recipe (every config): a ``torch.Generator`` seeded with ``1000 + config index`` draws, in
this order, x ~ N(0,1), router logits ~ N(0,1) (fp32), W1 and W3 ~ N(0, 1/sqrt(d)) as
[E, d, dff], W2 ~ N(0, 1/sqrt(dff)) as [E, dff, d], and (when asked) the upstream gradient
dY ~ N(0,1).  x, W and dY are rounded to bf16 (round to nearest even); logits stay fp32.
The large skewed workload adds a per-expert bias -1.2 * ln(e + 1) to the logits, a
Zipf(s = 1.2) popularity law over expert rank e + 1.
"""
from dataclasses import dataclass, field
import math

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    dff: int
    zipf_s: float = 0.0          # 0: no bias; else logits += -s * ln(e + 1)
    seed: int = 1000
    sweep: tuple = field(default=())   # token counts of a batch-invariance sweep
    gated: bool = True           # False: no W3 (squared-ReLU expert, d_ff = 1.5x for the
                                 # same parameter count)

    @property
    def pairs(self) -> int:
        return self.T * self.k


# The five workloads of the benchmark suite (tiny, mid, small-batch sweep, large skewed,
# forward+backward), with seed 1000 + position.
WORKLOADS = [
    Workload("tiny", T=64, d=128, E=8, k=2, dff=256, seed=1000),
    Workload("mid", T=4096, d=2048, E=64, k=6, dff=1024, seed=1001),
    Workload("sweep", T=128, d=7168, E=256, k=8, dff=2048, seed=1002,
             sweep=(1, 2, 4, 8, 16, 32, 64, 128)),
    Workload("large_skewed", T=16384, d=7168, E=256, k=8, dff=2048, zipf_s=1.2, seed=1003),
    Workload("fwd_bwd", T=8192, d=4096, E=128, k=8, dff=1536, seed=1004),
    # the large skewed layer with the cheap activation: the same parameter budget (two
    # projections of d_ff = 3072 instead of three of 2048)
    Workload("large_skewed_relu2", T=16384, d=7168, E=256, k=8, dff=3072, zipf_s=1.2,
             seed=1005, gated=False),
]


def by_name(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def custom(T, d, E, k, dff, seed=7, zipf_s=0.0, name="custom", gated=True) -> Workload:
    return Workload(name, T=T, d=d, E=E, k=k, dff=dff, zipf_s=zipf_s, seed=seed, gated=gated)


def generate(w: Workload, device="cpu", with_dy=False):
    """Draw the inputs of workload ``w`` on ``device``.

    Returns a dict of torch tensors: x [T,d] bf16, logits [T,E] fp32, W1/W3 [E,d,dff] bf16,
    W2 [E,dff,d] bf16 and, if ``with_dy``, dy [T,d] bf16.  The same seed on the same device
    type gives the same tensors.
    """
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)

    def randn(*shape, std=1.0):
        t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        return t

    out = {}
    out["x"] = randn(w.T, w.d).to(torch.bfloat16)
    logits = randn(w.T, w.E)
    if w.zipf_s:
        bias = -w.zipf_s * torch.log(torch.arange(1, w.E + 1, dtype=torch.float64))
        logits += bias.to(torch.float32).to(device)
    out["logits"] = logits
    out["W1"] = _randn_bf16(randn, (w.E, w.d, w.dff), 1.0 / math.sqrt(w.d))
    if w.gated:
        out["W3"] = _randn_bf16(randn, (w.E, w.d, w.dff), 1.0 / math.sqrt(w.d))
    out["W2"] = _randn_bf16(randn, (w.E, w.dff, w.d), 1.0 / math.sqrt(w.dff))
    if with_dy:
        out["dy"] = randn(w.T, w.d).to(torch.bfloat16)
    return out


def _randn_bf16(randn, shape, std):
    # Drawn expert by expert so the fp32 staging buffer stays small for the large workloads.
    E = shape[0]
    first = randn(*shape[1:], std=std).to(torch.bfloat16)
    out = torch.empty(shape, dtype=torch.bfloat16, device=first.device)
    out[0] = first
    for e in range(1, E):
        out[e] = randn(*shape[1:], std=std).to(torch.bfloat16)
    return out


def rows(inp, T):
    """The first ``T`` tokens of a drawn batch (x and logits; weights shared), used by the
    batch-invariance sweep."""
    out = dict(inp)
    out["x"] = inp["x"][:T].contiguous()
    out["logits"] = inp["logits"][:T].contiguous()
    if "dy" in inp:
        out["dy"] = inp["dy"][:T].contiguous()
    return out


def to_numpy(inp):
    """bf16 tensors as raw uint16 numpy arrays, fp32 as float32 numpy arrays (host copies)."""
    import numpy as np
    out = {}
    for key, t in inp.items():
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            out[key] = t.view(torch.int16).numpy().view(np.uint16)
        else:
            out[key] = t.numpy()
    return out
