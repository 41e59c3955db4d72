"""Dispatch on the GPU (moe_route_dispatch through the C ABI) against the oracle.

Bar: top-k indices, counts, offsets, perm and pos bit-exact; x_perm bitwise; the fp32 gate
within a few fp32 ulps of the fp64 softmax (exp, sum and one division in fp32: relative
error well under 1e-5).
"""
import numpy as np
import pytest
import torch

import moe_synth
import oracle
from moe_harness import route_dispatch, to_dev

pytestmark = pytest.mark.gpu

GATE_RTOL, GATE_ATOL = 1e-5, 1e-7


@pytest.fixture(scope="module")
def moe():
    import combine_fp32_router_gb300 as m
    return m


def _check_route(moe, g, k):
    out = route_dispatch(moe, g, k)
    logits = g["logits"].cpu().numpy()
    E = logits.shape[1]
    idx, gate = oracle.route(logits, k)
    counts, offsets, perm, pos = oracle.dispatch(idx, E)
    np.testing.assert_array_equal(out["topk_idx"].cpu().numpy(), idx)
    np.testing.assert_array_equal(out["counts"].cpu().numpy(), counts)
    np.testing.assert_array_equal(out["offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(out["perm"].cpu().numpy(), perm)
    np.testing.assert_array_equal(out["pos"].cpu().numpy(), pos)
    np.testing.assert_allclose(out["gate"].cpu().numpy(), gate, rtol=GATE_RTOL, atol=GATE_ATOL)
    ref_rows = g["x"][torch.from_numpy(perm // k).long().to(g["x"].device)]
    assert torch.equal(out["x_perm"].view(torch.int16), ref_rows.view(torch.int16))
    return out


@pytest.mark.parametrize("T,E,k", [
    (64, 8, 2),        # tiny workload shape
    (300, 40, 5),      # ragged T (3 routing CTAs, last one partial), E not a multiple of 32
    (1, 256, 8),       # one token
    (129, 1, 1),       # one expert
    (257, 16, 16),     # k = E
    (1000, 1024, 16),  # largest E and k
    (4096, 64, 6),     # mid workload routing
])
def test_route_dispatch_matches_oracle(moe, T, E, k):
    w = moe_synth.custom(T=T, d=64, E=E, k=k, dff=128, seed=T + E)
    g = to_dev(moe_synth.generate(w))
    _check_route(moe, g, k)


def test_route_ties_and_signed_zero(moe):
    rng = np.random.default_rng(1)
    T, E, k = 500, 24, 4
    logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    logits[::7] = 0.0
    logits[::11, ::2] = -0.0
    x = torch.randn(T, 64).to(torch.bfloat16)
    g = to_dev({"x": x, "logits": torch.from_numpy(logits)})
    _check_route(moe, g, k)


def test_route_all_tokens_one_expert(moe):
    T, E, k = 700, 32, 2
    logits = torch.randn(T, E)
    logits[:, 5] += 100.0
    g = to_dev({"x": torch.randn(T, 128).to(torch.bfloat16), "logits": logits})
    out = _check_route(moe, g, k)
    assert out["counts"][5].item() == T


def test_route_large_skewed_workload(moe):
    # routing and permutation of the T = 16384, E = 256, top-8, Zipf(1.2)-biased workload
    w = moe_synth.by_name("large_skewed")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(w.seed)
    x = torch.randn(w.T, w.d, generator=gen, device="cuda").to(torch.bfloat16)
    logits = torch.randn(w.T, w.E, generator=gen, device="cuda")
    logits += (-w.zipf_s * torch.log(torch.arange(1, w.E + 1, dtype=torch.float64))).float().cuda()
    out = _check_route(moe, {"x": x, "logits": logits}, w.k)
    c = out["counts"].cpu().numpy()
    assert c.max() > 10 * c.mean()   # the skew is real


def test_route_zero_tokens(moe):
    g = to_dev({"x": torch.zeros(0, 64, dtype=torch.bfloat16), "logits": torch.zeros(0, 8)})
    out = route_dispatch(moe, g, 2)
    assert (out["counts"] == 0).all() and (out["offsets"] == 0).all()
