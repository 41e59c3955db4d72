"""The expert without the gate projection (W3 absent: h = relu(x W1)^2, the cheap element-wise
activation) on the GPU against the oracle: forward and backward parity, batch invariance and
run-to-run determinism, as for the SwiGLU expert."""
import numpy as np
import pytest
import torch

import moe_synth
import oracle
from moe_harness import (backward, check_backward, check_forward, forward, np_of,
                         sample_tokens, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import combine_fp32_router_gb300 as m
    return m


def _w(T, d, E, k, dff, seed):
    return moe_synth.custom(T, d, E, k, dff, seed=seed, gated=False)


@pytest.mark.parametrize("T,d,E,k,dff", [
    (64, 128, 8, 2, 256),      # tiny shape
    (300, 256, 16, 4, 512),    # ragged tiles, pair + leftover launches
    (77, 384, 5, 3, 256),      # d % 256 != 0 (128-wide GEMM2 tiles)
    (513, 128, 1, 1, 256),     # one expert: a dense squared-ReLU MLP
    (200, 128, 64, 2, 256),    # many empty experts
])
def test_relu2_forward_matches_oracle(moe, T, d, E, k, dff):
    w = _w(T, d, E, k, dff, seed=T + d)
    inp = moe_synth.generate(w)
    assert "W3" not in inp
    g = to_dev(inp)
    out, ws = forward(moe, g, k)
    assert moe.moe_get_error(ws) == 0
    check_forward(out, moe_synth.to_numpy(inp), k, "out (relu2)")


@pytest.mark.parametrize("T,d,E,k,dff", [
    (64, 128, 8, 2, 256),
    (300, 256, 16, 4, 512),
    (77, 384, 5, 3, 256),
])
def test_relu2_backward_matches_oracle(moe, T, d, E, k, dff):
    w = _w(T, d, E, k, dff, seed=3 * T + d)
    inp = moe_synth.generate(w, with_dy=True)
    g = to_dev(inp)
    _, ws = forward(moe, g, k, save=True)
    res = backward(moe, g, k, ws)
    assert moe.moe_get_error(ws) == 0 and res["dW3"] is None
    npi = moe_synth.to_numpy(inp)
    used = check_backward(res, npi, k, " (relu2)")
    print("relu2 backward: elements that needed the flip allowance:", used)


def test_relu2_batch_invariance_and_determinism(moe):
    w = _w(400, 256, 16, 4, 512, seed=11)
    inp = moe_synth.generate(w, with_dy=True)
    g = to_dev(inp)
    full, _ = forward(moe, g, w.k)
    for T in (1, 3, 64, 129, 255):
        part, _ = forward(moe, moe_synth.rows(g, T), w.k)
        assert torch.equal(part.view(torch.int16), full[:T].view(torch.int16)), T
    out0, ws = forward(moe, g, w.k, save=True)
    ref = backward(moe, g, w.k, ws)
    for _ in range(3):
        out1, _ = forward(moe, g, w.k, save=True, ws=ws)
        res = backward(moe, g, w.k, ws)
        assert torch.equal(out1.view(torch.int16), out0.view(torch.int16))
        for kk, v in res.items():
            if v is None:
                continue
            a = v.view(torch.int16) if v.dtype == torch.bfloat16 else v.view(torch.int32)
            b = ref[kk].view(torch.int16) if v.dtype == torch.bfloat16 else ref[kk].view(torch.int32)
            assert torch.equal(a, b), kk


def test_relu2_rejects_d_ff_not_multiple_of_256(moe):
    w = _w(64, 128, 8, 2, 384, seed=1)
    g = to_dev(moe_synth.generate(w))
    with pytest.raises(moe.MoeError) as e:
        forward(moe, g, w.k)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED


def test_relu2_large_workload_sampled(moe):
    # T=16384, d=7168, E=256, top-8, d_ff=3072 (the same parameter budget as the SwiGLU
    # layer), Zipf(1.2)-biased logits
    w = moe_synth.by_name("large_skewed_relu2")
    g = moe_synth.generate(w, device="cuda")
    out, ws = forward(moe, g, w.k)
    assert moe.moe_get_error(ws) == 0
    npi = moe_synth.to_numpy(g)
    tok = sample_tokens(w.T, 16, seed=4)
    check_forward(out, npi, w.k, "out (large relu2, sampled tokens)", tokens=tok)
