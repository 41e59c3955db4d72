"""Backward of the layer on the GPU (moe_backward through the C ABI) against the oracle, and
run-to-run bitwise determinism of forward + backward.

Bar: every gradient element meets the stated bound |g - g_ref| <= 2e-2 |g_ref| + 2e-3 widened
by the oracle's rounding-flip allowance for that element (moe_harness.assert_close_flip): the
largest change that bf16 operands (h, dO, da, db) which may round the other way in fp32
arithmetic can cause there, derived from oracle values alone.  The tiny workload also meets
the stated bound alone."""
import numpy as np
import pytest
import torch

import moe_synth
import oracle
from moe_harness import (assert_close, backward, check_backward, check_forward, forward, np_of,
                         sample_tokens, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import combine_fp32_router_gb300 as m
    return m


def _run(moe, g, k):
    _, ws = forward(moe, g, k, save=True)
    res = backward(moe, g, k, ws)
    assert moe.moe_get_error(ws) == 0
    return res


def _check_all(moe, w, experts=None, plain=False):
    inp = moe_synth.generate(w, with_dy=True)
    g = to_dev(inp)
    res = _run(moe, g, w.k)
    npi = moe_synth.to_numpy(inp)
    used = check_backward(res, npi, w.k, experts=experts)
    print("%s: elements that needed the flip allowance: %s" % (w.name, used))
    if plain:  # the stated bound alone
        dx, dgate, dlog = oracle.backward_tokens(npi, npi["dy"], w.k)
        assert_close(np_of(res["dx"]), dx, "dx")
        assert_close(np_of(res["dgate"]), dgate, "dgate")
        assert_close(np_of(res["dlogits"]), dlog, "dlogits")
        r1, r3, r2 = oracle.backward_dw(npi, npi["dy"], w.k, np.arange(w.E))
        assert_close(np_of(res["dW1"]), r1, "dW1")
        assert_close(np_of(res["dW3"]), r3, "dW3")
        assert_close(np_of(res["dW2"]), r2, "dW2")


def test_backward_tiny_workload(moe):
    _check_all(moe, moe_synth.by_name("tiny"), plain=True)


@pytest.mark.parametrize("T,d,E,k,dff", [
    (300, 256, 16, 4, 384),   # ragged tiles, 128-wide dH tiles (dff % 256 != 0)
    (77, 384, 5, 3, 128),     # 128-wide dX / dW2 tiles (d % 256 != 0)
    (200, 128, 64, 2, 256),   # many experts with no rows: their dW must be exactly 0
])
def test_backward_small_shapes(moe, T, d, E, k, dff):
    _check_all(moe, moe_synth.custom(T, d, E, k, dff, seed=T + 3 * d))


def test_backward_empty_experts_are_zero(moe):
    w = moe_synth.custom(T=50, d=128, E=64, k=1, dff=128, seed=4)
    inp = moe_synth.generate(w, with_dy=True)
    g = to_dev(inp)
    res = _run(moe, g, w.k)
    idx, _ = oracle.route(inp["logits"].numpy(), w.k)
    unused = np.setdiff1d(np.arange(w.E), idx.reshape(-1))
    assert len(unused) > 0
    for name in ("dW1", "dW3", "dW2"):
        assert (res[name][torch.from_numpy(unused).cuda()] == 0).all()


def test_fwd_bwd_workload_sampled_and_deterministic(moe):
    # T=8192, d=4096, E=128, top-8, dff=1536: 10 identical runs, bitwise
    w = moe_synth.by_name("fwd_bwd")
    g = moe_synth.generate(w, device="cuda", with_dy=True)
    out0, ws = forward(moe, g, w.k, save=True)
    res0 = backward(moe, g, w.k, ws)
    assert moe.moe_get_error(ws) == 0
    ref = {kk: v.clone() for kk, v in res0.items()}
    ref["out"] = out0.clone()
    for _ in range(9):
        out, _ = forward(moe, g, w.k, save=True, ws=ws)
        res = backward(moe, g, w.k, ws)
        assert torch.equal(out.view(torch.int16), ref["out"].view(torch.int16))
        for kk, v in res.items():
            a = v.view(torch.int16) if v.dtype == torch.bfloat16 else v.view(torch.int32)
            b = ref[kk].view(torch.int16) if v.dtype == torch.bfloat16 else ref[kk].view(torch.int32)
            assert torch.equal(a, b), kk
    assert moe.moe_get_error(ws) == 0
    npi = moe_synth.to_numpy(g)
    tok = sample_tokens(w.T, 64, seed=2)
    check_forward(ref["out"], npi, w.k, "out (fwd_bwd, sampled tokens)", tokens=tok)
    # weight gradients of 10 experts: the most and the least loaded non-empty experts, and 8
    # drawn at random
    counts = np.bincount(oracle.route(npi["logits"], w.k)[0].reshape(-1), minlength=w.E)
    hot, cold = int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30)))
    rng = np.random.default_rng(5)
    ex = np.unique(np.concatenate([[hot, cold], rng.choice(w.E, 8, replace=False)]))
    assert len(ex) >= 8 and counts[ex].min() > 0
    used = check_backward(ref, npi, w.k, " (fwd_bwd)", tokens=tok, experts=ex)
    exl = ex.tolist()
    print("fwd_bwd: elements that needed the flip allowance:", used,
          "experts", exl, "rows", counts[ex].tolist())
