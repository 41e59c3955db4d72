"""Failure detection on the GPU without a GPU fault: a bounded device-side wait that runs
out must come back as MOE_ERR_TIMEOUT, and the context must stay usable afterwards.

The test hook (moe_debug_set_flags bit 0) makes the first CTA of each grouped-GEMM launch
skip its first operand load, so the matching wait can never complete; the wait limit is
lowered to 50 ms for the duration of the test.
"""
import pytest
import torch

import moe_synth
from moe_harness import forward, to_dev

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    import combine_fp32_router_gb300 as moe
    w = moe_synth.by_name("tiny")
    g = to_dev(moe_synth.generate(w))
    ref, ws = forward(moe, g, w.k)
    assert moe.moe_get_error(ws) == moe.MOE_OK
    try:
        moe.moe_set_wait_timeout_ns(50_000_000)
        moe.moe_debug_set_flags(1)
        forward(moe, g, w.k, ws=ws)
        assert moe.moe_get_error(ws) == moe.MOE_ERR_TIMEOUT
    finally:
        moe.moe_debug_set_flags(0)
        moe.moe_set_wait_timeout_ns(2_000_000_000)
    out, _ = forward(moe, g, w.k, ws=ws)
    assert moe.moe_get_error(ws) == moe.MOE_OK
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
