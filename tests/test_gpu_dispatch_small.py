"""The single-launch dispatch of small batches (T <= 128) in moe_forward.

moe_forward does the whole dispatch of a batch of at most 128 tokens in one launch: route,
count, scan, tile tables, stable permute and row copies.  The test hook
moe_debug_set_flags(2) makes it use the multi-kernel sequence of larger batches instead.

The two must leave bitwise the same output and workspace. The only region excluded is the
multi-kernel path's per-block histogram scratch (the error record, histogram and block bases
at the start of the workspace). The output must also meet the oracle's bound."""
import numpy as np
import pytest
import torch

import moe_synth
from moe_harness import check_forward, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import combine_fp32_router_gb300 as m
    return m


def _run(moe, g, k, flags, debug):
    x = g["x"]
    T, d = x.shape
    E, _, dff = g["W1"].shape
    ws = torch.zeros(moe.moe_workspace_bytes(T, d, E, k, dff, True), dtype=torch.uint8,
                     device=x.device)
    out = torch.zeros(T, d, dtype=torch.bfloat16, device=x.device)
    moe.moe_debug_set_flags(debug)
    try:
        moe.moe_forward(x, g["logits"], g["W1"], g.get("W3"), g["W2"], k, out, ws, flags=flags)
        torch.cuda.synchronize()
    finally:
        moe.moe_debug_set_flags(0)
    assert moe.moe_get_error(ws) == moe.MOE_OK
    return out, ws


def _scratch_end(E):
    # error record (256 bytes), then the histogram and block bases of one routing block
    return 256 + 2 * ((E * 4 + 255) // 256 * 256)


@pytest.mark.parametrize("T,d,E,k,dff", [
    (1, 256, 8, 2, 256),
    (37, 384, 33, 3, 256),      # two logits per lane, ragged expert count
    (128, 256, 256, 8, 256),    # the largest batch of the single launch
    (100, 128, 1000, 16, 128),  # 32 logits per lane, the largest k
    (90, 128, 100, 5, 128),     # 4 logits per lane
    (33, 128, 300, 6, 128),     # 16 logits per lane
    (64, 256, 1, 1, 256),       # one expert
])
@pytest.mark.parametrize("flags", [0, 1, 4])  # plain, save for backward, row gather
def test_small_dispatch_equals_multi_kernel_dispatch(moe, T, d, E, k, dff, flags):
    w = moe_synth.custom(T, d, E, k, dff, seed=T * 31 + E, zipf_s=1.2)
    inp = moe_synth.generate(w)
    g = to_dev(inp)
    out1, ws1 = _run(moe, g, k, flags, 0)
    out2, ws2 = _run(moe, g, k, flags, 2)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    s = _scratch_end(E)
    diff = (ws1[s:] != ws2[s:]).nonzero()
    assert diff.numel() == 0, f"workspace differs from byte {s + int(diff[0])}"
    check_forward(out1, moe_synth.to_numpy(inp), k, "out (single-launch dispatch)")


def test_small_dispatch_at_the_size_limit_boundary(moe):
    # T = 128 takes the single launch, T = 129 the multi-kernel sequence: both against the oracle
    for T in (128, 129):
        w = moe_synth.custom(T, 256, 16, 4, 256, seed=900 + T, zipf_s=1.2)
        inp = moe_synth.generate(w)
        out, _ = _run(moe, to_dev(inp), 4, 0, 0)
        check_forward(out, moe_synth.to_numpy(inp), 4, f"out T={T}")
