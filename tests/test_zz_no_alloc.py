"""moe_route_dispatch_noalloc: the dispatch entry point for callers that cannot allocate
device memory (a host framework that owns every allocation, serving loops where allocating is
not allowed, fixed device-memory budgets).  It must give the same outputs as
moe_route_dispatch, which takes a caller workspace, on consecutive calls that reuse its
built-in scratch, and must reject sizes beyond that scratch before launching anything.
"""
import numpy as np
import pytest
import torch

import moe_synth
from moe_harness import route_dispatch, to_dev

pytestmark = pytest.mark.gpu

GATE_RTOL, GATE_ATOL = 1e-5, 1e-7   # the routing tests' gate tolerance


def _noalloc(moe, g, k):
    x, logits = g["x"], g["logits"]
    T, d = x.shape
    E = logits.shape[1]
    dev = x.device
    out = dict(
        topk_idx=torch.full((T, k), -7, dtype=torch.int32, device=dev),
        gate=torch.full((T, k), -7.0, dtype=torch.float32, device=dev),
        counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
        offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        perm=torch.full((T * k,), -7, dtype=torch.int32, device=dev),
        pos=torch.full((T * k,), -7, dtype=torch.int32, device=dev),
        x_perm=torch.zeros(T * k, d, dtype=torch.bfloat16, device=dev),
    )
    moe.moe_route_dispatch_noalloc(x, logits, k, out["topk_idx"], out["gate"], out["counts"],
                                   out["offsets"], out["perm"], out["pos"], out["x_perm"])
    torch.cuda.synchronize()
    return out


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    import combine_fp32_router_gb300 as moe
    # two calls in a row with different sizes: the second reuses the scratch the first left
    for T, d, E, k, seed in [(3000, 256, 64, 6, 21), (777, 128, 40, 5, 22)]:
        g = to_dev(moe_synth.generate(moe_synth.custom(T, d, E, k, 128, seed=seed)))
        ref = route_dispatch(moe, g, k)
        got = _noalloc(moe, g, k)
        for key in ("topk_idx", "counts", "offsets", "perm", "pos"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["x_perm"].view(torch.int16), ref["x_perm"].view(torch.int16))
        np.testing.assert_allclose(got["gate"].cpu().numpy(), ref["gate"].cpu().numpy(),
                                   rtol=GATE_RTOL, atol=GATE_ATOL)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import combine_fp32_router_gb300 as moe
    T, E, k = 129 * 1024, 1024, 2     # ceil(T/128) * E = 1032192 > 262080
    g = {"x": torch.empty(T, 8, dtype=torch.bfloat16, device="cuda"),
         "logits": torch.empty(T, E, dtype=torch.float32, device="cuda")}
    with pytest.raises(moe.MoeError) as exc:
        _noalloc(moe, g, k)
    assert exc.value.status == moe.MOE_ERR_UNSUPPORTED


def test_noalloc_error_record_reads_ok_after_a_normal_call():
    import combine_fp32_router_gb300 as moe
    g = to_dev(moe_synth.generate(moe_synth.custom(500, 128, 16, 4, 128, seed=31)))
    _noalloc(moe, g, 4)
    assert moe.moe_route_dispatch_noalloc_get_error() == moe.MOE_OK


def test_noalloc_empty_batch_zeroes_counts_and_offsets():
    import combine_fp32_router_gb300 as moe
    E, k = 24, 3
    g = {"x": torch.empty(0, 128, dtype=torch.bfloat16, device="cuda"),
         "logits": torch.empty(0, E, dtype=torch.float32, device="cuda")}
    out = _noalloc(moe, g, k)
    assert (out["counts"] == 0).all() and (out["offsets"] == 0).all()
    assert moe.moe_route_dispatch_noalloc_get_error() == moe.MOE_OK


def test_noalloc_size_limit_is_exact():
    # ceil(T/128) * E <= 262080 is accepted (T = 273 * 128, E = 960 reaches it exactly) and
    # matches the workspace entry point; one more routing block is rejected
    import combine_fp32_router_gb300 as moe
    E, k, d = 960, 2, 8
    T = 273 * 128
    assert (T + 127) // 128 * E == 262080
    w = moe_synth.custom(T, d, E, k, 128, seed=41)
    g = to_dev(moe_synth.generate(w))
    ref = route_dispatch(moe, g, k)
    got = _noalloc(moe, g, k)
    for key in ("topk_idx", "counts", "offsets", "perm", "pos"):
        assert torch.equal(got[key], ref[key]), key
    assert torch.equal(got["x_perm"].view(torch.int16), ref["x_perm"].view(torch.int16))
    assert moe.moe_route_dispatch_noalloc_get_error() == moe.MOE_OK
    big = {"x": torch.zeros(T + 1, d, dtype=torch.bfloat16, device="cuda"),
           "logits": torch.zeros(T + 1, E, dtype=torch.float32, device="cuda")}
    with pytest.raises(moe.MoeError) as exc:
        _noalloc(moe, big, k)
    assert exc.value.status == moe.MOE_ERR_UNSUPPORTED
