"""Host-side logic of bench.py, on the CPU: the algorithmic FLOP and byte counts behind the
reported roofline fractions, and the launch counts that follow the library's rule for CTA
pairs (MOE_GEMM_PAIR: "0" never, "1" whenever T > 128, unset T > 128 and T k d d_ff >= 2^37) and
for the swapped-operand kinds (T <= 128, wherever row tiles pair, and from T k d d_ff >= 2^36).
"""
import pytest

import moe_synth


@pytest.fixture(scope="module")
def bench():
    import bench as b
    return b


def test_algorithmic_counts_of_the_large_workload(bench, monkeypatch):
    w = moe_synth.by_name("large_skewed")
    P = w.T * w.k
    a = bench._algorithmic(w, P)
    # SwiGLU expert: gate, up and down projections, 2 FLOP per multiply-add each, i.e. 6 d d_ff
    # per token-expert pair (report translation, section 1.4)
    assert a["gemm_flops"] == 6 * w.d * w.dff * P
    assert a["gemm1_flops"] + a["gemm2_flops"] == a["gemm_flops"]
    assert abs(a["gemm_flops"] / 1e12 - 11.545) < 5e-4
    # dispatch: logits read (fp32), 16 B of routing results per pair, x read and x_perm written
    assert a["dispatch_bytes"] == w.T * w.E * 4 + P * 16 + w.T * w.d * 2 + P * w.d * 2
    assert abs(a["dispatch_bytes"] / 1e9 - 2.133) < 5e-4
    # the routing part alone, when GEMM1 copies the rows (the default above T = 128)
    assert a["dispatch_route_bytes"] == w.T * w.E * 4 + P * 16
    monkeypatch.delenv("MOE_FWD_ROW_COPY", raising=False)
    monkeypatch.delenv("MOE_FWD_SWAP", raising=False)
    monkeypatch.delenv("MOE_GEMM_PAIR", raising=False)
    monkeypatch.delenv("MOE_FWD_FUSED", raising=False)
    assert bench._gemm_row_copy(w.T, w.k, w.d, w.dff)
    assert not bench._gemm_row_copy(128, w.k, w.d, w.dff)
    monkeypatch.setenv("MOE_FWD_ROW_COPY", "0")
    assert not bench._gemm_row_copy(w.T, w.k, w.d, w.dff)
    # combine: bf16 expert rows read, gate + pos read, bf16 output written
    assert a["combine_bytes"] == P * w.d * 2 + P * 8 + w.T * w.d * 2
    assert abs(a["combine_bytes"] / 1e9 - 2.115) < 5e-4


def test_algorithmic_counts_without_the_gate_projection(bench):
    w = moe_synth.by_name("large_skewed_relu2")
    P = w.T * w.k
    a = bench._algorithmic(w, P)
    assert a["gemm_flops"] == 4 * w.d * w.dff * P
    assert a["gemm1_flops"] == a["gemm2_flops"] == 2 * w.d * w.dff * P


@pytest.mark.parametrize("mode,name,pairs", [
    (None, "large_skewed", True),    # T k d d_ff = 1.9e12
    (None, "fwd_bwd", True),         # 4.1e11
    (None, "mid", False),            # 5.2e10 < 2^37
    (None, "tiny", False),           # T = 64 <= 128
    ("0", "large_skewed", False),
    ("1", "mid", True),
    ("1", "tiny", False),            # no expert can fill a pair tile
])
def test_pair_rule_and_launch_counts(bench, monkeypatch, mode, name, pairs):
    if mode is None:
        monkeypatch.delenv("MOE_GEMM_PAIR", raising=False)
    else:
        monkeypatch.setenv("MOE_GEMM_PAIR", mode)
    w = moe_synth.by_name(name)
    assert bench._row_pairs(w.T, w.k, w.d, w.dff) == pairs
    # the backward's row-grouped GEMMs add a single-CTA launch beside each pair launch; the
    # forward's swapped GEMMs (wherever row tiles would pair, and T <= 128) are one launch
    # each; a batch of T <= 128 is dispatched in one launch instead of five
    small = w.T <= 128
    monkeypatch.setenv("MOE_FWD_SWAP", "0")
    assert bench.fwd_launches(w.T, w.k, w.d, w.dff) == (10 if pairs else (4 if small else 8))
    monkeypatch.delenv("MOE_FWD_SWAP")
    assert bench._forward_swap(w.T, w.k, w.d, w.dff) == (mode != "0" and (pairs or small))
    # T <= 64: both swapped GEMMs in one launch
    fused = mode != "0" and w.T <= 64
    expect = (3 if fused else 4) if small else 8
    assert bench.fwd_launches(w.T, w.k, w.d, w.dff) == expect
    # saving for the backward adds the zeroing of the padding rows to the single dispatch
    assert bench.fwd_launches(w.T, w.k, w.d, w.dff, save=True) == expect + (1 if small else 0)
    # the backward's dH and dX run swapped (one launch each) wherever the forward's GEMMs
    # would; MOE_BWD_DH_SWAP overrides the rule for dH alone
    monkeypatch.setenv("MOE_BWD_SWAP", "0")
    assert bench.bwd_launches(w.T, w.k, w.d, w.dff) == (10 if pairs else 8)
    monkeypatch.setenv("MOE_BWD_DH_SWAP", "1")
    assert bench.bwd_launches(w.T, w.k, w.d, w.dff) == (9 if pairs else 8)
    monkeypatch.delenv("MOE_BWD_DH_SWAP")
    monkeypatch.delenv("MOE_BWD_SWAP")
    assert bench.bwd_launches(w.T, w.k, w.d, w.dff) == 8


@pytest.mark.parametrize("T,d,E,k,dff,swap", [
    (2048, 4096, 32, 8, 1536, True),    # 1.03e11: swapped, row tiles on single CTAs
    (1024, 4096, 64, 8, 1536, False),   # 5.2e10 < 2^36
    (4096, 2048, 64, 6, 1024, False),   # 5.2e10 (the mid workload)
    (128, 128, 8, 2, 128, True),        # T <= 128
])
def test_swap_size_rule_between_the_thresholds(bench, monkeypatch, T, d, E, k, dff, swap):
    # the swapped kinds start at T k d d_ff = 2^36, half the row-tile pair threshold
    for v in ("MOE_GEMM_PAIR", "MOE_FWD_SWAP", "MOE_BWD_SWAP", "MOE_BWD_DH_SWAP"):
        monkeypatch.delenv(v, raising=False)
    assert bench._forward_swap(T, k, d, dff) == swap
    assert bench._backward_swap(T, k, d, dff) == swap
    if T > 128:
        assert not bench._row_pairs(T, k, d, dff)
        assert bench.fwd_launches(T, k, d, dff) == 5 + 2 + 1
    # MOE_GEMM_PAIR "1" pairs every size above T = 128 and swaps with it; "0" never swaps
    monkeypatch.setenv("MOE_GEMM_PAIR", "1")
    assert bench._forward_swap(T, k, d, dff)
    monkeypatch.setenv("MOE_GEMM_PAIR", "0")
    assert not bench._forward_swap(T, k, d, dff)
