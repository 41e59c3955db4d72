"""The FP8 dispatch payload on the GPU against the oracle: the E4M3 weight copies and their
scales bitwise, the forward within the stated tolerance plus the oracle's rounding-flip
allowance of the bf16 h and output rows, batch invariance and run-to-run determinism bitwise,
and CTA-pair vs single-CTA schedules bitwise."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import moe_synth
import oracle
from moe_harness import assert_close_flip, np_of, sample_tokens, to_dev

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    import combine_fp32_router_gb300 as m
    return m


def _fp8_forward(moe, g, k, ws=None):
    x = g["x"]
    T, d = x.shape
    E, _, dff = g["W1"].shape
    W1q, s1 = moe.moe_quantize_weights_fp8(g["W1"])
    W3q, s3 = moe.moe_quantize_weights_fp8(g["W3"])
    if ws is None:
        ws = torch.empty(moe.moe_workspace_bytes(T, d, E, k, dff), dtype=torch.uint8,
                         device=x.device)
    out = torch.empty(T, d, dtype=torch.bfloat16, device=x.device)
    moe.moe_forward_fp8(x, g["logits"], W1q, W3q, s1, s3, g["W2"], k, out, ws)
    return out, ws


def test_weight_quantization_matches_oracle(moe):
    rng = np.random.default_rng(3)
    W = torch.from_numpy(rng.standard_normal((3, 256, 384)) / 16).to(torch.bfloat16)
    W[1, :, 5] = 0.0                                   # an all-zero column: scale 1
    Wq, sc = moe.moe_quantize_weights_fp8(W.cuda())
    q_ref, s_ref = oracle.quantize_cols_e4m3(W.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(sc.cpu().numpy().astype(np.float64), s_ref)
    got = Wq.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()     # [E, N, K]
    np.testing.assert_array_equal(got, q_ref.transpose(0, 2, 1))


@pytest.mark.parametrize("T,d,E,k,dff", [
    (64, 128, 8, 2, 256),      # tiny shape
    (300, 256, 16, 4, 384),    # ragged tiles, pair + leftover launches
    (77, 384, 5, 3, 128),      # d % 256 != 0 (128-wide GEMM2 tiles)
    (513, 128, 1, 1, 128),     # one expert
    (200, 128, 64, 2, 256),    # many empty experts
])
def test_fp8_forward_matches_oracle(moe, T, d, E, k, dff):
    w = moe_synth.custom(T, d, E, k, dff, seed=T * 3 + d)
    inp = moe_synth.generate(w)
    out, ws = _fp8_forward(moe, to_dev(inp), k)
    assert moe.moe_get_error(ws) == 0
    ref, allow = oracle.forward_tokens_fp8_flip(moe_synth.to_numpy(inp), k)
    assert_close_flip(np_of(out), ref, allow, "out (fp8)")


def test_fp8_batch_invariance_and_determinism(moe):
    w = moe_synth.custom(400, 256, 16, 4, 256, seed=21)
    g = to_dev(moe_synth.generate(w))
    full, ws = _fp8_forward(moe, g, w.k)
    for _ in range(3):
        again, _ = _fp8_forward(moe, g, w.k, ws=ws)
        assert torch.equal(again.view(torch.int16), full.view(torch.int16))
    for T in (1, 3, 64, 129, 255):
        part, _ = _fp8_forward(moe, moe_synth.rows(g, T), w.k)
        assert torch.equal(part.view(torch.int16), full[:T].view(torch.int16)), T


_SCRIPT = r"""
import hashlib, sys
sys.path.insert(0, %(root)r)
sys.path.insert(0, %(root)r + "/tests")
import torch
import moe_synth
import combine_fp32_router_gb300 as moe
from moe_harness import to_dev
from test_gpu_fp8 import _fp8_forward
w = moe_synth.custom(T=3000, d=512, E=64, k=4, dff=384, seed=78, zipf_s=1.2)
g = to_dev(moe_synth.generate(w))
out, ws = _fp8_forward(moe, g, w.k)
assert moe.moe_get_error(ws) == 0
print(hashlib.sha256(out.view(torch.uint8).cpu().numpy().tobytes()).hexdigest())
"""


def _digest(env_extra):
    env = dict(os.environ)
    env.update(env_extra)
    r = subprocess.run([sys.executable, "-c", _SCRIPT % {"root": ROOT}], env=env,
                       capture_output=True, text=True, timeout=600, cwd=os.path.join(ROOT, "tests"))
    assert r.returncode == 0, r.stderr[-3000:]
    return r.stdout.strip().splitlines()[-1]


def test_fp8_schedule_does_not_change_results():
    # single CTAs / CTA pairs with GEMM2 swapped / CTA pairs with row-tile GEMM2
    ref = _digest({"MOE_GEMM_PAIR": "0"})
    assert _digest({"MOE_GEMM_PAIR": "1"}) == ref
    assert _digest({"MOE_GEMM_PAIR": "1", "MOE_FWD_SWAP": "0"}) == ref


def test_fp8_large_workload_sampled(moe):
    w = moe_synth.by_name("large_skewed")
    g = moe_synth.generate(w, device="cuda")
    out, ws = _fp8_forward(moe, g, w.k)
    assert moe.moe_get_error(ws) == 0
    npi = moe_synth.to_numpy(g)
    tok = sample_tokens(w.T, 6, seed=5)
    ref, allow = oracle.forward_tokens_fp8_flip(npi, w.k, tokens=tok)
    assert_close_flip(np_of(out)[tok], ref, allow, "out (fp8, large workload, sampled tokens)")


@pytest.mark.parametrize("T", [5, 200])   # single dispatch launch for moe_forward / five kernels
def test_every_forward_clears_the_error_record(moe, T):
    # a workspace full of stale bytes: each forward entry point starts from a clean record
    w = moe_synth.custom(T, 128, 8, 2, 256, seed=T + 11)
    g = to_dev(moe_synth.generate(w))
    ws = torch.full((moe.moe_workspace_bytes(T, 128, 8, 2, 256),), 0x7F, dtype=torch.uint8,
                    device=g["x"].device)
    out = torch.empty(T, 128, dtype=torch.bfloat16, device=g["x"].device)
    moe.moe_forward(g["x"], g["logits"], g["W1"], g["W3"], g["W2"], 2, out, ws)
    assert moe.moe_get_error(ws) == moe.MOE_OK
    ws.fill_(0x7F)
    _fp8_forward(moe, g, 2, ws=ws)
    assert moe.moe_get_error(ws) == moe.MOE_OK
