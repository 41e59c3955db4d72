"""The tile schedule changes no bit of the results.

Forward and backward outputs (SwiGLU and squared-ReLU experts) must be bitwise the same
whether the forward GEMMs run with swapped operands (weight columns x blocks of up to 256
rows, CTA pairs; MOE_FWD_SWAP=1), or as row tiles: 256-row tiles on CTA pairs for the experts
the tile tables pick and the rest on single CTAs (MOE_FWD_SWAP=0, MOE_GEMM_PAIR=1), or
128-row tiles on single CTAs only (MOE_GEMM_PAIR=0); the backward's row-grouped GEMMs follow
MOE_GEMM_PAIR or the library's size rule (unset).  The swapped GEMMs also run as one launch
(MOE_FWD_FUSED=1: GEMM2 of a row block after its GEMM1 tiles), the swapped GEMM1 copies the
permuted rows itself or leaves them to the dispatch (MOE_FWD_ROW_COPY=0), and the backward's dX and dH
GEMMs run swapped (MOE_BWD_SWAP=1; MOE_BWD_DH_SWAP for dH alone) or as row tiles ("0").  The forward variant that gathers GEMM1's
rows from x and fuses the combine into GEMM2 must match the default forward bitwise.  Each
schedule runs in its own process (the switches are read once per process).
"""
import hashlib
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu

_SCRIPT = r"""
import hashlib, sys
sys.path.insert(0, %(root)r)
sys.path.insert(0, %(root)r + "/tests")
import torch
import moe_synth
import combine_fp32_router_gb300 as moe
from moe_harness import forward, backward, to_dev
w = moe_synth.custom(T=3000, d=512, E=%(E)d, k=4, dff=%(dff)d, seed=77, zipf_s=1.2,
                     gated=%(gated)s)
inp = moe_synth.generate(w, with_dy=True)
g = to_dev(inp)
h = hashlib.sha256()
out, ws = forward(moe, g, w.k, save=True)
res = backward(moe, g, w.k, ws)
assert moe.moe_get_error(ws) == 0
for t in [out] + [res[k] for k in sorted(res) if res[k] is not None]:
    h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())
o2 = torch.empty_like(out)
moe.moe_forward(g["x"], g["logits"], g["W1"], g.get("W3"), g["W2"], w.k, o2, ws,
                flags=moe.MOE_FWD_GATHER_ROWS | moe.MOE_FWD_FUSED_COMBINE)
assert moe.moe_get_error(ws) == 0
assert torch.equal(o2.view(torch.int16), out.view(torch.int16))
print(h.hexdigest())
"""


def _digest(env_extra, gated=True, E=64):
    env = {k: v for k, v in os.environ.items()
           if k not in ("MOE_GEMM_PAIR", "MOE_FWD_SWAP", "MOE_FWD_FUSED", "MOE_BWD_SWAP",
                        "MOE_BWD_DH_SWAP", "MOE_FWD_ROW_COPY")}
    env.update(env_extra)
    script = _SCRIPT % {"root": ROOT, "gated": gated, "dff": 384 if gated else 512, "E": E}
    r = subprocess.run([sys.executable, "-c", script], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return r.stdout.strip().splitlines()[-1]


@pytest.mark.parametrize("gated", [True, False])   # SwiGLU, squared ReLU (no W3)
def test_schedule_does_not_change_results(gated):
    ref = _digest({"MOE_GEMM_PAIR": "1", "MOE_FWD_SWAP": "0"}, gated)
    assert _digest({"MOE_GEMM_PAIR": "1", "MOE_FWD_SWAP": "1"}, gated) == ref
    assert _digest({"MOE_GEMM_PAIR": "1", "MOE_FWD_SWAP": "1", "MOE_FWD_FUSED": "1"}, gated) == ref
    # the swapped GEMM1 copying the permuted rows itself, or the dispatch's scatter copying them
    assert _digest({"MOE_GEMM_PAIR": "1", "MOE_FWD_SWAP": "1", "MOE_FWD_ROW_COPY": "0"},
                   gated) == ref
    assert _digest({"MOE_GEMM_PAIR": "0"}, gated) == ref
    assert _digest({}, gated) == ref
    # the backward's dX and dH GEMMs with swapped operands (CTA pairs, one launch each) or as
    # row tiles, together and each alone
    assert _digest({"MOE_GEMM_PAIR": "1", "MOE_BWD_SWAP": "1"}, gated) == ref
    assert _digest({"MOE_GEMM_PAIR": "1", "MOE_BWD_SWAP": "0"}, gated) == ref
    assert _digest({"MOE_GEMM_PAIR": "1", "MOE_BWD_SWAP": "0", "MOE_BWD_DH_SWAP": "1"},
                   gated) == ref
    assert _digest({"MOE_GEMM_PAIR": "1", "MOE_BWD_SWAP": "1", "MOE_BWD_DH_SWAP": "0"},
                   gated) == ref


@pytest.mark.parametrize("gated", [True, False])
def test_wide_epilogue_gemm1_matches_row_tiles(gated):
    # 16 experts for 12000 token-expert pairs (P >= 256 E): the swapped GEMM1 runs its 8-warp
    # epilogue form; bitwise the row-tile kernels' rows
    ref = _digest({"MOE_GEMM_PAIR": "1", "MOE_FWD_SWAP": "0"}, gated, E=16)
    assert _digest({"MOE_GEMM_PAIR": "1", "MOE_FWD_SWAP": "1"}, gated, E=16) == ref
    assert _digest({"MOE_GEMM_PAIR": "1", "MOE_FWD_SWAP": "1", "MOE_FWD_ROW_COPY": "0"},
                   gated, E=16) == ref
    assert _digest({}, gated, E=16) == ref
