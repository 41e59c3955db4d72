"""Forward (saving for the backward) and backward of seeded random layer shapes against the
oracle, element by element: T above the single-launch dispatch (129..700), d in 128..512,
1..40 experts, top-1..8, d_ff of 128, 256 or 384 (256 or 512 without the gate projection),
uniform or Zipf-skewed logits.  Each schedule runs in its own process (the switches are read
once per process): the library's choice, and the swapped kinds forced on (CTA pairs, the
row copy inside GEMM1, swapped dX and dH; or swapped dH with row-tile dX).  Larger layers
(T 700..2000, d up to 1024, up to 100 experts, top-10) are checked on 96 sampled tokens and
8 experts' weight gradients."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu

_SCRIPT = r"""
import random, sys
sys.path.insert(0, %(root)r)
sys.path.insert(0, %(root)r + "/tests")
import moe_synth
import combine_fp32_router_gb300 as moe
from moe_harness import forward, backward, to_dev, check_forward, check_backward
rng = random.Random(%(seed)d)
for i in range(%(n)d):
    if %(big)d:
        T = rng.randint(700, 2000)
        d = rng.choice([512, 768, 1024])
        E = rng.choice([16, 40, 64, 100])
        k = rng.randint(1, min(E, 10))
    else:
        T = rng.randint(129, 700)
        d = rng.choice([128, 256, 384, 512])
        E = rng.choice([1, 2, 3, 5, 8, 13, 16, 24, 40])
        k = rng.randint(1, min(E, 8))
    gated = rng.random() < 0.8
    dff = rng.choice([128, 256, 384]) if gated else rng.choice([256, 512])
    zipf = rng.choice([0.0, 1.2])
    w = moe_synth.custom(T, d, E, k, dff, seed=%(seed)d * 100 + i, zipf_s=zipf, gated=gated)
    inp = moe_synth.generate(w, with_dy=True)
    g = to_dev(inp)
    out, ws = forward(moe, g, k, save=True)
    res = backward(moe, g, k, ws)
    assert moe.moe_get_error(ws) == 0
    npi = moe_synth.to_numpy(inp)
    tag = " T=%%d d=%%d E=%%d k=%%d dff=%%d gated=%%s zipf=%%.1f" %% (T, d, E, k, dff, gated, zipf)
    # larger layers: sampled tokens, and the weight gradients of the first, the last and 6
    # random experts
    tok = sorted(rng.sample(range(T), 96)) if %(big)d else None
    ex = sorted(set([0, E - 1] + rng.sample(range(E), 6))) if %(big)d else None
    check_forward(out, npi, k, "out" + tag, tokens=tok)
    check_backward(res, npi, k, tag, tokens=tok, experts=ex)
print("ok")
"""

_KEYS = ("MOE_GEMM_PAIR", "MOE_FWD_SWAP", "MOE_FWD_FUSED", "MOE_BWD_SWAP", "MOE_BWD_DH_SWAP",
         "MOE_FWD_ROW_COPY")


@pytest.mark.parametrize("seed,env,big", [
    (11, {}, 0),
    (12, {"MOE_GEMM_PAIR": "1", "MOE_FWD_SWAP": "1", "MOE_BWD_SWAP": "1"}, 0),
    (13, {"MOE_GEMM_PAIR": "1", "MOE_FWD_SWAP": "1", "MOE_BWD_SWAP": "0", "MOE_BWD_DH_SWAP": "1"},
     0),
    (14, {}, 1),
    (15, {"MOE_GEMM_PAIR": "1", "MOE_FWD_SWAP": "1", "MOE_BWD_SWAP": "1"}, 1),
])
def test_random_shapes_match_the_oracle(seed, env, big):
    e = {k: v for k, v in os.environ.items() if k not in _KEYS}
    e.update(env)
    script = _SCRIPT % {"root": ROOT, "seed": seed, "n": 8, "big": big}
    r = subprocess.run([sys.executable, "-c", script], env=e, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    assert r.stdout.strip().splitlines()[-1] == "ok"
