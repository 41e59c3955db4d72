"""Pins of the oracle's rounding-flip allowance (CPU only).

The oracle and an fp32 implementation both round h, the expert output rows o = h W2 (the
combine's bf16 payload), dO = g dy, da and db to bf16, from pre-rounding values that differ by
the fp32 implementation's own rounding errors (and, for o, by the flips of h).  The oracle
bounds, from its fp64 values alone, how far the two roundings of each operand can lie apart
(a model of fp32 arithmetic: a probabilistic accumulation bound and an element-wise
evaluation bound), and turns that into an allowance for every gradient element.  These tests
tie the machinery to things other than itself:
  * the rounding spread against torch's bf16 cast;
  * the silu Lipschitz constants against sympy's derivatives on a fine grid;
  * the accumulation bound against real fp32 sums (numpy float32, sequential and pairwise);
  * an fp32 emulation of the layer (numpy float32 arithmetic, torch's bf16 rounding): its
    operands differ from the oracle's only where the oracle allows a flip, and by no more, and
    its gradients meet the stated tolerance plus the allowance; with the model switched off
    the same emulation does show flips, so the test has teeth;
  * random extreme choices of the flagged operands, propagated with numpy matmuls, stay
    inside the allowance.
"""
import math

import numpy as np
import pytest
import sympy
import torch

import oracle

RTOL, ATOL = 2e-2, 2e-3
F32 = np.float32


def _bf16_bits(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)


def _bits_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_round32(a):
    """float32 array -> nearest bf16 values (ties to even, torch), as float32."""
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def _inputs(seed, T, d, E, k, dff, gated=True):
    rng = np.random.default_rng(seed)
    inp = dict(x=_bf16_bits(rng.standard_normal((T, d))),
               logits=rng.standard_normal((T, E)).astype(np.float32),
               W1=_bf16_bits(rng.standard_normal((E, d, dff)) / math.sqrt(d)),
               W2=_bf16_bits(rng.standard_normal((E, dff, d)) / math.sqrt(dff)))
    if gated:
        inp["W3"] = _bf16_bits(rng.standard_normal((E, d, dff)) / math.sqrt(d))
    dy = _bf16_bits(rng.standard_normal((T, d)))
    return inp, dy


# --------------------------------------------------------------------- building blocks


def test_round_spread_matches_torch_bf16_cast():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(4000) * np.exp2(rng.integers(-20, 20, 4000))).astype(np.float32)
    # offsets of up to 3 bf16 half-ulps (2^15 fp32 ulps each), whole fp32 ulps of v so that
    # v +- dv stay fp32 values
    ulp32 = np.exp2(np.floor(np.log2(np.abs(v.astype(np.float64)))) - 23)
    dv = (ulp32 * rng.integers(0, 3 * 2 ** 15, 4000)).astype(np.float32)
    hi = (v.astype(np.float64) + dv).astype(np.float32)
    lo = (v.astype(np.float64) - dv).astype(np.float32)
    exact = (hi.astype(np.float64) - v == dv) & (v - lo.astype(np.float64) == dv)
    assert exact.mean() > 0.9
    r, rh, rl = (_bf16_round32(a).astype(np.float64) for a in (v, hi, lo))
    want = np.maximum(np.abs(rh - r), np.abs(rl - r))
    got = np.array([oracle.round_spread(float(a), float(b)) for a, b in zip(v, dv)])
    assert np.array_equal(got[exact], want[exact])
    assert (got[exact] > 0).mean() > 0.3  # many offsets cross a rounding midpoint


def test_silu_lipschitz_constants():
    # the allowance uses |silu'| <= 1.1 and |silu''| <= 0.5 over the whole real line
    a = sympy.symbols("a", real=True)
    silu = a / (1 + sympy.exp(-a))
    d1 = sympy.lambdify(a, sympy.diff(silu, a), "numpy")
    d2 = sympy.lambdify(a, sympy.diff(silu, a, 2), "numpy")
    grid = np.linspace(-60, 60, 2_400_001)
    m1 = np.max(np.abs(d1(grid)))
    m2 = np.max(np.abs(d2(grid)))
    assert 1.09 < m1 <= 1.1 and abs(m2 - 0.5) < 1e-9
    # the oracle's own closed forms (sigmoid products) agree with sympy's derivatives
    s = 1 / (1 + np.exp(-grid))
    np.testing.assert_allclose(s * (1 + grid * (1 - s)), d1(grid), rtol=1e-12, atol=1e-14)


def test_sum_bound_covers_real_fp32_sums():
    rng = np.random.default_rng(7)
    worst = 0.0
    for n in (16, 256, 4096, 8192):
        for trial in range(40):
            t64 = (rng.standard_normal(n) * rng.random(n) ** 3).astype(np.float32) \
                .astype(np.float64)
            exact, bound = oracle.sum_bound(t64)
            seq = float(np.cumsum(t64.astype(F32), dtype=F32)[-1])
            pairwise = float(np.sum(t64.astype(F32), dtype=F32))
            err = max(abs(seq - exact), abs(pairwise - exact))
            assert err <= bound, (n, trial, err, bound)
            worst = max(worst, err / bound)
            # not a worst-case bound either: far below n eps sum|t| for long sums
            if n >= 4096:
                assert bound < 0.05 * n * oracle.EPS32 * np.abs(t64).sum()
    assert worst > 1e-3  # the bound is exercised, not vacuous


# ------------------------------------------------------------- fp32 emulation of the layer


def _emulate_fp32(inp, dy, k, gated):
    """The layer in float32 arithmetic with products accumulated in order (as a tensor core
    with fp32 accumulation would, up to the order), h, the output rows Y, dO, da, db rounded
    to bf16 by torch."""
    x = _bits_to_f64(inp["x"]).astype(F32)
    W1 = _bits_to_f64(inp["W1"]).astype(F32)
    W3 = _bits_to_f64(inp["W3"]).astype(F32) if gated else None
    W2 = _bits_to_f64(inp["W2"]).astype(F32)
    dyf = _bits_to_f64(dy).astype(F32)
    T, d = x.shape
    E, _, dff = W1.shape
    idx, _ = oracle.route(inp["logits"], k)
    lg = inp["logits"].astype(F32)
    sel = np.take_along_axis(lg, idx, 1)
    ex = np.exp(sel - sel[:, :1]).astype(F32)
    s = np.zeros(T, F32)
    for j in range(k):
        s = (s + ex[:, j]).astype(F32)
    g = (ex / s[:, None]).astype(F32)
    P = T * k
    tok = np.repeat(np.arange(T), k)
    ep = idx.reshape(-1)
    xp = x[tok]
    A = np.zeros((P, dff), F32)
    B = np.zeros((P, dff), F32)
    for c in range(d):
        A += xp[:, c:c + 1] * W1[ep, c, :]
        if gated:
            B += xp[:, c:c + 1] * W3[ep, c, :]
    if gated:
        sg = (F32(1) / (F32(1) + np.exp(-A))).astype(F32)
        h = _bf16_round32((A * sg) * B)
    else:
        r = np.maximum(A, F32(0))
        h = _bf16_round32(r * r)
    Y = np.zeros((P, d), F32)
    for f in range(dff):
        Y += h[:, f:f + 1] * W2[ep, f, :]
    Y = _bf16_round32(Y)
    dyp = dyf[tok]
    dO = _bf16_round32(g.reshape(-1)[:, None] * dyp)
    dH = np.zeros((P, dff), F32)
    for c in range(d):
        dH += dO[:, c:c + 1] * W2[ep, :, c]
    if gated:
        sp = sg * (F32(1) + A * (F32(1) - sg))
        da = _bf16_round32(dH * B * sp)
        db = _bf16_round32(dH * (A * sg))
    else:
        da = _bf16_round32(dH * (F32(2) * np.maximum(A, F32(0))))
        db = np.zeros_like(da)
    dxp = np.zeros((P, d), F32)
    for f in range(dff):
        dxp += da[:, f:f + 1] * W1[ep, :, f]
    if gated:
        for f in range(dff):
            dxp += db[:, f:f + 1] * W3[ep, :, f]
    dx = np.zeros((T, d), F32)
    for j in range(k):
        dx += dxp[j::k]
    dgate = np.zeros(P, F32)
    for c in range(d):
        dgate += Y[:, c] * dyp[:, c]
    dW1 = np.zeros((E, d, dff), F32)
    dW3 = np.zeros((E, d, dff), F32)
    dW2 = np.zeros((E, dff, d), F32)
    for p in range(P):  # rows in token order within each expert, as the oracle sums them
        e = ep[p]
        dW1[e] += np.outer(xp[p], da[p])
        if gated:
            dW3[e] += np.outer(xp[p], db[p])
        dW2[e] += np.outer(h[p], dO[p])
    out = np.zeros((T, d), F32)
    for j in range(k):
        out += g[:, j:j + 1] * Y[j::k]
    return dict(h=h, o=Y, dO=dO, da=da, db=db, dx=dx, dgate=dgate.reshape(T, k), dW1=dW1,
                dW3=dW3, dW2=dW2, idx=idx, out=out)


def _within(got, ref, allow, what):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    bad = err > RTOL * np.abs(ref) + ATOL + allow
    assert not bad.any(), "%s: %d outside; worst %r" % (
        what, int(bad.sum()), np.max(err - RTOL * np.abs(ref) - ATOL - allow))


@pytest.mark.parametrize("gated", [True, False])
def test_fp32_emulation_flips_only_where_allowed(gated):
    T, d, E, k = 24, 512, 4, 2
    dff = 256
    inp, dy = _inputs(11 if gated else 12, T, d, E, k, dff, gated)
    emu = _emulate_fp32(inp, dy, k, gated)
    flips = {"h": 0, "o": 0, "dO": 0, "da": 0, "db": 0}
    unflagged_flips_without_model = 0
    for t in range(T):
        for j in range(k):
            op = oracle.pair_operands(inp, dy, k, t, j)
            off = oracle.pair_operands(inp, dy, k, t, j, model=(0.0, 0.0, 0.0))
            p = t * k + j
            for name, D in (("h", "Dh"), ("o", "Do"), ("dO", "DdO"), ("da", "Dda"),
                            ("db", "Ddb")):
                diff = emu[name][p].astype(np.float64) - op[name]
                lo, hi = op[D][:, 0], op[D][:, 1]
                assert (lo <= 0).all() and (hi >= 0).all()
                assert ((diff >= lo) & (diff <= hi)).all(), (name, t, j)
                flips[name] += int((diff != 0).sum())
                unflagged_flips_without_model += int(
                    ((diff != 0) & (off[D][:, 0] == 0) & (off[D][:, 1] == 0)).sum())
    # the emulation does flip operands, and a model that allows nothing would miss them
    assert flips["h"] + flips["da"] > 0
    assert unflagged_flips_without_model > 0
    y, ay = oracle.forward_tokens_flip(inp, k)
    _within(emu["out"], y, ay, "out")
    (dx, dgate, dlog), (adx, adg, adl) = oracle.backward_tokens_flip(inp, dy, k)
    _within(emu["dx"], dx, adx, "dx")
    _within(emu["dgate"], dgate, adg, "dgate")
    ex = np.arange(E)
    (r1, r3, r2), (a1, a3, a2) = oracle.backward_dw_flip(inp, dy, k, ex)
    _within(emu["dW1"], r1, a1, "dW1")
    _within(emu["dW2"], r2, a2, "dW2")
    if gated:
        _within(emu["dW3"], r3, a3, "dW3")


def test_forward_flip_that_breaks_the_stated_bound_is_covered():
    # T=2000, d=256, E=32, top-2, d_ff=256, every token's expert 0 logit raised by 50 (seed
    # 2013): for token 1088, h[2] of expert 0 lies 8.4e-8 from a bf16 rounding midpoint before
    # rounding (-2.0078125843 between -2.0 and -2.015625).  fp32 arithmetic rounds it up, the
    # oracle down, and that one ulp times W2[2][13] = -0.168 moves the near-cancelled output
    # out[1088, 13] by 0.0026, past the stated absolute term.  The allowance covers it.
    import moe_synth
    w = moe_synth.custom(2000, 256, 32, 2, 256, seed=2013)
    inp = moe_synth.generate(w)
    inp["logits"][:, 0] += 50.0
    npi = moe_synth.to_numpy(inp)
    t, c = 1088, 13
    y, ay = oracle.forward_tokens_flip(npi, 2, tokens=[t])
    op = oracle.pair_operands(npi, npi["x"], 2, t, 0)
    assert op["e"] == 0 and 0 < -2.0078125 - op["vh"][2] < 1e-7
    assert op["h"][2] == -2.015625 and op["Dh"][2].tolist() == [0.0, 0.015625]
    # the fp32 evaluation of h[2] (sequential fp32 sums, fp32 silu), rounded by torch
    x = _bits_to_f64(npi["x"][t]).astype(F32)
    W1 = _bits_to_f64(npi["W1"][0]).astype(F32)
    W3 = _bits_to_f64(npi["W3"][0]).astype(F32)
    W2 = _bits_to_f64(npi["W2"][0]).astype(F32)
    a = np.zeros(256, F32)
    b = np.zeros(256, F32)
    for cc in range(256):
        a += x[cc] * W1[cc]
        b += x[cc] * W3[cc]
    h32 = _bf16_round32((a / (F32(1) + np.exp(-a))) * b).astype(np.float64)
    assert h32[2] == -2.0
    moved = (h32[2] - op["h"][2]) * float(W2[2, c])
    assert abs(moved) > RTOL * abs(y[0, c]) + ATOL
    assert abs(moved) <= ay[0, c]


def test_flip_allowance_values_equal_the_plain_backward():
    inp, dy = _inputs(3, 16, 128, 4, 2, 128)
    y, _ = oracle.forward_tokens_flip(inp, 2)
    assert np.array_equal(y, oracle.forward_tokens(inp, 2))
    (dx, dgate, dlog), _ = oracle.backward_tokens_flip(inp, dy, 2)
    dx0, dg0, dl0 = oracle.backward_tokens(inp, dy, 2)
    assert np.array_equal(dx, dx0) and np.array_equal(dgate, dg0) and np.array_equal(dlog, dl0)
    (r1, r3, r2), _ = oracle.backward_dw_flip(inp, dy, 2, [0, 3])
    q1, q3, q2 = oracle.backward_dw(inp, dy, 2, [0, 3])
    assert np.array_equal(r1, q1) and np.array_equal(r3, q3) and np.array_equal(r2, q2)


def test_zero_model_gives_zero_allowance():
    inp, dy = _inputs(4, 16, 128, 4, 2, 128)
    _, (adx, adg, adl) = oracle.backward_tokens_flip(inp, dy, 2, model=(0.0, 0.0, 0.0))
    _, (a1, a3, a2) = oracle.backward_dw_flip(inp, dy, 2, [0, 1, 2, 3], model=(0.0, 0.0, 0.0))
    for a in (adx, adg, adl, a1, a3, a2):
        assert not a.any()


@pytest.mark.parametrize("gated", [True, False])
def test_extreme_operand_choices_stay_inside_the_allowance(gated):
    # A loose model flags many operands.  (1) Picking, for each flagged operand, either end of
    # its interval at random and recomputing the gradients with numpy matmuls stays within
    # the allowance.  (2) The allowance is attained: for a given output element, taking each
    # operand's end that pushes that element up (or down) reproduces the allowance exactly.
    T, d, E, k, dff = 12, 64, 3, 2, 128
    inp, dy = _inputs(21 if gated else 22, T, d, E, k, dff, gated)
    model = (2e-3, 1e-3, 2e-3)
    (dx, dgate, dlog), (adx, adg, adl) = oracle.backward_tokens_flip(inp, dy, k, model=model)
    (r1, r3, r2), (a1, a3, a2) = oracle.backward_dw_flip(inp, dy, k, np.arange(E), model=model)
    W1 = _bits_to_f64(inp["W1"])
    W3 = _bits_to_f64(inp["W3"]) if gated else None
    W2 = _bits_to_f64(inp["W2"])
    x = _bits_to_f64(inp["x"])
    dyf = _bits_to_f64(dy)
    ops = {(t, j): oracle.pair_operands(inp, dy, k, t, j, model=model)
           for t in range(T) for j in range(k)}
    frac = np.mean([(o["Dh"][:, 1] - o["Dh"][:, 0] > 0).mean() for o in ops.values()])
    assert frac > 0.2  # the loose model flags a good share of h
    rng = np.random.default_rng(0)
    slack = 1e-9

    def gradients(choose):
        pdx = np.zeros((T, d))
        pdg = np.zeros((T, k))
        pW1, pW3, pW2 = np.zeros((E, d, dff)), np.zeros((E, d, dff)), np.zeros((E, dff, d))
        for (t, j), o in ops.items():
            e = o["e"]
            h, dO = o["h"] + choose(o["Dh"]), o["dO"] + choose(o["DdO"])
            da, db = o["da"] + choose(o["Dda"]), o["db"] + choose(o["Ddb"])
            pdx[t] += W1[e] @ da + (W3[e] @ db if gated else 0.0)
            pdg[t, j] = (o["o"] + choose(o["Do"])) @ dyf[t]   # dgate reads the bf16 output row
            pW1[e] += np.outer(x[t], da)
            if gated:
                pW3[e] += np.outer(x[t], db)
            pW2[e] += np.outer(h, dO)
        return pdx, pdg, pW1, pW3, pW2

    def random_end(D):
        return np.where(rng.random(len(D)) < 0.5, D[:, 0], D[:, 1])

    # forward: out = sum_j g_j o_j with o_j the bf16 output row; its flip interval Do takes in
    # the h flips (any h choice moves the pre-rounding row by at most sum_f |W2| |Dh|)
    y, ay = oracle.forward_tokens_flip(inp, k, model=model)
    for trial in range(6):
        py = np.zeros((T, d))
        for (t, j), o in ops.items():
            py[t] += o["g"] * (o["o"] + random_end(o["Do"]))
        assert (np.abs(py - y) <= ay + slack).all()
    for (t, j), o in ops.items():   # the h flips' reach stays inside the row's interval
        hb = o["h"] + random_end(o["Dh"])
        pre = hb @ W2[o["e"]]
        assert (np.abs(pre - (o["h"] @ W2[o["e"]])) <= np.abs(W2[o["e"]]).T @ np.maximum(
            -o["Dh"][:, 0], o["Dh"][:, 1]) + slack).all()
    t, c = 4, 9
    up = dn = 0.0
    for j in range(k):
        o = ops[(t, j)]
        prod = o["g"] * o["Do"][c]
        up += prod.max()
        dn += prod.min()
    assert math.isclose(max(up, -dn), ay[t, c], rel_tol=1e-12, abs_tol=1e-15)

    for trial in range(6):
        pdx, pdg, pW1, pW3, pW2 = gradients(random_end)
        assert (np.abs(pdx - dx) <= adx + slack).all()
        assert (np.abs(pdg - dgate) <= adg + slack).all()
        assert (np.abs(pW1 - r1) <= a1 + slack).all()
        assert (np.abs(pW2 - r2) <= a2 + slack).all()
        if gated:
            assert (np.abs(pW3 - r3) <= a3 + slack).all()

    # attainment for dx[t, c]: each da_f / db_f takes the end whose product with W[c, f] is
    # largest (or smallest); the dx element then moves by exactly the allowance
    for t, c in ((0, 3), (5, 17), (11, 40)):
        up, dn = 0.0, 0.0
        for j in range(k):
            o = ops[(t, j)]
            for D, W in ((o["Dda"], W1), (o["Ddb"], W3)):
                if W is None:
                    continue
                prod = W[o["e"]][c][:, None] * D  # [dff, 2]
                up += prod.max(axis=1).sum()
                dn += prod.min(axis=1).sum()
        assert math.isclose(max(up, -dn), adx[t, c], rel_tol=1e-12, abs_tol=1e-15)
    # attainment for dgate[t, j]: the multiplier of o_c is dy_t[c]
    for t, j in ((1, 0), (7, 1)):
        o = ops[(t, j)]
        prod = dyf[t][:, None] * o["Do"]
        want = max(prod.max(axis=1).sum(), -prod.min(axis=1).sum())
        assert math.isclose(want, adg[t, j], rel_tol=1e-12, abs_tol=1e-15)
    # dlogits: a linear map of the dgate intervals through the softmax Jacobian
    assert (adl >= 0).all() and (adl[dlog == 0] == 0).all()


def test_fp8_forward_allowance_values_and_zero_model():
    # the FP8 forward's allowance comes with values equal to the plain FP8 forward; a model that
    # allows nothing gives none; an fp32 emulation of the FP8 expert (dequantized operands,
    # fp32 sums, torch's bf16 rounding of h and the output rows) stays inside it
    inp, _ = _inputs(31, 20, 256, 4, 2, 256)
    y0 = oracle.forward_tokens_fp8(inp, 2)
    y, ay = oracle.forward_tokens_fp8_flip(inp, 2)
    assert np.array_equal(y0, y)
    _, az = oracle.forward_tokens_fp8_flip(inp, 2, model=(0.0, 0.0, 0.0))
    assert not az.any()
    xq, _ = oracle.quantize_rows_e4m3(inp["x"])
    q1, s1 = oracle.quantize_cols_e4m3(inp["W1"])
    q3, s3 = oracle.quantize_cols_e4m3(inp["W3"])
    W2 = _bits_to_f64(inp["W2"]).astype(F32)
    idx, g = oracle.route(inp["logits"], 2)
    out = np.zeros(y.shape, F32)
    for t in range(y.shape[0]):
        for j in range(2):
            e = idx[t, j]
            W1 = (q1[e] * s1[e][None, :]).astype(F32)
            W3 = (q3[e] * s3[e][None, :]).astype(F32)
            xr = xq[t].astype(F32)
            A = np.zeros(W1.shape[1], F32)
            B = np.zeros(W1.shape[1], F32)
            for c in range(xr.shape[0]):
                A += xr[c] * W1[c]
                B += xr[c] * W3[c]
            h = _bf16_round32((A / (F32(1) + np.exp(-A))) * B)
            o = np.zeros(W2.shape[2], F32)
            for f in range(h.shape[0]):
                o += h[f] * W2[e, f]
            out[t] += F32(g[t, j]) * _bf16_round32(o)
    _within(out, y, ay, "out (fp8 emulation)")
