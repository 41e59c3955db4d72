"""Pins of the fp64 CPU oracle against things other than itself (CPU only).

Each test ties one oracle function to an independent fact: a hand-worked example from the
definitions, a library routine that computes the same quantity a different way (numpy's
stable sort and lexsort, scipy's softmax, numpy matmul, torch's bf16 cast), a closed form
(k = 1 with one expert is a dense SwiGLU MLP; k = E is a softmax-weighted dense sum), or
central finite differences of the oracle's own forward for the backward pass.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_bits(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)


def _bits_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rand_inputs(rng, T, d, E, k, dff, ties=False, as_bf16=True):
    x = rng.standard_normal((T, d))
    if ties:
        logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    else:
        logits = rng.standard_normal((T, E)).astype(np.float32)
    W1 = rng.standard_normal((E, d, dff)) / math.sqrt(d)
    W3 = rng.standard_normal((E, d, dff)) / math.sqrt(d)
    W2 = rng.standard_normal((E, dff, d)) / math.sqrt(dff)
    if as_bf16:
        return dict(x=_bf16_bits(x), logits=logits, W1=_bf16_bits(W1), W3=_bf16_bits(W3),
                    W2=_bf16_bits(W2))
    return dict(x=x, logits=logits, W1=W1, W3=W3, W2=W2)


# ----------------------------------------------------------------------------- routing


def test_route_and_dispatch_hand_worked_example():
    g = _golden("route_example.json")
    logits = np.array(g["logits"], np.float32)
    idx, gate = oracle.route(logits, g["k"])
    assert idx.tolist() == g["topk_idx"]
    np.testing.assert_allclose(gate, np.array(g["gate"]), rtol=1e-15, atol=0)
    counts, offsets, perm, pos = oracle.dispatch(idx, g["E"])
    assert counts.tolist() == g["counts"]
    assert offsets.tolist() == g["offsets"]
    assert perm.tolist() == g["perm"]
    assert pos.tolist() == g["pos"]


@pytest.mark.parametrize("T,E,k", [(50, 8, 2), (40, 37, 5), (30, 64, 8), (7, 5, 5), (9, 3, 1)])
@pytest.mark.parametrize("ties", [False, True])
def test_route_matches_lexsort_and_scipy_softmax(T, E, k, ties):
    from scipy.special import softmax
    rng = np.random.default_rng(T * 100 + E + k)
    logits = (rng.integers(-2, 3, size=(T, E)) if ties else rng.standard_normal((T, E))) \
        .astype(np.float32)
    idx, gate = oracle.route(logits, k)
    for t in range(T):
        # lexsort: last key is primary -> sort by -logit, then by index
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))
        assert idx[t].tolist() == order[:k].tolist()
        ref = softmax(logits[t, order[:k]].astype(np.float64))
        np.testing.assert_allclose(gate[t], ref, rtol=1e-14, atol=1e-16)


def test_route_signed_zero_is_a_tie():
    logits = np.array([[-0.0, 0.0, -1.0], [0.0, -0.0, -1.0]], np.float32)
    idx, gate = oracle.route(logits, 1)
    assert idx[:, 0].tolist() == [0, 0]
    np.testing.assert_array_equal(gate, 1.0)


def test_route_all_equal_logits():
    logits = np.full((3, 11), 0.25, np.float32)
    idx, gate = oracle.route(logits, 4)
    assert (idx == np.arange(4)).all()
    np.testing.assert_allclose(gate, 0.25, rtol=1e-15)


def test_route_k1_gate_is_one():
    rng = np.random.default_rng(3)
    idx, gate = oracle.route(rng.standard_normal((20, 9)).astype(np.float32), 1)
    np.testing.assert_array_equal(gate, 1.0)


@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (100, 33, 6), (1, 4, 4), (0, 5, 2)])
def test_dispatch_invariants_and_stable_sort(T, E, k):
    rng = np.random.default_rng(T + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = oracle.route(logits, k)
    counts, offsets, perm, pos = oracle.dispatch(idx, E)
    P = T * k
    assert counts.sum() == P
    assert offsets[0] == 0 and offsets[-1] == P
    assert (np.diff(offsets) == counts).all()
    assert sorted(perm.tolist()) == list(range(P))           # bijection
    assert (pos[perm] == np.arange(P)).all()                  # pos is its inverse
    flat = idx.reshape(-1)
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert (flat[seg] == e).all()
        assert (np.diff(seg // k) > 0).all()                  # ascending token order
    # numpy stable argsort by expert gives the same row order
    assert (np.argsort(flat, kind="stable") == perm).all()


# ----------------------------------------------------------------------------- bf16 rounding


def test_round_bf16_matches_torch_cast():
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000),
        [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -130, 3.5 * 2.0 ** -133,
         3.4e38, 1e-45, -2.5 * 2.0 ** -133],
    ]).astype(np.float32)
    ref = torch.tensor(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in vals])
    np.testing.assert_array_equal(got, ref)


# ----------------------------------------------------------------------------- forward


def test_ffn_hand_worked_example():
    g = _golden("ffn_example.json")
    inp = dict(x=np.array(g["x"], np.float64), logits=np.zeros((2, 1), np.float32),
               W1=np.array(g["W1"], np.float64), W3=np.array(g["W3"], np.float64),
               W2=np.array(g["W2"], np.float64))
    y = oracle.forward_tokens(inp, 1, round_h=False)
    np.testing.assert_allclose(y, np.array(g["y_exact_h"]), rtol=1e-15, atol=0)
    y = oracle.forward_tokens(inp, 1, round_h=True)
    np.testing.assert_array_equal(y, np.array(g["y_bf16_h"]))
    # same example through the bf16 entry point (every input is exactly bf16)
    inpb = {kk: (_bf16_bits(v) if kk != "logits" else v) for kk, v in inp.items()}
    y = oracle.forward_tokens(inpb, 1, round_h=True)
    np.testing.assert_array_equal(y, np.array(g["y_bf16_h"]))


def _silu(a):
    return a / (1.0 + np.exp(-a))


def _torch_bf16(a):
    return torch.tensor(a).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def test_k1_single_expert_is_dense_swiglu_mlp():
    rng = np.random.default_rng(11)
    inp = _rand_inputs(rng, T=16, d=32, E=1, k=1, dff=48)
    X = _bits_to_f64(inp["x"])
    W1, W3, W2 = (_bits_to_f64(inp[n])[0] for n in ("W1", "W3", "W2"))
    h = _silu(X @ W1) * (X @ W3)
    np.testing.assert_allclose(oracle.forward_tokens(inp, 1, round_h=False), h @ W2,
                               rtol=1e-12, atol=1e-13)
    # rounding h, then the expert's output row, to bf16 (the BF16 combine payload); with one
    # expert and k = 1 the gate is 1 and the output is that row (the values are float64 here;
    # rounding via float32 first can only differ on exact float32 ties, which this random draw
    # does not produce)
    y = oracle.forward_tokens(inp, 1, round_h=True)
    np.testing.assert_array_equal(y, _torch_bf16(_torch_bf16(h) @ W2))


def test_k_equals_E_is_softmax_weighted_dense_sum():
    from scipy.special import softmax
    rng = np.random.default_rng(12)
    T, d, E, dff = 10, 16, 5, 24
    inp = _rand_inputs(rng, T=T, d=d, E=E, k=E, dff=dff)
    X = _bits_to_f64(inp["x"])
    p = softmax(inp["logits"].astype(np.float64), axis=1)
    ref = np.zeros((T, d))
    for e in range(E):
        W1, W3, W2 = (_bits_to_f64(inp[n])[e] for n in ("W1", "W3", "W2"))
        ref += p[:, e:e + 1] * ((_silu(X @ W1) * (X @ W3)) @ W2)
    np.testing.assert_allclose(oracle.forward_tokens(inp, E, round_h=False), ref,
                               rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("T,d,E,k,dff", [(40, 16, 6, 2, 24), (25, 8, 9, 4, 16)])
def test_bruteforce_and_permuted_forward_agree(T, d, E, k, dff):
    rng = np.random.default_rng(T)
    inp = _rand_inputs(rng, T, d, E, k, dff)
    y_bf = oracle.forward_tokens(inp, k)
    y_pm, x_perm, o_perm = oracle.forward_permuted(inp, k)
    np.testing.assert_allclose(y_pm, y_bf, rtol=1e-13, atol=1e-14)
    idx, _ = oracle.route(inp["logits"], k)
    _, _, perm, _ = oracle.dispatch(idx, E)
    np.testing.assert_array_equal(x_perm, inp["x"][perm // k])
    # a token subset gives the same rows as the full batch
    sub = np.array([T - 1, 0, T // 2])
    np.testing.assert_array_equal(oracle.forward_tokens(inp, k, tokens=sub), y_bf[sub])


# ----------------------------------------------------------------------------- backward


def _loss(inp, dy, k):
    return float((oracle.forward_tokens(inp, k, round_h=False) * dy).sum())


def _fd(inp, dy, k, name, eps):
    base = inp[name]
    g = np.zeros(base.shape)
    it = np.nditer(base, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        plus, minus = dict(inp), dict(inp)
        bp, bm = base.copy(), base.copy()
        bp[i] += eps
        bm[i] -= eps
        plus[name], minus[name] = bp, bm
        g[i] = (_loss(plus, dy, k) - _loss(minus, dy, k)) / (2 * eps)
    return g


def test_backward_matches_central_finite_differences():
    rng = np.random.default_rng(21)
    T, d, E, k, dff = 3, 4, 3, 2, 5
    inp = _rand_inputs(rng, T, d, E, k, dff, as_bf16=False)
    inp["logits"] = inp["logits"].astype(np.float64)   # perturbable
    dy = rng.standard_normal((T, d))
    dx, dgate, dlog = oracle.backward_tokens(inp, dy, k, round_h=False, round_grad=False)
    dW1, dW3, dW2 = oracle.backward_dw(inp, dy, k, np.arange(E), round_h=False, round_grad=False)
    tol = dict(rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dx, _fd(inp, dy, k, "x", 1e-6), **tol)
    np.testing.assert_allclose(dW1, _fd(inp, dy, k, "W1", 1e-6), **tol)
    np.testing.assert_allclose(dW3, _fd(inp, dy, k, "W3", 1e-6), **tol)
    np.testing.assert_allclose(dW2, _fd(inp, dy, k, "W2", 1e-6), **tol)
    # logits: the top-k selection is locally constant, so the derivative flows only through
    # the gate softmax (the draw keeps every gap between logits far above eps)
    np.testing.assert_allclose(dlog, _fd(inp, dy, k, "logits", 1e-6), **tol)
    # dgate_j = <o_j, dy>: with o_j from the permuted forward (an independent path)
    idx, _ = oracle.route(inp["logits"], k)
    _, _, _, pos = oracle.dispatch(idx, E)
    inpb = _rand_inputs(np.random.default_rng(21), T, d, E, k, dff)   # bf16 copy for o_perm
    _, _, o_perm = oracle.forward_permuted(inpb, k, round_h=False)
    _, dg_b, _ = oracle.backward_tokens(inpb, _bf16_bits(dy), k, round_h=False)
    dyb = _bits_to_f64(_bf16_bits(dy))
    ref = np.einsum("tjc,tc->tj", o_perm[oracle.dispatch(oracle.route(inpb["logits"], k)[0], E)[3]]
                    .reshape(T, k, d), dyb)
    np.testing.assert_allclose(dg_b, ref, rtol=1e-12, atol=1e-14)


def test_backward_closed_form_with_sympy():
    sp = pytest.importorskip("sympy")
    g = _golden("ffn_example.json")
    x0, x1 = sp.symbols("x0 x1")
    W1 = sp.Matrix(g["W1"][0])
    W3 = sp.Matrix(g["W3"][0])
    W2 = sp.Matrix(g["W2"][0])
    X = sp.Matrix([[x0, x1]])
    a, b = X * W1, X * W3
    h = sp.Matrix([[a[i] / (1 + sp.exp(-a[i])) * b[i] for i in range(2)]])
    y = h * W2
    dy = [0.75, -1.25]
    L = y[0] * dy[0] + y[1] * dy[1]
    pts = [(1.0, 0.0), (0.0, -2.0)]
    inp = dict(x=np.array(pts), logits=np.zeros((2, 1)), W1=np.array(g["W1"], np.float64),
               W3=np.array(g["W3"], np.float64), W2=np.array(g["W2"], np.float64))
    dx, dgate, dlog = oracle.backward_tokens(inp, np.array([dy, dy]), 1, round_h=False,
                                             round_grad=False)
    for t, (p0, p1) in enumerate(pts):
        sub = {x0: p0, x1: p1}
        ref = [float(sp.diff(L, v).subs(sub).evalf(30)) for v in (x0, x1)]
        np.testing.assert_allclose(dx[t], ref, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(dgate[t, 0], float(L.subs(sub).evalf(30)), rtol=1e-13)
    np.testing.assert_array_equal(dlog, 0.0)   # k = 1: the gate is constant 1


def test_backward_round_grad_rounds_exactly_the_product_operands():
    # With round_grad the oracle rounds dO = g*dy, da and db to bf16 before they enter a
    # product.  Rebuild dW2 = sum h^T dO, dW1 = sum x^T da, dW3 = sum x^T db and
    # dx = sum (da W1^T + db W3^T) for one expert with numpy products and torch's bf16 cast.
    from scipy.special import softmax
    rng = np.random.default_rng(31)
    T, d, E, k, dff = 12, 16, 3, 2, 24
    inp = _rand_inputs(rng, T, d, E, k, dff)
    dy = _bf16_bits(rng.standard_normal((T, d)))
    X, DY = _bits_to_f64(inp["x"]), _bits_to_f64(dy)
    W1, W3, W2 = (_bits_to_f64(inp[n]) for n in ("W1", "W3", "W2"))
    logits = inp["logits"].astype(np.float64)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    gates = softmax(np.take_along_axis(logits, order, 1), axis=1)
    e = 1
    ref2 = np.zeros((dff, d)); ref1 = np.zeros((d, dff)); ref3 = np.zeros((d, dff))
    dx_ref = np.zeros((T, d))
    for t in range(T):
        for j in range(k):
            ee = order[t, j]
            a, b = X[t] @ W1[ee], X[t] @ W3[ee]
            h = _torch_bf16(_silu(a) * b)
            dO = _torch_bf16(gates[t, j] * DY[t])
            dh = W2[ee] @ dO
            sg = 1 / (1 + np.exp(-a))
            da = _torch_bf16(dh * b * sg * (1 + a * (1 - sg)))
            db = _torch_bf16(dh * a * sg)
            dx_ref[t] += W1[ee] @ da + W3[ee] @ db
            if ee == e:
                ref2 += np.outer(h, dO)
                ref1 += np.outer(X[t], da)
                ref3 += np.outer(X[t], db)
    dW1, dW3, dW2 = oracle.backward_dw(inp, dy, k, [e])
    np.testing.assert_allclose(dW2[0], ref2, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dW1[0], ref1, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dW3[0], ref3, rtol=1e-10, atol=1e-12)
    dx, _, _ = oracle.backward_tokens(inp, dy, k)
    np.testing.assert_allclose(dx, dx_ref, rtol=1e-10, atol=1e-12)
    # and the rounding is really applied: the unrounded gradients differ
    dW1u, _, _ = oracle.backward_dw(inp, dy, k, [e], round_grad=False)
    assert np.abs(dW1u - dW1).max() > 0


def test_layer_flops_is_six_h_d_per_pair():
    # the report's section 1.4 counts 6hd FLOP per token-expert pair (gate, up, down)
    assert oracle.layer_flops(1, 7168, 2048) == 6 * 7168 * 2048
    assert oracle.layer_flops(16384 * 8, 7168, 2048) == 11544872091648


# ----------------------------------------------------------- cheap activation (no W3)


def _no_w3(inp):
    return {kk: v for kk, v in inp.items() if kk != "W3"}


def _relu2(a):
    return np.maximum(a, 0.0) ** 2


def test_cheap_activation_k1_single_expert_is_dense_relu2_mlp():
    # without the gate projection the expert is y = relu(x W1)^2 W2: with one expert and k = 1
    # the layer is that dense MLP (numpy products)
    rng = np.random.default_rng(41)
    inp = _no_w3(_rand_inputs(rng, T=16, d=32, E=1, k=1, dff=48))
    X = _bits_to_f64(inp["x"])
    W1, W2 = (_bits_to_f64(inp[n])[0] for n in ("W1", "W2"))
    h = _relu2(X @ W1)
    assert (X @ W1 < 0).any() and (X @ W1 > 0).any()      # both sides of the kink occur
    np.testing.assert_allclose(oracle.forward_tokens(inp, 1, round_h=False), h @ W2,
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(oracle.forward_tokens(inp, 1, round_h=True),
                                  _torch_bf16(_torch_bf16(h) @ W2))


def test_cheap_activation_k_equals_E_and_permuted_forward():
    from scipy.special import softmax
    rng = np.random.default_rng(42)
    T, d, E, dff = 10, 16, 5, 24
    inp = _no_w3(_rand_inputs(rng, T=T, d=d, E=E, k=E, dff=dff))
    X = _bits_to_f64(inp["x"])
    p = softmax(inp["logits"].astype(np.float64), axis=1)
    ref = np.zeros((T, d))
    for e in range(E):
        W1, W2 = (_bits_to_f64(inp[n])[e] for n in ("W1", "W2"))
        ref += p[:, e:e + 1] * (_relu2(X @ W1) @ W2)
    np.testing.assert_allclose(oracle.forward_tokens(inp, E, round_h=False), ref,
                               rtol=1e-12, atol=1e-13)
    k = 2
    y_pm, _, _ = oracle.forward_permuted(inp, k)
    np.testing.assert_allclose(y_pm, oracle.forward_tokens(inp, k), rtol=1e-13, atol=1e-14)


def test_cheap_activation_backward_matches_central_finite_differences():
    rng = np.random.default_rng(43)
    T, d, E, k, dff = 3, 4, 3, 2, 5
    inp = _no_w3(_rand_inputs(rng, T, d, E, k, dff, as_bf16=False))
    inp["logits"] = inp["logits"].astype(np.float64)
    dy = rng.standard_normal((T, d))
    dx, dgate, dlog = oracle.backward_tokens(inp, dy, k, round_h=False, round_grad=False)
    dW1, dW3, dW2 = oracle.backward_dw(inp, dy, k, np.arange(E), round_h=False, round_grad=False)
    assert dW3 is None
    # relu(a)^2 is continuously differentiable, so central differences converge at the kink too
    tol = dict(rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dx, _fd(inp, dy, k, "x", 1e-6), **tol)
    np.testing.assert_allclose(dW1, _fd(inp, dy, k, "W1", 1e-6), **tol)
    np.testing.assert_allclose(dW2, _fd(inp, dy, k, "W2", 1e-6), **tol)
    np.testing.assert_allclose(dlog, _fd(inp, dy, k, "logits", 1e-6), **tol)


def test_cheap_activation_round_grad_rounds_exactly_the_product_operands():
    from scipy.special import softmax
    rng = np.random.default_rng(44)
    T, d, E, k, dff = 12, 16, 3, 2, 24
    inp = _no_w3(_rand_inputs(rng, T, d, E, k, dff))
    dy = _bf16_bits(rng.standard_normal((T, d)))
    X, DY = _bits_to_f64(inp["x"]), _bits_to_f64(dy)
    W1, W2 = (_bits_to_f64(inp[n]) for n in ("W1", "W2"))
    logits = inp["logits"].astype(np.float64)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    gates = softmax(np.take_along_axis(logits, order, 1), axis=1)
    e = 2
    ref2 = np.zeros((dff, d)); ref1 = np.zeros((d, dff)); dx_ref = np.zeros((T, d))
    for t in range(T):
        for j in range(k):
            ee = order[t, j]
            a = X[t] @ W1[ee]
            h = _torch_bf16(_relu2(a))
            dO = _torch_bf16(gates[t, j] * DY[t])
            da = _torch_bf16((W2[ee] @ dO) * 2.0 * np.maximum(a, 0.0))
            dx_ref[t] += W1[ee] @ da
            if ee == e:
                ref2 += np.outer(h, dO)
                ref1 += np.outer(X[t], da)
    dW1, dW3, dW2 = oracle.backward_dw(inp, dy, k, [e])
    np.testing.assert_allclose(dW2[0], ref2, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dW1[0], ref1, rtol=1e-10, atol=1e-12)
    dx, _, _ = oracle.backward_tokens(inp, dy, k)
    np.testing.assert_allclose(dx, dx_ref, rtol=1e-10, atol=1e-12)


def test_layer_flops_without_the_gate_projection():
    assert oracle.layer_flops(1, 7168, 3072, gated=False) == 4 * 7168 * 3072
    # the same parameter budget (d_ff' = 1.5 d_ff) keeps the FLOP count
    assert oracle.layer_flops(5, 7168, 3072, gated=False) == oracle.layer_flops(5, 7168, 2048)


# ------------------------------------------------------------------ FP8 dispatch payload


def _torch_e4m3(v):
    return torch.tensor(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).to(torch.float64) \
        .numpy()


def test_round_e4m3_matches_torch_float8_cast():
    rng = np.random.default_rng(51)
    v = np.concatenate([
        rng.uniform(-448, 448, 4000),
        rng.uniform(-2.0 ** -5, 2.0 ** -5, 2000),             # subnormals and the normal edge
        np.ldexp(rng.integers(-16, 17, 400) + 0.5, -9),        # exact subnormal ties
        np.array([0.0, -0.0, 448.0, -448.0, 1.0625, 1.1875, 2.0 ** -6, 2.0 ** -10]),
    ]).astype(np.float32).astype(np.float64)
    got = np.array([oracle.round_e4m3(x) for x in v])
    np.testing.assert_array_equal(got, _torch_e4m3(v))
    # saturation above the largest finite value (torch's cast gives NaN there)
    assert oracle.round_e4m3(1000.0) == 448.0 and oracle.round_e4m3(-470.0) == -448.0


def test_quantize_rows_e4m3_matches_float32_division_and_torch_cast():
    rng = np.random.default_rng(52)
    x = rng.standard_normal((9, 64)) * np.exp(rng.uniform(-6, 6, (9, 1)))
    x[3] = 0.0                                                  # all-zero row: scale 1
    xb = _bf16_bits(x)
    xq, s = oracle.quantize_rows_e4m3(xb)
    X32 = _bits_to_f64(xb).astype(np.float32)
    amax = np.abs(X32).max(axis=1)
    s_ref = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    np.testing.assert_array_equal(s, s_ref.astype(np.float64))
    q_ref = _torch_e4m3(X32 / s_ref[:, None])
    np.testing.assert_array_equal(xq, q_ref * s_ref[:, None].astype(np.float64))
    assert np.abs(q_ref).max() == 448.0                         # each row's amax maps to 448


def test_quantize_cols_e4m3_matches_float32_division_and_torch_cast():
    rng = np.random.default_rng(53)
    W = rng.standard_normal((3, 40, 24)) / 6.0
    Wb = _bf16_bits(W)
    q, s = oracle.quantize_cols_e4m3(Wb)
    W32 = _bits_to_f64(Wb).astype(np.float32)
    s_ref = (np.abs(W32).max(axis=1) / np.float32(448.0)).astype(np.float32)   # [E, N]
    np.testing.assert_array_equal(s, s_ref.astype(np.float64))
    np.testing.assert_array_equal(q, _torch_e4m3(W32 / s_ref[:, None, :]))


def test_fp8_forward_k1_single_expert_is_dense_mlp_on_dequantized_values():
    rng = np.random.default_rng(54)
    inp = _rand_inputs(rng, T=12, d=32, E=1, k=1, dff=40)
    xq, _ = oracle.quantize_rows_e4m3(inp["x"])
    q1, s1 = oracle.quantize_cols_e4m3(inp["W1"])
    q3, s3 = oracle.quantize_cols_e4m3(inp["W3"])
    W1 = q1[0] * s1[0][None, :]
    W3 = q3[0] * s3[0][None, :]
    W2 = _bits_to_f64(inp["W2"])[0]
    h = _silu(xq @ W1) * (xq @ W3)
    np.testing.assert_allclose(oracle.forward_tokens_fp8(inp, 1, round_h=False), h @ W2,
                               rtol=1e-12, atol=1e-13)
    # bf16 h, then the bf16 output row (gate 1 with one expert and k = 1)
    np.testing.assert_array_equal(oracle.forward_tokens_fp8(inp, 1),
                                  _torch_bf16(_torch_bf16(h) @ W2))


def test_fp8_forward_equals_bf16_forward_when_quantization_is_exact():
    # rows and weight columns whose largest magnitude is 448 and whose values are E4M3
    # numbers quantize to themselves (scale 1): the FP8 forward is then the bf16 forward
    rng = np.random.default_rng(55)
    T, d, E, k, dff = 8, 16, 4, 2, 24
    grid = np.unique(_torch_e4m3(rng.uniform(-448, 448, 5000)))
    def pick(shape):
        v = rng.choice(grid, size=shape)
        return v
    x = pick((T, d)); x[:, 0] = 448.0
    W1 = pick((E, d, dff)); W1[:, 0, :] = 448.0
    W3 = pick((E, d, dff)); W3[:, 0, :] = -448.0
    W2 = rng.standard_normal((E, dff, d)) / 100
    inp = dict(x=_bf16_bits(x), logits=rng.standard_normal((T, E)).astype(np.float32),
               W1=_bf16_bits(W1), W3=_bf16_bits(W3), W2=_bf16_bits(W2))
    np.testing.assert_array_equal(oracle.forward_tokens_fp8(inp, k), oracle.forward_tokens(inp, k))
