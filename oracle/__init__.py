"""numpy front end of the fp64 CPU oracle of the MoE expert layer.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` leg of ``bench.py`` may import this package.  It shares no code with the
CUDA implementation and never imports it.

Arrays: bf16 tensors travel as their raw 16-bit patterns (``numpy.uint16``); fp32 router
logits are widened to fp64 exactly before they reach the C code.  Every function below
calls one entry point of ``moe_oracle.cpp``; the docstrings of that file name the
passages of the pages each step follows.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_i64 = ctypes.c_int64
_int = ctypes.c_int
_p = ctypes.c_void_p


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dims = [_i64, _int, _int, _int, _int]
        lib.oracle_num_threads.restype = _int
        lib.oracle_round_bf16.restype = ctypes.c_double
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_route.argtypes = [_p, _i64, _int, _int, _p, _p]
        lib.oracle_round_e4m3.restype = ctypes.c_double
        lib.oracle_round_e4m3.argtypes = [ctypes.c_double]
        lib.oracle_quantize_rows_e4m3.argtypes = [_p, _i64, _int, _p, _p]
        lib.oracle_quantize_cols_e4m3.argtypes = [_p, _int, _int, _int, _p, _p]
        lib.oracle_forward_tokens_fp8.argtypes = [_p] * 5 + dims + [_int, _p, _i64, _p]
        lib.oracle_dispatch.argtypes = [_p, _i64, _int, _int, _p, _p, _p, _p]
        for n in ("oracle_forward_tokens_bf16", "oracle_forward_tokens_f64"):
            getattr(lib, n).argtypes = [_p] * 5 + dims + [_int, _p, _i64, _p]
        lib.oracle_forward_permuted_bf16.argtypes = [_p] * 5 + dims + [_int, _p, _p, _p]
        for n in ("oracle_backward_tokens_bf16", "oracle_backward_tokens_f64"):
            getattr(lib, n).argtypes = [_p] * 6 + dims + [_int, _int, _p, _i64, _p, _p, _p]
        for n in ("oracle_backward_dw_bf16", "oracle_backward_dw_f64"):
            getattr(lib, n).argtypes = [_p] * 6 + dims + [_int, _int, _p, _int, _p, _p, _p]
        lib.oracle_round_spread_bf16.restype = ctypes.c_double
        lib.oracle_round_spread_bf16.argtypes = [ctypes.c_double, ctypes.c_double]
        lib.oracle_sum_bound.restype = ctypes.c_double
        lib.oracle_sum_bound.argtypes = [_p, _i64, ctypes.c_double, _p]
        lib.oracle_forward_tokens_flip_bf16.argtypes = [_p] * 5 + dims + [_p, _p, _i64, _p, _p]
        lib.oracle_forward_tokens_fp8_flip.argtypes = [_p] * 5 + dims + [_p, _p, _i64, _p, _p]
        lib.oracle_backward_tokens_flip_bf16.argtypes = \
            [_p] * 6 + dims + [_int, _p, _p, _i64] + [_p] * 6
        lib.oracle_backward_dw_flip_bf16.argtypes = \
            [_p] * 6 + dims + [_int, _p, _p, _int] + [_p] * 6
        lib.oracle_pair_operands_bf16.argtypes = [_p] * 6 + dims + [_i64, _int] + [_p] * 14
        _lib = lib
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc):
    if rc != 0:
        raise ValueError("oracle rejected its arguments (rc=%d)" % rc)


def num_threads() -> int:
    return _load().oracle_num_threads()


def round_bf16(v: float) -> float:
    """Nearest bf16 value of ``v`` (ties to even), as a float."""
    return _load().oracle_round_bf16(float(v))


def round_e4m3(v: float) -> float:
    """Nearest FP8 E4M3 value of ``v`` (ties to even, saturating at 448), as a float."""
    return _load().oracle_round_e4m3(float(v))


def quantize_rows_e4m3(x):
    """Per-row E4M3 quantization of bf16 rows x [T, d] (raw uint16): returns the dequantized
    values q*s [T, d] (float64) and the row scales s [T] (fp32 values as float64)."""
    x = _c(x, np.uint16)
    T, d = x.shape
    xq = np.empty((T, d), np.float64)
    s = np.empty(T, np.float64)
    _check(_load().oracle_quantize_rows_e4m3(_ptr(x), T, d, _ptr(xq), _ptr(s)))
    return xq, s


def quantize_cols_e4m3(W):
    """Per-(expert, column) E4M3 quantization of bf16 weights W [E, K, N] (raw uint16) over
    K: returns the E4M3 values q [E, K, N] (float64) and the scales s [E, N]."""
    W = _c(W, np.uint16)
    E, K, N = W.shape
    q = np.empty((E, K, N), np.float64)
    s = np.empty((E, N), np.float64)
    _check(_load().oracle_quantize_cols_e4m3(_ptr(W), E, K, N, _ptr(q), _ptr(s)))
    return q, s


def forward_tokens_fp8(inp, k, tokens=None, round_h=True):
    """Forward with the FP8 dispatch payload (rows and W1 / W3 quantized to E4M3 with fp32
    scales, then the SwiGLU expert on the dequantized values), bf16 inputs.  Returns [n, d]."""
    x, l64, W1, W3, W2, T, d, E, dff = _unpack(inp)
    x, W1, W3, W2 = (_prep(a, "bf16") for a in (x, W1, W3, W2))
    tok = None if tokens is None else _c(tokens, np.int64)
    n = T if tok is None else len(tok)
    y = np.empty((n, d), np.float64)
    _check(_load().oracle_forward_tokens_fp8(_ptr(x), _ptr(l64), _ptr(W1), _ptr(W3), _ptr(W2),
                                             T, d, E, k, dff, int(round_h), _ptr(tok), n,
                                             _ptr(y)))
    return y


def _logits64(logits):
    return _c(logits, np.float64)


def route(logits, k):
    """Top-k experts per token (descending logit, ties to the lower index) and the
    softmax gate over the selected logits.  Returns (idx int32 [T,k], gate float64 [T,k])."""
    l64 = _logits64(logits)
    T, E = l64.shape
    idx = np.empty((T, k), np.int32)
    gate = np.empty((T, k), np.float64)
    _check(_load().oracle_route(_ptr(l64), T, E, k, _ptr(idx), _ptr(gate)))
    return idx, gate


def dispatch(idx, E):
    """counts [E], exclusive offsets [E+1], perm [T*k] (row -> pair t*k+j) and
    pos [T*k] (pair -> row); rows ordered by (expert, token)."""
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    pos = np.empty(T * k, np.int32)
    _check(_load().oracle_dispatch(_ptr(idx), T, E, k, _ptr(counts), _ptr(offsets), _ptr(perm),
                                   _ptr(pos)))
    return counts, offsets, perm, pos


def _unpack(inp):
    # W3 absent or None: the cheap-activation expert, h = relu(x W1)^2
    x, logits, W1, W3, W2 = inp["x"], inp["logits"], inp["W1"], inp.get("W3"), inp["W2"]
    T, d = x.shape
    E, _, dff = W1.shape
    return x, _logits64(logits), W1, W3, W2, T, d, E, dff


def _wtype(x):
    return "bf16" if x.dtype == np.uint16 else "f64"


def _prep(a, wt):
    if a is None:
        return None
    return _c(a, np.uint16 if wt == "bf16" else np.float64)


def forward_tokens(inp, k, tokens=None, round_h=True):
    """Brute-force forward for the listed tokens (all if None): route each token, run its
    k experts on its own row, sum the gate-weighted outputs in fp64.  Returns [n, d]."""
    x, l64, W1, W3, W2, T, d, E, dff = _unpack(inp)
    wt = _wtype(x)
    x, W1, W3, W2 = (_prep(a, wt) for a in (x, W1, W3, W2))
    tok = None if tokens is None else _c(tokens, np.int64)
    n = T if tok is None else len(tok)
    y = np.empty((n, d), np.float64)
    fn = getattr(_load(), "oracle_forward_tokens_" + wt)
    _check(fn(_ptr(x), _ptr(l64), _ptr(W1), _ptr(W3), _ptr(W2), T, d, E, k, dff, int(round_h),
              _ptr(tok), n, _ptr(y)))
    return y


def forward_permuted(inp, k, round_h=True):
    """Permuted forward (route, dispatch, row copy, per-row expert FFN, combine), bf16
    inputs.  Returns (y [T,d] f64, x_perm [T*k,d] uint16, o_perm [T*k,d] f64)."""
    x, l64, W1, W3, W2, T, d, E, dff = _unpack(inp)
    x, W1, W3, W2 = (_prep(a, "bf16") for a in (x, W1, W3, W2))
    y = np.empty((T, d), np.float64)
    xp = np.empty((T * k, d), np.uint16)
    op = np.empty((T * k, d), np.float64)
    _check(_load().oracle_forward_permuted_bf16(_ptr(x), _ptr(l64), _ptr(W1), _ptr(W3), _ptr(W2),
                                                T, d, E, k, dff, int(round_h), _ptr(y), _ptr(xp),
                                                _ptr(op)))
    return y, xp, op


def backward_tokens(inp, dy, k, tokens=None, round_h=True, round_grad=True):
    """Per-token backward: dx [n,d], dgate [n,k], dlogits [n,E] (all f64).  With round_grad,
    the product operands dO = g dy, da and db are rounded to bf16 (as h is in the forward)."""
    x, l64, W1, W3, W2, T, d, E, dff = _unpack(inp)
    wt = _wtype(x)
    x, W1, W3, W2, dy = (_prep(a, wt) for a in (x, W1, W3, W2, dy))
    tok = None if tokens is None else _c(tokens, np.int64)
    n = T if tok is None else len(tok)
    dx = np.empty((n, d), np.float64)
    dgate = np.empty((n, k), np.float64)
    dlog = np.empty((n, E), np.float64)
    fn = getattr(_load(), "oracle_backward_tokens_" + wt)
    _check(fn(_ptr(x), _ptr(l64), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(dy), T, d, E, k, dff,
              int(round_h), int(round_grad), _ptr(tok), n, _ptr(dx), _ptr(dgate), _ptr(dlog)))
    return dx, dgate, dlog


def backward_dw(inp, dy, k, experts, round_h=True, round_grad=True):
    """Weight gradients of the listed experts: dW1, dW3 [n,d,dff] and dW2 [n,dff,d], f64
    (round_grad as in backward_tokens); dW3 is None for the cheap-activation expert."""
    x, l64, W1, W3, W2, T, d, E, dff = _unpack(inp)
    wt = _wtype(x)
    x, W1, W3, W2, dy = (_prep(a, wt) for a in (x, W1, W3, W2, dy))
    ex = _c(experts, np.int32)
    n = len(ex)
    dW1 = np.empty((n, d, dff), np.float64)
    dW3 = np.empty((n, d, dff), np.float64) if W3 is not None else None
    dW2 = np.empty((n, dff, d), np.float64)
    fn = getattr(_load(), "oracle_backward_dw_" + wt)
    _check(fn(_ptr(x), _ptr(l64), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(dy), T, d, E, k, dff,
              int(round_h), int(round_grad), _ptr(ex), n, _ptr(dW1), _ptr(dW3), _ptr(dW2)))
    return dW1, dW3, dW2


def layer_flops(pairs: int, d: int, dff: int, gated: bool = True) -> int:
    """Algorithmic FLOP of the expert stage: 6*d*dff per token-expert pair (gate, up and
    down projections: three d x dff multiply-adds), as the report's section 1.4 counts it;
    4*d*dff without the gate projection (the cheap activation)."""
    return (6 if gated else 4) * d * dff * pairs


# --------------------------------------------------------- rounding-flip allowance
# Model of fp32 arithmetic behind the allowance (see the oracle's FlipModel): an fp32 sum lies
# within ACC = lambda * eps * sqrt(sum of its squared running partial sums) of the exact sum,
# with eps = 2^-23, twice the unit roundoff of round-to-nearest (a margin for the hardware's
# order of accumulation), and lambda = 6, so that under the independent-error model a sum
# leaves the bound with probability below 2 exp(-18) = 3e-8 (and far less with errors of at
# most 2^-24); an element-wise fp32 evaluation lies within 16 eps of its value; the fp32
# softmax gate within 32 eps.
EPS32 = 2.0 ** -23
FLIP_MODEL = (6 * EPS32, 16 * EPS32, 32 * EPS32)


def _model(model):
    m = np.asarray(FLIP_MODEL if model is None else model, np.float64)
    assert m.shape == (3,)
    return m


def round_spread(v: float, dv: float) -> float:
    """Largest change of the bf16 rounding of v when v moves by at most dv."""
    return _load().oracle_round_spread_bf16(float(v), float(dv))


def sum_bound(t, acc=FLIP_MODEL[0]):
    """(exact sum of t in index order, the flip model's bound on an fp32 evaluation of it)."""
    t = _c(t, np.float64)
    s = ctypes.c_double(0.0)
    b = _load().oracle_sum_bound(_ptr(t), t.size, float(acc), ctypes.byref(s))
    return s.value, b


def forward_tokens_fp8_flip(inp, k, tokens=None, model=None):
    """forward_tokens_fp8 (h and the output rows rounded) plus the rounding-flip allowance of
    each output element, as forward_tokens_flip: returns (y [n,d], ay [n,d])."""
    x, l64, W1, W3, W2, T, d, E, dff = _unpack(inp)
    x, W1, W3, W2 = (_prep(a, "bf16") for a in (x, W1, W3, W2))
    tok = None if tokens is None else _c(tokens, np.int64)
    n = T if tok is None else len(tok)
    y = np.empty((n, d), np.float64)
    ay = np.empty((n, d), np.float64)
    m = _model(model)
    _check(_load().oracle_forward_tokens_fp8_flip(
        _ptr(x), _ptr(l64), _ptr(W1), _ptr(W3), _ptr(W2), T, d, E, k, dff, _ptr(m), _ptr(tok),
        n, _ptr(y), _ptr(ay)))
    return y, ay


def forward_tokens_flip(inp, k, tokens=None, model=None):
    """forward_tokens (h and the output rows rounded, bf16 inputs) plus the rounding-flip
    allowance of each output element: returns (y [n,d], ay [n,d]), ay the largest change that
    output-row values which may round the other way in fp32 arithmetic (taking in the h values
    that may) can cause in that element."""
    x, l64, W1, W3, W2, T, d, E, dff = _unpack(inp)
    x, W1, W3, W2 = (_prep(a, "bf16") for a in (x, W1, W3, W2))
    tok = None if tokens is None else _c(tokens, np.int64)
    n = T if tok is None else len(tok)
    y = np.empty((n, d), np.float64)
    ay = np.empty((n, d), np.float64)
    m = _model(model)
    _check(_load().oracle_forward_tokens_flip_bf16(
        _ptr(x), _ptr(l64), _ptr(W1), _ptr(W3), _ptr(W2), T, d, E, k, dff, _ptr(m), _ptr(tok),
        n, _ptr(y), _ptr(ay)))
    return y, ay


def backward_tokens_flip(inp, dy, k, tokens=None, round_h=True, model=None):
    """backward_tokens (round_grad on, bf16 inputs) plus the rounding-flip allowance of each
    output: returns ((dx, dgate, dlogits), (adx, adgate, adlogits)).  An implementation that
    rounds h, dO, da and db to bf16 after fp32 arithmetic obeying the flip model matches
    within the stated tolerance plus these allowances."""
    x, l64, W1, W3, W2, T, d, E, dff = _unpack(inp)
    x, W1, W3, W2, dy = (_prep(a, "bf16") for a in (x, W1, W3, W2, dy))
    tok = None if tokens is None else _c(tokens, np.int64)
    n = T if tok is None else len(tok)
    out = [np.empty(s, np.float64) for s in ((n, d), (n, k), (n, E)) * 2]
    m = _model(model)
    _check(_load().oracle_backward_tokens_flip_bf16(
        _ptr(x), _ptr(l64), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(dy), T, d, E, k, dff,
        int(round_h), _ptr(m), _ptr(tok), n, *[_ptr(a) for a in out]))
    return tuple(out[:3]), tuple(out[3:])


def backward_dw_flip(inp, dy, k, experts, round_h=True, model=None):
    """backward_dw (round_grad on, bf16 inputs) plus the rounding-flip allowances: returns
    ((dW1, dW3, dW2), (a1, a3, a2)); dW3 and a3 are None without W3."""
    x, l64, W1, W3, W2, T, d, E, dff = _unpack(inp)
    x, W1, W3, W2, dy = (_prep(a, "bf16") for a in (x, W1, W3, W2, dy))
    ex = _c(experts, np.int32)
    n = len(ex)
    g = W3 is not None
    dW1, a1 = np.empty((n, d, dff)), np.empty((n, d, dff))
    dW3, a3 = (np.empty((n, d, dff)), np.empty((n, d, dff))) if g else (None, None)
    dW2, a2 = np.empty((n, dff, d)), np.empty((n, dff, d))
    m = _model(model)
    _check(_load().oracle_backward_dw_flip_bf16(
        _ptr(x), _ptr(l64), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(dy), T, d, E, k, dff,
        int(round_h), _ptr(m), _ptr(ex), n, _ptr(dW1), _ptr(dW3), _ptr(dW2), _ptr(a1),
        _ptr(a3), _ptr(a2)))
    return (dW1, dW3, dW2), (a1, a3, a2)


def pair_operands(inp, dy, k, t, j, model=None):
    """The bf16 operands of token t's slot-j pair and their flip intervals (test support): a
    dict with e, g, h, vh (h before rounding), dO, da, db, o (the bf16 output row), and Dh,
    DdO, Dda, Ddb, Do of shape [n, 2]: the signed interval (lo <= 0 <= hi) within which
    another rounding may lie."""
    x, l64, W1, W3, W2, T, d, E, dff = _unpack(inp)
    x, W1, W3, W2, dy = (_prep(a, "bf16") for a in (x, W1, W3, W2, dy))
    names = ("h", "vh", "Dh", "dO", "DdO", "da", "Dda", "db", "Ddb", "o", "Do")
    sizes = (dff, dff, (dff, 2), d, (d, 2), dff, (dff, 2), dff, (dff, 2), d, (d, 2))
    r = {nm: np.empty(sz, np.float64) for nm, sz in zip(names, sizes)}
    e = ctypes.c_int(0)
    g = ctypes.c_double(0.0)
    m = _model(model)
    _check(_load().oracle_pair_operands_bf16(
        _ptr(x), _ptr(l64), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(dy), T, d, E, k, dff, int(t),
        int(j), _ptr(m), ctypes.byref(e), ctypes.byref(g), *[_ptr(r[nm]) for nm in names]))
    r["e"], r["g"] = e.value, g.value
    return r
