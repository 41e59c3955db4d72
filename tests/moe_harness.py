"""Helpers shared by the GPU tests: run the CUDA path through the C ABI, run the oracle on
the same inputs, compare with the stated tolerance."""
import numpy as np
import torch

import moe_synth

# Output tolerance of the layer (forward and gradients), elementwise against the fp64
# oracle on the same bf16 inputs with h rounded to bf16 on both sides.
RTOL = 2e-2
ATOL = 2e-3


def assert_close(got, ref, what, rtol=RTOL, atol=ATOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref)
    bad = err > rtol * np.abs(ref) + atol
    if bad.any():
        i = np.unravel_index(np.argmax(err - rtol * np.abs(ref)), err.shape)
        raise AssertionError("%s: %d / %d outside |d| <= %g|ref| + %g; worst at %s: got %r ref %r"
                             % (what, int(bad.sum()), bad.size, rtol, atol, i, got[i], ref[i]))


def assert_close_flip(got, ref, allow, what, rtol=RTOL, atol=ATOL):
    """The stated bound, widened element by element by the oracle's rounding-flip allowance
    (oracle.forward_tokens_flip, backward_tokens_flip, ...): both sides round h, the expert
    output rows, dO, da and db to bf16, and an operand whose pre-rounding value lies near a
    bf16 rounding midpoint may
    round the other way on the GPU (its value comes from fp32 accumulation, the oracle's from
    fp64).  `allow` is, per element, the largest change those operands can cause there,
    computed from oracle values alone.  Returns how many elements needed it."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    allow = np.asarray(allow, np.float64)
    assert got.shape == ref.shape == allow.shape, (what, got.shape, ref.shape, allow.shape)
    err = np.abs(got - ref)
    stated = rtol * np.abs(ref) + atol
    bad = err > stated + allow
    if bad.any():
        i = np.unravel_index(np.argmax(err - stated - allow), err.shape)
        raise AssertionError("%s: %d / %d outside |d| <= %g|ref| + %g + allowance; worst at %s: "
                             "got %r ref %r allowance %r" % (what, int(bad.sum()), bad.size, rtol,
                                                             atol, i, got[i], ref[i], allow[i]))
    return int((err > stated).sum())


def check_forward(out, npi, k, what, tokens=None):
    """Layer output (rows `tokens` of the batch, or all) against the oracle: the stated bound
    plus the oracle's per-element rounding-flip allowance of h and the bf16 expert output
    rows.  Returns how many elements needed the allowance."""
    import oracle
    y, ay = oracle.forward_tokens_flip(npi, k, tokens=tokens)
    got = np_of(out) if tokens is None else np_of(out)[tokens]
    return assert_close_flip(got, y, ay, what)


def check_backward(res, npi, k, what="", tokens=None, experts=None):
    """Gradients of a moe_backward against the oracle with its per-element rounding-flip
    allowance: dx, dgate, dlogits of `tokens` (all if None) and dW1, dW3, dW2 of `experts`
    (all if None).  Returns {name: elements that needed the allowance}."""
    import oracle
    (dx, dgate, dlog), (adx, adg, adl) = oracle.backward_tokens_flip(npi, npi["dy"], k,
                                                                      tokens=tokens)
    sel = (lambda a: a) if tokens is None else (lambda a: a[tokens])
    used = {}
    used["dx"] = assert_close_flip(sel(np_of(res["dx"])), dx, adx, "dx" + what)
    used["dgate"] = assert_close_flip(sel(np_of(res["dgate"])), dgate, adg, "dgate" + what)
    used["dlogits"] = assert_close_flip(sel(np_of(res["dlogits"])), dlog, adl, "dlogits" + what)
    E = npi["W1"].shape[0]
    ex = np.arange(E) if experts is None else np.asarray(experts)
    (r1, r3, r2), (a1, a3, a2) = oracle.backward_dw_flip(npi, npi["dy"], k, ex)
    exl = ex.tolist()
    used["dW1"] = assert_close_flip(np_of(res["dW1"][exl]), r1, a1, "dW1" + what)
    if r3 is not None:
        used["dW3"] = assert_close_flip(np_of(res["dW3"][exl]), r3, a3, "dW3" + what)
    used["dW2"] = assert_close_flip(np_of(res["dW2"][exl]), r2, a2, "dW2" + what)
    return used


def to_dev(inp, dev="cuda"):
    return {k: v.to(dev) for k, v in inp.items()}


def route_dispatch(moe, g, k):
    x, logits = g["x"], g["logits"]
    T, d = x.shape
    E = logits.shape[1]
    dev = x.device
    P = T * k
    out = dict(
        topk_idx=torch.empty(T, k, dtype=torch.int32, device=dev),
        gate=torch.empty(T, k, dtype=torch.float32, device=dev),
        counts=torch.empty(E, dtype=torch.int32, device=dev),
        offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
        perm=torch.empty(P, dtype=torch.int32, device=dev),
        pos=torch.empty(P, dtype=torch.int32, device=dev),
        x_perm=torch.empty(P, d, dtype=torch.bfloat16, device=dev),
    )
    ws = torch.empty(max(moe.moe_route_workspace_bytes(T, E, k), 256), dtype=torch.uint8,
                     device=dev)
    moe.moe_route_dispatch(x, logits, k, out["topk_idx"], out["gate"], out["counts"],
                           out["offsets"], out["perm"], out["pos"], out["x_perm"], ws)
    assert moe.moe_get_error(ws) == 0
    return out


def forward(moe, g, k, save=False, ws=None):
    x = g["x"]
    T, d = x.shape
    E, _, dff = g["W1"].shape
    if ws is None:
        ws = torch.empty(moe.moe_workspace_bytes(T, d, E, k, dff, save), dtype=torch.uint8,
                         device=x.device)
    out = torch.empty(T, d, dtype=torch.bfloat16, device=x.device)
    moe.moe_forward(x, g["logits"], g["W1"], g.get("W3"), g["W2"], k, out, ws,
                    flags=moe.MOE_FWD_SAVE_FOR_BACKWARD if save else 0)
    return out, ws


def backward(moe, g, k, ws):
    x = g["x"]
    T, d = x.shape
    E, _, dff = g["W1"].shape
    dev = x.device
    res = dict(
        dx=torch.empty(T, d, dtype=torch.bfloat16, device=dev),
        dW1=torch.empty(E, d, dff, dtype=torch.float32, device=dev),
        dW3=torch.empty(E, d, dff, dtype=torch.float32, device=dev) if "W3" in g else None,
        dW2=torch.empty(E, dff, d, dtype=torch.float32, device=dev),
        dgate=torch.empty(T, k, dtype=torch.float32, device=dev),
        dlogits=torch.empty(T, E, dtype=torch.float32, device=dev),
    )
    moe.moe_backward(g["dy"], x, g["logits"], g["W1"], g.get("W3"), g["W2"], k, res["dx"],
                     res["dW1"], res["dW3"], res["dW2"], res["dgate"], res["dlogits"], ws)
    return res


def np_of(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.float().numpy().astype(np.float64)
    return t.numpy()


def sample_tokens(T, n, seed=0):
    rng = np.random.default_rng(seed)
    pick = {0, T - 1}
    pick.update(rng.choice(T, size=min(n, T), replace=False).tolist())
    return np.array(sorted(pick), np.int64)
