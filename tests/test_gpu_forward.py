"""Forward of the whole layer on the GPU (moe_forward through the C ABI) against the oracle,
batch invariance and run-to-run determinism (bitwise).

Bar: every output element meets the stated bound |y - y_ref| <= 2e-2 |y_ref| + 2e-3 widened by
the oracle's rounding-flip allowance for that element (moe_harness.check_forward): the
largest change that h values which may round to the other bf16 neighbour in fp32 arithmetic
can cause there.  The tiny workload also meets the stated bound alone."""
import numpy as np
import pytest
import torch

import moe_synth
import oracle
from moe_harness import (assert_close, backward, check_forward, forward, np_of,
                         sample_tokens, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import combine_fp32_router_gb300 as m
    return m


def _full_check(moe, w, plain=False):
    inp = moe_synth.generate(w)
    g = to_dev(inp)
    out, ws = forward(moe, g, w.k)
    assert moe.moe_get_error(ws) == 0
    npi = moe_synth.to_numpy(inp)
    check_forward(out, npi, w.k, "out")
    if plain:  # the stated bound alone
        assert_close(np_of(out), oracle.forward_tokens(npi, w.k), "out")
    return g, out


def _oracle_check(out, g, k, what, n_sample=64):
    """out against the oracle on the same inputs: every token for small layers, a sample of
    tokens (first and last included) for large ones."""
    npi = moe_synth.to_numpy(g)
    T = npi["x"].shape[0]
    tok = None if T <= 2048 else sample_tokens(T, n_sample, seed=T)
    check_forward(out, npi, k, what, tokens=tok)


def test_forward_tiny_workload(moe):
    _full_check(moe, moe_synth.by_name("tiny"), plain=True)


@pytest.mark.parametrize("T,d,E,k,dff", [
    (300, 256, 16, 4, 384),    # ragged tiles, d % 256 == 0, dff % 256 != 0
    (77, 384, 5, 3, 128),      # d % 256 != 0 (128-wide N tiles), one 128-wide h block
    (1, 128, 4, 4, 256),       # a single token, k = E
    (513, 128, 1, 1, 128),     # one expert: a dense SwiGLU MLP with 5 row tiles
    (200, 128, 64, 2, 256),    # many empty experts
])
def test_forward_small_shapes(moe, T, d, E, k, dff):
    _full_check(moe, moe_synth.custom(T, d, E, k, dff, seed=T * 7 + d))


@pytest.mark.parametrize("gated", [True, False])
def test_forward_expert_row_counts_at_block_edges(moe, gated):
    # one expert per row count around the swapped GEMMs' block sizes (a CTA takes 16, 32, 64 or
    # 128 rows of a block of up to 256): 1, 16, 17, 32, 33, 64, 65, 128, 129, 255, 256, 257, 300
    counts = [1, 16, 17, 32, 33, 64, 65, 128, 129, 255, 256, 257, 300]
    E, k, d, dff = len(counts), 1, 384, 256   # d % 256 == 128: GEMM2's last column block is half
    T = sum(counts)
    w = moe_synth.custom(T, d, E, k, dff, seed=123, gated=gated)
    inp = moe_synth.generate(w)
    owner = torch.repeat_interleave(torch.arange(E), torch.tensor(counts))
    owner = owner[torch.randperm(T, generator=torch.Generator().manual_seed(5))]
    inp["logits"][torch.arange(T), owner] += 40.0
    g = to_dev(inp)
    out, ws = forward(moe, g, k)
    assert moe.moe_get_error(ws) == 0
    npi = moe_synth.to_numpy(inp)
    assert np.bincount(oracle.route(npi["logits"], k)[0].reshape(-1), minlength=E).tolist() == counts
    check_forward(out, npi, k, "out (block edges)")


def test_forward_mid_workload_sampled(moe):
    w = moe_synth.by_name("mid")
    inp = moe_synth.generate(w)
    g = to_dev(inp)
    out, ws = forward(moe, g, w.k)
    assert moe.moe_get_error(ws) == 0
    tok = sample_tokens(w.T, 96, seed=1)
    check_forward(out, moe_synth.to_numpy(inp), w.k, "out (mid, sampled tokens)", tokens=tok)


def test_forward_skewed_one_expert_hot(moe):
    # 90% of the pairs on expert 0: one expert spans many 128-row tiles, most are empty
    w = moe_synth.custom(T=2000, d=256, E=32, k=2, dff=256, seed=5)
    inp = moe_synth.generate(w)
    inp["logits"][:1800, 0] += 50.0
    g = to_dev(inp)
    out, ws = forward(moe, g, w.k)
    assert moe.moe_get_error(ws) == 0
    check_forward(out, moe_synth.to_numpy(inp), w.k, "out (hot expert)")


def test_forward_deterministic_and_ws_reuse(moe):
    w = moe_synth.custom(T=1000, d=256, E=16, k=4, dff=256, seed=9)
    g = to_dev(moe_synth.generate(w))
    out0, ws = forward(moe, g, w.k)
    for _ in range(5):
        out1, _ = forward(moe, g, w.k, ws=ws)
        assert torch.equal(out0.view(torch.int16), out1.view(torch.int16))


def test_forward_batch_invariance_small(moe):
    # each token's output is bitwise the same whatever the batch it sits in
    w = moe_synth.custom(T=400, d=256, E=16, k=4, dff=256, seed=11)
    g = to_dev(moe_synth.generate(w))
    full, _ = forward(moe, g, w.k)
    for T in (1, 3, 64, 129, 255):
        part, _ = forward(moe, moe_synth.rows(g, T), w.k)
        assert torch.equal(part.view(torch.int16), full[:T].view(torch.int16)), T
    # a token placed in a different batch (reversed order) gives the same bits
    rev = {kk: (v.flip(0).contiguous() if kk in ("x", "logits") else v) for kk, v in g.items()}
    out_rev, _ = forward(moe, rev, w.k)
    assert torch.equal(out_rev.flip(0).view(torch.int16), full.view(torch.int16))


@pytest.mark.parametrize("T,d,E,k,dff", [
    (64, 128, 8, 2, 256),       # tiny
    (300, 256, 16, 4, 384),     # ragged tiles
    (77, 384, 5, 3, 128),       # 128-wide GEMM2 tiles
    (2000, 256, 32, 2, 256),    # one expert takes most tokens
    (4096, 2048, 64, 6, 1024),  # mid workload
])
def test_fused_combine_equals_separate_stages(moe, T, d, E, k, dff):
    # GEMM2 with the combine fused in gives bitwise the same output as GEMM2 + combine kernel
    w = moe_synth.custom(T, d, E, k, dff, seed=T + 13)
    inp = moe_synth.generate(w)
    if T == 2000:
        inp["logits"][:, 0] += 50.0
    g = to_dev(inp)
    sep, ws = forward(moe, g, k)
    fused = torch.empty_like(sep)
    moe.moe_forward(g["x"], g["logits"], g["W1"], g["W3"], g["W2"], k, fused, ws,
                    flags=moe.MOE_FWD_FUSED_COMBINE)
    assert moe.moe_get_error(ws) == 0
    assert torch.equal(fused.view(torch.int16), sep.view(torch.int16))
    _oracle_check(fused, g, k, "out (fused combine)")


@pytest.mark.parametrize("T,d,E,k,dff,flags", [
    (64, 128, 8, 2, 256, 0),          # tiny
    (300, 256, 16, 4, 384, 0),        # ragged tiles: padding rows gather token 0, never stored
    (77, 384, 5, 3, 128, 0),          # 128-wide GEMM2 tiles
    (2000, 256, 32, 2, 256, 0),       # one expert takes most tokens
    (4096, 2048, 64, 6, 1024, 0),     # mid workload
    (4096, 2048, 64, 6, 1024, 2),     # gather + fused combine: the overlapped waves together
])
def test_row_gather_equals_permuted_copy(moe, T, d, E, k, dff, flags):
    # GEMM1 gathering its rows from x (cp.async) gives bitwise the same output as GEMM1
    # reading the dispatch's permuted copy
    w = moe_synth.custom(T, d, E, k, dff, seed=T + 17)
    inp = moe_synth.generate(w)
    if T == 2000:
        inp["logits"][:, 0] += 50.0
    g = to_dev(inp)
    sep, ws = forward(moe, g, k)
    got = torch.empty_like(sep)
    moe.moe_forward(g["x"], g["logits"], g["W1"], g["W3"], g["W2"], k, got, ws,
                    flags=moe.MOE_FWD_GATHER_ROWS | flags)
    assert moe.moe_get_error(ws) == 0
    assert torch.equal(got.view(torch.int16), sep.view(torch.int16))
    _oracle_check(got, g, k, "out (row gather, flags %d)" % flags)


@pytest.mark.parametrize("T,pinned,save", [
    (300, True, False),
    (300, False, False),   # pageable host buffers
    (1, True, False),
    (0, True, False),
    (200, True, True),     # saving for backward: moe_backward then runs on the same ws
])
def test_forward_host_equals_device(moe, T, pinned, save):
    d, E, k, dff = 256, 16, 4, 384
    w = moe_synth.custom(max(T, 1), d, E, k, dff, seed=77)
    inp = moe_synth.generate(w, with_dy=True)
    inp = moe_synth.rows(inp, T)
    g = to_dev(inp)
    ref, ws_ref = forward(moe, g, k, save=save)
    ws = torch.empty(moe.moe_workspace_bytes(T, d, E, k, dff, save, host_io=True),
                     dtype=torch.uint8, device="cuda")
    hx = inp["x"].clone().pin_memory() if pinned else inp["x"].clone()
    hl = inp["logits"].clone().pin_memory() if pinned else inp["logits"].clone()
    ho = torch.empty(T, d, dtype=torch.bfloat16)
    ho = ho.pin_memory() if pinned else ho
    ho.fill_(7.0)
    moe.moe_forward_host(hx, hl, g["W1"], g["W3"], g["W2"], k, ho, ws,
                         flags=moe.MOE_FWD_SAVE_FOR_BACKWARD if save else 0)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    assert torch.equal(ho.view(torch.int16), ref.cpu().view(torch.int16))
    if save:
        r_dev = backward(moe, g, k, ws_ref)
        r_host = backward(moe, g, k, ws)
        for name, v in r_dev.items():
            a = v.view(torch.int16) if v.dtype == torch.bfloat16 else v.view(torch.int32)
            b = r_host[name].view(torch.int16) if v.dtype == torch.bfloat16 else r_host[name].view(torch.int32)
            assert torch.equal(a, b), name


def test_forward_host_pipelined_back_to_back(moe):
    # six different batches through two workspaces, layers on one compute stream, copies on
    # one copy stream per workspace: each output is bitwise the device forward of its batch
    # (a copy that overtook a layer on a shared workspace would mix batches)
    T, d, E, k, dff = 1024, 512, 32, 4, 384
    nb = 6
    w = moe_synth.custom(T * nb, d, E, k, dff, seed=91, zipf_s=1.2)
    inp = moe_synth.generate(w)
    g = to_dev(inp)
    batches = [{"x": g["x"][i * T:(i + 1) * T].contiguous(),
                "logits": g["logits"][i * T:(i + 1) * T].contiguous(),
                "W1": g["W1"], "W3": g["W3"], "W2": g["W2"]} for i in range(nb)]
    refs = [forward(moe, b, k)[0].cpu() for b in batches]
    ws = [torch.empty(moe.moe_workspace_bytes(T, d, E, k, dff, False, host_io=True),
                      dtype=torch.uint8, device="cuda") for _ in range(2)]
    compute = torch.cuda.Stream()
    copies = [torch.cuda.Stream() for _ in range(2)]
    events = [[torch.cuda.Event(), torch.cuda.Event()] for _ in range(2)]
    hx = [b["x"].cpu().pin_memory() for b in batches]
    hl = [b["logits"].cpu().pin_memory() for b in batches]
    ho = [torch.full((T, d), 7.0, dtype=torch.bfloat16).pin_memory() for _ in range(nb)]
    torch.cuda.synchronize()
    for i in range(nb):
        j = i % 2
        moe.moe_forward_host_pipelined(hx[i], hl[i], g["W1"], g["W3"], g["W2"], k, ho[i], ws[j],
                                       copy_stream=copies[j], events=events[j], stream=compute)
    torch.cuda.synchronize()
    for x in ws:
        assert moe.moe_get_error(x) == 0
    for i in range(nb):
        assert torch.equal(ho[i].view(torch.int16), refs[i].view(torch.int16)), i
    # an empty batch between full ones: nothing to copy, the events still order the streams
    h0 = torch.empty(0, d, dtype=torch.bfloat16).pin_memory()
    l0 = torch.empty(0, E, dtype=torch.float32).pin_memory()
    moe.moe_forward_host_pipelined(h0, l0, g["W1"], g["W3"], g["W2"], k, h0, ws[0],
                                   copy_stream=copies[0], events=events[0], stream=compute)
    ho[0].fill_(7.0)
    moe.moe_forward_host_pipelined(hx[0], hl[0], g["W1"], g["W3"], g["W2"], k, ho[0], ws[0],
                                   copy_stream=copies[0], events=events[0], stream=compute)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws[0]) == 0
    assert torch.equal(ho[0].view(torch.int16), refs[0].view(torch.int16))


@pytest.mark.parametrize("T,flags", [(1, 0), (64, 0), (300, 0), (300, 2)])
def test_forward_graph_replays_the_layer(moe, T, flags):
    # a captured forward, replayed after the inputs are rewritten in place, gives bitwise
    # what a direct moe_forward gives on the new inputs
    d, E, k, dff = 256, 16, 4, 384
    w = moe_synth.custom(T, d, E, k, dff, seed=500 + T)
    g = to_dev(moe_synth.generate(w))
    x, logits = g["x"].clone(), g["logits"].clone()
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(moe.moe_workspace_bytes(T, d, E, k, dff), dtype=torch.uint8, device="cuda")
    graph = moe.moe_forward_graph_create(x, logits, g["W1"], g["W3"], g["W2"], k, out, ws,
                                         flags=flags)
    try:
        for rep in range(3):
            gen = torch.Generator(device="cuda")
            gen.manual_seed(rep)
            x.copy_(torch.randn(T, d, generator=gen, device="cuda").to(torch.bfloat16))
            logits.copy_(torch.randn(T, E, generator=gen, device="cuda"))
            graph.launch()
            ref, ws_ref = forward(moe, {**g, "x": x, "logits": logits}, k)
            torch.cuda.synchronize()
            assert moe.moe_get_error(ws) == 0 and moe.moe_get_error(ws_ref) == 0
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), rep
            _oracle_check(out, {**g, "x": x, "logits": logits}, k, "out (graph replay %d)" % rep)
    finally:
        graph.close()


def _device_workload(name):
    w = moe_synth.by_name(name)
    return w, moe_synth.generate(w, device="cuda")


def test_forward_sweep_batch_invariance(moe):
    # T in {1, 2, 4, ..., 128} over the same 128 token rows, d=7168, E=256, top-8, dff=2048
    w, g = _device_workload("sweep")
    outs = {}
    ws = torch.empty(moe.moe_workspace_bytes(128, w.d, w.E, w.k, w.dff, False),
                     dtype=torch.uint8, device="cuda")
    for T in w.sweep:
        out, _ = forward(moe, moe_synth.rows(g, T), w.k, ws=ws)
        assert moe.moe_get_error(ws) == 0
        outs[T] = out.clone()
    full = outs[128].view(torch.int16)
    for T in w.sweep:
        assert torch.equal(outs[T].view(torch.int16), full[:T]), T
    tok = np.array([0, 1, 5, 77, 127])
    npi = moe_synth.to_numpy(g)
    check_forward(outs[128], npi, w.k, "out (sweep, sampled tokens)", tokens=tok)


def test_forward_large_skewed_sampled(moe):
    w, g = _device_workload("large_skewed")
    out, ws = forward(moe, g, w.k)
    assert moe.moe_get_error(ws) == 0
    npi = moe_synth.to_numpy(g)
    idx, _ = oracle.route(npi["logits"], w.k)
    # sampled tokens plus tokens of the most and least loaded non-empty experts
    counts = np.bincount(idx.reshape(-1), minlength=w.E)
    hot = int(np.argmax(counts))
    cold = int(np.argmin(np.where(counts > 0, counts, 1 << 30)))
    extra = [int(np.nonzero((idx == e).any(1))[0][-1]) for e in (hot, cold)]
    tok = np.unique(np.concatenate([sample_tokens(w.T, 24, seed=3), extra]))
    check_forward(out, npi, w.k, "out (large skewed, sampled tokens)", tokens=tok)
