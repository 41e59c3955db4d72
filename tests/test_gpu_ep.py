"""The pull-based row copies of the expert-parallel path (moe_ep_copy_rows) on one GPU.

Three ranks are emulated on one device: each holds its own batch and its own permuted rows
from moe_route_dispatch, and the "peer" pointers are these buffers on the same GPU (no rank
waits on another, so the emulation is exact).  The tests check two things:
- Owner side: the rows each owner pulls with moe_ep_plan's segments are bitwise the rows that
  a single-GPU dispatch of the concatenated batch gives its experts, in the same order.
- Source side: the output rows each rank pulls back with moe_ep_return_plan land bitwise in
  its permuted slots.
A segment outside its buffers is rejected on the device (MOE_ERR_DEVICE_BOUNDS) and writes
nothing.
"""
import numpy as np
import pytest
import torch

import moe_synth
from moe_harness import route_dispatch, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import combine_fp32_router_gb300 as m
    return m


def _segments(dev, src_rank, src_row, dst_row, rows):
    t = lambda a: torch.tensor(np.asarray(a, np.int32), dtype=torch.int32, device=dev)
    return t(src_rank), t(src_row), t(dst_row), t(rows)


def test_ep_pull_and_return_match_the_single_gpu_dispatch(moe):
    R, Tl, d, E, k = 3, 300, 256, 10, 3
    w = moe_synth.custom(R * Tl, d, E, k, 128, seed=71, zipf_s=1.2)
    g = to_dev(moe_synth.generate(w))
    dev = g["x"].device
    ranks = [route_dispatch(moe, {"x": g["x"][r * Tl:(r + 1) * Tl].contiguous(),
                                  "logits": g["logits"][r * Tl:(r + 1) * Tl].contiguous()}, k)
             for r in range(R)]
    whole = route_dispatch(moe, g, k)
    counts_all = np.stack([rk["counts"].cpu().numpy() for rk in ranks]).astype(np.int32)
    assert np.array_equal(counts_all.sum(0), whole["counts"].cpu().numpy())
    peers = torch.tensor([rk["x_perm"].data_ptr() for rk in ranks], dtype=torch.int64,
                         device=dev)
    peer_rows = torch.tensor([rk["x_perm"].shape[0] for rk in ranks], dtype=torch.int64,
                             device=dev)
    err = torch.zeros(64, dtype=torch.uint8, device=dev)
    woff = whole["offsets"].cpu().numpy()
    y_recv = []
    for r in range(R):
        pl = moe.moe_ep_plan(counts_all, r, row_align=128, wave_experts=2)
        e0 = moe.moe_ep_first_expert(E, R, r)
        nloc = pl["recv_counts"].shape[0]
        recv = torch.full((max(pl["rows"], 1), d), 7.0, dtype=torch.bfloat16, device=dev)
        # one launch per wave, as the pipelined path would issue them
        for wv in range(len(pl["waves"]) - 1):
            seg = [(s, pl["src_off"][i, s], pl["recv_off"][i, s], counts_all[s, e0 + i])
                   for i in range(pl["waves"][wv], pl["waves"][wv + 1]) for s in range(R)]
            moe.moe_ep_copy_rows(peers, peer_rows, *_segments(dev, *zip(*seg)), recv, err)
        assert moe.moe_get_error(err) == moe.MOE_OK
        for i in range(nloc):
            e = e0 + i
            a, n = pl["recv_off"][i, 0], pl["recv_counts"][i]
            got = recv[a:a + n].view(torch.int16)
            ref = whole["x_perm"][woff[e]:woff[e] + n].view(torch.int16)
            assert torch.equal(got, ref), e
        # stand-in expert outputs of this owner (fp32 rows, distinct per row)
        y = torch.randn(max(pl["rows"], 1), d, device=dev,
                        generator=torch.Generator(device=dev).manual_seed(r))
        y_recv.append(y)
    # return leg: every rank pulls its rows back from the owners
    ypeers = torch.tensor([y.data_ptr() for y in y_recv], dtype=torch.int64, device=dev)
    yrows = torch.tensor([y.shape[0] for y in y_recv], dtype=torch.int64, device=dev)
    for s in range(R):
        owner, orow, own = moe.moe_ep_return_plan(counts_all, s, row_align=128)
        seg = [(owner[e], orow[e], own[e], counts_all[s, e]) for e in range(E)]
        y_perm = torch.full((Tl * k, d), -3.0, dtype=torch.float32, device=dev)
        moe.moe_ep_copy_rows(ypeers, yrows, *_segments(dev, *zip(*seg)), y_perm, err)
        assert moe.moe_get_error(err) == moe.MOE_OK
        own_off = np.concatenate([[0], np.cumsum(counts_all[s])])
        for e in range(E):
            n = counts_all[s, e]
            if n:
                assert torch.equal(y_perm[own_off[e]:own_off[e] + n],
                                   y_recv[owner[e]][orow[e]:orow[e] + n]), (s, e)
        assert (y_perm != -3.0).all()   # every slot was filled


def test_ep_copy_rows_rejects_segments_outside_the_buffers(moe):
    dev = torch.device("cuda")
    src = torch.arange(64 * 32, dtype=torch.float32, device=dev).view(64, 32)
    peers = torch.tensor([src.data_ptr()], dtype=torch.int64, device=dev)
    rows = torch.tensor([64], dtype=torch.int64, device=dev)
    dst = torch.zeros(16, 32, dtype=torch.float32, device=dev)
    err = torch.zeros(64, dtype=torch.uint8, device=dev)
    # the second segment reads past the source's 64 rows; the third writes past dst's 16
    moe.moe_ep_copy_rows(peers, rows, *_segments(dev, [0, 0, 0], [2, 60, 0], [0, 4, 10],
                                                 [4, 8, 8]), dst, err)
    assert moe.moe_get_error(err) == moe.MOE_ERR_DEVICE_BOUNDS
    assert torch.equal(dst[:4], src[2:6])
    assert (dst[4:] == 0).all()


@pytest.mark.parametrize("gated,waves", [(True, False), (False, False), (True, True)])
def test_ep_layer_end_to_end_matches_the_single_gpu_forward(moe, gated, waves):
    # Three emulated ranks run the whole expert-parallel layer: dispatch their own tokens,
    # owners pull their experts' rows, run the expert stage on the receive buffer
    # (moe_expert_forward), every rank pulls its rows' outputs back and combines them
    # (moe_combine).  Each rank's output is bitwise the single-GPU forward's rows for its
    # tokens.  With waves, an owner pulls wave i+1's rows on a copy stream while the expert
    # stage of wave i runs on its own slice of the receive buffer.
    from moe_harness import forward
    R, Tl, d, E, k = 3, 300, 256, 10, 3
    dff = 384 if gated else 256
    w = moe_synth.custom(R * Tl, d, E, k, dff, seed=72, zipf_s=1.2, gated=gated)
    g = to_dev(moe_synth.generate(w))
    dev = g["x"].device
    ref, ws_ref = forward(moe, g, k)
    assert moe.moe_get_error(ws_ref) == moe.MOE_OK
    ranks = [route_dispatch(moe, {"x": g["x"][r * Tl:(r + 1) * Tl].contiguous(),
                                  "logits": g["logits"][r * Tl:(r + 1) * Tl].contiguous()}, k)
             for r in range(R)]
    counts_all = np.stack([rk["counts"].cpu().numpy() for rk in ranks]).astype(np.int32)
    peers = torch.tensor([rk["x_perm"].data_ptr() for rk in ranks], dtype=torch.int64,
                         device=dev)
    peer_rows = torch.tensor([rk["x_perm"].shape[0] for rk in ranks], dtype=torch.int64,
                             device=dev)
    err = torch.zeros(64, dtype=torch.uint8, device=dev)
    y_out = []
    for r in range(R):
        pl = moe.moe_ep_plan(counts_all, r, row_align=128, wave_experts=2)
        e0 = moe.moe_ep_first_expert(E, R, r)
        nloc = pl["recv_counts"].shape[0]
        rows = max(pl["rows"], 1)
        recv = torch.full((rows, d), 7.0, dtype=torch.bfloat16, device=dev)
        cnt = torch.tensor(np.asarray(pl["recv_counts"], np.int32), device=dev)
        y = torch.full((rows, d), -5.0, dtype=torch.bfloat16, device=dev)
        W3 = g["W3"] if gated else None
        # waves of experts [a, b): their rows are [recv_off[a, 0], recv_off[b, 0]) of the
        # receive buffer, each expert's from a 128-row boundary
        bounds = list(pl["waves"]) if waves else [0, nloc]
        copy, comp = torch.cuda.Stream(dev), torch.cuda.current_stream(dev)
        pulled = []
        for wv in range(len(bounds) - 1):
            a, b = bounds[wv], bounds[wv + 1]
            seg = [(s, pl["src_off"][i, s], pl["recv_off"][i, s], counts_all[s, e0 + i])
                   for i in range(a, b) for s in range(R)]
            with torch.cuda.stream(copy):
                moe.moe_ep_copy_rows(peers, peer_rows, *_segments(dev, *zip(*seg)), recv, err,
                                     stream=copy)
                ev = torch.cuda.Event()
                ev.record(copy)
            pulled.append(ev)
        for wv in range(len(bounds) - 1):
            a, b = bounds[wv], bounds[wv + 1]
            r0 = int(pl["recv_off"][a, 0])
            r1 = int(pl["recv_off"][b, 0]) if b < nloc else pl["rows"]
            if r1 == r0:
                continue
            comp.wait_event(pulled[wv])
            ws = torch.empty(moe.moe_expert_workspace_bytes(r1 - r0, d, b - a, dff),
                             dtype=torch.uint8, device=dev)
            moe.moe_expert_forward(recv[r0:r1], cnt[a:b], g["W1"][e0 + a:e0 + b],
                                   W3[e0 + a:e0 + b] if gated else None,
                                   g["W2"][e0 + a:e0 + b], y[r0:r1], ws)
            assert moe.moe_get_error(ws) == moe.MOE_OK
        assert moe.moe_get_error(err) == moe.MOE_OK
        y_out.append(y)
    ypeers = torch.tensor([y.data_ptr() for y in y_out], dtype=torch.int64, device=dev)
    yrows = torch.tensor([y.shape[0] for y in y_out], dtype=torch.int64, device=dev)
    for s in range(R):
        owner, orow, own = moe.moe_ep_return_plan(counts_all, s, row_align=128)
        seg = [(owner[e], orow[e], own[e], counts_all[s, e]) for e in range(E)]
        y_perm = torch.empty(Tl * k, d, dtype=torch.bfloat16, device=dev)
        moe.moe_ep_copy_rows(ypeers, yrows, *_segments(dev, *zip(*seg)), y_perm, err)
        out = torch.empty(Tl, d, dtype=torch.bfloat16, device=dev)
        moe.moe_combine(y_perm, ranks[s]["gate"], ranks[s]["pos"], out, err)
        assert moe.moe_get_error(err) == moe.MOE_OK
        assert torch.equal(out.view(torch.int16), ref[s * Tl:(s + 1) * Tl].view(torch.int16)), s


def test_combine_rejects_rows_outside_its_buffer(moe):
    dev = torch.device("cuda")
    y = torch.ones(8, 128, dtype=torch.bfloat16, device=dev)
    gate = torch.full((2, 2), 0.5, dtype=torch.float32, device=dev)
    pos = torch.tensor([[0, 1], [2, 8]], dtype=torch.int32, device=dev)   # row 8 is past y
    out = torch.empty(2, 128, dtype=torch.bfloat16, device=dev)
    err = torch.zeros(64, dtype=torch.uint8, device=dev)
    moe.moe_combine(y, gate, pos, out, err)
    assert moe.moe_get_error(err) == moe.MOE_ERR_DEVICE_BOUNDS
    assert (out[0] == 1.0).all()
