"""Fine-grained expert parallelism across GPUs: the exchange protocol on the CPU (gloo).

The layer is split across R ranks, each of which routes and dispatches its own tokens, with
experts owned in contiguous blocks.  The path then runs:
1. all-gather the per-expert counts;
2. each owner pulls the rows of its experts from every rank, at the offsets moe_ep_plan
   gives (here an all-gather of the ranks' permuted buffers stands in for the peer reads of
   moe_ep_copy_rows);
3. the owner computes the experts on the received rows;
4. each rank pulls its rows' outputs back at the offsets moe_ep_return_plan gives;
5. each rank combines them in slot order.

The result must be bitwise the single-process oracle's forward of the concatenated batch:
the plan must deliver each expert's rows in the single-GPU (expert, token) order, and every
output row back to the slot it came from.  Expert math and routing come from the fp64
oracle; the plans come from the library's C entry points (host code, no GPU).
"""
import math
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bf16_bits(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)


def _global_batch(T, d, E, dff, seed):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits -= (1.2 * np.log(np.arange(E) + 1.0)).astype(np.float32)  # skewed loads
    return dict(x=_bf16_bits(rng.standard_normal((T, d))), logits=logits,
                W1=_bf16_bits(rng.standard_normal((E, d, dff)) / math.sqrt(d)),
                W3=_bf16_bits(rng.standard_normal((E, d, dff)) / math.sqrt(d)),
                W2=_bf16_bits(rng.standard_normal((E, dff, d)) / math.sqrt(dff)))


def _expert_rows(inp, rows_x, e):
    """Expert e on the given bf16 rows: the oracle's forward with one expert selected (k=1,
    gate exactly 1)."""
    n = rows_x.shape[0]
    E = inp["W1"].shape[0]
    lg = np.zeros((n, E), np.float32)
    lg[:, e] = 1.0
    return oracle_forward({**inp, "x": rows_x, "logits": lg}, 1)


def oracle_forward(inp, k, tokens=None):
    sys.path.insert(0, ROOT)
    import oracle
    return oracle.forward_tokens(inp, k, tokens=tokens)


def _rank_main(rank, R, port, shape, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import oracle
    import combine_fp32_router_gb300 as moe
    dist.init_process_group("gloo", rank=rank, world_size=R)
    try:
        Tl, d, E, k, dff, seed = shape
        inp = _global_batch(Tl * R, d, E, dff, seed)
        t0 = rank * Tl
        mine = {**inp, "x": inp["x"][t0:t0 + Tl], "logits": inp["logits"][t0:t0 + Tl]}
        # local route + dispatch (the oracle stands in for moe_route_dispatch on this rank)
        idx, gate = oracle.route(mine["logits"], k)
        counts, offsets, perm, pos = oracle.dispatch(idx, E)
        x_perm = mine["x"][perm // k]                           # [Tl k, d] bf16 bits
        parts = [torch.zeros(E, dtype=torch.int32) for _ in range(R)]
        dist.all_gather(parts, torch.from_numpy(counts.astype(np.int32)))
        counts_all = torch.stack(parts).numpy()
        # every rank's permuted rows, padded to the largest (the stand-in for peer reads)
        P = Tl * k
        allx = [torch.zeros(P, d // 2, dtype=torch.int32) for _ in range(R)]  # bf16 pairs
        dist.all_gather(allx, torch.from_numpy(np.ascontiguousarray(x_perm).view(np.int32)))
        allx = [a.numpy().view(np.uint16) for a in allx]
        # 1-2: this rank's receive buffer, filled wave by wave from the plan
        plan = moe.moe_ep_plan(counts_all, rank, row_align=128, wave_experts=2)
        e0 = moe.moe_ep_first_expert(E, R, rank)
        nloc = moe.moe_ep_first_expert(E, R, rank + 1) - e0
        recv = np.zeros((plan["rows"], d), np.uint16)
        waves = plan["waves"]
        assert waves[0] == 0 and waves[-1] == nloc and len(waves) == (nloc + 1) // 2 + 1
        for w in range(len(waves) - 1):
            for i in range(waves[w], waves[w + 1]):
                for s in range(R):
                    n = counts_all[s, e0 + i]
                    a, b = plan["recv_off"][i, s], plan["src_off"][i, s]
                    recv[a:a + n] = allx[s][b:b + n]
        # 3: the experts on the received rows (the oracle's bf16 output rows, held as fp64)
        y_recv = np.zeros((plan["rows"], d))
        for i in range(nloc):
            a, n = plan["recv_off"][i, 0], plan["recv_counts"][i]
            assert n == counts_all[:, e0 + i].sum()
            if n:
                y_recv[a:a + n] = _expert_rows(inp, recv[a:a + n], e0 + i)
        # 4: pull this rank's output rows back from their owners
        top = max(_all_rows(counts_all, R, moe))   # every owner's buffer, padded alike
        ally = [torch.zeros(max(top, 1), d, dtype=torch.float64) for _ in range(R)]
        dist.all_gather(ally, _pad(y_recv, top, d))
        owner, owner_row, own_row = moe.moe_ep_return_plan(counts_all, rank, row_align=128)
        y_perm = np.zeros((P, d))
        for e in range(E):
            n = counts_all[rank, e]
            y_perm[own_row[e]:own_row[e] + n] = \
                ally[owner[e]].numpy()[owner_row[e]:owner_row[e] + n]
        # 5: combine in slot order
        out = np.zeros((Tl, d))
        for j in range(k):
            out += gate[:, j:j + 1] * y_perm[pos.reshape(Tl, k)[:, j]]
        ref = oracle.forward_tokens(inp, k, tokens=np.arange(t0, t0 + Tl))
        q.put((rank, bool(np.array_equal(out, ref)), float(np.abs(out - ref).max())))
    finally:
        dist.destroy_process_group()


def _all_rows(counts_all, R, moe):
    return [moe.moe_ep_plan(counts_all, r)["rows"] for r in range(R)]


def _pad(a, rows, d):
    out = torch.zeros(max(rows, 1), d, dtype=torch.float64)
    out[:a.shape[0]] = torch.from_numpy(a)
    return out


@pytest.mark.parametrize("R,shape", [
    (2, (48, 128, 8, 2, 128, 1)),
    (3, (40, 128, 7, 3, 128, 2)),   # E not a multiple of R: blocks of 2, 2 and 3 experts
])
def test_ep_protocol_matches_the_single_process_layer(R, shape):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, R, port, shape, q)) for r in range(R)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(R))
    assert all(ok for _, ok, _ in got), got


def test_ep_plan_invariants():
    sys.path.insert(0, ROOT)
    import combine_fp32_router_gb300 as moe
    rng = np.random.default_rng(3)
    for R, E in ((1, 5), (2, 8), (3, 7), (4, 32), (8, 256)):
        counts = rng.integers(0, 300, size=(R, E)).astype(np.int32)
        counts[:, rng.integers(0, E)] = 0   # an expert nobody routes to
        firsts = [moe.moe_ep_first_expert(E, R, r) for r in range(R + 1)]
        assert firsts[0] == 0 and firsts[-1] == E and all(np.diff(firsts) >= 1)
        for r in range(R):
            pl = moe.moe_ep_plan(counts, r, row_align=128, wave_experts=3)
            e0, e1 = firsts[r], firsts[r + 1]
            assert np.array_equal(pl["recv_counts"], counts[:, e0:e1].sum(0))
            # every expert's rows start on a 128-row boundary, sources back to back
            starts = pl["recv_off"][:, 0]
            assert (starts % 128 == 0).all()
            for i in range(e1 - e0):
                assert np.array_equal(np.diff(pl["recv_off"][i]), counts[:-1, e0 + i])
            ends = starts + pl["recv_counts"]
            assert (ends <= np.append(starts[1:], pl["rows"])).all()
            # the layout moe_expert_forward reads: expert i from the exclusive prefix of the
            # counts rounded up to 128, the buffer exactly their sum
            padded = -(-pl["recv_counts"].astype(np.int64) // 128) * 128
            assert np.array_equal(starts, np.concatenate([[0], np.cumsum(padded)[:-1]]))
            assert pl["rows"] == int(padded.sum())
            # sources: the exclusive prefix of each rank's counts (its dispatch offsets)
            excl = np.concatenate([np.zeros((R, 1), np.int64), np.cumsum(counts, 1)], 1)
            assert np.array_equal(pl["src_off"], excl[:, e0:e1].T)
            # return plan of every rank points at the same rows from the other side
            for s in range(R):
                owner, orow, own = moe.moe_ep_return_plan(counts, s, row_align=128)
                for i in range(e1 - e0):
                    assert owner[e0 + i] == r and orow[e0 + i] == pl["recv_off"][i, s]
                    assert own[e0 + i] == pl["src_off"][i, s]


def test_ep_plan_rejects_bad_arguments():
    sys.path.insert(0, ROOT)
    import combine_fp32_router_gb300 as moe
    c = np.ones((2, 4), np.int32)
    with pytest.raises(moe.MoeError):
        moe.moe_ep_plan(c, 2)                 # rank out of range
    bad = c.copy()
    bad[1, 2] = -1
    with pytest.raises(moe.MoeError):
        moe.moe_ep_plan(bad, 0)               # negative count
    with pytest.raises(moe.MoeError):
        moe.moe_ep_plan(np.ones((5, 4), np.int32), 0)   # more ranks than experts
    assert moe.moe_ep_first_expert(4, 0, 0) == -1
