"""The exchange plan of expert parallelism on the CPU: W gloo ranks, no GPU.

Each rank routes its own slice of the tokens with the CPU oracle and dispatches it
(orc_dispatch over its slice).  The rows it sends are labels -- the global token id and the
global slot of each dispatched row -- so that what arrives can be checked exactly:
  * counts: the segment counts a rank receives are the other ranks' per-expert counts of its
    experts;
  * dispatch: for every local expert, the rows received from source 0, 1, ... in that order
    are exactly the rows of that expert in the oracle's dispatch of ALL tokens (stable in
    token order), bit for bit;
  * combine: rows sent back land in each source's own dispatch order, so row p of the source
    gets back the label it sent as row p.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CASES = {
    # name: (T, d, E, k, W, zipf)
    "w2_even": (256, 32, 8, 2, 2, False),
    "w2_skewed_ragged": (300, 32, 16, 4, 2, True),    # one rank receives most rows, empty segments
    "w4": (512, 32, 16, 4, 4, False),
}


def _routing(case):
    from top_routing_grouped_gb300.workloads import MoEShape, make_inputs
    import oracle
    T, d, E, k, W, zipf = case
    s = MoEShape("ep", T=T, d=d, E=E, k=k, F=8, dtype="f32", zipf_bias=zipf)
    inp = make_inputs(s, seed=11, parts=("x", "wr")).numpy_for_oracle()
    return s, inp, oracle


def _rank_main(rank, world, port, case, q):
    from top_routing_grouped_gb300 import ep
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        s, inp, oracle = _routing(case)
        T, d, E, k, W, _ = case
        Tl, El = T // W, E // W
        t0 = rank * Tl
        orc = oracle.Oracle(Tl, d, E, k, 8)
        _, _, idx, _ = orc.router(np.ascontiguousarray(inp["x"][t0:t0 + Tl]), inp["wr"], inp["bias"])
        counts, offsets, perm_src, perm_slot = orc.dispatch(idx)
        # labels of the dispatched rows: global token and global slot
        rows = torch.stack([torch.as_tensor(perm_src.astype(np.int64) + t0),
                            torch.as_tensor(perm_slot.astype(np.int64) + t0 * k)], dim=1)
        c = torch.as_tensor(counts)
        seg = ep.exchange_counts(c, W)
        send = ep.rows_per_rank(c, W)
        recv = ep.rows_per_rank(seg, W)
        out = torch.full((W * Tl * min(k, El), 2), -1, dtype=torch.int64)
        got = ep.exchange_rows(out, rows, send, recv).clone()
        # the expert stage would compute here; send the labels back unchanged
        back = torch.full_like(rows, -1)
        ep.exchange_rows(back, got, recv, send)
        q.put((rank, seg.numpy().copy(), got.numpy().copy(), back.numpy().copy(), rows.numpy().copy(),
               np.asarray(send), np.asarray(recv), counts.copy()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name", sorted(CASES))
def test_exchange_plan_matches_the_global_dispatch(name):
    case = CASES[name]
    T, d, E, k, W, _ = case
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, W, port, case, q)) for r in range(W)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(W):
        r, *vals = q.get(timeout=180)
        res[r] = vals
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # the oracle's dispatch of all T tokens at once
    s, inp, oracle = _routing(case)
    orc = oracle.Oracle(T, d, E, k, 8)
    _, _, idx, _ = orc.router(inp["x"], inp["wr"], inp["bias"])
    counts, offsets, perm_src, perm_slot = orc.dispatch(idx)
    El, Tl = E // W, T // W
    for r in range(W):
        seg, got, back, rows, send, recv, _ = res[r]
        seg = seg.reshape(W, El)
        # counts: row j = source j's per-expert counts of my experts
        for j in range(W):
            np.testing.assert_array_equal(seg[j], res[j][6][r * El:(r + 1) * El])
        np.testing.assert_array_equal(seg.sum(axis=0), counts[r * El:(r + 1) * El])
        assert got.shape[0] == seg.sum() == recv.sum()
        # dispatch: per local expert, rows from source 0, 1, ... = the global dispatch's rows
        off = np.concatenate([[0], np.cumsum(seg.reshape(-1))])
        for e in range(El):
            ge = r * El + e
            mine = np.concatenate([got[off[j * El + e]:off[j * El + e + 1]] for j in range(W)])
            np.testing.assert_array_equal(mine[:, 0], perm_src[offsets[ge]:offsets[ge + 1]])
            np.testing.assert_array_equal(mine[:, 1], perm_slot[offsets[ge]:offsets[ge + 1]])
        # combine: every row comes back to its own place
        np.testing.assert_array_equal(back, rows)
        assert send.sum() == Tl * k
    # every segment of every rank accounted for; the skewed case leaves some empty
    all_seg = np.concatenate([res[r][0] for r in range(W)])
    assert all_seg.sum() == T * k
    if case[5]:
        assert (all_seg == 0).any()


def test_rows_per_rank_sums_each_destination():
    from top_routing_grouped_gb300 import ep
    assert ep.rows_per_rank(torch.tensor([1, 2, 3, 4, 0, 6], dtype=torch.int32), 3) == [3, 7, 6]
    assert ep.rows_per_rank(torch.tensor([5, 0], dtype=torch.int32), 1) == [5]
