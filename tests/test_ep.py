"""Expert parallelism on one GPU: W ranks emulated in one process.

Each emulated rank holds a slice of the tokens and E/W experts' weights and runs its phases
through the library (route + permute over all experts, the expert stage on the rows it
receives, combine); the exchanges between ranks, which NCCL all-to-alls do between GPUs, are
done here by copying each rank's row runs into the others' receive buffers in the same order.
Nothing waits on another rank inside a kernel.  Checked against the CPU oracle of the whole
layer (all T tokens, all E experts):
  * routing of every token (expert sets on clear tokens, gates), as in the parity tests;
  * y on every token, |y - y_ref| <= tol (1 + |y_ref|);
  * the balancing scalar over all ranks (counts and softmax sums summed over the ranks, then
    moe_aux_from_totals) within 1e-5 of the oracle's;
  * y equal, within the same tolerance, to the single-GPU forward of the whole layer.
The exchange plan itself is checked bit-exact on the CPU with gloo ranks in
tests/test_ep_exchange.py.
"""
import numpy as np
import pytest
import torch

from top_routing_grouped_gb300.workloads import MoEShape, make_inputs

pytestmark = pytest.mark.gpu

CASES = [
    # (T, d, E, k, F, W, zipf, tau, path)
    (512, 256, 8, 2, 256, 2, False, 1.0, "auto"),
    (600, 256, 16, 4, 128, 2, True, 1.0, "auto"),    # ragged slices, one rank takes most rows, empty segments
    (1024, 256, 16, 4, 192, 4, False, 0.7, "auto"),
    (600, 256, 16, 4, 128, 2, True, 1.0, "tc1"),
    (600, 256, 16, 4, 128, 2, True, 1.0, "simt"),
    (4096, 2048, 8, 2, 8192, 2, False, 1.0, "auto"),  # the coarse-expert layer split over two ranks
]


def emulate_all_to_all(outs, sends, splits):
    """splits[r][j] rows of sends[r] (in order of j) go to rank j; rank j receives them source
    by source.  What one NCCL all-to-all per rank does, for every rank at once."""
    W = len(sends)
    for j in range(W):
        pieces = []
        for r in range(W):
            off = sum(splits[r][:j])
            pieces.append(sends[r][off:off + splits[r][j]])
        cat = torch.cat(pieces)
        outs[j][:cat.shape[0]].copy_(cat)


def run_ep(T, d, E, k, F, W, tau, path, inp):
    """One expert-parallel step over W emulated ranks; returns (ranks, y [T,d] host fp64, aux, segs)."""
    import parity
    from top_routing_grouped_gb300 import moe
    from top_routing_grouped_gb300.ep import EPRank, rows_per_rank
    dev = inp.to("cuda")
    has_bias = inp.bias is not None
    Tl, El = T // W, E // W
    ranks = [EPRank(Tl, d, E, k, F, W, r, dtype="bf16", tau=tau, has_bias=has_bias, path=path) for r in range(W)]
    xs = [dev.x[r * Tl:(r + 1) * Tl].contiguous() for r in range(W)]
    ys = [torch.empty(Tl, d, dtype=ranks[0].src.out_dtype, device="cuda") for _ in range(W)]
    w1 = [dev.w1[r * El:(r + 1) * El].contiguous() for r in range(W)]
    w3 = [dev.w3[r * El:(r + 1) * El].contiguous() for r in range(W)]
    w2 = [dev.w2[r * El:(r + 1) * El].contiguous() for r in range(W)]

    for r, rk in enumerate(ranks):                        # 1. route + dispatch, every rank
        rk.dispatch(xs[r], dev.w_router, dev.bias, ys[r])
    counts = [rk.counts().cpu() for rk in ranks]          # 2. counts exchange
    segs = [torch.cat([counts[j][r * El:(r + 1) * El] for j in range(W)]).cuda() for r in range(W)]
    send = [rows_per_rank(counts[r], W) for r in range(W)]
    recv = [rows_per_rank(segs[r].cpu(), W) for r in range(W)]
    N = Tl * k                                            # 3. rows and gates exchange
    emulate_all_to_all([rk.x_recv for rk in ranks], [rk.views["xp"][:N] for rk in ranks], send)
    emulate_all_to_all([rk.g_recv for rk in ranks], [rk.views["gate_perm"][:N] for rk in ranks], send)
    for r, rk in enumerate(ranks):                        # 4. the local experts
        rk.experts(segs[r], w1[r], w3[r], w2[r])
    emulate_all_to_all([rk.views["yp"] for rk in ranks], [rk.y_recv for rk in ranks], recv)   # 5. back
    for r, rk in enumerate(ranks):                        # 6. combine
        rk.combine(xs[r], dev.w_router, dev.bias, ys[r])
    tot_c = sum(rk.views["expert_counts"].clone() for rk in ranks)      # 7. aux over all ranks
    tot_p = sum(rk.views["expert_psum"].clone() for rk in ranks)
    aux = float(moe.aux_from_totals(E, k, T, tot_c.to(torch.int32), tot_p).item())
    torch.cuda.synchronize()
    for rk in ranks:
        assert rk.src.device_status(rk.ws) == moe.MOE_OK
        assert rk.exp.device_status(rk.ws_exp) == moe.MOE_OK
    assert sum(sum(rc) for rc in recv) == T * k
    y = np.concatenate([parity.to_np(yy) for yy in ys])
    return ranks, y, aux, segs


def check_against_oracle(T, d, E, k, F, tau, inp, ranks, y, aux, full_tokens):
    import oracle
    import parity
    host = inp.numpy_for_oracle()
    orc = oracle.Oracle(T, d, E, k, F, tau=tau, dtype="bf16")
    z, p, oidx, _ = orc.router(host["x"], host["wr"], host["bias"])
    gidx = np.concatenate([rk.views["topk_idx"].cpu().numpy() for rk in ranks])
    ggate = np.concatenate([rk.views["topk_gate"].cpu().numpy() for rk in ranks]).astype(np.float64)
    clear = parity.clear_tokens(z, k)
    np.testing.assert_array_equal(np.sort(gidx[clear], 1), np.sort(oidx[clear], 1))
    gref = np.take_along_axis(p, gidx, axis=1)
    assert np.max(np.abs(ggate - gref) / (gref + 1e-12)) <= parity.GATE_RTOL
    Tl = T // len(ranks)
    tokens = None if full_tokens else np.unique(np.concatenate([np.arange(0, T, 17), np.arange(Tl - 40, Tl + 40)]))
    yref = orc.combine(host["x"], host["w1"], host["w3"], host["w2"], gidx, gref, tokens)
    yg = y if tokens is None else y[tokens]
    err = np.abs(yg - yref) / (1 + np.abs(yref))
    assert err.max() <= parity.Y_TOL["bf16"], err.max()
    counts_all, _, _, _ = orc.dispatch(gidx)
    aux_ref = orc.aux(p, counts_all)
    assert abs(aux - aux_ref) <= parity.AUX_RTOL * abs(aux_ref), (aux, aux_ref)
    return float(err.max())


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T{}_d{}_E{}_k{}_F{}_W{}{}_{}".format(
    *c[:6], "_zipf" if c[6] else "", c[8]))
def test_expert_parallel_step_matches_the_oracle(case):
    import parity
    from top_routing_grouped_gb300 import moe
    T, d, E, k, F, W, zipf, tau, path = case
    s = MoEShape("ep", T=T, d=d, E=E, k=k, F=F, dtype="bf16", tau=tau, zipf_bias=zipf)
    inp = make_inputs(s, seed=5)
    ranks, y, aux, segs = run_ep(T, d, E, k, F, W, tau, path, inp)
    err = check_against_oracle(T, d, E, k, F, tau, inp, ranks, y, aux, full_tokens=T * d * F <= (1 << 31))
    print(f"\n[ep {case}] y max err {err:.2e}; segments {[sg.cpu().tolist() for sg in segs]}")
    # against the single-GPU forward of the whole layer
    plan = moe.MoEPlan(T, d, E, k, F, dtype="bf16", tau=tau, has_bias=zipf, path=path)
    got = parity.run_gpu(plan, inp.to("cuda"))
    y1 = parity.to_np(got["y"])
    assert np.max(np.abs(y - y1) / (1 + np.abs(y1))) <= parity.Y_TOL["bf16"]


def test_expert_parallel_degenerate_layouts():
    """W = 1 (one rank holds every expert: one segment per expert), and W = 2 with a router
    bias that keeps every token off rank 1's experts (rank 1 receives no rows, its expert
    stage has an empty tile table, and it sends none back)."""
    T, d, E, k, F, tau = 256, 256, 8, 2, 128, 1.0
    s = MoEShape("ep1", T=T, d=d, E=E, k=k, F=F, dtype="bf16", tau=tau)
    inp = make_inputs(s, seed=9)
    ranks, y, aux, segs = run_ep(T, d, E, k, F, 1, tau, "auto", inp)
    check_against_oracle(T, d, E, k, F, tau, inp, ranks, y, aux, full_tokens=True)
    inp.bias = torch.zeros(E, dtype=torch.float32)
    inp.bias[E // 2:] = -100.0
    ranks, y, aux, segs = run_ep(T, d, E, k, F, 2, tau, "auto", inp)
    assert int(segs[1].sum()) == 0 and int(segs[0].sum()) == T * k
    check_against_oracle(T, d, E, k, F, tau, inp, ranks, y, aux, full_tokens=True)


def test_expert_stage_rejects_counts_beyond_its_rows():
    """Segment counts that add up to more rows than the plan holds are reported on the device
    (MOE_ERR_INTERNAL) and no tile runs."""
    from top_routing_grouped_gb300 import moe
    plan = moe.ExpertPlan(256, 128, 2, 2, 64)
    ws = plan.new_workspace()
    x = torch.zeros(256, 128, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(256, dtype=torch.float32, device="cuda")
    y = torch.full((256, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(2, 64, 128, dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros(2, 128, 64, dtype=torch.bfloat16, device="cuda")
    seg = torch.tensor([100, 100, 100, 0], dtype=torch.int32, device="cuda")   # 300 > 256
    plan.forward(seg, x, g, w, w, w2, y, ws)
    assert plan.device_status(ws) == moe.MOE_ERR_INTERNAL
    assert torch.all(y == 7.0), "no row may be written"
    seg = torch.tensor([100, -1, 0, 0], dtype=torch.int32, device="cuda")
    plan.forward(seg, x, g, w, w, w2, y, ws)
    assert plan.device_status(ws) == moe.MOE_ERR_INTERNAL
    seg = torch.tensor([100, 50, 0, 106], dtype=torch.int32, device="cuda")    # exactly 256: fine
    plan.forward(seg, x, g, w, w, w2, y, ws)
    assert plan.device_status(ws) == moe.MOE_OK
    torch.cuda.synchronize()
    assert torch.all(y == 0.0)
