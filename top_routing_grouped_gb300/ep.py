"""Expert parallelism over W ranks ("Distributed Training Part 4", §4 Expert Parallelism:
the experts are spread over the GPUs; Dispatch sends every routed row to the GPU that holds
its expert, the experts run there, Combine sends the outputs back to their tokens).

Rank r holds its own T_local tokens, the whole router, and the weights of E_l = E / W
experts (global experts r*E_l .. (r+1)*E_l - 1).  Its dispatch order (the permute of
moe_forward) is expert-contiguous, hence destination-rank-contiguous, so the row exchange is
one all-to-all of the rows as they lie; what a rank receives is W*E_l segments, source-major,
on which the library's expert stage (moe_expert_forward) runs the grouped GEMMs in place.

The exchange plan -- rows per destination, segment counts -- is host logic in this module and
runs on CPU tensors too (the gloo tests); the collectives are torch.distributed (NCCL between
GPUs).  Every arithmetic step of the layer runs in the library's kernels; this module only
moves rows between ranks and marshals arguments.  The library itself is imported lazily, so
the exchange plan can be used and tested without a GPU.
"""
import torch
import torch.distributed as dist


def rows_per_rank(counts, world):
    """Rows a rank sends to each destination: its per-expert counts [E] summed over each
    destination's E/W experts (host list of W ints)."""
    c = torch.as_tensor(counts).reshape(world, -1)
    return [int(v) for v in c.sum(dim=1).tolist()]


def exchange_counts(counts, world, group=None):
    """All-to-all of the per-expert counts viewed [W, E_l]: returns this rank's segment counts
    [W * E_l] (row s = source s, column = local expert), in the tensor's device and dtype."""
    seg = torch.empty_like(counts)
    dist.all_to_all_single(seg, counts.contiguous(), group=group)
    return seg


def exchange_rows(out, send, send_splits, recv_splits, group=None):
    """All-to-all of rows: send[ sum(send_splits[:j]) : +send_splits[j] ] goes to rank j;
    what rank i sends lands in out[ sum(recv_splits[:i]) : +recv_splits[i] ].  Returns the
    filled prefix of `out`."""
    n = sum(recv_splits)
    view = out[:n]
    dist.all_to_all_single(view, send[:sum(send_splits)].contiguous(), output_split_sizes=list(recv_splits),
                           input_split_sizes=list(send_splits), group=group)
    return view


class EPRank:
    """One rank's part of an expert-parallel MoE layer.

    T_local tokens on this rank; d, E (all experts), k, F as in the layer; world = W ranks,
    rank = r.  The step is split into the phases below so that the ranks' exchanges can be
    driven either by torch.distributed (forward) or by a caller that holds every rank
    (the single-process emulation in the tests)."""

    def __init__(self, T_local, d, E, k, F, world, rank, dtype="bf16", tau=1.0, has_bias=False, path="auto",
                 renorm_gates=False, device="cuda"):
        from . import moe
        if E % world != 0:
            raise ValueError("the experts must split evenly over the ranks")
        self.moe = moe
        self.T, self.d, self.E, self.k, self.F = int(T_local), int(d), int(E), int(k), int(F)
        self.world, self.rank = int(world), int(rank)
        self.E_l = self.E // self.world
        self.src = moe.MoEPlan(T_local, d, E, k, F, dtype=dtype, tau=tau, has_bias=has_bias, path=path,
                               renorm_gates=renorm_gates)
        # dropless: every token of every rank may send up to min(k, E_l) rows here
        self.max_rows = self.world * self.T * min(self.k, self.E_l)
        self.exp = moe.ExpertPlan(self.max_rows, d, self.E_l, self.world, F, dtype=dtype, path=path)
        self.ws = self.src.new_workspace(device)
        self.ws_exp = self.exp.new_workspace(device)
        self.views = self.src.views(self.ws)
        act = self.src.act_dtype
        self.x_recv = torch.empty(self.max_rows, d, dtype=act, device=device)
        self.g_recv = torch.empty(self.max_rows, dtype=torch.float32, device=device)
        self.y_recv = torch.empty(self.max_rows, d, dtype=act, device=device)
        self.N = self.T * self.k

    # phase 1: route and dispatch the rank's own tokens over all E experts
    def dispatch(self, x, w_router, bias, y, stream=None):
        for stage in ("route", "permute"):
            self.src.forward_stage(self.src.stage_names.index(stage), x, w_router, bias, x, x, x, y, self.ws,
                                   stream=stream)

    def counts(self):
        """Per-expert counts of this rank's rows [E] (device, int32), = [W, E_l] by destination."""
        return self.views["expert_counts"]

    def send_rows(self):
        """Dispatched rows and their gates, destination-major (device views of N rows)."""
        return self.views["xp"], self.views["gate_perm"]

    # phase 4: the local experts on the received segments
    def experts(self, seg_counts, w1_local, w3_local, w2_local, stream=None):
        self.exp.forward(seg_counts, self.x_recv, self.g_recv, w1_local, w3_local, w2_local, self.y_recv, self.ws_exp,
                         stream=stream)

    # phase 6: combine the returned rows (already in this rank's Yp) into y
    def combine(self, x, w_router, bias, y, stream=None):
        self.src.forward_stage(self.src.stage_names.index("combine"), x, w_router, bias, x, x, x, y, self.ws,
                               stream=stream)

    def forward(self, x, w_router, bias, w1_local, w3_local, w2_local, y, group=None):
        """The whole step with torch.distributed collectives (every rank calls it)."""
        self.dispatch(x, w_router, bias, y)
        counts = self.counts()
        seg = exchange_counts(counts, self.world, group)
        send = rows_per_rank(counts.cpu(), self.world)
        recv = rows_per_rank(seg.cpu(), self.world)
        xp, gp = self.send_rows()
        exchange_rows(self.x_recv, xp, send, recv, group)
        exchange_rows(self.g_recv, gp, send, recv, group)
        self.experts(seg, w1_local, w3_local, w2_local)
        exchange_rows(self.views["yp"], self.y_recv, recv, send, group)
        self.combine(x, w_router, bias, y)

    def aux_loss(self, T_total, group=None, out=None):
        """The balancing scalar over every rank's tokens: counts and softmax sums all-reduced,
        then moe_aux_from_totals (every rank calls it)."""
        c = self.views["expert_counts"].clone()
        p = self.views["expert_psum"].clone()
        dist.all_reduce(c, group=group)
        dist.all_reduce(p, group=group)
        return self.moe.aux_from_totals(self.E, self.k, T_total, c, p, out=out)
