"""Helpers that run the CUDA path through the C ABI and compare it with the CPU oracle.

Comparison rules (tolerances derived in the design notes):
  * logits:   |z_gpu - z| <= 1e-5 (1 + |z|)
  * routing:  for every *clear* token, i.e. one whose fp32 logits have
              z_(k) - z_(k+1) > 1e-4 (k = E: every token is clear), the chosen expert set is
              bit-exact and the slot order descends in the oracle's logits up to 1e-4 (two
              chosen experts closer than that may swap slots); every other token is checked
              against the oracle run with the GPU's own choice;
  * gates:    |g_gpu - g| <= 1e-4 (g + 1e-12)   (g = oracle softmax at the GPU's indices)
  * dispatch: counts, offsets, perm_src, perm_slot bit-exact against the oracle's
              dispatch of the GPU's indices; Xp = x[perm_src] bit-exact (a copy);
  * order:    on every *decided* token (all adjacent gaps among its k+1 largest fp32 logits
              exceed 1e-4; for k = E among its k) the ordered topk_idx equals the oracle's,
              and wherever an expert's rows are the oracle's, those rows carry the oracle's
              perm_slot bit-exact;
  * H rows:   |h_gpu - h| <= tol (1 + |h|), Yp rows: |yp_gpu - g o| <= tol (1 + |g o|)
              (o the oracle's expert output, g the oracle's gate at the GPU's index),
              y: |y_gpu - y| <= tol (1 + |y|), with tol = 1e-4 for fp32 layers and 2e-2 for
              bf16 layers.  At full size the rows checked cover every 128-row m-tile of
              the expert GEMMs (one row each), the first and last row of every non-empty
              expert, and every row of each expert's last 256-row pair tile (where the
              pair kernel's partial and odd tiles live);
  * aux:      |aux_gpu - aux| <= 1e-5 aux, aux from the oracle's softmax and the GPU's counts.
"""
import time

import numpy as np
import torch

import oracle

Y_TOL = {"f32": 1e-4, "bf16": 2e-2}
LOGIT_RTOL = 1e-5
GATE_RTOL = 1e-4
GATE_FLOOR = 1e-12   # gates below this (fp32 denormals) contribute nothing measurable
AUX_RTOL = 1e-5
MARGIN = 1e-4


def to_np(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.float().numpy().astype(np.float64)
    return t.numpy()


def run_gpu(plan, dev_inputs, y=None, ws=None, stream=None):
    s = dev_inputs.shape
    if y is None:
        y = torch.empty(s.T, s.d, dtype=plan.out_dtype, device="cuda")
    if ws is None:
        ws = plan.new_workspace()
    plan.forward(dev_inputs.x, dev_inputs.w_router, dev_inputs.bias, dev_inputs.w1, dev_inputs.w3,
                 dev_inputs.w2, y, ws, stream=stream)
    status = plan.device_status(ws, stream=stream)
    aux = plan.aux_loss(ws, stream=stream)
    torch.cuda.synchronize()
    return dict(y=y, ws=ws, status=status, aux=float(aux.item()), views=plan.views(ws))


def decided_tokens(z, k):
    """Tokens whose slot order is decided: every gap between neighbours among the k+1
    largest fp32 logits (the k largest when k = E) exceeds MARGIN."""
    E = z.shape[1]
    m = min(k + 1, E)
    zs = -np.sort(-z.astype(np.float32), axis=1)[:, :m].astype(np.float64)
    if m < 2:
        return np.ones(z.shape[0], bool)
    return np.all(zs[:, :-1] - zs[:, 1:] > MARGIN, axis=1)


def clear_tokens(z, k):
    """Tokens whose fp32 logit margin between the k-th and (k+1)-th largest exceeds MARGIN."""
    E = z.shape[1]
    if k == E:
        return np.ones(z.shape[0], bool)
    zs = -np.sort(-z.astype(np.float32), axis=1)
    return (zs[:, k - 1].astype(np.float64) - zs[:, k].astype(np.float64)) > MARGIN


class Report:
    def __init__(self):
        self.lines = []

    def add(self, name, value):
        self.lines.append(f"{name}: {value}")

    def __str__(self):
        return "\n".join(self.lines)


def check_routing(orc, host, bias, got, rep):
    """Router, top-k, gates, counts, dispatch and aux; returns (z, p, gpu_idx, gates_ref)."""
    v = got["views"]
    T, k, E = orc.T, orc.k, orc.E
    z, p, oidx, _ = orc.router(host["x"], host["wr"], bias)
    gidx = v["topk_idx"].cpu().numpy()
    ggate = v["topk_gate"].cpu().numpy().astype(np.float64)
    assert got["status"] == 0, f"device status {got['status']}"
    if v["logits"] is not None:
        zl = v["logits"].cpu().numpy().astype(np.float64)
        err = np.abs(zl - z) / (1.0 + np.abs(z))
        rep.add("logit max rel err", float(err.max()))
        assert err.max() <= LOGIT_RTOL, f"logits off by {err.max()}"
    clear = clear_tokens(z, k)
    rep.add("clear tokens", f"{int(clear.sum())}/{T}")
    # indices: on clear tokens the chosen set is exactly the oracle's; the order inside it
    # follows the oracle's logits wherever neighbours differ by more than the margin (two
    # chosen experts within the margin of each other may come in either order)
    zs32 = z.astype(np.float32)
    bad = np.where(clear & np.any(np.sort(gidx, axis=1) != np.sort(oidx, axis=1), axis=1))[0]
    assert bad.size == 0, f"{bad.size} clear tokens chose a different expert set, e.g. token {bad[:5]}"
    assert gidx.min() >= 0 and gidx.max() < E
    assert all(len(set(r)) == k for r in gidx.tolist())
    gz = np.take_along_axis(zs32, gidx, axis=1).astype(np.float64)
    assert np.all(gz[:, :-1] - gz[:, 1:] >= -MARGIN), "chosen experts not in descending logit order"
    rep.add("slots in oracle order", f"{int(np.all(gidx == oidx, axis=1).sum())}/{T}")
    dec = decided_tokens(z, k)
    bad = np.where(dec & np.any(gidx != oidx, axis=1))[0]
    rep.add("decided tokens (ordered idx bit-exact)", f"{int(dec.sum())}/{T}")
    assert bad.size == 0, f"{bad.size} decided tokens differ in slot order, e.g. token {bad[:5]}"
    # gates: the oracle's softmax at the GPU's indices (renormalised over them in that variant)
    gref = np.take_along_axis(p, gidx, axis=1)
    if getattr(orc, "renorm", False):
        gref = gref / gref.sum(axis=1, keepdims=True)
    gerr = np.abs(ggate - gref) / (gref + GATE_FLOOR)
    rep.add("gate max rel err", float(gerr.max()))
    assert gerr.max() <= GATE_RTOL, f"gates off by {gerr.max()}"
    # dispatch: bit-exact against the oracle's counting sort of the GPU's indices
    counts, offsets, perm_src, perm_slot = orc.dispatch(gidx)
    np.testing.assert_array_equal(v["expert_counts"].cpu().numpy(), counts)
    np.testing.assert_array_equal(v["expert_offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(v["perm_src"].cpu().numpy(), perm_src)
    np.testing.assert_array_equal(v["perm_slot"].cpu().numpy(), perm_slot)
    slot_pos = np.empty_like(perm_slot)
    slot_pos[perm_slot] = np.arange(perm_slot.size, dtype=np.int32)
    np.testing.assert_array_equal(v["slot_pos"].cpu().numpy(), slot_pos)
    np.testing.assert_array_equal(v["gate_perm"].cpu().numpy(), ggate.reshape(-1)[perm_slot].astype(np.float32))
    rep.add("counts min/max/#zero", f"{counts.min()}/{counts.max()}/{int((counts == 0).sum())}")
    # perm_slot against the oracle's own dispatch: on every expert whose rows (tokens, in
    # order) are the oracle's, rows of decided tokens carry the oracle's slot
    ocounts, ooff, osrc, oslot = orc.dispatch(oidx)
    gsrc, gslot = v["perm_src"].cpu().numpy(), v["perm_slot"].cpu().numpy()
    checked = 0
    for e in range(E):
        a, b = ooff[e], ooff[e + 1]
        if counts[e] != ocounts[e] or not np.array_equal(gsrc[a:b], osrc[a:b]):
            continue
        rows = np.arange(a, b)[dec[osrc[a:b]]]
        np.testing.assert_array_equal(gslot[rows], oslot[rows], err_msg=f"perm_slot of expert {e}")
        checked += rows.size
    rep.add("rows with perm_slot = oracle's", f"{checked}/{T * k}")
    # aux: the oracle's softmax with the routed counts
    aux_ref = orc.aux(p, counts)
    rep.add("aux gpu/ref", f"{got['aux']:.7f}/{aux_ref:.7f}")
    assert abs(got["aux"] - aux_ref) <= AUX_RTOL * abs(aux_ref), f"aux {got['aux']} vs {aux_ref}"
    return z, p, gidx, gref, perm_src, perm_slot, counts, offsets


def check_xp(dev_x, got, perm_src, rows=None):
    xp = got["views"]["xp"]
    if rows is None:
        ref = dev_x[torch.as_tensor(perm_src, device="cuda").long()]
        assert torch.equal(xp, ref), "Xp is not x[perm_src]"
    else:
        r = torch.as_tensor(rows, device="cuda").long()
        ref = dev_x[torch.as_tensor(perm_src[rows], device="cuda").long()]
        assert torch.equal(xp[r], ref), "Xp rows are not x[perm_src]"


def tile_rows(counts, offsets, rng):
    """Routed rows that cover the expert GEMMs' tiles: one seeded row inside every 128-row
    m-tile of every expert, the first and last row of every non-empty expert, and every row
    of each expert's last 256-row pair tile."""
    rows = []
    for e, c in enumerate(counts):
        if c == 0:
            continue
        a = int(offsets[e])
        for m0 in range(0, int(c), 128):
            rows.append(a + m0 + int(rng.integers(0, min(128, int(c) - m0))))
        rows += [a, a + int(c) - 1]
        last_pair = (int(c) - 1) // 256 * 256
        rows += list(range(a + last_pair, a + int(c)))
    return np.unique(np.asarray(rows, dtype=np.int64))


def check_rows(orc, host, got, perm_src, perm_slot, gidx, gref, rows, tol, rep):
    """H rows and Yp rows (the two expert GEMMs' outputs) against the oracle, batched."""
    rows = np.asarray(rows, dtype=np.int64)
    t0 = time.perf_counter()
    tokens = perm_src[rows].astype(np.int64)
    experts = gidx.reshape(-1)[perm_slot[rows]]
    href, oref = orc.expert_rows(host["x"], host["w1"], host["w3"], host["w2"], tokens, experts)
    rep.add("oracle s (rows)", round(time.perf_counter() - t0, 1))
    r = torch.as_tensor(rows, device="cuda")
    h = to_np(got["views"]["h"][r])
    err = np.abs(h - href) / (1.0 + np.abs(href))
    rep.add("rows checked (H, Yp)", rows.size)
    rep.add("H max err/(1+|h|)", float(err.max()))
    assert err.max() <= tol, f"H rows off by {err.max()}, worst row {rows[np.argmax(err.max(axis=1))]}"
    yp = to_np(got["views"]["yp"][r])
    ypref = gref.reshape(-1)[perm_slot[rows]][:, None] * oref
    err = np.abs(yp - ypref) / (1.0 + np.abs(ypref))
    rep.add("Yp max err/(1+|yp|)", float(err.max()))
    assert err.max() <= tol, f"Yp rows off by {err.max()}, worst row {rows[np.argmax(err.max(axis=1))]}"


def check_y(orc, host, got, gidx, gref, tokens, tol, rep):
    t0 = time.perf_counter()
    yref = orc.combine(host["x"], host["w1"], host["w3"], host["w2"], gidx, gref, tokens)
    rep.add("oracle s (y)", round(time.perf_counter() - t0, 1))
    rep.add("y tokens checked", orc.T if tokens is None else len(tokens))
    y = got["y"]
    yg = to_np(y if tokens is None else y[torch.as_tensor(tokens, device="cuda").long()])
    err = np.abs(yg - yref) / (1.0 + np.abs(yref))
    rep.add("y max err/(1+|y|)", float(err.max()))
    rep.add("y rms", float(np.sqrt(np.mean(yref ** 2))))
    assert err.max() <= tol, f"y off by {err.max()} (tol {tol})"


def full_check(shape, inputs, plan, y_tokens=None, h_rows=None, seed=0):
    """Run the plan on `inputs` and check every stage; returns (report, result).

    h_rows: routed rows whose H and Yp are checked; None = every row when the layer is
    small, else "tiles"; "tiles" = the rows tile_rows() picks.  y_tokens: tokens whose y is
    checked; None = every token; "tiles" = 48 seeded tokens, every token of the smallest
    non-empty expert, and up to 1024 tokens owning rows of the experts' last pair tiles."""
    rep = Report()
    host = inputs.numpy_for_oracle()
    dev = inputs.to("cuda")
    got = run_gpu(plan, dev)
    orc = oracle.Oracle(shape.T, shape.d, shape.E, shape.k, shape.F, tau=shape.tau, dtype=shape.dtype,
                        renorm=getattr(plan, "renorm_gates", False))
    bias = host["bias"]
    z, p, gidx, gref, perm_src, perm_slot, counts, offsets = check_routing(orc, host, bias, got, rep)
    check_xp(dev.x, got, perm_src)
    tol = Y_TOL[shape.dtype]
    rng = np.random.default_rng(seed)
    N = shape.T * shape.k
    if h_rows is None:
        h_rows = np.arange(N) if N * shape.d * shape.F <= (1 << 31) else "tiles"
    if isinstance(h_rows, str):
        h_rows = tile_rows(counts, offsets, rng)
    check_rows(orc, host, got, perm_src, perm_slot, gidx, gref, h_rows, tol, rep)
    if isinstance(y_tokens, str):
        nz = np.where(counts > 0)[0]
        e_min = nz[np.argmin(counts[nz])]
        last = []
        for e in nz:
            a, c = int(offsets[e]), int(counts[e])
            last.append(perm_src[a + (c - 1) // 256 * 256:a + c])
        last = np.unique(np.concatenate(last))
        if last.size > 1024:
            last = rng.choice(last, 1024, replace=False)
        y_tokens = np.unique(np.concatenate([rng.integers(0, shape.T, size=48),
                                             perm_src[offsets[e_min]:offsets[e_min + 1]], last]))
    check_y(orc, host, got, gidx, gref, y_tokens, tol, rep)
    return rep, got
