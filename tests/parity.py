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
  * H rows:   |h_gpu - h| <= tol (1 + |h|), y: |y_gpu - y| <= tol (1 + |y|), with
              tol = 1e-4 for fp32 layers and 2e-2 for bf16 layers;
  * aux:      |aux_gpu - aux| <= 1e-5 aux, aux from the oracle's softmax and the GPU's counts.
"""
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


def check_h_rows(orc, host, got, perm_src, perm_slot, gidx, rows, tol, rep):
    h = to_np(got["views"]["h"][torch.as_tensor(rows, device="cuda").long()])
    worst = 0.0
    for i, p in enumerate(rows):
        t = int(perm_src[p])
        e = int(gidx.reshape(-1)[perm_slot[p]])
        href, _ = orc.expert(host["x"], host["w1"], host["w3"], host["w2"], t, e)
        err = np.abs(h[i] - href) / (1.0 + np.abs(href))
        worst = max(worst, float(err.max()))
    rep.add("H max err/(1+|h|)", worst)
    assert worst <= tol, f"H rows off by {worst}"


def check_y(orc, host, got, gidx, gref, tokens, tol, rep):
    yref = orc.combine(host["x"], host["w1"], host["w3"], host["w2"], gidx, gref, tokens)
    y = got["y"]
    yg = to_np(y if tokens is None else y[torch.as_tensor(tokens, device="cuda").long()])
    err = np.abs(yg - yref) / (1.0 + np.abs(yref))
    rep.add("y max err/(1+|y|)", float(err.max()))
    rep.add("y rms", float(np.sqrt(np.mean(yref ** 2))))
    assert err.max() <= tol, f"y off by {err.max()} (tol {tol})"


def full_check(shape, inputs, plan, y_tokens=None, h_rows=None, seed=0):
    """Run the plan on `inputs` and check every stage; returns the report."""
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
        h_rows = np.unique(np.concatenate([rng.integers(0, N, size=min(N, 48)), [0, N - 1]]))
    check_h_rows(orc, host, got, perm_src, perm_slot, gidx, h_rows, tol, rep)
    check_y(orc, host, got, gidx, gref, y_tokens, tol, rep)
    return rep, got
