"""Pins for the oracle's backward pass (gradients of L = sum(dy * y) + alpha * aux).

* central finite differences of the oracle's own forward (fp64 loss; the routing is
  piecewise constant, so the steps are kept far below the smallest top-k margin);
* an independent float64 torch-autograd implementation of the layer on tiny shapes;
* mutation check: plausible mistakes planted in a copy of the backward fail a pin.
"""
import os
import shutil
import tempfile

import numpy as np
import pytest
import torch

import oracle
from oracle import build as obuild
from top_routing_grouped_gb300.workloads import MoEShape, make_inputs


def tiny(seed=0, E=4, k=2, renorm=False):
    s = MoEShape("bwd", T=7, d=8, E=E, k=k, F=6, dtype="f32", tau=0.9)
    inp = make_inputs(s, seed=seed).numpy_for_oracle()
    inp["bias"] = np.linspace(-0.3, 0.4, E).astype(np.float32)
    rng = np.random.default_rng(seed + 100)
    dy = rng.standard_normal((s.T, s.d))
    return s, inp, dy


def loss(o, inp, dy, alpha):
    r = o.forward(inp["x"], inp["wr"], inp["bias"], inp["w1"], inp["w3"], inp["w2"])
    return float((dy * r["y"]).sum() + alpha * r["aux"]), r


def torch_reference(s, inp, dy, alpha, renorm):
    """The layer written with torch ops in float64; gradients by autograd."""
    t = {n: torch.tensor(inp[n].astype(np.float64), requires_grad=True) for n in ("x", "wr", "w1", "w3", "w2", "bias")}
    z = (t["x"] @ t["wr"].T + t["bias"]) / s.tau
    p = torch.softmax(z, dim=1)
    idx = torch.topk(z.detach().float(), s.k, dim=1).indices  # fp32 decision, descending
    gate = p.gather(1, idx)
    if renorm:
        gate = gate / gate.sum(dim=1, keepdim=True)
    y = torch.zeros(s.T, s.d, dtype=torch.float64)
    rows = []
    for ti in range(s.T):
        acc = torch.zeros(s.d, dtype=torch.float64)
        for j in range(s.k):
            e = int(idx[ti, j])
            a = t["w1"][e] @ t["x"][ti]
            b = t["w3"][e] @ t["x"][ti]
            acc = acc + gate[ti, j] * (t["w2"][e] @ (torch.nn.functional.silu(a) * b))
        rows.append(acc)
    y = torch.stack(rows)
    counts = torch.bincount(idx.reshape(-1), minlength=s.E).double()
    aux = s.E * ((counts / (s.T * s.k)) * p.mean(dim=0)).sum()
    L = (torch.tensor(dy) * y).sum() + alpha * aux
    L.backward()
    return {"dx": t["x"].grad.numpy(), "dwr": t["wr"].grad.numpy(), "dbias": t["bias"].grad.numpy(),
            "dw1": t["w1"].grad.numpy(), "dw3": t["w3"].grad.numpy(), "dw2": t["w2"].grad.numpy()}


def pin_autograd(lib):
    for renorm in (False, True):
        for seed, alpha in ((0, 0.0), (1, 0.7)):
            s, inp, dy = tiny(seed, renorm=renorm)
            o = oracle.Oracle(s.T, s.d, s.E, s.k, s.F, tau=s.tau, lib=lib, renorm=renorm)
            g = o.backward(inp["x"], inp["wr"], inp["bias"], inp["w1"], inp["w3"], inp["w2"], dy, alpha)
            ref = torch_reference(s, inp, dy, alpha, renorm)
            for name in ref:
                np.testing.assert_allclose(g[name], ref[name], rtol=1e-9, atol=1e-11, err_msg=name)


def pin_finite_differences(lib):
    s, inp, dy = tiny(3)
    alpha = 0.5
    o = oracle.Oracle(s.T, s.d, s.E, s.k, s.F, tau=s.tau, lib=lib)
    g = o.backward(inp["x"], inp["wr"], inp["bias"], inp["w1"], inp["w3"], inp["w2"], dy, alpha)
    z, _, _, _ = o.router(inp["x"], inp["wr"], inp["bias"])
    zs = -np.sort(-z, axis=1)
    assert (zs[:, s.k - 1] - zs[:, s.k]).min() > 1e-3  # steps below stay far from a routing change
    rng = np.random.default_rng(7)
    names = {"x": "dx", "wr": "dwr", "bias": "dbias", "w1": "dw1", "w3": "dw3", "w2": "dw2"}
    for name, gname in names.items():
        for _ in range(6):
            flat = rng.integers(0, inp[name].size)
            hi, lo = ({k: v.copy() for k, v in inp.items()} for _ in range(2))
            base = inp[name].reshape(-1)[flat]
            step = np.float32(2e-3) * np.float32(max(1.0, abs(base)))
            hi[name].reshape(-1)[flat] = base + step
            lo[name].reshape(-1)[flat] = base - step
            actual = float(hi[name].reshape(-1)[flat]) - float(lo[name].reshape(-1)[flat])
            fd = (loss(o, hi, dy, alpha)[0] - loss(o, lo, dy, alpha)[0]) / actual
            an = g[gname].reshape(-1)[flat]
            assert abs(fd - an) <= 2e-5 * (1 + abs(an)), f"{gname}[{flat}]: fd {fd} vs analytic {an}"


PINS = [pin_autograd, pin_finite_differences]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_backward_pin(pin):
    pin(oracle.load())


MUTANTS = {
    "silu_grad_sign": ("s * (1.0 + av[f] * (1.0 - s))", "s * (1.0 - av[f] * (1.0 - s))"),
    "aux_grad_dropped": ("dp[e] = alpha * (double)E", "dp[e] = 0.0 * (double)E"),
    "gate_not_in_dh": ("* g * dyt[r];", "* dyt[r];"),
    "softmax_grad_no_centering": ("const double dl = pt[e] * (dp[e] - pdp) / c->tau;",
                                  "const double dl = pt[e] * dp[e] / c->tau;"),
    "renorm_grad_uncorrected": ("dp[idx[t * k + j]] += (dg[t * k + j] - gdg) / S;",
                                "dp[idx[t * k + j]] += dg[t * k + j];"),
    "w3_grad_uses_da": ("g3[col] += db * xv;", "g3[col] += da * xv;"),
    "w2_grad_wrong_token": ("const double gdy = gate[slot] * dy[t * d + r];",
                            "const double gdy = gate[slot] * dy[(slot % T) * d + r];"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="orc_bmut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_backward_mistake_is_caught(name, mutant_dir):
    src = open(obuild.SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = os.path.join(mutant_dir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.load(obuild.compile_oracle(path, os.path.join(mutant_dir, f"lib{name}.so"),
                                            extra=("-Wno-unused-parameter", "-Wno-unused-variable",
                                                   "-Wno-unused-but-set-variable")))
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
