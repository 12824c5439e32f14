"""Pins for the CPU oracle: checks against things the page and the mathematics fix,
independent of the oracle's own code.

* dense reduction: E = 1, k = 1 makes the layer a plain SwiGLU FFN (gate = 1); checked
  against numpy matrix products;
* router / top-k: numpy logits, scipy softmax and a stable argsort;
* brute force on tiny inputs: every expert evaluated densely for every token, then masked
  to the top-k (§3 output formula);
* invariants: gates are the softmax entries at the chosen experts, counts sum to T k,
  the dispatch is a bijection, stable in token order;
* a hand-worked routing/dispatch example (tests/golden/);
* the balancing scalar: exactly 1 for a uniform router, E for a collapsed one, invariant
  under relabelling the experts;
* mutation check: plausible mistakes planted in a copy of the oracle each fail a pin.
"""
import json
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import build as obuild
from top_routing_grouped_gb300.workloads import MoEShape, make_inputs, SHAPES

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def shape(T, d, E, k, F, dtype="f32", tau=1.0, zipf=False):
    return MoEShape("test", T=T, d=d, E=E, k=k, F=F, dtype=dtype, tau=tau, zipf_bias=zipf)


def widen(a):
    """fp32 / bf16-bit-pattern numpy array -> float64."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def silu(a):
    return a / (1.0 + np.exp(-a))


def dense_swiglu(xr, w1, w3, w2):
    """Textbook SwiGLU FFN for rows xr [n, d]: W2 (silu(W1 x) * (W3 x))."""
    return (silu(xr @ w1.T) * (xr @ w3.T)) @ w2.T


# ---------------------------------------------------------------- pin functions
# Each takes a liboracle handle so the mutation test can run them on planted mistakes.

def pin_dense_reduction(lib):
    for dtype in ("f32", "bf16"):
        s = shape(T=9, d=24, E=1, k=1, F=40, dtype=dtype)
        inp = make_inputs(s, seed=3).numpy_for_oracle()
        o = oracle.Oracle(s.T, s.d, s.E, s.k, s.F, dtype=dtype, lib=lib)
        r = o.forward(inp["x"], inp["wr"], None, inp["w1"], inp["w3"], inp["w2"])
        x, w1, w3, w2 = (widen(inp[n]) for n in ("x", "w1", "w3", "w2"))
        ref = dense_swiglu(x, w1[0], w3[0], w2[0])
        np.testing.assert_allclose(r["gate"], 1.0, rtol=0, atol=0)
        np.testing.assert_allclose(r["y"], ref, rtol=1e-12, atol=1e-12)


def pin_router_library(lib):
    s = shape(T=70, d=32, E=8, k=3, F=8, tau=0.7)
    inp = make_inputs(s, seed=5).numpy_for_oracle()
    bias = np.linspace(-0.5, 0.5, s.E).astype(np.float32)
    o = oracle.Oracle(s.T, s.d, s.E, s.k, s.F, tau=s.tau, lib=lib)
    z, p, idx, gate = o.router(inp["x"], inp["wr"], bias)
    zr = (widen(inp["x"]) @ widen(inp["wr"]).T + bias.astype(np.float64)) / s.tau
    pr = scipy.special.softmax(zr, axis=1)
    idxr = np.argsort(-zr.astype(np.float32), axis=1, kind="stable")[:, : s.k]
    np.testing.assert_allclose(z, zr, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(p, pr, rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(idx, idxr)
    np.testing.assert_allclose(gate, np.take_along_axis(pr, idxr, axis=1), rtol=1e-12)


def pin_bruteforce(lib):
    s = shape(T=17, d=8, E=5, k=2, F=12, tau=1.3)
    inp = make_inputs(s, seed=11).numpy_for_oracle()
    bias = np.array([0.3, -0.2, 0.0, 0.1, -0.4], np.float32)
    o = oracle.Oracle(s.T, s.d, s.E, s.k, s.F, tau=s.tau, lib=lib)
    r = o.forward(inp["x"], inp["wr"], bias, inp["w1"], inp["w3"], inp["w2"])
    x, wr, w1, w3, w2 = (widen(inp[n]) for n in ("x", "wr", "w1", "w3", "w2"))
    # every expert on every token, densely
    allout = np.stack([dense_swiglu(x, w1[e], w3[e], w2[e]) for e in range(s.E)], axis=1)
    z = (x @ wr.T + bias) / s.tau
    p = scipy.special.softmax(z, axis=1)
    y = np.zeros((s.T, s.d))
    for t in range(s.T):
        order = sorted(range(s.E), key=lambda e: (-np.float32(z[t, e]), e))[: s.k]
        for e in order:
            y[t] += p[t, e] * allout[t, e]
    np.testing.assert_allclose(r["y"], y, rtol=1e-11, atol=1e-12)


def pin_invariants(lib):
    s = shape(T=300, d=16, E=6, k=3, F=8)
    inp = make_inputs(s, seed=7).numpy_for_oracle()
    o = oracle.Oracle(s.T, s.d, s.E, s.k, s.F, lib=lib)
    z, p, idx, gate = o.router(inp["x"], inp["wr"])
    np.testing.assert_array_equal(gate, np.take_along_axis(p, idx, axis=1))
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    zs = np.take_along_axis(z.astype(np.float32), idx, axis=1)
    assert np.all(zs[:, :-1] >= zs[:, 1:])                       # descending
    assert all(len(set(r)) == s.k for r in idx.tolist())          # distinct experts
    counts, offsets, perm_src, perm_slot = o.dispatch(idx)
    assert counts.sum() == s.T * s.k                               # every slot routed once
    np.testing.assert_array_equal(np.diff(offsets), counts)
    assert offsets[0] == 0 and offsets[-1] == s.T * s.k
    np.testing.assert_array_equal(np.sort(perm_slot), np.arange(s.T * s.k))   # bijection
    np.testing.assert_array_equal(perm_src, perm_slot // s.k)
    flat = idx.reshape(-1)
    for e in range(s.E):
        rows = perm_slot[offsets[e]:offsets[e + 1]]
        assert np.all(flat[rows] == e)
        assert np.all(np.diff(rows) > 0)                           # stable in token order


def pin_golden(lib):
    g = json.load(open(os.path.join(GOLDEN, "routing_dispatch_worked_example.json")))
    T, d, E, k = g["T"], g["d"], g["E"], g["k"]
    o = oracle.Oracle(T, d, E, k, 4, lib=lib)
    x = np.array(g["x"], np.float32)
    wr = np.eye(E, d, dtype=np.float32)
    z, p, idx, gate = o.router(x, wr)
    np.testing.assert_array_equal(idx, np.array(g["idx"]))
    counts, offsets, perm_src, perm_slot = o.dispatch(idx)
    np.testing.assert_array_equal(counts, g["counts"])
    np.testing.assert_array_equal(offsets, g["offsets"])
    np.testing.assert_array_equal(perm_src, g["perm_src"])
    np.testing.assert_array_equal(perm_slot, g["perm_slot"])
    tx = np.array(g["ties"]["x"], np.float32)
    o2 = oracle.Oracle(len(tx), d, E, k, 4, lib=lib)
    _, _, tidx, _ = o2.router(tx, wr)
    np.testing.assert_array_equal(tidx, np.array(g["ties"]["idx"]))


def pin_aux(lib):
    # uniform router: every logit equal -> p = 1/E exactly (E a power of two) -> aux = 1
    for E, k in ((8, 2), (32, 8), (64, 4), (128, 8), (1, 1)):
        s = shape(T=64, d=16, E=E, k=k, F=8)
        inp = make_inputs(s, seed=1).numpy_for_oracle()
        o = oracle.Oracle(s.T, s.d, E, k, s.F, lib=lib)
        r = o.forward(inp["x"], np.zeros_like(inp["wr"]), None, inp["w1"], inp["w3"], inp["w2"])
        assert r["aux"] == 1.0
    # collapse: every token certain of expert 0 with k = 1 -> aux = E (f_0 = P_0 = 1)
    s = shape(T=50, d=16, E=8, k=1, F=8)
    inp = make_inputs(s, seed=2).numpy_for_oracle()
    bias = np.zeros(s.E, np.float32)
    bias[0] = 100.0
    o = oracle.Oracle(s.T, s.d, s.E, s.k, s.F, lib=lib)
    r = o.forward(inp["x"], inp["wr"], bias, inp["w1"], inp["w3"], inp["w2"])
    assert np.all(r["idx"] == 0)
    assert abs(r["aux"] - s.E) < 1e-9
    # relabelling experts (permuting router rows and expert weights) changes nothing
    s = shape(T=40, d=16, E=6, k=2, F=8)
    inp = make_inputs(s, seed=9).numpy_for_oracle()
    o = oracle.Oracle(s.T, s.d, s.E, s.k, s.F, lib=lib)
    r = o.forward(inp["x"], inp["wr"], None, inp["w1"], inp["w3"], inp["w2"])
    perm = np.array([3, 0, 5, 1, 4, 2])
    rp = o.forward(inp["x"], inp["wr"][perm].copy(), None, inp["w1"][perm].copy(),
                   inp["w3"][perm].copy(), inp["w2"][perm].copy())
    assert abs(r["aux"] - rp["aux"]) < 1e-12
    np.testing.assert_allclose(r["y"], rp["y"], rtol=1e-12, atol=1e-13)


def pin_expert_rows(lib):
    s = shape(T=5, d=12, E=3, k=2, F=20, dtype="bf16")
    inp = make_inputs(s, seed=4).numpy_for_oracle()
    o = oracle.Oracle(s.T, s.d, s.E, s.k, s.F, dtype="bf16", lib=lib)
    x, w1, w3, w2 = (widen(inp[n]) for n in ("x", "w1", "w3", "w2"))
    for t in range(s.T):
        for e in range(s.E):
            h, out = o.expert(inp["x"], inp["w1"], inp["w3"], inp["w2"], t, e)
            href = silu(w1[e] @ x[t]) * (w3[e] @ x[t])
            np.testing.assert_allclose(h, href, rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(out, w2[e] @ href, rtol=1e-11, atol=1e-13)
    # many rows at once, in an arbitrary order with repeats (the batched form the full-size
    # parity checks use)
    tk = np.array([4, 0, 2, 2, 1, 4, 3, 0])
    ex = np.array([2, 1, 0, 2, 1, 0, 2, 0])
    hs, outs = o.expert_rows(inp["x"], inp["w1"], inp["w3"], inp["w2"], tk, ex)
    for i, (t, e) in enumerate(zip(tk, ex)):
        href = silu(w1[e] @ x[t]) * (w3[e] @ x[t])
        np.testing.assert_allclose(hs[i], href, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(outs[i], w2[e] @ href, rtol=1e-11, atol=1e-13)


def pin_renormalised_gates(lib):
    """Variant: gates renormalised over the k chosen = a softmax over the chosen logits."""
    s = shape(T=60, d=16, E=8, k=3, F=8, tau=0.8)
    inp = make_inputs(s, seed=12).numpy_for_oracle()
    o = oracle.Oracle(s.T, s.d, s.E, s.k, s.F, tau=s.tau, lib=lib, renorm=True)
    z, p, idx, gate = o.router(inp["x"], inp["wr"])
    zc = np.take_along_axis(z, idx, axis=1)
    np.testing.assert_allclose(gate, scipy.special.softmax(zc, axis=1), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(gate.sum(axis=1), 1.0, atol=1e-14)
    # k = 1: the single gate is exactly 1; k = E: the renormalised gates are the softmax itself
    o1 = oracle.Oracle(s.T, s.d, s.E, 1, s.F, tau=s.tau, lib=lib, renorm=True)
    assert np.all(o1.router(inp["x"], inp["wr"])[3] == 1.0)
    oE = oracle.Oracle(s.T, s.d, s.E, s.E, s.F, tau=s.tau, lib=lib, renorm=True)
    _, pE, idxE, gE = oE.router(inp["x"], inp["wr"])
    np.testing.assert_allclose(gE, np.take_along_axis(pE, idxE, axis=1), rtol=1e-12)


PINS = [pin_dense_reduction, pin_router_library, pin_bruteforce, pin_invariants, pin_golden,
        pin_aux, pin_expert_rows, pin_renormalised_gates]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.load())


def test_active_fraction_two_of_eight():
    """§3: with 8 experts and top-2, each token runs 2 of 8 expert FFNs (25 % of the
    expert parameters); the oracle's dispatch routes exactly T*2 rows."""
    s = shape(T=128, d=16, E=8, k=2, F=8)
    inp = make_inputs(s, seed=0).numpy_for_oracle()
    o = oracle.Oracle(s.T, s.d, s.E, s.k, s.F)
    r = o.forward(inp["x"], inp["wr"], None, inp["w1"], inp["w3"], inp["w2"])
    assert r["counts"].sum() / (s.T * s.E) == 0.25
    assert s.with_(T=s.T).expert_flops == 6 * s.T * s.k * s.d * s.F


def test_combine_subset_matches_full():
    s = shape(T=40, d=16, E=4, k=2, F=8, dtype="bf16")
    inp = make_inputs(s, seed=6).numpy_for_oracle()
    o = oracle.Oracle(s.T, s.d, s.E, s.k, s.F, dtype="bf16")
    r = o.forward(inp["x"], inp["wr"], None, inp["w1"], inp["w3"], inp["w2"])
    toks = np.array([39, 0, 17, 17, 5])
    ys = o.combine(inp["x"], inp["w1"], inp["w3"], inp["w2"], r["idx"], r["gate"], toks)
    np.testing.assert_array_equal(ys, r["y"][toks])


def test_zipf_bias_leaves_experts_empty():
    """The skewed workload (E = 128, Zipf-like logit bias) must leave some experts with
    no tokens at seed 0; routing only needs x and W_r."""
    s = SHAPES["skewed_e128"]
    inp = make_inputs(s, seed=0, parts=("x", "wr")).numpy_for_oracle()
    o = oracle.Oracle(s.T, s.d, s.E, s.k, s.F, dtype="bf16")
    z, p, idx, gate = o.router(inp["x"], inp["wr"], inp["bias"])
    counts, offsets, _, _ = o.dispatch(idx)
    assert counts.sum() == s.T * s.k
    assert (counts == 0).sum() >= 1
    assert counts[0] == counts.max()


def test_bad_arguments_rejected():
    o = oracle.Oracle(4, 8, 2, 3, 8)      # k > E
    with pytest.raises(RuntimeError):
        o.router(np.zeros((4, 8), np.float32), np.zeros((2, 8), np.float32))


# ---------------------------------------------------------------- mutation check
MUTANTS = {
    "bias_dropped": ("if (bias) acc += (double)bias[e];", ""),
    "tau_multiplied": ("zt[e] = acc / c->tau;", "zt[e] = acc * c->tau;"),
    "silu_sign": ("h[f] = a / (1.0 + exp(-a)) * g;", "h[f] = a / (1.0 + exp(a)) * g;"),
    "w1_w3_swapped": ("h[f] = a / (1.0 + exp(-a)) * g;", "h[f] = g / (1.0 + exp(-g)) * a;"),
    "w2_transposed": ("wbase + (int64_t)r * F + f", "wbase + (int64_t)f * d + r"),
    "tie_to_higher": ("if (best < 0 || v > bestv) {", "if (best < 0 || v >= bestv) {"),
    "dispatch_reversed": ("int32_t pos = offsets[e] + cursor[e]++;",
                          "int32_t pos = offsets[e + 1] - 1 - cursor[e]++;"),
    "gate_dropped": ("yr[col] += gate[t * k + j] * o[col];", "yr[col] += o[col];"),
    "gate_renormalised": ("gate[t * k + j] = pt[best];",
                          "gate[t * k + j] = pt[best] / pt[idx[t * k]];"),
    "aux_without_k": ("double f = (double)counts[i] / ((double)T * (double)c->k);",
                      "double f = (double)counts[i] / (double)T;"),
    "softmax_unnormalised": ("for (int32_t e = 0; e < E; ++e) pt[e] /= s;", ""),
    "renorm_ignored": ("for (int32_t j = 0; j < k; ++j) gate[t * k + j] /= chosen;", ""),
    "rows_token_ignored": ("xr[col] = orc_load(x, c->dtype, t[i] * d + col);",
                           "xr[col] = orc_load(x, c->dtype, i * d + col);"),
    "renorm_over_all": ("for (int32_t j = 0; j < k; ++j) chosen += gate[t * k + j];",
                        "for (int32_t e = 0; e < E; ++e) chosen += pt[e];"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="orc_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, mutant_dir):
    src = open(obuild.SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = os.path.join(mutant_dir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.load(obuild.compile_oracle(path, os.path.join(mutant_dir, f"lib{name}.so"),
                                            extra=("-Wno-unused-parameter",
                                                   "-Wno-unused-variable",
                                                   "-Wno-unused-but-set-variable")))
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, RuntimeError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
