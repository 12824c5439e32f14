"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Such callers (a fixed device-memory budget, a runtime that owns every allocation, a step
that must not fail half-way on an allocation) cannot hand moe_forward a workspace.  The
no-alloc entry point keeps its scratch in a static device array inside the library.  These
tests call it through the C ABI twice in a row (the second call reuses the array the first
one left behind) and check both results:
  * against the routing moe_forward leaves in its workspace, under the parity rules: the
    chosen expert set bit-exact on every token whose logit margin exceeds 1e-4 (slots may
    swap only between experts within that margin of each other), gates within 1e-4, counts
    exact (or, if a token is not clear, consistent with the returned indices), aux within
    1e-5 relative;
  * for a plan made for training (whose forward also keeps the softmax), against the CPU
    oracle directly: the same rules, with the oracle's logits, softmax and dispatch;
  * the device status output: 0 on clean input, MOE_ERR_INTERNAL when a logit is NaN, and
    0 again on the next clean call (each call clears the status it starts from).

This file is named to be collected last, so that a run stopping at its first failure has
already run every other test; it also passes when run alone in a fresh process.  The host
side argument checks of the entry point are covered without a GPU in test_abi.py.
"""
import ctypes

import numpy as np
import pytest
import torch

from top_routing_grouped_gb300.workloads import SHAPES, MoEShape, make_inputs

pytestmark = pytest.mark.gpu

MARGIN = 1e-4
CASES = [SHAPES["tiny_f32"],
         MoEShape("ragged_bias", T=300, d=256, E=16, k=4, F=128, dtype="bf16", tau=0.7, zipf_bias=True),
         SHAPES["fine_e32"]]


def clear_tokens(z, k):
    zs = -np.sort(-z.astype(np.float32), axis=1)
    if k == z.shape[1]:
        return np.ones(z.shape[0], bool)
    return (zs[:, k - 1].astype(np.float64) - zs[:, k].astype(np.float64)) > MARGIN


def call_noalloc(moe, plan, shape, dev):
    """One call through the C ABI into fresh, poisoned output tensors; returns host arrays."""
    lib = moe.lib()
    stream = torch.cuda.current_stream()
    idx = torch.full((shape.T, shape.k), -7, dtype=torch.int32, device="cuda")
    gate = torch.full((shape.T, shape.k), -1.0, dtype=torch.float32, device="cuda")
    counts = torch.full((shape.E,), -1, dtype=torch.int32, device="cuda")
    aux = torch.full((4,), -1.0, dtype=torch.float32, device="cuda")
    status = torch.full((4,), 77, dtype=torch.int32, device="cuda")
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = lib.moe_route_noalloc(plan.handle, P(dev.x), P(dev.w_router), P(dev.bias), P(idx), P(gate), P(counts),
                               P(aux), P(status), ctypes.c_void_p(stream.cuda_stream))
    assert st == moe.MOE_OK, lib.moe_last_error().decode()
    torch.cuda.synchronize()
    return dict(idx=idx.cpu().numpy(), gate=gate.cpu().numpy().astype(np.float64), counts=counts.cpu().numpy(),
                aux=float(aux[0].item()), status=int(status[0].item()))


def check_against(got, logits, ref_idx, gate_of, ref_counts, ref_aux, shape, what):
    """The parity rules for routing: `gate_of(idx)` gives the reference gates at indices idx."""
    clear = clear_tokens(logits, shape.k)
    gi = got["idx"]
    assert got["status"] == 0, f"{what}: device status {got['status']}"
    np.testing.assert_array_equal(np.sort(gi[clear], axis=1), np.sort(ref_idx[clear], axis=1),
                                  err_msg=f"{what}: expert sets")
    assert gi.min() >= 0 and gi.max() < shape.E
    assert all(len(set(r)) == shape.k for r in gi.tolist()), f"{what}: repeated expert"
    zl = np.take_along_axis(logits.astype(np.float32), gi, axis=1).astype(np.float64)
    assert np.all(zl[:, :-1] - zl[:, 1:] >= -MARGIN), f"{what}: slots out of logit order"
    gref = gate_of(gi)
    gerr = np.abs(got["gate"] - gref) / (gref + 1e-12)
    assert gerr.max() <= 1e-4, f"{what}: gates off by {gerr.max()}"
    np.testing.assert_array_equal(got["counts"], np.bincount(gi.reshape(-1), minlength=shape.E), err_msg=what)
    if clear.all():
        np.testing.assert_array_equal(got["counts"], ref_counts, err_msg=f"{what}: counts")
    aux_ref = ref_aux(got["counts"])
    assert abs(got["aux"] - aux_ref) <= 1e-5 * abs(aux_ref), f"{what}: aux {got['aux']} vs {aux_ref}"


@pytest.mark.parametrize("shape", CASES, ids=lambda s: s.name)
def test_route_noalloc_matches_forward_twice(shape):
    from top_routing_grouped_gb300 import moe

    inp = make_inputs(shape, seed=0)
    dev = inp.to("cuda")
    plan = moe.MoEPlan.for_shape(shape, keep_logits=True)

    # the existing entry point, with its caller-owned workspace
    ws = plan.new_workspace()
    y = torch.empty(shape.T, shape.d, dtype=plan.out_dtype, device="cuda")
    plan.forward(dev.x, dev.w_router, dev.bias, dev.w1, dev.w3, dev.w2, y, ws)
    assert plan.device_status(ws) == moe.MOE_OK
    v = plan.views(ws)
    ref_idx = v["topk_idx"].cpu().numpy()
    ref_gate = v["topk_gate"].cpu().numpy().astype(np.float64)
    ref_counts = v["expert_counts"].cpu().numpy()
    ref_aux = float(v["aux"].item())
    logits = v["logits"].cpu().numpy()

    clear = clear_tokens(logits, shape.k)
    for call in range(2):
        got = call_noalloc(moe, plan, shape, dev)
        gi, gg, gc = got["idx"], got["gate"], got["counts"]
        assert got["status"] == 0, f"call {call}: device status {got['status']}"
        # same expert set on every clear token; inside it, slots may swap only between
        # experts whose logits lie within the 1e-4 margin of each other
        np.testing.assert_array_equal(np.sort(gi[clear], axis=1), np.sort(ref_idx[clear], axis=1),
                                      err_msg=f"call {call}: expert sets")
        assert gi.min() >= 0 and gi.max() < shape.E
        zl = np.take_along_axis(logits.astype(np.float32), gi, axis=1).astype(np.float64)
        assert np.all(zl[:, :-1] - zl[:, 1:] >= -MARGIN), f"call {call}: slots out of logit order"
        same = np.all(gi == ref_idx, axis=1)
        gerr = np.abs(gg[same] - ref_gate[same]) / (ref_gate[same] + 1e-12)
        assert gerr.max() <= 1e-4, f"call {call}: gates off by {gerr.max()}"
        np.testing.assert_array_equal(gc, np.bincount(gi.reshape(-1), minlength=shape.E), err_msg=f"call {call}")
        if clear.all():
            np.testing.assert_array_equal(gc, ref_counts, err_msg=f"call {call}: counts")
        assert abs(got["aux"] - ref_aux) <= 1e-5 * abs(ref_aux), f"call {call}: aux {got['aux']} vs {ref_aux}"


def test_route_noalloc_training_plan_matches_oracle():
    """A plan made for training asks the forward to keep the router softmax for its
    backward; the routing-only call has no room for it and must not store it.  Its results
    match the oracle on two calls in a row."""
    import oracle
    from top_routing_grouped_gb300 import moe

    shape = MoEShape("train_bias", T=300, d=256, E=16, k=4, F=128, dtype="bf16", tau=0.7, zipf_bias=True)
    inp = make_inputs(shape, seed=0)
    dev = inp.to("cuda")
    plan = moe.MoEPlan.for_shape(shape, training=True)
    host = inp.numpy_for_oracle()
    orc = oracle.Oracle(shape.T, shape.d, shape.E, shape.k, shape.F, tau=shape.tau, dtype=shape.dtype)
    z, p, oidx, _ = orc.router(host["x"], host["wr"], host["bias"])
    ocounts, _, _, _ = orc.dispatch(oidx)
    for call in range(2):
        got = call_noalloc(moe, plan, shape, dev)
        check_against(got, z, oidx, lambda gi: np.take_along_axis(p, gi, axis=1), ocounts,
                      lambda c: orc.aux(p, c), shape, f"training plan, call {call}")


def test_route_noalloc_reports_a_nan_logit():
    """A NaN in x makes every logit of that token NaN: the call records MOE_ERR_INTERNAL in
    its status output (the other outputs are then unspecified but stay in range); the next
    call on clean input starts from a cleared status and reports 0."""
    from top_routing_grouped_gb300 import moe

    shape = MoEShape("nan_x", T=300, d=256, E=16, k=4, F=128, dtype="bf16", tau=1.0)
    inp = make_inputs(shape, seed=3)
    plan = moe.MoEPlan.for_shape(shape)
    bad = inp.to("cuda")
    bad.x = bad.x.clone()
    bad.x[123, 7] = float("nan")
    got = call_noalloc(moe, plan, shape, bad)
    assert got["status"] == moe.MOE_ERR_INTERNAL
    assert got["idx"].min() >= 0 and got["idx"].max() < shape.E
    assert got["counts"].sum() == shape.T * shape.k
    clean = call_noalloc(moe, plan, shape, inp.to("cuda"))
    assert clean["status"] == 0
    assert clean["counts"].sum() == shape.T * shape.k
