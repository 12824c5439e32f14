"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Such callers (a fixed device-memory budget, a runtime that owns every allocation, a step
that must not fail half-way on an allocation) cannot hand moe_forward a workspace.  The
no-alloc entry point keeps its scratch in a static device array inside the library.  This
test calls it through the C ABI twice in a row (the second call reuses the array the first
one left behind) and checks both results against the routing that moe_forward leaves in its
workspace, under the same rules as the parity tests: the chosen expert set bit-exact on
every token whose logit margin exceeds 1e-4 (slots may swap only between experts within that
margin of each other), gates within 1e-4, counts exact (or, if a token is not clear,
consistent with the returned indices), aux within 1e-5 relative.

This file is named to be collected last, so that a run stopping at its first failure has
already run every other test; it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from top_routing_grouped_gb300.workloads import SHAPES, MoEShape, make_inputs

pytestmark = pytest.mark.gpu

CASES = [SHAPES["tiny_f32"],
         MoEShape("ragged_bias", T=300, d=256, E=16, k=4, F=128, dtype="bf16", tau=0.7, zipf_bias=True),
         SHAPES["fine_e32"]]


def clear_tokens(z, k):
    zs = -np.sort(-z.astype(np.float32), axis=1)
    if k == z.shape[1]:
        return np.ones(z.shape[0], bool)
    return (zs[:, k - 1].astype(np.float64) - zs[:, k].astype(np.float64)) > 1e-4


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

    lib = moe.lib()
    stream = torch.cuda.current_stream()
    for call in range(2):
        idx = torch.full((shape.T, shape.k), -7, dtype=torch.int32, device="cuda")
        gate = torch.full((shape.T, shape.k), -1.0, dtype=torch.float32, device="cuda")
        counts = torch.full((shape.E,), -1, dtype=torch.int32, device="cuda")
        aux = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
        P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
        st = lib.moe_route_noalloc(plan.handle, P(dev.x), P(dev.w_router), P(dev.bias), P(idx), P(gate),
                                   P(counts), P(aux), ctypes.c_void_p(stream.cuda_stream))
        assert st == moe.MOE_OK, lib.moe_last_error().decode()
        torch.cuda.synchronize()
        gi = idx.cpu().numpy()
        gg = gate.cpu().numpy().astype(np.float64)
        gc = counts.cpu().numpy()
        ga = float(aux.item())
        # same expert set on every clear token; inside it, slots may swap only between
        # experts whose logits lie within the 1e-4 margin of each other
        np.testing.assert_array_equal(np.sort(gi[clear], axis=1), np.sort(ref_idx[clear], axis=1),
                                      err_msg=f"call {call}: expert sets")
        assert gi.min() >= 0 and gi.max() < shape.E
        zl = np.take_along_axis(logits.astype(np.float32), gi, axis=1).astype(np.float64)
        assert np.all(zl[:, :-1] - zl[:, 1:] >= -1e-4), f"call {call}: slots out of logit order"
        same = np.all(gi == ref_idx, axis=1)
        gerr = np.abs(gg[same] - ref_gate[same]) / (ref_gate[same] + 1e-12)
        assert gerr.max() <= 1e-4, f"call {call}: gates off by {gerr.max()}"
        np.testing.assert_array_equal(gc, np.bincount(gi.reshape(-1), minlength=shape.E), err_msg=f"call {call}")
        if clear.all():
            np.testing.assert_array_equal(gc, ref_counts, err_msg=f"call {call}: counts")
        assert abs(ga - ref_aux) <= 1e-5 * abs(ref_aux), f"call {call}: aux {ga} vs {ref_aux}"


def test_route_noalloc_rejects_shapes_beyond_its_buffer():
    from top_routing_grouped_gb300 import moe

    # 2M tokens x k=8 needs 64 MiB of per-slot ranks: more than the static buffer holds
    big = moe.MoEPlan(2_000_000, 64, 8, 8, 64, dtype="bf16")
    lib = moe.lib()
    x = torch.empty(8, dtype=torch.bfloat16, device="cuda")  # never read: rejected first
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.moe_route_noalloc(big.handle, P(x), P(x), None, P(x), P(x), P(x), P(x), None)
    assert st == moe.MOE_ERR_UNSUPPORTED
    assert b"MOE_NOALLOC_SCRATCH_BYTES" in lib.moe_last_error()
