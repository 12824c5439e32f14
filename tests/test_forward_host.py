"""The host-buffer forward (moe_forward_host): x in from pinned host memory and y out to it.
Its y must equal the device forward's bit for bit, for every path and for ragged token
counts, and successive calls must not see each other's data."""
import pytest
import torch

from top_routing_grouped_gb300.workloads import MoEShape, make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path", ["auto", "tc1", "simt"])
@pytest.mark.parametrize("T", [1, 300, 2000])
def test_host_forward_equals_device_forward(path, T):
    from top_routing_grouped_gb300 import moe
    s = MoEShape("host", T=T, d=256, E=8, k=2, F=192, dtype="bf16")
    plan = moe.MoEPlan(s.T, s.d, s.E, s.k, s.F, path=path)
    ws = plan.new_workspace()
    outs = []
    for seed in (3, 4):  # two calls in a row with different x: nothing stale carries over
        dev = make_inputs(s, seed=seed).to("cuda")
        y = torch.empty(T, s.d, dtype=torch.bfloat16, device="cuda")
        plan.forward(dev.x, dev.w_router, dev.bias, dev.w1, dev.w3, dev.w2, y, ws)
        torch.cuda.synchronize()
        ref = y.cpu()
        aux_ref = plan.aux_loss(ws).item()
        x_host = dev.x.cpu().pin_memory()
        x_dev = torch.empty_like(dev.x)
        y_host = torch.full((T, s.d), float("nan"), dtype=torch.bfloat16).pin_memory()
        y_dev = torch.empty_like(y)
        plan.forward_host(x_host, x_dev, dev.w_router, dev.bias, dev.w1, dev.w3, dev.w2, y_dev, y_host, ws)
        torch.cuda.current_stream().synchronize()
        assert plan.device_status(ws) == moe.MOE_OK
        assert torch.equal(y_host, ref)
        assert plan.aux_loss(ws).item() == aux_ref
        outs.append(y_host.clone())
    assert not torch.equal(outs[0], outs[1])
