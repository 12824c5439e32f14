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


@pytest.mark.parametrize("path", ["auto", "simt"])
def test_two_streams_in_flight(path):
    """Serving-loop use: successive batches alternate between two streams, each with its own
    workspace and device/host buffers, so one batch's copies overlap the other's kernels.  Every
    batch's y must equal its own device forward."""
    from top_routing_grouped_gb300 import moe
    s = MoEShape("host2", T=1000, d=256, E=8, k=2, F=192, dtype="bf16")
    plan = moe.MoEPlan(s.T, s.d, s.E, s.k, s.F, path=path)
    w = make_inputs(s, seed=5).to("cuda")
    xs = [make_inputs(s, seed=10 + i).x for i in range(6)]
    refs = []
    ws_ref = plan.new_workspace()
    for x in xs:
        y = torch.empty(s.T, s.d, dtype=torch.bfloat16, device="cuda")
        plan.forward(x.to("cuda"), w.w_router, w.bias, w.w1, w.w3, w.w2, y, ws_ref)
        refs.append(y.cpu())
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [plan.new_workspace(), plan.new_workspace()]
    x_dev = [torch.empty(s.T, s.d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    y_dev = [torch.empty(s.T, s.d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    x_host = [x.pin_memory() for x in xs]
    y_host = [torch.full((s.T, s.d), float("nan"), dtype=torch.bfloat16).pin_memory() for _ in xs]
    for i in range(len(xs)):
        b = i % 2
        plan.forward_host(x_host[i], x_dev[b], w.w_router, w.bias, w.w1, w.w3, w.w2, y_dev[b], y_host[i], wss[b],
                          stream=streams[b])
    torch.cuda.synchronize()
    for b in range(2):
        assert plan.device_status(wss[b], stream=streams[b]) == moe.MOE_OK
    for i in range(len(xs)):
        assert torch.equal(y_host[i], refs[i]), i
