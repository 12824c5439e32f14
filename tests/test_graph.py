"""The forward and the backward captured into a CUDA graph.

moe_forward and moe_backward only enqueue work (kernels chained by programmatic dependent
launch, one memset, no allocation, no synchronisation), so a caller can capture them into a
CUDA graph once and replay it.  A replay must give exactly the eager result, and must read
the buffers' current contents (new x values give the new x's output).
"""
import pytest
import torch

from top_routing_grouped_gb300.workloads import MoEShape, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from top_routing_grouped_gb300 import moe as m
    return m


def capture(fn):
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    return g


@pytest.mark.parametrize("path", ["auto", "tc1", "simt"])
@pytest.mark.parametrize("dims", [
    (300, 256, 8, 2, 192),      # ragged T, several n-tiles
    (2048, 512, 16, 4, 1024),   # several pair tiles per expert
], ids=lambda d: "x".join(map(str, d)))
def test_forward_graph_replay(moe, path, dims):
    T, d, E, k, F = dims
    s = MoEShape("graph", T=T, d=d, E=E, k=k, F=F, dtype="bf16")
    dev = make_inputs(s, seed=21).to("cuda")
    x2 = make_inputs(s, seed=22).x.to("cuda")
    plan = moe.MoEPlan.for_shape(s, path=path)
    ws = plan.new_workspace()
    y = torch.empty(T, d, dtype=plan.out_dtype, device="cuda")
    args = (dev.w_router, dev.bias, dev.w1, dev.w3, dev.w2, y, ws)
    x = dev.x.clone()

    plan.forward(x, *args)
    torch.cuda.synchronize()
    y_eager = y.clone()
    aux_eager = plan.aux_loss(ws).item()
    plan.forward(x2, *args)
    torch.cuda.synchronize()
    y2_eager = y.clone()

    g = capture(lambda: plan.forward(x, *args))
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert plan.device_status(ws) == 0
    assert torch.equal(y, y_eager)
    assert plan.aux_loss(ws).item() == aux_eager
    x.copy_(x2)  # the graph reads x's current contents
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert plan.device_status(ws) == 0
    assert torch.equal(y, y2_eager)


def test_train_step_graph_replay(moe):
    """Forward + backward of a training plan in one graph."""
    T, d, E, k, F = 512, 256, 8, 2, 512
    s = MoEShape("graph_train", T=T, d=d, E=E, k=k, F=F, dtype="bf16")
    dev = make_inputs(s, seed=23).to("cuda")
    plan = moe.MoEPlan.for_shape(s, training=True)
    ws = plan.new_workspace()
    y = torch.empty(T, d, dtype=plan.out_dtype, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(5)
    dy = torch.randn(T, d, device="cuda", generator=gen).to(plan.out_dtype)
    f32 = dict(device="cuda", dtype=torch.float32)
    outs = dict(dx=torch.empty(T, d, **f32), dwr=torch.empty(E, d, **f32), db=None,
                dw1=torch.empty(E, F, d, **f32), dw3=torch.empty(E, F, d, **f32), dw2=torch.empty(E, d, F, **f32))
    w = (dev.w_router, dev.bias, dev.w1, dev.w3, dev.w2)

    def step():
        plan.forward(dev.x, *w, y, ws)
        plan.backward(dev.x, *w, dy, 0.01, outs["dx"], outs["dwr"], outs["db"], outs["dw1"], outs["dw3"],
                      outs["dw2"], ws)

    step()
    torch.cuda.synchronize()
    ref = {n: t.clone() for n, t in outs.items() if t is not None}
    y_ref = y.clone()
    g = capture(step)
    for t in list(outs.values()) + [y]:
        if t is not None:
            t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert plan.device_status(ws) == 0
    assert torch.equal(y, y_ref)
    for n, t in ref.items():
        assert torch.equal(outs[n], t), n
