"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small shapes are checked in full (every token, every routed row of Xp, H and Yp, every y).
The listed workloads are checked at full size in the launch configuration the benchmark
uses: routing, gates, dispatch, Xp and aux on every token; H and Yp on rows that cover
every m-tile of the expert GEMMs and every row of each expert's last pair tile; y on every
token of the two smaller bf16 workloads and on the tokens of those tiles for the larger
two.
"""
import numpy as np
import pytest
import torch

from top_routing_grouped_gb300.workloads import SHAPES, ORDER, MoEShape, make_inputs

pytestmark = pytest.mark.gpu

PATHS = ["auto", "tc1", "simt"]


@pytest.fixture(scope="module")
def moe():
    from top_routing_grouped_gb300 import moe as m
    return m


def small(name, T, d, E, k, F, dtype="bf16", tau=1.0):
    return MoEShape(name, T=T, d=d, E=E, k=k, F=F, dtype=dtype, tau=tau)


def check(moe, shape, inputs, path="auto", y_tokens=None, h_rows=None, has_bias=None):
    import parity
    plan = moe.MoEPlan(shape.T, shape.d, shape.E, shape.k, shape.F, dtype=shape.dtype, tau=shape.tau,
                       has_bias=(inputs.bias is not None) if has_bias is None else has_bias,
                       path=path, keep_logits=True, renorm_gates=shape.renorm)
    rep, got = parity.full_check(shape, inputs, plan, y_tokens=y_tokens, h_rows=h_rows)
    print(f"\n[{shape.name} path={path}]\n{rep}")
    return rep, got


def test_tiny_f32_full(moe):
    s = SHAPES["tiny_f32"]
    check(moe, s, make_inputs(s, seed=0))


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dims", [
    (300, 256, 8, 2, 192),    # ragged T (not a multiple of the 128-token blocks), 3 n-tiles
    (1, 128, 8, 2, 128),      # a single token
    (257, 128, 1, 1, 64),     # E = 1, k = 1: a dense SwiGLU FFN
    (130, 192, 4, 4, 128),    # k = E: every expert on every token
    (512, 128, 16, 8, 320),   # k = 8 (the largest), F not a power of two
    (40, 64, 64, 2, 64),      # more experts than routed rows per expert: counts of 0, 1, 2
], ids=lambda d: "x".join(map(str, d)))
def test_small_bf16(moe, path, dims):
    T, d, E, k, F = dims
    s = small("small", T, d, E, k, F)
    check(moe, s, make_inputs(s, seed=1), path=path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dims", [
    (300, 256, 256, 16, 64),   # the most experts and the largest top-k the plan accepts
    (200, 128, 200, 8, 64),    # E above 128 and not a multiple of 16 (four threads finish a token)
    (100, 2048, 33, 3, 64),    # one token block, long d: d split over a cluster of four, deepest ring
    (130, 4096, 160, 5, 64),   # many experts: the kept exp(z - max) no longer fits, the softmax sums recompute it
], ids=lambda d: "x".join(map(str, d)))
def test_maximum_sizes(moe, path, dims):
    """The largest expert counts and top-k, and the router shapes whose shared memory is
    tightest (split-d clusters with a receive buffer, many experts)."""
    T, d, E, k, F = dims
    s = small("maximum", T, d, E, k, F)
    check(moe, s, make_inputs(s, seed=8), path=path)


@pytest.mark.parametrize("path", PATHS)
def test_temperature_and_bias(moe, path):
    s = small("tau_bias", 384, 256, 16, 4, 128, tau=0.5)
    inp = make_inputs(s, seed=2)
    inp.bias = torch.linspace(-1.0, 1.0, s.E, dtype=torch.float32)
    check(moe, s, inp, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_all_tokens_to_one_expert(moe, path):
    """A +100 logit bias on expert 0: every token routes its first slot there."""
    s = small("collapse", 300, 128, 8, 2, 128)
    inp = make_inputs(s, seed=3)
    inp.bias = torch.zeros(s.E, dtype=torch.float32)
    inp.bias[0] = 100.0
    rep, got = check(moe, s, inp, path=path)
    idx = got["views"]["topk_idx"].cpu()
    assert torch.all(idx[:, 0] == 0)
    assert got["views"]["expert_counts"][0].item() == s.T


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T", [2048, 2049, 2176, 2304, 4097])
def test_scheduling_group_boundaries(moe, path, T):
    """k = 1 and a +100 logit bias on expert 0: all T rows in one expert, so its m-tiles (128
    rows) fill scheduling groups of 16 exactly (T = 2048), spill one row into a second group
    (2049: a half-empty pair of one row), fill a 17th m-tile (2176: an odd group of one full
    m-tile), an 18th (2304: a whole second pair) or a third group (4097).  Every row of H, Yp
    and y is compared."""
    s = small("groups", T, 128, 4, 1, 64)
    inp = make_inputs(s, seed=7)
    inp.bias = torch.zeros(s.E, dtype=torch.float32)
    inp.bias[0] = 100.0
    rep, got = check(moe, s, inp, path=path)
    assert got["views"]["expert_counts"][0].item() == T


@pytest.mark.parametrize("path", PATHS)
def test_uniform_router_aux_is_one(moe, path):
    """W_r = 0: every logit equal, p = 1/E; the balancing scalar is exactly 1 (k slots
    always sum to 1 whatever the tie-break) and top-k takes the lowest indices."""
    s = small("uniform", 256, 128, 8, 2, 64)
    inp = make_inputs(s, seed=4)
    inp.w_router = torch.zeros_like(inp.w_router)
    rep, got = check(moe, s, inp, path=path)
    assert abs(got["aux"] - 1.0) <= 1e-6
    assert torch.all(got["views"]["topk_idx"].cpu() == torch.tensor([0, 1], dtype=torch.int32))


@pytest.mark.parametrize("path", PATHS)
def test_out_dtype_f32(moe, path):
    import parity
    s = small("outf32", 200, 128, 8, 2, 128)
    inp = make_inputs(s, seed=5)
    plan = moe.MoEPlan(s.T, s.d, s.E, s.k, s.F, dtype="bf16", out_dtype="f32", path=path)
    got = parity.run_gpu(plan, inp.to("cuda"))
    plan_b = moe.MoEPlan(s.T, s.d, s.E, s.k, s.F, dtype="bf16", path=path)
    got_b = parity.run_gpu(plan_b, inp.to("cuda"))
    assert got["y"].dtype == torch.float32
    # same arithmetic; only the final rounding differs
    assert torch.allclose(got["y"].bfloat16().float(), got_b["y"].float(), atol=0, rtol=0)


@pytest.mark.parametrize("path", PATHS)
def test_deterministic(moe, path):
    import parity
    s = small("det", 640, 256, 16, 4, 256)
    dev = make_inputs(s, seed=6).to("cuda")
    plan = moe.MoEPlan(s.T, s.d, s.E, s.k, s.F, path=path)
    a = parity.run_gpu(plan, dev)
    b = parity.run_gpu(plan, dev)
    assert torch.equal(a["y"], b["y"])
    assert a["aux"] == b["aux"]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dims", [
    (300, 256, 8, 1, 128),     # k = 1 (Switch-style routing)
    (256, 128, 32, 16, 64),    # k = 16, the largest top-k
    (200, 128, 8, 4, 128),
], ids=lambda d: "x".join(map(str, d)))
@pytest.mark.parametrize("renorm", [False, True], ids=["softmax_gates", "renorm_gates"])
def test_variants(moe, path, dims, renorm):
    """Variants the page leaves open: k = 1, large k, gates renormalised over the chosen."""
    T, d, E, k, F = dims
    s = small("variant", T, d, E, k, F).with_(renorm=renorm)
    rep, got = check(moe, s, make_inputs(s, seed=7), path=path)
    if renorm:
        g = got["views"]["topk_gate"].cpu().double()
        assert torch.allclose(g.sum(dim=1), torch.ones(T, dtype=torch.float64), atol=1e-6)


@pytest.mark.parametrize("name", ORDER[1:])
@pytest.mark.parametrize("path", ["auto", "tc1"])
def test_full_size_workloads(moe, name, path):
    """The listed workloads at full size, in the launch configuration the benchmark times:
    every token's routing and dispatch (ordered indices on decided tokens), Xp on every
    row, H and Yp on rows covering every m-tile and each expert's last pair tile, and y on
    every token (coarse_e8, fine_e32 on the benchmark's path) or on the tokens of the
    experts' last pair tiles, the smallest expert and a seeded sample (the larger two, and
    the one-CTA path).  Yp rows carry what the combine gathers, whose indices (slot_pos)
    are checked bit-exact on every slot, so the tile-covering Yp rows stand for y there."""
    import parity
    s = SHAPES[name]
    inp = make_inputs(s, seed=0)
    plan = moe.MoEPlan.for_shape(s, path=path, keep_logits=True)
    every_token = path == "auto" and name in ("coarse_e8", "fine_e32")
    rep, got = parity.full_check(s, inp, plan, y_tokens=None if every_token else "tiles", h_rows="tiles")
    print(f"\n[{name} path={path}]\n{rep}")
    if name == "skewed_e128":
        assert (got["views"]["expert_counts"] == 0).sum().item() >= 1
