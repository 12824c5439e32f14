"""Parity with the CPU oracle on seeded random layer shapes.

Each case draws T, d, E, k, F, the router temperature, the Zipf router bias, renormalised gates,
the output dtype and the kernel path from one seeded generator, so that the combinations the
hand-picked cases do not name are covered too: odd and single tokens, one or many experts, k up
to min(E, 16), d and F any multiple of 64 on the tensor-core paths (any multiple of 4 on the fp32
SIMT path).  Every routed row and every token is compared under the same rules as the other parity
tests (routing, dispatch, H, Yp, y, the balancing scalar)."""
import numpy as np
import pytest

from top_routing_grouped_gb300.workloads import MoEShape, make_inputs

pytestmark = pytest.mark.gpu

N_CASES = 24


def draw_case(i):
    rng = np.random.default_rng(1000 + i)
    path = ["auto", "auto", "tc1", "simt"][i % 4]
    dtype = "f32" if path == "simt" and i % 8 == 3 else "bf16"
    T = int(rng.choice([1, 2, 37, 128, 129, 255, 511, 700, 1024, 1500]))
    E = int(rng.choice([1, 2, 3, 5, 8, 16, 31, 64]))
    k = int(rng.integers(1, min(E, 16) + 1))
    step = 4 if dtype == "f32" else 64
    d = int(rng.choice([64, 128, 192, 256, 384] if dtype == "bf16" else [4, 12, 68, 132, 256]))
    F = int(rng.choice([64, 128, 192, 320, 384] if dtype == "bf16" else [8, 36, 100, 192]))
    assert d % step == 0
    tau = float(rng.choice([0.5, 1.0, 2.0]))
    zipf = bool(rng.integers(0, 2))
    renorm = bool(rng.integers(0, 2))
    out_f32 = bool(rng.integers(0, 4) == 0)
    return dict(T=T, d=d, E=E, k=k, F=F, dtype=dtype, tau=tau, zipf=zipf, renorm=renorm, out_f32=out_f32,
                path=path, seed=2000 + i)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(i):
    import parity
    from top_routing_grouped_gb300 import moe
    c = draw_case(i)
    s = MoEShape(f"random{i}", T=c["T"], d=c["d"], E=c["E"], k=c["k"], F=c["F"], dtype=c["dtype"], tau=c["tau"],
                 zipf_bias=c["zipf"], renorm=c["renorm"])
    inp = make_inputs(s, seed=c["seed"])
    plan = moe.MoEPlan(s.T, s.d, s.E, s.k, s.F, dtype=s.dtype, out_dtype="f32" if c["out_f32"] else None, tau=s.tau,
                       has_bias=s.zipf_bias, path=c["path"], keep_logits=True, renorm_gates=s.renorm)
    rep, got = parity.full_check(s, inp, plan)
    print(f"\n[{c}]\n{rep}")
    assert got["status"] == moe.MOE_OK
