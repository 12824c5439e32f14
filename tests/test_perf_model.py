"""The operator-level performance model ("Compute-Optimal Is Not Cluster-Optimal", gist.science
summary, Methodology item 2: an MoE layer priced per operator -- grouped GEMMs, data
movement, dispatch latency -- fitted to measurements and judged by its prediction error).

CPU: the fit recovers known latencies and rates from exact synthetic samples; the pair-tile
count follows its closed forms; the wave efficiency charges a partial last wave.
GPU: the pair-tile count the model prices equals the count the router's scan writes for the
expert GEMMs, on every listed bf16 workload and every granularity-sweep layer.
"""
import math

import numpy as np
import pytest

from top_routing_grouped_gb300 import perf_model as pm
from top_routing_grouped_gb300.workloads import SHAPES, ORDER, granularity_sweep, make_inputs


def test_fit_recovers_known_latency_and_rate():
    rng = np.random.default_rng(0)
    truth = {st: (0.002 * (i + 1), 1e-9 * (i + 3)) for i, st in enumerate(pm.STAGES)}
    samples = []
    for _ in range(6):
        f = {st: float(rng.uniform(1e6, 1e9)) for st in pm.STAGES}
        m = {st: truth[st][0] + truth[st][1] * f[st] for st in pm.STAGES}
        samples.append((f, m))
    params = pm.fit(samples)
    for st in pm.STAGES:
        L, slope = params[st]
        assert L == pytest.approx(truth[st][0], rel=1e-6, abs=1e-12)
        assert slope == pytest.approx(truth[st][1], rel=1e-9)
    # predictions of a held-out point are then exact, and so its error is zero
    f = {st: 5e8 for st in pm.STAGES}
    meas = {st: truth[st][0] + truth[st][1] * 5e8 for st in pm.STAGES}
    meas["total"] = sum(meas.values())
    pred = pm.predict(params, f)
    assert max(pm.mape(pred, meas).values()) < 1e-6
    # rates: B = 1 / slope in GB/s for movers (slope in ms per byte), R in TFLOP/s for GEMMs
    r = pm.rates(params)
    assert r["permute_GBps"] == pytest.approx(1e-6 / truth["permute"][1], rel=1e-9)
    assert r["gemm1_swiglu_TFLOPs"] == pytest.approx(1e-9 / truth["gemm1_swiglu"][1], rel=1e-9)


def test_fit_never_returns_a_negative_latency():
    x = np.array([1.0, 2.0, 3.0, 4.0]) * 1e8
    y = 2e-9 * x - 0.05
    samples = [({st: v for st in pm.STAGES}, {st: t for st in pm.STAGES}) for v, t in zip(x, y)]
    # through the origin, relative errors: minimise sum((s x / y - 1)^2)
    xw = x / y
    for L, slope in pm.fit(samples).values():
        assert L == 0.0
        assert slope == pytest.approx(float(xw.sum() / (xw @ xw)), rel=1e-12)


def test_fit_weighs_layers_by_relative_error():
    """Three layers a decade apart in size with +10 %, 0, -10 % deviations from one rate: the
    fit keeps every layer's relative error under 5 %, where an unweighted least-squares fit
    (dominated by the largest layer) misses the smallest by about 30 %."""
    x = np.array([1e8, 1e9, 1e10])
    y = np.array([1.1e-9 * 1e8, 1.0e-9 * 1e9, 0.9e-9 * 1e10]) + 0.02
    samples = [({st: v for st in pm.STAGES}, {st: t for st in pm.STAGES}) for v, t in zip(x, y)]
    L, slope = pm.fit(samples)["gemm1_swiglu"]
    assert np.max(np.abs(L + slope * x - y) / y) < 0.05
    (L0, s0), *_ = np.linalg.lstsq(np.stack([np.ones_like(x), x], axis=1), y, rcond=None)
    assert np.max(np.abs(L0 + s0 * x - y) / y) > 0.25


@pytest.mark.parametrize("counts, pairs", [
    ([0], 0), ([1], 1), ([128], 1), ([129], 1), ([256], 1), ([257], 2),
    ([1024], 4),               # 8 m-tiles: 4 pairs
    ([1025], 5),               # 9 m-tiles: 4 whole pairs and a half-empty one
    ([16 * 128 + 128], 9),     # 17 m-tiles: a whole group of 16 (8 pairs), then a group of one m-tile
    ([16 * 128 * 3 + 3 * 128], 26),  # 51 m-tiles: 3 groups of 8 pairs + a group of 3 (2 pairs)
    ([0, 1, 0, 300, 2048], 1 + 2 + 8),
])
def test_pair_tiles_closed_forms(counts, pairs):
    assert pm.pair_tiles(counts) == pairs


def test_features_charge_padding_and_the_last_wave():
    s = SHAPES["coarse_e8"]
    counts = [s.N // s.E] * s.E                     # 1024 rows each: 4 pairs, no padding
    f = pm.features(s, counts)
    pairs = pm.pair_tiles(counts)
    t1 = pairs * math.ceil(s.F / pm.GEMM1_TILE_N)   # 32 * 64 = 2048 tiles on 76 slots
    eff = t1 / (76 * math.ceil(t1 / 76))
    assert f["gemm1_swiglu"] == pytest.approx(4.0 * pairs * 256 * s.d * s.F / eff)
    assert f["gemm1_swiglu"] >= 4.0 * s.N * s.d * s.F
    # one row more in the first expert: a ninth m-tile, i.e. a fifth, half-empty pair
    f2 = pm.features(s, [counts[0] + 1] + counts[1:-1] + [counts[-1] - 1])
    assert f2["gemm1_swiglu"] > f["gemm1_swiglu"]
    assert f["route"] == s.T * s.d * 2 + s.N * 8


def test_features_count_gemm_work_at_the_reference_clock():
    """A layer that ran at a lower SM clock carries proportionally more GEMM work (the tensor
    cores' rate scales with the clock); the movers' bytes do not depend on it."""
    s = SHAPES["large_e64"]
    counts = [s.N // s.E] * s.E
    f = pm.features(s, counts)
    f_max = pm.features(s, counts, sm_mhz=pm.REF_MHZ)
    f_cap = pm.features(s, counts, sm_mhz=pm.REF_MHZ / 1.25)
    for st in pm.STAGES:
        assert f_max[st] == pytest.approx(f[st])
    for st in ("gemm1_swiglu", "gemm2_gate"):
        assert f_cap[st] == pytest.approx(1.25 * f[st])
    for st in ("route", "permute", "combine"):
        assert f_cap[st] == f[st]


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [SHAPES[n] for n in ORDER[1:]] + granularity_sweep(), ids=lambda s: s.name)
def test_pair_tiles_match_the_scan_kernel(shape):
    """The route stage only (the router, whose last CTA builds the tile table) on the
    workload's own inputs; the model's pair count for the routed counts equals the kernel's."""
    import torch
    from top_routing_grouped_gb300 import moe
    inp = make_inputs(shape, seed=0, parts=("x", "wr"))
    x = inp.x.to("cuda")
    wr = inp.w_router.to("cuda")
    bias = None if inp.bias is None else inp.bias.to("cuda")
    plan = moe.MoEPlan.for_shape(shape)
    ws = plan.new_workspace()
    # the route stage reads x, W_r and the bias only; the other pointers must merely be valid
    plan.forward_stage(0, x, wr, bias, x, x, x, x, ws)
    assert plan.device_status(ws) == moe.MOE_OK
    v = plan.views(ws)
    counts = v["expert_counts"].cpu().numpy()
    hdr = v["status"].cpu().numpy()
    assert counts.sum() == shape.N
    assert pm.pair_tiles(counts) == int(hdr[4]), (pm.pair_tiles(counts), int(hdr[4]))
    mt = (counts.astype(np.int64) + 127) // 128
    assert int(hdr[3]) == mt.sum()
    del ws
    torch.cuda.empty_cache()
