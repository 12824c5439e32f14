"""Operator-level performance model of this MoE layer on one GPU.

"Compute-Optimal Is Not Cluster-Optimal" (gist.science summary, Methodology item 2) prices
an MoE layer per operator -- dense and grouped GEMMs, data movement, dispatch latency --
and reports how well that predicts measured utilisation.  This module does the same for the
kernels of this library, from quantities the layer shape and the routing fix:

  mover kernels (router with its scan, permute, combine):  t = L + bytes / B
  grouped GEMMs:                                           t = L + FLOP_padded / (R * wave_efficiency)

FLOP_padded counts the rows the tensor cores actually process (256-row CTA-pair tiles of
each expert, so padding and odd m-tiles count), and wave_efficiency = tiles / (slots *
ceil(tiles / slots)) charges the last partial wave of the persistent grid.  The tensor-core
rate scales with the SM clock, which the 1.4 kW power cap pulls down on the largest layers:
given the median SM clock f seen while a layer ran, the GEMM work is counted at the reference
clock, FLOP_padded * f_ref / f.  L, B, R are fitted per kernel by least squares on measured
stage times (fit), then used to predict others (predict); mape() reports the mean absolute
percentage error.
"""
import math

import numpy as np

STAGES = ("route", "permute", "gemm1_swiglu", "gemm2_gate", "combine")
PAIR_ROWS = 256      # rows of one CTA-pair tile
GROUP_MTILES = 16    # 128-row m-tiles per scheduling group
GEMM1_TILE_N = 128   # output columns of a SwiGLU tile (W1 and W3 halves)
GEMM2_TILE_N = 256


def pair_tiles(counts):
    """CTA-pair m-tiles per expert: groups of up to GROUP_MTILES m-tiles, ceil(m/2) pairs per
    group (GROUP_MTILES is even, so this is ceil(m/2) per expert whatever the group size)."""
    pairs = 0
    for c in counts:
        mt = (int(c) + 127) // 128
        full, last = divmod(mt, GROUP_MTILES)
        pairs += full * (GROUP_MTILES // 2) + (last + 1) // 2
    return pairs


REF_MHZ = 2070.0  # the GB300's maximum SM clock


def features(shape, counts, slots=76, sm_mhz=None):
    """Per-stage work of one forward: bytes for movers, padded FLOPs over the wave efficiency
    for the GEMMs, counted at REF_MHZ when the layer's SM clock sm_mhz is given."""
    T, d, E, k, F = shape.T, shape.d, shape.E, shape.k, shape.F
    N = T * k
    pairs = pair_tiles(counts)
    rows = pairs * PAIR_ROWS
    t1 = pairs * math.ceil(F / GEMM1_TILE_N)
    t2 = pairs * math.ceil(d / GEMM2_TILE_N)
    wave = lambda n: n / (slots * math.ceil(n / slots)) if n else 1.0
    clk = REF_MHZ / sm_mhz if sm_mhz else 1.0
    return {
        "route": T * d * 2 + N * 8,
        "permute": T * d * 2 + N * d * 2 + 28 * N,
        "gemm1_swiglu": 4.0 * rows * d * F / wave(t1) * clk,
        "gemm2_gate": 2.0 * rows * d * F / wave(t2) * clk,
        "combine": N * d * 2 + T * d * 2,
    }


def fit(samples):
    """samples: list of (features dict, measured stage_ms dict).  Returns, per stage, the
    (L [ms], slope [ms per unit]) fit of t = L + slope * work (L >= 0) that minimises the
    squared RELATIVE errors, so that every layer weighs the same whatever its size."""
    params = {}
    for st in STAGES:
        x = np.array([f[st] for f, _ in samples], dtype=np.float64)
        y = np.array([m[st] for _, m in samples], dtype=np.float64)
        w = 1.0 / y
        A = np.stack([np.ones_like(x), x], axis=1) * w[:, None]
        (L, slope), *_ = np.linalg.lstsq(A, y * w, rcond=None)
        if L < 0:  # a negative launch latency is not physical: refit through the origin
            xw, yw = x * w, y * w
            L, slope = 0.0, float((xw @ yw) / (xw @ xw))
        params[st] = (float(L), float(slope))
    return params


def predict(params, feats):
    stage = {st: params[st][0] + params[st][1] * feats[st] for st in STAGES}
    stage["total"] = sum(stage[st] for st in STAGES)
    return stage


def mape(pred, meas, keys=STAGES + ("total",)):
    return {k: abs(pred[k] - meas[k]) / meas[k] for k in keys}


def rates(params):
    """Fitted throughputs: B in GB/s for the movers, R in TFLOP/s for the GEMMs."""
    out = {}
    for st in ("route", "permute", "combine"):
        out[st + "_GBps"] = 1e-6 / params[st][1] if params[st][1] > 0 else None
    for st in ("gemm1_swiglu", "gemm2_gate"):
        out[st + "_TFLOPs"] = 1e-9 / params[st][1] if params[st][1] > 0 else None
    return out
