"""Benchmark of the sparse-MoE forward on GB300 (one JSON line on stdout, rank 0).

Workload (default): the large layer, T=32768 tokens, d_model=4096, E=64 experts, top-4,
d_expert=2048, router temperature 0.5, bf16 inputs, seeded synthetic data (the largest of the
listed layers; --workload picks another).  A step is one whole forward (router with its scan, permute,
grouped SwiGLU GEMM, grouped down-projection with gate and un-permute, combine, balancing
scalar) through the C ABI.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Under torchrun (N > 1) every rank runs an independent replica of the layer on its own GPU
(the forward has no exchange step on one device; "replicas only"), the timed region is
bracketed by barriers, and the max time over ranks is used.

--impl reference times the CPU oracle (the plain fp64 C implementation) on the host cores
on a bounded sample of the same workload; it is the baseline the GPU path is compared to.
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE fwd tokens/s and grouped-GEMM TFLOP/s (% of GB300 BF16 peak), 1 GPU"
STAGES = ["route", "permute", "gemm1_swiglu", "gemm2_gate", "combine"]
L2_FLUSH_BYTES = 256 << 20  # > 129 MB of L2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="large_e64")
    ap.add_argument("--tokens", type=int, default=0, help="override T (profiling a smaller case)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU work of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sweep", choices=["granularity"], default=None,
                    help="granularity sweep at equal active FLOPs (one JSON line with every G)")
    ap.add_argument("--train", action="store_true",
                    help="time the training step: forward (keeping activations) + backward")
    ap.add_argument("--perf-model", action="store_true",
                    help="fit the operator-level model on the listed workloads, predict the sweep")
    ap.add_argument("--ep-stage", type=int, default=0, metavar="W",
                    help="time the expert-parallel expert stage of W ranks emulated on this GPU")
    return ap.parse_args()


def reduce_max(value, device):
    """Max of a per-rank float over all ranks (the rank's own value when not distributed)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(units_per_rank_step, steps, world, max_ms):
    """Whole-job rate: the units every rank processed, over the slowest rank's time."""
    return units_per_rank_step * steps * world / (max_ms / 1e3)


def workload_config(shape, world):
    return {"workload": shape.name, "T": shape.T, "d_model": shape.d, "E": shape.E, "k": shape.k,
            "d_expert": shape.F, "dtype": shape.dtype, "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": "flushed between steps (256 MiB write outside the timed events)"}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sust=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


# sources each profiled kernel is built from: a recorded ncu traffic figure is only used
# while these files are unchanged
KERNEL_SOURCES = {
    "gemm1_swiglu": ["gemm_tc2.cu", "gemm_tc.h", "tc_ptx.cuh", "device_common.cuh", "moe_internal.h"],
}


def kernel_source_digest(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "top_routing_grouped_gb300", "csrc")
    for fn in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was taken on
    the current kernel sources (else None).  The summary gives either the full-size launch's
    bytes, or (for layers too large to capture whole) the bytes extrapolated to the full
    launch from captures at reduced T, with the fit it used."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.ncu.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_sources") != kernel_source_digest(kernel):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.dev), "-lms", "100"], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
            # nvidia-smi's first query initialises NVML, which can stall the GPU for a while:
            # let it finish (the first sample is written) before the timed region starts
            t0 = time.time()
            while time.time() - t0 < 5.0 and os.path.getsize(self.file.name) == 0:
                time.sleep(0.05)
            time.sleep(0.2)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), hw=parts[5], hwt=parts[6],
                                     swt=parts[7], pcap=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sms = sorted(r["sm"] for r in rows)
        reasons = set()
        for r in rows:
            if r["hw"] == "Active":
                reasons.add("hw_slowdown")
            if r["hwt"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def cpu_baseline(shape, inputs, target_s):
    """Time the oracle's whole forward on the first n tokens of the workload (a bounded
    sample: about target_s seconds of CPU work).  Returns the cpu_baseline dict."""
    import numpy as np
    import oracle
    host = inputs.numpy_for_oracle()

    def run(n):
        o = oracle.Oracle(n, shape.d, shape.E, shape.k, shape.F, tau=shape.tau, dtype=shape.dtype)
        t0 = time.perf_counter()
        o.forward(np.ascontiguousarray(host["x"][:n]), host["wr"], host["bias"], host["w1"], host["w3"], host["w2"])
        return time.perf_counter() - t0

    n0 = min(shape.T, 16)
    t_small = run(n0)
    n = int(min(shape.T, max(n0, n0 * target_s / max(t_small, 1e-6))))
    t = run(n) if n != n0 else t_small
    return {"value": n / t, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"whole forward of the first {n} of {shape.T} tokens of {shape.name} (fp64 C oracle, "
                      f"OpenMP over tokens), {t:.1f} s wall"}


def measure_shape(shape, steps, warmup):
    """Per-stage CUDA-event times (staged pass) and whole-forward time of one layer shape."""
    import torch
    from top_routing_grouped_gb300 import moe
    from top_routing_grouped_gb300.workloads import make_inputs
    dev = make_inputs(shape, seed=0).to("cuda")
    plan = moe.MoEPlan.for_shape(shape)
    ws = plan.new_workspace()
    y = torch.empty(shape.T, shape.d, dtype=plan.out_dtype, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    a = (dev.x, dev.w_router, dev.bias, dev.w1, dev.w3, dev.w2, y, ws)
    for _ in range(warmup):
        plan.forward(*a)
    whole, staged = [], [[0.0] * len(STAGES)]
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        evs[i][0].record()
        plan.forward(*a)
        evs[i][1].record()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)] for _ in range(steps)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        for i in range(steps):
            flush.zero_()
            for s_ in range(len(STAGES)):
                ev[i][s_].record()
                plan.forward_stage(s_, *a)
            ev[i][len(STAGES)].record()
        torch.cuda.synchronize()
    if plan.device_status(ws) != 0:
        raise RuntimeError(f"device status error on {shape.name}")
    step_ms = sum(b.elapsed_time(e) for b, e in evs) / steps
    stage_ms = {st: sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)) / steps
                for j, st in enumerate(STAGES)}
    counts = plan.views(ws)["expert_counts"].cpu().tolist()
    g_ms = stage_ms["gemm1_swiglu"] + stage_ms["gemm2_gate"]
    out = {"workload": shape.name, "T": shape.T, "d_model": shape.d, "E": shape.E, "k": shape.k, "d_expert": shape.F,
           "G": None, "tokens_per_s": shape.T / (step_ms / 1e3), "ms_per_step": step_ms,
           "grouped_gemm_tflops": shape.expert_flops / (g_ms / 1e3) / 1e12, "stage_ms": stage_ms, "counts": counts,
           "clocks": clk.summary()}
    del dev, plan, ws, y, flush
    torch.cuda.empty_cache()
    return out


def run_sweep(args):
    from top_routing_grouped_gb300.workloads import granularity_sweep
    pk = peaks()
    rows = []
    for sh in granularity_sweep():
        r = measure_shape(sh, max(10, args.steps // 5), args.warmup)
        r["G"] = 8192 // sh.F
        r["grouped_gemm_frac_of_bf16_peak"] = r["grouped_gemm_tflops"] / pk["bf16"]
        r.pop("counts")
        rows.append(r)
    print(json.dumps({"metric": METRIC, "sweep": "granularity G = d_ff/d_expert at equal active FLOPs "
                      "(T=8192, d=2048, d_ff=8192, E=8G, k=2G)", "unit": "tokens/s", "rows": rows}), flush=True)


def run_perf_model(args):
    from top_routing_grouped_gb300 import perf_model as pm
    from top_routing_grouped_gb300.workloads import SHAPES, granularity_sweep
    steps = max(10, args.steps // 5)
    train = [SHAPES[n] for n in ("coarse_e8", "fine_e32", "skewed_e128", "large_e64")]
    test = granularity_sweep()
    meas = {sh.name: measure_shape(sh, steps, args.warmup) for sh in train + test}
    mhz = {n: m["clocks"]["sm_mhz"] for n, m in meas.items()}
    feats = {sh.name: pm.features(sh, meas[sh.name]["counts"], sm_mhz=mhz[sh.name]) for sh in train + test}
    samples = [(feats[sh.name], meas[sh.name]["stage_ms"]) for sh in train]
    params = pm.fit(samples)
    # the same model without the clock term, for comparison
    feats0 = {sh.name: pm.features(sh, meas[sh.name]["counts"]) for sh in train + test}
    params0 = pm.fit([(feats0[sh.name], meas[sh.name]["stage_ms"]) for sh in train])
    report = []
    for sh in train + test:
        m = dict(meas[sh.name]["stage_ms"])
        m["total"] = sum(m[st] for st in pm.STAGES)
        pred = pm.predict(params, feats[sh.name])
        err = pm.mape(pred, m)
        err0 = pm.mape(pm.predict(params0, feats0[sh.name]), m)
        report.append({"workload": sh.name, "role": "fit" if sh in train else "held out", "sm_mhz": mhz[sh.name],
                       "total_err_pct_without_clock": round(100 * err0["total"], 2),
                       "measured_ms": {k: round(v, 4) for k, v in m.items()},
                       "predicted_ms": {k: round(v, 4) for k, v in pred.items()},
                       "abs_pct_err": {k: round(100 * v, 2) for k, v in err.items()}})
    held = [r for r in report if r["role"] == "held out"]
    print(json.dumps({"perf_model": "t = L + work / rate per kernel, fitted on the four listed bf16 workloads; "
                                    "GEMM work counted at the reference SM clock (work * 2070 MHz / the layer's "
                                    "median SM clock)",
                      "params": {st: {"L_ms": round(L, 5), "per_unit_ms": slope} for st, (L, slope) in params.items()},
                      "fitted_rates": pm.rates(params),
                      "held_out_total_mape_pct": round(sum(r["abs_pct_err"]["total"] for r in held) / len(held), 2),
                      "held_out_total_mape_pct_without_clock":
                          round(sum(r["total_err_pct_without_clock"] for r in held) / len(held), 2),
                      "rows": report}), flush=True)


def run_train(args):
    """Forward (training mode) + backward of the workload: one JSON line."""
    import torch
    from top_routing_grouped_gb300 import moe
    from top_routing_grouped_gb300.workloads import SHAPES, make_inputs
    shape = SHAPES[args.workload]
    if args.tokens:
        shape = shape.with_(T=args.tokens)
    inputs = make_inputs(shape, seed=0)
    dev = inputs.to("cuda")
    plan = moe.MoEPlan.for_shape(shape, training=True)
    ws = plan.new_workspace()
    y = torch.empty(shape.T, shape.d, dtype=torch.bfloat16, device="cuda")
    g = torch.Generator().manual_seed(1)
    dy = torch.randn(shape.T, shape.d, generator=g).to(torch.bfloat16).to("cuda")
    f32 = lambda *sz: torch.empty(*sz, dtype=torch.float32, device="cuda")
    E, d, F, T = shape.E, shape.d, shape.F, shape.T
    grads = (f32(T, d), f32(E, d), f32(E) if dev.bias is not None else None, f32(E, F, d), f32(E, F, d), f32(E, d, F))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    fa = (dev.x, dev.w_router, dev.bias, dev.w1, dev.w3, dev.w2, y, ws)
    ba = lambda: (dev.x, dev.w_router, dev.bias, dev.w1, dev.w3, dev.w2, dy, 0.01) + grads + (ws,)
    names = plan.backward_stage_names
    for _ in range(args.warmup):
        plan.forward(*fa)
        for i in range(len(names)):
            plan.backward_stage(i, *ba())
    K = max(10, args.steps // 5)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 2)] for _ in range(K)]
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        for k in range(K):
            flush.zero_()
            ev[k][0].record()
            plan.forward(*fa)
            for i in range(len(names)):
                ev[k][i + 1].record()
                plan.backward_stage(i, *ba())
            ev[k][len(names) + 1].record()
        torch.cuda.synchronize()
    if plan.device_status(ws) != 0:
        raise RuntimeError("device status error in the training step")
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    st_ms = {n: sum(e[i + 1].elapsed_time(e[i + 2]) for e in ev) / K for i, n in enumerate(names)}
    bwd_ms = sum(st_ms.values())
    N = shape.N
    gemm_flops = {"bwd_dh_swiglu": 2 * N * d * F, "bwd_dx_gemm": 4 * N * d * F, "bwd_dw13": 4 * N * d * F,
                  "bwd_dw2": 2 * N * d * F}
    pk = peaks()
    g_ms = sum(st_ms[n] for n in gemm_flops)
    g_tf = sum(gemm_flops.values()) / (g_ms / 1e3) / 1e12
    top = max(gemm_flops, key=lambda n: st_ms[n])
    top_tf = gemm_flops[top] / (st_ms[top] / 1e3) / 1e12
    print(json.dumps({
        "metric": "MoE training step (forward + backward) tokens/s; backward grouped-GEMM TFLOP/s", "unit": "tokens/s",
        "value": T / ((fwd_ms + bwd_ms) / 1e3), "ms_per_step": fwd_ms + bwd_ms, "forward_ms": fwd_ms, "backward_ms": bwd_ms,
        "steps": K, "warmup": args.warmup, "config": workload_config(shape, 1), "dtype": "bf16",
        "backward_stage_ms": st_ms, "backward_gemm_tflops": g_tf, "backward_gemm_frac_of_bf16_peak": g_tf / pk["bf16"],
        "roofline": {"kernel": top, "bound": "tensor", "achieved": top_tf, "peak": pk["bf16"], "unit": "TFLOP/s",
                     "frac": top_tf / pk["bf16"], "peak_source": f"{pk['src']} bf16 burst"},
        "clocks": clk.summary()}), flush=True)


def run_reference(args):
    """--impl reference: the oracle on the host cores, rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from top_routing_grouped_gb300.workloads import SHAPES, make_inputs
    import oracle
    shape = SHAPES[args.workload]
    inputs = make_inputs(shape, seed=0)
    # each step: a sample sized to ~per_step seconds, so the whole run stays within a few minutes
    per_step = min(20.0, max(0.05, 60.0 / max(args.steps + args.warmup, 1)))
    import numpy as np
    host = inputs.numpy_for_oracle()

    def run(n):
        o = oracle.Oracle(n, shape.d, shape.E, shape.k, shape.F, tau=shape.tau, dtype=shape.dtype)
        t0 = time.perf_counter()
        o.forward(np.ascontiguousarray(host["x"][:n]), host["wr"], host["bias"], host["w1"], host["w3"], host["w2"])
        return time.perf_counter() - t0

    n0 = min(4, shape.T)
    t0 = run(n0)
    n = int(min(shape.T, max(1, n0 * per_step / max(t0, 1e-6))))
    for _ in range(args.warmup):
        run(n)
    times = [run(n) for _ in range(args.steps)]
    tot = sum(times)
    value = n * len(times) / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(workload_config(shape, args.gpus), tokens_per_step=n),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"each step: whole forward of the first {n} of {shape.T} tokens"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ep_stage(args):
    """The expert stage of expert parallelism (moe_expert_forward: segment scan + the grouped
    SwiGLU GEMM and down-projection over the rows a rank receives), for W ranks emulated on this
    GPU: every rank routes and dispatches its token slice, the row all-to-all is done by copies,
    then each rank's expert stage is timed alone (CUDA events, L2 flushed before each step).
    Beside it, the same layer's two GEMMs in the single-GPU forward (staged events), which
    multiply the same rows without the per-source segments."""
    import torch
    from top_routing_grouped_gb300 import moe
    from top_routing_grouped_gb300.ep import EPRank, rows_per_rank
    from top_routing_grouped_gb300.workloads import SHAPES, make_inputs
    shape = SHAPES[args.workload]
    W = args.ep_stage
    if shape.T % W or shape.E % W:
        raise SystemExit(f"{shape.name}: T and E must split evenly over {W} ranks")
    dev = make_inputs(shape, seed=0).to("cuda")
    Tl, El = shape.T // W, shape.E // W
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    ranks = [EPRank(Tl, shape.d, shape.E, shape.k, shape.F, W, r, tau=shape.tau, has_bias=shape.zipf_bias,
                    renorm_gates=shape.renorm) for r in range(W)]
    xs = [dev.x[r * Tl:(r + 1) * Tl].contiguous() for r in range(W)]
    ys = [torch.empty(Tl, shape.d, dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    wl = [(dev.w1[r * El:(r + 1) * El].contiguous(), dev.w3[r * El:(r + 1) * El].contiguous(),
           dev.w2[r * El:(r + 1) * El].contiguous()) for r in range(W)]
    for r, rk in enumerate(ranks):
        rk.dispatch(xs[r], dev.w_router, dev.bias, ys[r])
    counts = [rk.counts().cpu() for rk in ranks]
    segs = [torch.cat([counts[j][r * El:(r + 1) * El] for j in range(W)]).cuda() for r in range(W)]
    send = [rows_per_rank(counts[r], W) for r in range(W)]
    for j in range(W):  # the row and gate all-to-alls, as copies
        for dst, src in ((ranks[j].x_recv, "xp"), (ranks[j].g_recv, "gate_perm")):
            parts = [ranks[r].views[src][sum(send[r][:j]):sum(send[r][:j + 1])] for r in range(W)]
            cat = torch.cat(parts)
            dst[:cat.shape[0]].copy_(cat)
    per_rank = []
    for r, rk in enumerate(ranks):
        for _ in range(args.warmup):
            rk.experts(segs[r], *wl[r])
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record()
            rk.experts(segs[r], *wl[r])
            ev[i][1].record()
        torch.cuda.synchronize()
        if rk.exp.device_status(rk.ws_exp) != moe.MOE_OK:
            raise RuntimeError(f"device status error in rank {r}'s expert stage")
        per_rank.append(sum(a.elapsed_time(b) for a, b in ev) / args.steps)
    rows = [int(sg.sum()) for sg in segs]
    seg_rows = [sg.cpu().tolist() for sg in segs]
    exec_rows = [128 * sum((c + 127) // 128 for c in sr) for sr in seg_rows]
    del ranks
    torch.cuda.empty_cache()
    single = measure_shape(shape, max(10, args.steps // 5), args.warmup)
    g_single = single["stage_ms"]["gemm1_swiglu"] + single["stage_ms"]["gemm2_gate"]
    flops = shape.expert_flops
    print(json.dumps({
        "ep_stage": {"workload": shape.name, "ranks": W, "tokens_per_rank": Tl, "experts_per_rank": El,
                     "rows_per_rank": rows, "m_tile_rows_per_rank": exec_rows,
                     "expert_stage_ms_per_rank": [round(t, 4) for t in per_rank],
                     "sum_ms": round(sum(per_rank), 4), "max_ms": round(max(per_rank), 4),
                     "single_gpu_gemms_ms": round(g_single, 4),
                     "sum_tflops": flops / (sum(per_rank) / 1e3) / 1e12,
                     "single_gpu_gemm_tflops": flops / (g_single / 1e3) / 1e12,
                     "from": "CUDA events around moe_expert_forward per rank (ranks emulated on one GPU, "
                             "all-to-alls by copies); single-GPU GEMMs from the staged forward"}}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.ep_stage:
        return run_ep_stage(args)
    if args.sweep:
        return run_sweep(args)
    if args.perf_model:
        return run_perf_model(args)
    if args.train:
        return run_train(args)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from top_routing_grouped_gb300 import moe
    from top_routing_grouped_gb300.workloads import SHAPES, make_inputs

    shape = SHAPES[args.workload]
    if args.tokens:
        shape = shape.with_(T=args.tokens)
    inputs = make_inputs(shape, seed=0)
    dev = inputs.to("cuda")
    plan = moe.MoEPlan.for_shape(shape)
    assert plan.stage_names == STAGES
    ws = plan.new_workspace()
    y = torch.empty(shape.T, shape.d, dtype=plan.out_dtype, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    targs = (dev.x, dev.w_router, dev.bias, dev.w1, dev.w3, dev.w2, y, ws)

    for _ in range(args.warmup):
        plan.forward(*targs)
    st = plan.device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")
    # rows the pair GEMMs multiply: each expert's rows rounded up to whole 256-row pair tiles
    counts = plan.views(ws)["expert_counts"].cpu().tolist()
    pair_rows = 256 * sum((c + 255) // 256 for c in counts)

    K = args.steps
    # timed region 1: whole forwards (one event pair per step; the kernels of a forward are
    # chained with programmatic dependent launch, so nothing is placed between them)
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        for i in range(K):
            flush.zero_()  # L2 flush between steps, outside the events
            ev_s[i].record(stream)
            plan.forward(*targs)
            ev_e[i].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    st = plan.device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region")
    step_times = sorted(ev_s[i].elapsed_time(ev_e[i]) for i in range(K))
    step_ms = sum(step_times) / K
    step_ms_median = step_times[K // 2]
    max_ms = reduce_max(step_ms * K, "cuda")
    value = throughput(shape.T, K, world, max_ms)

    # timed region 2: the same steps with an event between every two kernels, for the
    # per-kernel durations (and the roofline of the dominant kernel)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)] for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        flush.zero_()
        for s_ in range(len(STAGES)):
            ev[i][s_].record(stream)
            plan.forward_stage(s_, *targs)
        ev[i][len(STAGES)].record(stream)
    torch.cuda.synchronize()
    st = plan.device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after the per-stage timing")
    stage_ms = [sum(ev[i][s_].elapsed_time(ev[i][s_ + 1]) for i in range(K)) / K for s_ in range(len(STAGES))]
    staged_step_ms = sum(ev[i][0].elapsed_time(ev[i][len(STAGES)]) for i in range(K)) / K

    # timed region 3: each kernel launched R times back to back (every stage recomputes the
    # same result from the same workspace, and each launch is chained to the previous one as
    # in the forward, so launch gaps are hidden as they are there); one L2 flush before each
    # batch; the per-launch time of the movers is their bandwidth figure
    R = 20
    chained_ms = []
    for s_ in range(len(STAGES)):
        flush.zero_()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(R):
            plan.forward_stage(s_, *targs)
        b1.record(stream)
        torch.cuda.synchronize()
        chained_ms.append(b0.elapsed_time(b1) / R)
    st = plan.device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after the back-to-back kernel timing")

    # timed region 4: the forward captured once into a CUDA graph and replayed K times (the
    # same flush between steps, outside the events)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        plan.forward(*targs)
    for _ in range(3):
        graph.replay()
    gev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    gev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        flush.zero_()
        gev_s[i].record(stream)
        graph.replay()
        gev_e[i].record(stream)
    torch.cuda.synchronize()
    st = plan.device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after the graph replays")
    graph_ms = sum(gev_s[i].elapsed_time(gev_e[i]) for i in range(K)) / K
    graph_max_ms = reduce_max(graph_ms * K, "cuda")
    del graph

    # end to end through the host-buffer entry point: pinned x in, pinned y out, every step.
    # As a serving loop runs it: successive steps alternate between two streams, each with its
    # own workspace and device buffers, so one step's copies overlap the other's kernels (every
    # step still moves its own x in and y out).  The one-stream loop is reported beside it.
    e2e = None
    if not args.no_e2e:
        x_host = inputs.x.pin_memory()
        y_host = [torch.empty(shape.T, shape.d, dtype=plan.out_dtype).pin_memory() for _ in range(2)]
        x_dev = [torch.empty_like(dev.x) for _ in range(2)]
        y_dev = [y, torch.empty_like(y)]
        wss = [ws, plan.new_workspace()]
        streams = [stream, torch.cuda.Stream()]

        def host_step(i, two_streams):
            b = i % 2 if two_streams else 0
            plan.forward_host(x_host, x_dev[b], dev.w_router, dev.bias, dev.w1, dev.w3, dev.w2, y_dev[b], y_host[b],
                              wss[b], stream=streams[b])

        def timed(two_streams):
            for i in range(4):
                host_step(i, two_streams)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(streams[0])
            streams[1].wait_event(e0)
            for i in range(K):
                host_step(i, two_streams)
            streams[0].wait_stream(streams[1])
            e1.record(streams[0])
            torch.cuda.synchronize()
            return reduce_max(e0.elapsed_time(e1), "cuda")

        e_ms = timed(True)
        for b in range(2):
            st = plan.device_status(wss[b], stream=streams[b])
            if st != 0:
                raise RuntimeError(f"device status {st} after the host-buffer steps")
            assert torch.equal(y_host[b].to("cuda"), y), "host-buffer forward disagrees with the device forward"
        e_serial_ms = timed(False)
        e2e = {"value": throughput(shape.T, K, world, e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
               "d2h_bytes_per_step": y_host[0].numel() * y_host[0].element_size(),
               "mode": "moe_forward_host, steps alternating between two streams (own workspace and buffers each)",
               "one_stream_value": throughput(shape.T, K, world, e_serial_ms)}
        del wss, x_dev, y_dev

    if rank == 0:
        pk = peaks()
        gemm_flops = shape.expert_flops
        g1_ms, g2_ms = stage_ms[STAGES.index("gemm1_swiglu")], stage_ms[STAGES.index("gemm2_gate")]
        g1_flops = 4 * shape.N * shape.d * shape.F  # the dominant kernel: SwiGLU GEMM (W1 and W3)
        g1_tflops = g1_flops / (g1_ms / 1e3) / 1e12
        gemm_tflops = gemm_flops / ((g1_ms + g2_ms) / 1e3) / 1e12
        # the committed ncu figure is for the listed layer's full size only
        traffic = recorded_traffic(shape.name, "gemm1_swiglu") if shape.T == SHAPES[shape.name].T else None
        x_bytes = shape.T * shape.d * 2
        perm_bytes = x_bytes + shape.N * shape.d * 2 + 16 * shape.N
        comb_bytes = shape.N * shape.d * 2 + shape.T * shape.d * 2
        route_bytes = x_bytes + 8 * shape.N  # x once, the indices and gates out (the scan's tables are small)
        chained = chained_ms
        line = {
            "metric": METRIC,
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": max_ms / K, "ms_per_step_median": step_ms_median,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded Gaussian, fan-in scaled)",
            "config": workload_config(shape, world),
            "grouped_gemm_tflops": gemm_tflops,
            "grouped_gemm_frac_of_bf16_peak": gemm_tflops / pk["bf16"],
            "stage_ms": dict(zip(STAGES, stage_ms)),  # from timed region 2
            "stage_ms_back_to_back": dict(zip(STAGES, chained_ms)),  # timed region 3
            "mover_gbs": {"permute": perm_bytes / (chained[STAGES.index("permute")] / 1e3) / 1e9,
                          "combine": comb_bytes / (chained[STAGES.index("combine")] / 1e3) / 1e9,
                          "route": route_bytes / (chained[0] / 1e3) / 1e9,
                          "frac_of_measured_hbm": {
                              "permute": perm_bytes / (chained[STAGES.index("permute")] / 1e3) / 1e9 / pk["hbm"],
                              "combine": comb_bytes / (chained[STAGES.index("combine")] / 1e3) / 1e9 / pk["hbm"],
                              "route": route_bytes / (chained[0] / 1e3) / 1e9 / pk["hbm"]},
                          "from": "bytes / per-launch time of 20 back-to-back launches (timed region 3)"},
            "roofline": {"kernel": "gemm1_swiglu", "bound": "tensor", "achieved": g1_tflops, "peak": pk["bf16"],
                         "unit": "TFLOP/s", "frac": g1_tflops / pk["bf16"], "traffic": traffic,
                         "peak_source": f"{pk['src']} bf16 burst", "frac_of_sustained": g1_tflops / pk["bf16_sust"],
                         "algorithmic": f"4*N*d*F = {g1_flops} FLOP per launch (N = T*k = {shape.N} rows)",
                         "executed": {"rows": pair_rows, "tflops": g1_tflops * pair_rows / shape.N,
                                      "frac_of_sustained": g1_tflops * pair_rows / shape.N / pk["bf16_sust"],
                                      "note": "the tensor cores also multiply the padding of each expert's last "
                                              "256-row pair tile; achieved counts the N routed rows only"}},
            "graph": {"ms_per_step": graph_max_ms / K, "tokens_per_s": throughput(shape.T, K, world, graph_max_ms),
                      "from": "one forward captured into a CUDA graph, K replays (timed region 4)"},
            "e2e": e2e,
            "gpu_launches": len(STAGES) * K,
            "ms_per_step_with_stage_events": staged_step_ms,
            "clocks": clk.summary(),
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(shape, inputs, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
