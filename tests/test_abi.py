"""The C ABI without a GPU: the library loads, exports every function include/moe.h
declares, and plans validate their configuration (plan creation is host-only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def declared_functions():
    names = set()
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = re.sub(r"^\s*#[^\n]*", "", text, flags=re.M)   # preprocessor lines
        for m in re.finditer(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\(([^;{]*)\)\s*;", text):
            if not m.group(1).startswith(("typedef",)) and m.group(1) not in ("sizeof",):
                names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def moe():
    from top_routing_grouped_gb300 import build as b
    if not b.up_to_date():
        b.build()
    from top_routing_grouped_gb300 import moe as m
    return m


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("moe_plan", "moe_forward", "moe_aux_loss", "moe_plan_destroy", "moe_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(moe):
    lib = moe.lib()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_plan_workspace_and_stages(moe):
    p = moe.MoEPlan(4096, 2048, 8, 2, 8192, dtype="bf16")
    N = 4096 * 2
    # the workspace holds at least Xp, H and Yslot
    assert p.workspace_bytes >= N * 2048 * 2 * 2 + N * 8192 * 2
    assert p.stage_names == ["route", "permute", "gemm1_swiglu", "gemm2_gate", "combine"]
    p2 = moe.MoEPlan(4096, 2048, 8, 2, 8192, dtype="bf16", keep_logits=True)
    assert p2.workspace_bytes >= p.workspace_bytes + 4096 * 8 * 4


@pytest.mark.parametrize("kw, status", [
    (dict(T=0), "MOE_ERR_INVALID_ARG"),
    (dict(E=0), "MOE_ERR_INVALID_ARG"),
    (dict(E=300), "MOE_ERR_INVALID_ARG"),
    (dict(k=17, E=32), "MOE_ERR_INVALID_ARG"),
    (dict(k=5, E=4), "MOE_ERR_INVALID_ARG"),
    (dict(tau=0.0), "MOE_ERR_INVALID_ARG"),
    (dict(tau=float("inf")), "MOE_ERR_INVALID_ARG"),
    (dict(d=100, dtype="bf16"), "MOE_ERR_UNSUPPORTED"),
    (dict(d=130, dtype="f32"), "MOE_ERR_UNSUPPORTED"),
])
def test_plan_rejects_bad_configs(moe, kw, status):
    args = dict(T=64, d=128, E=8, k=2, F=256, dtype="f32", tau=1.0)
    args.update(kw)
    with pytest.raises(moe.MoEError) as ei:
        moe.MoEPlan(args["T"], args["d"], args["E"], args["k"], args["F"], dtype=args["dtype"], tau=args["tau"])
    assert status in str(ei.value)


def test_forward_rejects_bad_pointers_without_touching_the_device(moe):
    """Argument checks run on the host before any CUDA call."""
    lib = moe.lib()
    p = moe.MoEPlan(64, 128, 8, 2, 256, dtype="f32")
    P = ctypes.c_void_p
    # null x
    st = lib.moe_forward(p.handle, None, P(256), None, P(256), P(256), P(256), P(256), P(256), p.workspace_bytes, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # misaligned workspace
    st = lib.moe_forward(p.handle, P(256), P(256), None, P(256), P(256), P(256), P(256), P(128), p.workspace_bytes, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # workspace too small
    st = lib.moe_forward(p.handle, P(256), P(256), None, P(256), P(256), P(256), P(256), P(256), 16, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    assert b"workspace too small" in lib.moe_last_error()
    # bias required by the plan but missing
    pb = moe.MoEPlan(64, 128, 8, 2, 256, dtype="f32", has_bias=True)
    st = lib.moe_forward(pb.handle, P(256), P(256), None, P(256), P(256), P(256), P(256), P(256), pb.workspace_bytes, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    # stage out of range
    st = lib.moe_forward_stage(p.handle, 7, P(256), P(256), None, P(256), P(256), P(256), P(256), P(256),
                               p.workspace_bytes, None)
    assert st != moe.MOE_OK


def test_status_strings(moe):
    lib = moe.lib()
    assert lib.moe_status_string(moe.MOE_ERR_TIMEOUT) == b"MOE_ERR_TIMEOUT"
    assert lib.moe_status_string(99) == b"MOE_ERR_UNKNOWN"


def test_route_noalloc_checks_arguments_before_any_cuda_call(moe):
    """moe_route_noalloc validates everything on the host first: null or misaligned
    pointers, a missing bias, a shape beyond the static scratch.  The fake addresses are
    never dereferenced (every case is rejected before the first CUDA call)."""
    lib = moe.lib()
    P = ctypes.c_void_p
    p = moe.MoEPlan(300, 256, 16, 4, 128, dtype="bf16", training=True)
    ok = [P(4096 * (i + 1)) for i in range(8)]   # x, w_router, idx, gate, counts, aux, status
    x, wr, idx, gate, counts, aux, status = ok[:7]

    def call(plan=p, x=x, wr=wr, bias=None, idx=idx, gate=gate, counts=counts, aux=aux, status=status):
        return lib.moe_route_noalloc(plan.handle, x, wr, bias, idx, gate, counts, aux, status, None)

    for name in ("x", "wr", "idx", "gate", "counts", "aux", "status"):
        assert call(**{name: None}) == moe.MOE_ERR_INVALID_ARG, name
        assert call(**{name: P(4096 + 4)}) == moe.MOE_ERR_INVALID_ARG, name + " misaligned"
    pb = moe.MoEPlan(300, 256, 16, 4, 128, dtype="bf16", has_bias=True)
    assert call(plan=pb) == moe.MOE_ERR_INVALID_ARG
    assert b"router_bias" in lib.moe_last_error()
    # 2M tokens x k=8 needs 64 MiB of per-slot ranks: more than the static buffer holds
    big = moe.MoEPlan(2_000_000, 64, 8, 8, 64, dtype="bf16")
    assert call(plan=big) == moe.MOE_ERR_UNSUPPORTED
    assert b"MOE_NOALLOC_SCRATCH_BYTES" in lib.moe_last_error()
