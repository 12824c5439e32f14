"""Failure detection without faulting the GPU.

Device side: every wait in the tensor-core kernels is bounded.  The test hook
MOE_FLAG_TEST_STALL makes the SwiGLU GEMM's producer withhold one shared-memory stage, so
the MMA issuer's wait runs out (a barrier nothing will complete); the kernel must record
MOE_ERR_TIMEOUT in the workspace status word, leave its loops, drain its copies, free TMEM
and return, and the context must stay usable for the next forward.

Host side: invalid arguments come back as status codes before any device work
(tests/test_abi.py covers the plan and pointer checks on the CPU).
"""
import pytest
import torch

from top_routing_grouped_gb300.workloads import MoEShape, make_inputs


# sites a timeout of the SwiGLU GEMM may be recorded at: producer / MMA issuer / epilogue of
# the one-SM kernel, then of the CTA-pair kernel
GEMM1_TIMEOUT_SITES = (b"0x501", b"0x511", b"0x531", b"0x541", b"0x551", b"0x571")


@pytest.mark.gpu
@pytest.mark.parametrize("path", ["auto", "tc1"])
def test_stalled_pipeline_times_out_and_the_context_survives(path):
    from top_routing_grouped_gb300 import moe
    import parity

    s = MoEShape("stall", T=256, d=128, E=4, k=2, F=128, dtype="bf16")
    dev = make_inputs(s, seed=0).to("cuda")
    stalled = moe.MoEPlan(s.T, s.d, s.E, s.k, s.F, test_stall=True, wait_timeout_ns=50_000_000, path=path)
    ws = stalled.new_workspace()
    y = torch.empty(s.T, s.d, dtype=torch.bfloat16, device="cuda")
    stalled.forward(dev.x, dev.w_router, None, dev.w1, dev.w3, dev.w2, y, ws)
    assert stalled.device_status(ws) == moe.MOE_ERR_TIMEOUT
    msg = moe.lib().moe_last_error()
    assert any(site in msg for site in GEMM1_TIMEOUT_SITES), msg

    # the same context still runs a correct forward afterwards
    plan = moe.MoEPlan.for_shape(s, keep_logits=True, path=path)
    rep, got = parity.full_check(s, make_inputs(s, seed=0), plan)
    assert got["status"] == moe.MOE_OK


def test_stall_hook_needs_the_tensor_core_path():
    from top_routing_grouped_gb300 import build as b
    if not b.up_to_date():
        b.build()
    from top_routing_grouped_gb300 import moe
    with pytest.raises(moe.MoEError) as ei:
        moe.MoEPlan(64, 128, 4, 2, 128, dtype="f32", test_stall=True)
    assert "MOE_ERR_INVALID_ARG" in str(ei.value)
