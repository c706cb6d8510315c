"""Failure detection on the GPU without a fault: a bounded device wait that
runs out is reported through the status word, and the context and the
workspace stay usable.

The overlapped projections make the down-projection wait, per expert group,
for a count of stored hidden tiles that the up-projection raises (the
counters live at byte 8192 of the workspace header).  Setting those counters
far below zero before a call makes that count unreachable: the wait gives up
after its one-second limit, the kernel drains and returns, moe_check_status
reports MOE_ERR_TIMEOUT, and the grid's last CTA clears the counters, so the
next call runs normally."""

import numpy as np
import pytest
import torch

from sparse_mixture_experts_52_b300 import moe, synth

pytestmark = pytest.mark.gpu

READY_OFFSET = 8192   # int32 per expert group, zero between calls


def test_unreachable_wait_reports_timeout_and_the_next_call_recovers():
    cfg = synth.workload("switch_top1_cap", T=512, d_model=128, d_ff=256, E=16)
    inp = synth.make_inputs(cfg, device="cuda")
    layer = moe.MoELayer(cfg, inp, device="cuda")
    first = layer(inp["x"])["out"].clone()
    moe.check_status(layer.ws)
    G = cfg["E"] + cfg.get("n_shared", 0)
    poison = torch.full((G,), -(1 << 30), dtype=torch.int32, device="cuda")
    layer.ws[READY_OFFSET:READY_OFFSET + 4 * G].copy_(poison.view(torch.uint8))
    layer(inp["x"])
    with pytest.raises(moe.MoEError) as err:
        moe.check_status(layer.ws)
    assert err.value.status == 5   # MOE_ERR_TIMEOUT
    counters = layer.ws[READY_OFFSET:READY_OFFSET + 4 * G].view(torch.int32)
    assert int(counters.abs().max()) == 0, "the last CTA clears the counters"
    again = layer(inp["x"])["out"]
    moe.check_status(layer.ws)
    assert torch.equal(again, first)
