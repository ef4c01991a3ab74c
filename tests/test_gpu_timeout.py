"""Bounded device-side waits: a wait that runs out is reported, and the GPU stays usable.

Every wait of the library's kernels on a copy or an MMA is bounded.  The test
hook moe_debug_set_waits(limit, stall=1) makes the first wait of the chained
decode, segmented GEMV and tensor-core kernels wait on a barrier that nothing
completes (no faulty input, no fault): the call must return, the status word
must read MOE_ERR_TIMEOUT after the caller's sync, and the next normal call on
the same workspace must give the bits of a call made before, with MOE_OK.
"""
from __future__ import annotations

import pytest
import torch

import synth
from helpers import make_layer
from quantized_routed_expert_sigmoid_gb300 import _native as N

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000          # 2 ms


@pytest.mark.parametrize("T, tc_min, path", [(2, 0, "decode_chain"), (9, 1 << 30, "gemv"), (200, 0, "tensor")])
def test_wait_that_runs_out_is_reported(T, tc_min, path):
    tl = make_layer(synth.DECODE, 70 + T, T, exact_all=(path == "tensor"))
    layer = tl.moe_layer(tc_min_tokens=tc_min)
    assert layer.path(T) == path
    x = tl.x.cuda()
    ref = layer(x).clone()
    torch.cuda.synchronize()
    assert layer.device_status(T) == N.MOE_OK
    try:
        N.moe_debug_set_waits(LIMIT_NS, 1)
        layer(x)
        torch.cuda.synchronize()
    finally:
        N.moe_debug_set_waits(0, 0)
    assert layer.device_status(T) == N.MOE_ERR_TIMEOUT
    again = layer(x)
    torch.cuda.synchronize()
    assert layer.device_status(T) == N.MOE_OK
    assert torch.equal(again, ref), "the call after a timeout differs from the one before"
