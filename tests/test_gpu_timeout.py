"""The bounded waits of the GEMM pipeline give up cleanly.

Every mbarrier wait in the GEMM kernels has a time limit (1 s of the GPU's
global timer).  The MOE_DEBUG_FC1_SKIP_STAGE test hook makes the producer of
the first FC1 CTA leave one pipeline stage unissued -- no copy and no arrival
on that stage's barriers, so nothing is in flight against them -- and the
MMA thread's wait on it runs out.  Nothing faults and nothing hangs: the CTA
raises the timeout bit in the device status word, drains and exits, and the
next forward on the same workspace is clean and in parity with the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from nvfp4_mixture_experts_router_gb300 import api, build, synth

from gpu_parity import (check_fc2_input, check_routing, check_x_quant, check_y, make_inputs, oracle_layer,
                        scales_for)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    api.lib()


@pytest.mark.parametrize("mode", [synth.MODE_PER_TENSOR, synth.MODE_PER_TOKEN])
def test_bounded_wait_gives_up_then_next_forward_is_clean(mode):
    c = synth.config(0).with_(mode=mode, gemm_swap="never")
    inp = make_inputs(c)
    G1, G2 = scales_for(inp)
    flags = c.flags()
    layer = api.MoELayer.create(c.T, c.H, c.I, c.E, c.K, flags | api.MOE_DEBUG_FC1_SKIP_STAGE)
    layer.prepare(inp.w1, inp.w2)
    g1 = None if G1 is None else torch.tensor([G1], dtype=torch.float32, device="cuda")
    g2 = None if G2 is None else torch.tensor([G2], dtype=torch.float32, device="cuda")

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    layer.forward(inp.x, inp.logits, inp.bias, g1, g2)
    status = api.moe_nvfp4_last_device_status(layer.workspace)   # synchronizes
    waited = time.perf_counter() - t0
    assert status == api.MOE_ERR_TIMEOUT, api.STATUS_NAMES.get(status)
    assert waited >= 0.9, f"the wait gave up after {waited:.3f} s, before its 1 s limit"
    assert waited < 30.0

    # the same workspace and weights, hook off: a clean forward in parity
    layer.flags = flags
    y = layer.forward(inp.x, inp.logits, inp.bias, g1, g2)
    torch.cuda.synchronize()
    assert api.moe_nvfp4_last_device_status(layer.workspace) == api.MOE_OK
    prepared = {}
    ref = oracle.forward(oracle_layer(c), inp.x_np, inp.logits_np, inp.bias_np,
                         lambda e: (inp.w1_np[e], inp.w2_np[e]), G1=G1, G2=G2, prepared=prepared)
    ror = check_routing(layer, ref)
    check_x_quant(layer, ref, ror)
    frac, slack = check_fc2_input(layer, ref, ror, G2, prepared)
    check_y(y, ref, slack)
    assert frac >= 0.999
