"""The allocation-free routing entry point (moe_nvfp4_route_noalloc).

It serves callers that cannot allocate device memory: instead of a
caller-sized workspace it keeps its scratch in a fixed array inside the
library.  Its results must equal the routing intermediates that
moe_nvfp4_forward (the existing entry point) leaves in its workspace, bit
for bit, on consecutive calls that reuse the shared array.  This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""
import pytest
import torch

from nvfp4_mixture_experts_router_gb300 import api, build, synth

pytestmark = pytest.mark.gpu


def _forward_routing(c):
    dev = "cuda"
    x = synth.gen_x(c, dev)
    logits = synth.gen_logits(c, dev, x)
    bias = synth.gen_bias(c, dev)
    layer = api.MoELayer.create(c.T, c.H, c.I, c.E, c.K, c.flags())
    layer.prepare(synth.gen_w1(c, dev), synth.gen_w2(c, dev))
    layer.forward(x, logits, bias)
    torch.cuda.synchronize()
    T, E, K = c.T, c.E, c.K
    rows = int(layer.view("meta", torch.int32, 4)[0])
    ref = {
        "topk_ids": layer.view("topk_ids", torch.int32, T * K).clone(),
        "topk_w": layer.view("topk_w", torch.float32, T * K).clone(),
        "count": layer.view("count", torch.int32, E).clone(),
        "offsets": layer.view("offsets", torch.int32, E + 1).clone(),
        "padded_offsets": layer.view("padded_offsets", torch.int32, E + 1).clone(),
        "row_of_route": layer.view("row_of_route", torch.int32, T * K).clone(),
        "route_of_row": layer.view("route_of_row", torch.int32, rows).clone(),
    }
    return logits, bias, ref, rows


def _noalloc(c, logits, bias):
    T, E, K = c.T, c.E, c.K
    cap = api.moe_nvfp4_workspace_layout(api.shape(T, c.H, c.I, E, K), c.flags())["rows_cap"]
    i32 = dict(dtype=torch.int32, device="cuda")
    out = {
        "topk_ids": torch.full((T * K,), -7, **i32),
        "topk_w": torch.full((T * K,), -7.0, dtype=torch.float32, device="cuda"),
        "count": torch.full((E,), -7, **i32),
        "offsets": torch.full((E + 1,), -7, **i32),
        "padded_offsets": torch.full((E + 1,), -7, **i32),
        "row_of_route": torch.full((T * K,), -7, **i32),
        "route_of_row": torch.full((cap,), -7, **i32),
    }
    api.moe_nvfp4_route_noalloc(T, E, K, c.flags() & api.MOE_ROUTE_NO_RENORM, logits, bias, out)
    torch.cuda.synchronize()
    return out


def test_route_noalloc_matches_forward_on_consecutive_calls():
    build.build()
    cases = [synth.config(1),                                              # T=512, E=64, top-6, biased logits
             synth.MoEConfig("b", 300, 256, 128, 16, 4, mode=synth.MODE_PER_TOKEN, seed=21,
                             logits="normal", renorm=False),
             # decode sizes: the forward routes T <= 32 with its one-block
             # router + scan; here E = 40 is not a multiple of 32
             synth.config(0).with_(mode=synth.MODE_PER_TOKEN),             # T=16, E=8, top-2
             synth.MoEConfig("d", 24, 256, 128, 40, 3, mode=synth.MODE_PER_TOKEN, seed=22,
                             logits="normal")]
    refs = [_forward_routing(c) for c in cases]
    # calls in a row on the shared scratch, then the first shape again
    for c, (logits, bias, ref, rows) in list(zip(cases, refs)) + [(cases[0], refs[0])]:
        out = _noalloc(c, logits, bias)
        for name in ["topk_ids", "count", "offsets", "padded_offsets", "row_of_route"]:
            assert torch.equal(out[name], ref[name]), name
        assert torch.equal(out["route_of_row"][:rows], ref["route_of_row"])
        assert torch.equal(out["topk_w"], ref["topk_w"])     # same kernel: exact


def test_route_noalloc_rejects_oversized_shapes():
    build.build()
    T, E, K = 1 << 17, 1024, 8      # needs more than the fixed scratch
    logits = torch.zeros(1, device="cuda")
    out = {n: torch.zeros(1, dtype=torch.int32, device="cuda") for n in
           ["topk_ids", "topk_w", "count", "offsets", "padded_offsets", "row_of_route", "route_of_row"]}
    with pytest.raises(api.MoEError) as ei:
        api.moe_nvfp4_route_noalloc(T, E, K, 0, logits, None, out)
    assert ei.value.code == api.MOE_ERR_WORKSPACE
