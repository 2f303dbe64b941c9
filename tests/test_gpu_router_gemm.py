"""GPU parity of the router-logit GEMM (logits = x . W_g^T on the tensor cores)
and of the forward that starts from it (moe_nvfp4_forward_gate).

Acceptance:
  * logits: |l_gpu - l_ref| <= (H/16 + 2) * 2^-24 * sum_h |x_h w_h| per element,
    l_ref the oracle's exactly summed logit rounded once to FP32.  The BF16
    products are exact; the tensor core rounds at most once per K = 16
    instruction when it adds into the FP32 accumulator, plus the final
    rounding -- H/16 + 1 roundings of partial sums no larger than the sum of
    the absolute products.
  * routing: the expert ids of every token are bit-exact, except for tokens
    whose oracle logits (with the bias) have two of their K+1 largest values
    closer than twice that token's bound -- a near tie the FP32 accumulation
    may legitimately order either way.  The test counts them.
  * router weights: softmax of logits that may each be off by the bound b_t
    (the token's largest): relative error up to 2 b_t on top of the
    launch sequence's 2e-6.
  * layer output: when no id differs, the full parity of the launch sequence
    (tests/gpu_parity.py); otherwise the same per-token checks on the tokens
    whose ids match (routing and grouping of the others differ by design).
"""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_mixture_experts_router_gb300 import api, build, synth

from gpu_parity import (bits, check_fc2_input, check_routing, check_x_quant, check_y, oracle_layer)

pytestmark = pytest.mark.gpu

ROUNDINGS_PER_K = 16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    api.lib()


def logit_bound(x_bits: np.ndarray, wg_bits: np.ndarray) -> np.ndarray:
    H = x_bits.shape[1]
    ax = np.abs(oracle.bf16_bits_to_f64(x_bits))
    aw = np.abs(oracle.bf16_bits_to_f64(wg_bits))
    return (H // ROUNDINGS_PER_K + 2) * 2.0 ** -24 * (ax @ aw.T)


def near_tie_tokens(logits: np.ndarray, bias, K: int, bound: np.ndarray) -> np.ndarray:
    """Tokens whose K+1 largest biased logits hold two values within twice
    the token's largest bound."""
    l = logits if bias is None else (logits + bias[None, :]).astype(np.float32)
    top = -np.sort(-l.astype(np.float64), axis=1)[:, :K + 1]
    gaps = top[:, :-1] - top[:, 1:]
    return np.nonzero(np.min(gaps, axis=1) <= 2.0 * bound.max(axis=1))[0]


@pytest.mark.parametrize("T,H,E", [(1, 256, 8), (16, 256, 8), (300, 384, 40), (512, 2048, 64), (200, 512, 300),
                                   (129, 7168, 256)])
def test_router_logits_match_oracle(T, H, E):
    c = synth.MoEConfig("rl", T, H, 128, E, 1, seed=31 + T)
    x = synth.gen_x(c, "cuda")
    wg = synth.gen_wg(c, "cuda")
    out = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    api.moe_nvfp4_router_logits(x, wg, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    xb, wb = bits(x), bits(wg)
    ref = oracle.router_logits(xb, wb).astype(np.float64)
    bound = logit_bound(xb, wb)
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"{int(np.sum(err > bound))} logits beyond the bound; worst {float((err / bound).max()):.3g}x"


@pytest.mark.parametrize("cfg", ["tiny", "mid", "mid_per_tensor_det", "odd_E"])
def test_forward_gate_parity(cfg):
    if cfg == "tiny":
        c = synth.config(0)
    elif cfg == "mid":
        c = synth.config(1)
    elif cfg == "mid_per_tensor_det":
        c = synth.config(1).with_(mode=synth.MODE_PER_TENSOR, deterministic=True, router_on_input=False)
    else:
        c = synth.MoEConfig("gate_oddE", 200, 384, 256, 40, 3, mode=synth.MODE_PER_TOKEN, seed=41, bias="normal")
    dev = "cuda"
    x = synth.gen_x(c, dev)
    wg = synth.gen_wg(c, dev)
    bias = synth.gen_bias(c, dev)
    w1 = synth.gen_w1(c, dev)
    w2 = synth.gen_w2(c, dev)
    x_np, wg_np = bits(x), bits(wg)
    w1_np, w2_np = bits(w1), bits(w2)
    bias_np = None if bias is None else bias.cpu().numpy()
    weights = lambda e: (w1_np[e], w2_np[e])
    L = oracle_layer(c)
    logits_ref = oracle.router_logits(x_np, wg_np)
    G1 = G2 = None
    if c.mode == synth.MODE_PER_TENSOR:
        G1 = np.float32(oracle.tensor_global_scale(oracle.bf16_bits_to_f64(x_np).astype(np.float32)))
        G2 = np.float32(oracle.fc2_input_scale(L, x_np, logits_ref, bias_np, weights, G1))
    flags = c.flags() | api.MOE_ROUTER_GEMM
    layer = api.MoELayer.create(c.T, c.H, c.I, c.E, c.K, flags)
    layer.prepare(w1, w2)
    g1 = None if G1 is None else torch.tensor([G1], device=dev)
    g2 = None if G2 is None else torch.tensor([G2], device=dev)
    y = layer.forward_gate(x, wg, bias, g1, g2)
    torch.cuda.synchronize()
    assert api.moe_nvfp4_last_device_status(layer.workspace) == api.MOE_OK

    # logits in the workspace
    got = layer.view("logits", torch.float32, c.T * c.E).cpu().numpy().reshape(c.T, c.E).astype(np.float64)
    bound = logit_bound(x_np, wg_np)
    assert np.all(np.abs(got - logits_ref) <= bound)

    # routing
    ids_ref, _ = oracle.router(logits_ref, bias_np, c.K, c.renorm)
    ids = layer.view("topk_ids", torch.int32, c.T * c.K).cpu().numpy().reshape(c.T, c.K)
    ties = set(near_tie_tokens(logits_ref, bias_np, c.K, bound).tolist())
    differ = set(np.nonzero((ids != ids_ref).any(axis=1))[0].tolist())
    assert differ <= ties, f"ids differ on tokens without a near tie: {sorted(differ - ties)[:8]}"
    print(f"{cfg}: {len(ties)} near-tie token(s) of {c.T}, {len(differ)} with different ids")

    prepared = {}
    if not differ:
        ref = oracle.forward(L, x_np, logits_ref, bias_np, weights, G1=G1, G2=G2, prepared=prepared)
        ror = check_routing(layer, ref, w_rel_tol=2e-6 + 2.0 * bound.max(axis=1, keepdims=True))
    else:
        keep = [t for t in range(c.T) if t not in differ]
        ref = oracle.forward(L, x_np, logits_ref, bias_np, weights, G1=G1, G2=G2, tokens=keep, prepared=prepared)
        ror = layer.view("row_of_route", torch.int32, c.T * c.K).cpu().numpy()
    check_x_quant(layer, ref, ror)
    frac, slack = check_fc2_input(layer, ref, ror, G2, prepared)
    check_y(y, ref, slack)
    assert frac >= 0.999


def test_forward_gate_rejects_misuse():
    c = synth.config(0)
    s = api.shape(c.T, c.H, c.I, c.E, c.K)
    layer = api.MoELayer.create(c.T, c.H, c.I, c.E, c.K, c.flags() | api.MOE_ROUTER_GEMM)
    x = torch.zeros(c.T, c.H, dtype=torch.bfloat16, device="cuda")
    logits = torch.zeros(c.T, c.E, device="cuda")
    y = torch.empty(c.T, c.H, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(1, device="cuda")
    with pytest.raises(api.MoEError):      # the plain forward takes the caller's logits: flag invalid there
        api.moe_nvfp4_forward(s, c.flags() | api.MOE_ROUTER_GEMM, x, logits, None, g, g, layer.prepared,
                              layer.workspace, y)
    with pytest.raises(api.MoEError):      # the gate forward needs the flag (it sizes the logits region)
        plain = api.MoELayer.create(c.T, c.H, c.I, c.E, c.K, c.flags())
        api.moe_nvfp4_forward_gate(s, c.flags(), x, torch.zeros(c.E, c.H, dtype=torch.bfloat16, device="cuda"),
                                   None, g, g, plain.prepared, plain.workspace, y)
