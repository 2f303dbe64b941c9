"""Shared driver for the GPU parity tests: run one layer configuration
through the CUDA library (C ABI) and through the CPU oracle on the same
seeded inputs, and compare every stage.

Acceptance (stated once, used everywhere):
  * bit-exact: expert ids, counts, offsets, padded offsets, the permutation
    (row_of_route, route_of_row, M-tile -> expert map), the NVFP4 codes and
    scales of x (and the per-token G1), the prepared weight codes/scales/G.
  * router weights: |w - w_ref| <= 2e-6 * w_ref + 1e-7 (float32 expf vs FP64).
  * FC2-input codes: >= 99.9 % of E2M1 codes identical (accumulation order
    may move a value across a rounding boundary); in samples too small for
    0.1 % to be a whole value, one value may differ.  The same rule for the
    FC2-input block scales (E4M3 / E8M0 bytes, read back through the
    atom layout).  Per-token G2 of every checked route within a relative
    2^-12 of the oracle's: G2 = amax/2688 of a row whose values differ from
    the oracle's only by the FP32 accumulation and the approximate
    exponential / division of the activation (a few 1e-7 relative at the
    row maximum), so only a wrong row, a wrong formula or a wrong placement
    can exceed it.  W4A16 (BF16 FC2 input):
    >= 99.9 % identical and every value within one BF16 ulp of the oracle's
    plus 1e-5 of its row's largest magnitude (values that cancel to ~1e-8 of
    their row carry the FP32 accumulation error of the whole row).
  * y: |y - y_ref| <= 2e-2 * rms(y_ref) + ulp_bf16(y_ref)/2 + slack_t per
    element, y_ref the oracle's FP64 output.  The half ulp is the rounding
    of the BF16 output itself (for outliers beyond ~8x the RMS it alone
    exceeds 2e-2 * rms).  slack_t is zero unless a route of token t has an
    FC2 input that differs from the oracle's within the identity rules
    above (a code or scale moved across a rounding boundary, or a per-token
    G2 a few ulp away); then it is the exact worst-case effect of that
    difference on the output:
        sum_k w'_k * Gw2 * sum_j |a_gpu_j*G2_gpu - a_ref_j*G2_ref| * max_n |W2q[n,j]|
    with W2q the oracle's dequantized FC2 weight of the route's expert.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

import oracle
from nvfp4_mixture_experts_router_gb300 import api, synth

Y_TOL = 2e-2
CODE_MATCH = 0.999
G2_REL_TOL = 2.0 ** -12


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def sf_rowmajor(buf: np.ndarray, rows: Sequence[int], cols: int) -> np.ndarray:
    """Scales of the given rows, row-major [len(rows), cols/16], read from a
    buffer in the 512-byte atom layout [rows/128][cols/64][512]."""
    r = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(cols // 16, dtype=np.int64)[None, :]
    off = ((r >> 7) * (cols >> 6) + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3)
    return buf[off]


def sf_rowmajor_mx(buf: np.ndarray, rows: Sequence[int], cols: int) -> np.ndarray:
    """MXFP8 scales (one per 32) of the given rows, row-major [len(rows),
    cols/32], from the atom layout [rows/128][cols/128][512]."""
    r = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(cols // 32, dtype=np.int64)[None, :]
    off = ((r >> 7) * (cols >> 7) + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3)
    return buf[off]


def is_mx(layer) -> bool:
    return (layer.flags & (3 << 2)) == api.MOE_W8A8_MXFP8


def is_per_token(layer) -> bool:
    return (layer.flags & (3 << 2)) == api.MOE_W4A4_PER_TOKEN


def nibbles(codes: np.ndarray) -> np.ndarray:
    return np.stack([codes & 15, codes >> 4], axis=-1).reshape(codes.shape[0], -1)


def canonical_w1_rows(N1: int, I: int, swiglu: bool) -> np.ndarray:
    """prepared row -> checkpoint row of FC1 (inverse of the gate/up interleave)."""
    p = np.arange(N1)
    if not swiglu:
        return p
    tile, within = p // 128, p % 128
    up = within >= 64
    j = tile * 64 + (within % 64)
    return np.where(up, I + j, j)


@dataclass
class Inputs:
    c: synth.MoEConfig
    x: torch.Tensor            # device BF16 [T, H]
    logits: torch.Tensor       # device FP32 [T, E]
    bias: Optional[torch.Tensor]
    w1: torch.Tensor           # device BF16 [E, N1, H]
    w2: torch.Tensor           # device BF16 [E, H, I]
    x_np: np.ndarray
    logits_np: np.ndarray
    bias_np: Optional[np.ndarray]
    w1_np: np.ndarray
    w2_np: np.ndarray


def make_inputs(c: synth.MoEConfig, device="cuda", host_gen: bool = False) -> Inputs:
    """The workload's seeded inputs on `device`.  host_gen: draw them on the
    CPU and copy each tensor to the device once (a handful of copies instead
    of the generator's many small elementwise kernels; the values are the
    same bit for bit)."""
    g = "cpu" if host_gen else device
    x = synth.gen_x(c, g)
    logits = synth.gen_logits(c, g, x)
    bias = synth.gen_bias(c, g)
    w1 = synth.gen_w1(c, g)
    w2 = synth.gen_w2(c, g)
    if host_gen:
        x, logits, w1, w2 = (t.to(device) for t in (x, logits, w1, w2))
        bias = None if bias is None else bias.to(device)
    return Inputs(c, x, logits, bias, w1, w2, bits(x), logits.cpu().numpy(),
                  None if bias is None else bias.cpu().numpy(), bits(w1), bits(w2))


def oracle_layer(c: synth.MoEConfig) -> oracle.Layer:
    return oracle.Layer(c.H, c.I, c.E, c.K, act=c.act, mode=c.mode, router_on_input=c.router_on_input,
                        renorm=c.renorm, four_over_six=c.four_over_six)


def scales_for(inp: Inputs, tokens=None):
    """Per-tensor calibration (oracle): G1 over all of x, G2 over the FC2
    inputs of the given tokens."""
    c = inp.c
    if c.mode != synth.MODE_PER_TENSOR:
        return None, None
    G1 = oracle.tensor_global_scale(oracle.bf16_bits_to_f64(inp.x_np).astype(np.float32))
    G2 = oracle.fc2_input_scale(oracle_layer(c), inp.x_np, inp.logits_np, inp.bias_np,
                                lambda e: (inp.w1_np[e], inp.w2_np[e]), G1, tokens=tokens)
    return np.float32(G1), np.float32(G2)


def run_gpu(inp: Inputs, G1, G2):
    c = inp.c
    layer = api.MoELayer.create(c.T, c.H, c.I, c.E, c.K, c.flags())
    layer.prepare(inp.w1, inp.w2)
    g1 = None if G1 is None else torch.tensor([G1], dtype=torch.float32, device="cuda")
    g2 = None if G2 is None else torch.tensor([G2], dtype=torch.float32, device="cuda")
    y = layer.forward(inp.x, inp.logits, inp.bias, g1, g2)
    torch.cuda.synchronize()
    assert api.moe_nvfp4_last_device_status(layer.workspace) == api.MOE_OK
    return layer, y


def check_routing(layer: api.MoELayer, ref: oracle.Result, w_rel_tol=2e-6):
    """w_rel_tol: relative tolerance of the router weights (scalar, or per
    token [T, 1] when the GPU's logits themselves carry an error)."""
    T, K, E = layer.T, layer.K, layer.E
    ids = layer.view("topk_ids", torch.int32, T * K).cpu().numpy().reshape(T, K)
    w = layer.view("topk_w", torch.float32, T * K).cpu().numpy().reshape(T, K)
    assert np.array_equal(ids, ref.ids), "expert ids differ"
    assert np.all(np.abs(w - ref.w) <= w_rel_tol * ref.w + 1e-7), f"router weights: max err {np.abs(w - ref.w).max()}"
    g = ref.grouping
    assert np.array_equal(layer.view("count", torch.int32, E).cpu().numpy(), g.count)
    assert np.array_equal(layer.view("offsets", torch.int32, E + 1).cpu().numpy(), g.offsets)
    assert np.array_equal(layer.view("padded_offsets", torch.int32, E + 1).cpu().numpy(), g.padded_offsets)
    meta = layer.view("meta", torch.int32, 4).cpu().numpy()
    assert meta[0] == g.rows and meta[1] == g.rows // 128
    ror = layer.view("row_of_route", torch.int32, T * K).cpu().numpy()
    assert np.array_equal(ror, g.row_of_route), "row_of_route differs"
    rrow = layer.view("route_of_row", torch.int32, g.rows).cpu().numpy()
    assert np.array_equal(rrow, g.route_of_row[:g.rows]), "route_of_row differs"
    tiles = layer.view("tile_expert", torch.int32, g.rows // 128).cpu().numpy()
    want = np.repeat(np.arange(E), (g.padded_offsets[1:] - g.padded_offsets[:-1]) // 128)
    assert np.array_equal(tiles, want), "tile -> expert map differs"
    # pairs of consecutive M tiles of one expert: (first << 1) | has_second
    pairs = []
    for e in range(E):
        t0, nt = g.padded_offsets[e] // 128, (g.padded_offsets[e + 1] - g.padded_offsets[e]) // 128
        pairs += [((t0 + i) << 1) | int(i + 1 < nt) for i in range(0, nt, 2)]
    assert meta[2] == len(pairs), "M-tile pair count differs"
    got_pairs = layer.view("tile_pair", torch.int32, max(1, len(pairs))).cpu().numpy()[:len(pairs)]
    assert np.array_equal(got_pairs, np.array(pairs, dtype=np.int32)), "M-tile pair map differs"
    # 64-row halves of the M tiles that hold routes, expert by expert, in order
    halves = []
    for e in range(E):
        for j in range((int(g.count[e]) + 63) // 64):
            halves.append(((int(g.padded_offsets[e]) // 128 + j // 2) << 1) | (j & 1))
    assert meta[3] == len(halves), "occupied-half count differs"
    got_halves = layer.view("tile_half", torch.int32, max(1, len(halves))).cpu().numpy()[:len(halves)]
    assert np.array_equal(got_halves, np.array(halves, dtype=np.int32)), "occupied-half list differs"
    return ror


def check_x_quant(layer: api.MoELayer, ref: oracle.Result, ror: np.ndarray):
    T, K, H = layer.T, layer.K, layer.H
    lay = layer.layout()
    cap = lay["rows_cap"]
    mx = is_mx(layer)
    cb = H if mx else H // 2
    codes = layer.view("xq_codes", torch.uint8, cap * cb).cpu().numpy().reshape(cap, cb)
    sfbuf = layer.view("xq_sf", torch.uint8, cap * H // (32 if mx else 16)).cpu().numpy()
    sf_of = sf_rowmajor_mx if mx else sf_rowmajor
    toks = ref.tokens
    for k in range(K):
        rows = ror.reshape(T, K)[toks, k]
        kept = rows >= 0                      # dropped routes (caller-supplied routing) have no row
        assert np.array_equal(codes[rows[kept]], ref.x_codes[kept]), f"x codes differ (slot {k})"
        assert np.array_equal(sf_of(sfbuf, rows[kept], H), ref.x_sf[kept]), f"x scales differ (slot {k})"
    if is_per_token(layer):
        g1 = layer.view("g1", torch.float32, T).cpu().numpy()[toks]
        assert np.array_equal(g1, ref.G1), "per-token G1 differs"


def assert_mostly_identical(got: np.ndarray, want: np.ndarray, what: str):
    """>= 99.9 % identical; on tiny samples at least one value may differ."""
    n = got.size
    n_diff = int(np.sum(got != want))
    allowed = max(1, int((1.0 - CODE_MATCH) * n))
    assert n_diff <= allowed, f"{what}: {n_diff} of {n} differ (allowed {allowed})"


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def _e2m1_values(n: np.ndarray) -> np.ndarray:
    mag = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    return mag[n & 7] * np.where(n & 8, -1.0, 1.0)


def _e4m3_values(b: np.ndarray) -> np.ndarray:
    e, m = (b >> 3) & 15, b & 7
    return np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * 2.0 ** (e.astype(np.float64) - 7))


class W2Colmax:
    """Per-expert (max_n |W2q[n, j]| over the oracle's dequantized FC2
    weight, Gw2), from an oracle `prepared` cache or computed on demand."""

    def __init__(self, prepared=None, weights=None, mx=False):
        self.prepared, self.weights, self.mx, self.cache = prepared, weights, mx, {}

    def __getitem__(self, e):
        if e not in self.cache:
            if self.prepared is not None and e in self.prepared:
                w2op, gw2 = self.prepared[e][2], self.prepared[e][3]
            else:
                pm = (oracle.prepare_matrix_mx if self.mx else oracle.prepare_matrix)(self.weights(e)[1])
                w2op, gw2 = pm.operand(), float(pm.G)
            self.cache[e] = (np.abs(w2op).max(axis=0), gw2)
        return self.cache[e]


def check_fc2_input(layer: api.MoELayer, ref: oracle.Result, ror: np.ndarray, G2, prepared):
    """FC2-input code identity and the per-token output slack of the routes
    whose FC2 input differs (see module docstring)."""
    n_tok = len(ref.tokens)
    slack = np.zeros(n_tok)
    if not isinstance(prepared, W2Colmax):
        prepared = W2Colmax(prepared)
    if (layer.flags & (3 << 2)) == api.MOE_W4A16:
        return _check_fc2_input_bf16(layer, ref, ror, prepared, slack)
    if is_mx(layer):
        return _check_fc2_input_mx(layer, ref, ror, prepared, slack)
    I, K = layer.I, layer.K
    cap = layer.layout()["rows_cap"]
    codes = layer.view("hq_codes", torch.uint8, cap * I // 2).cpu().numpy().reshape(cap, I // 2)
    sfbuf = layer.view("hq_sf", torch.uint8, cap * I // 16).cpu().numpy()
    per_token = is_per_token(layer)
    g2_gpu = layer.view("g2", torch.float32, cap).cpu().numpy() if per_token else None
    routes = sorted(ref.h_codes)
    rows = ror[routes]
    got = nibbles(codes[rows])
    want = nibbles(np.stack([ref.h_codes[r] for r in routes]))
    frac = float(np.mean(got == want))
    assert_mostly_identical(got, want, "FC2-input codes")
    got_sf = sf_rowmajor(sfbuf, rows, I)
    want_sf = np.stack([ref.h_sf[r] for r in routes])
    assert_mostly_identical(got_sf, want_sf, "FC2-input scales")
    if per_token:
        g2g_all = g2_gpu[rows].astype(np.float64)
        g2r_all = np.array([float(ref.G2[r]) for r in routes])
        rel = np.abs(g2g_all - g2r_all) / g2r_all
        assert np.all(rel <= G2_REL_TOL), (f"per-token G2: {int(np.sum(rel > G2_REL_TOL))} of {len(routes)} "
                                           f"routes beyond 2^-12 relative (worst {float(rel.max()):.3g})")
    pos = {int(t): i for i, t in enumerate(ref.tokens)}
    for i, r in enumerate(routes):
        g2g = float(g2_gpu[rows[i]]) if per_token else float(G2)
        g2r = float(ref.G2[r])
        same = np.array_equal(got[i], want[i]) and np.array_equal(got_sf[i], ref.h_sf[r]) and g2g == g2r
        if same:
            continue
        t, k = divmod(r, K)
        colmax, gw2 = prepared[int(ref.ids[t, k])]
        sg = np.repeat(_e4m3_values(got_sf[i]), 16)
        sr = np.repeat(_e4m3_values(ref.h_sf[r]), 16)
        d = np.abs(_e2m1_values(got[i]) * sg * g2g - _e2m1_values(want[i]) * sr * g2r)
        wk = 1.0 if layer.flags & api.MOE_ROUTER_W_ON_INPUT else float(ref.w[t, k])
        slack[pos[t]] += wk * gw2 * float(np.dot(d, colmax))
    return frac, slack


def _mx_values(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    v = _e4m3_values(codes) * np.where(codes & 0x80, -1.0, 1.0)
    return v * np.exp2(np.repeat(sf.astype(np.float64) - 127, 32, axis=-1))


def _check_fc2_input_mx(layer, ref, ror, prepared, slack):
    """MXFP8: E4M3 codes >= 99.9 % identical; a token whose FC2 input
    differs gets the exact worst-case effect of the difference as slack."""
    I, K = layer.I, layer.K
    cap = layer.layout()["rows_cap"]
    codes = layer.view("hq_codes", torch.uint8, cap * I).cpu().numpy().reshape(cap, I)
    sfbuf = layer.view("hq_sf", torch.uint8, cap * I // 32).cpu().numpy()
    routes = sorted(ref.h_codes)
    rows = ror[routes]
    got = codes[rows]
    want = np.stack([ref.h_codes[r] for r in routes])
    frac = float(np.mean(got == want))
    assert_mostly_identical(got, want, "FC2-input codes")
    got_sf = sf_rowmajor_mx(sfbuf, rows, I)
    assert_mostly_identical(got_sf, np.stack([ref.h_sf[r] for r in routes]), "FC2-input scales")
    pos = {int(t): i for i, t in enumerate(ref.tokens)}
    for i, r in enumerate(routes):
        if np.array_equal(got[i], want[i]) and np.array_equal(got_sf[i], ref.h_sf[r]):
            continue
        t, k = divmod(r, K)
        colmax, gw2 = prepared[int(ref.ids[t, k])]
        d = np.abs(_mx_values(got[i], got_sf[i]) - _mx_values(want[i], ref.h_sf[r]))
        wk = 1.0 if layer.flags & api.MOE_ROUTER_W_ON_INPUT else float(ref.w[t, k])
        slack[pos[t]] += wk * gw2 * float(np.dot(d, colmax))
    return frac, slack


def _check_fc2_input_bf16(layer, ref, ror, prepared, slack):
    """W4A16: the FC2 input is the BF16 rounding of h; the same identity
    rule and slack as for the NVFP4 codes (a value on a BF16 rounding
    boundary may round either way)."""
    I, K = layer.I, layer.K
    cap = layer.layout()["rows_cap"]
    hb = layer.view("h_bf16", torch.bfloat16, cap * I).view(cap, I)
    routes = sorted(ref.h_bf16)
    got = bits(hb[torch.as_tensor(ror[routes], device=hb.device, dtype=torch.long)])
    want = np.stack([ref.h_bf16[r] for r in routes])
    frac = float(np.mean(got == want))
    assert_mostly_identical(got, want, "FC2-input BF16 values")
    gv, wv = oracle.bf16_bits_to_f64(got), oracle.bf16_bits_to_f64(want)
    ulp = ulp_bf16(np.maximum(np.abs(gv), np.abs(wv)))
    rowmax = np.stack([np.abs(ref.h[r]).max() for r in routes])[:, None]
    far = np.abs(gv - wv) > ulp + 1e-5 * rowmax
    assert not far.any(), f"FC2-input BF16 values beyond one ulp + 1e-5 * row max: {int(far.sum())}"
    pos = {int(t): i for i, t in enumerate(ref.tokens)}
    for i, r in enumerate(routes):
        if np.array_equal(got[i], want[i]):
            continue
        t, k = divmod(r, K)
        colmax, gw2 = prepared[int(ref.ids[t, k])]
        d = np.abs(oracle.bf16_bits_to_f64(got[i]) - oracle.bf16_bits_to_f64(want[i]))
        wk = 1.0 if layer.flags & api.MOE_ROUTER_W_ON_INPUT else float(ref.w[t, k])
        slack[pos[t]] += wk * gw2 * float(np.dot(d, colmax))
    return frac, slack


def check_y(y: torch.Tensor, ref: oracle.Result, slack=None) -> float:
    yg = y.float().cpu().numpy()[ref.tokens].astype(np.float64)
    assert np.isfinite(yg).all(), "non-finite output"
    rms = float(np.sqrt(np.mean(ref.y64 ** 2)))
    tol = Y_TOL * rms + 0.5 * ulp_bf16(ref.y64)
    if slack is not None:
        tol = tol + slack[:, None] * (1 + 1e-6)
    err = np.abs(yg - ref.y64)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (f"{len(bad)} outputs out of tolerance; worst err/rms "
                           f"{float(np.max(err / rms)):.4g} at token {ref.tokens[bad[0][0]]}")
    return float(np.max(err) / rms)


def full_parity(c: synth.MoEConfig, tokens=None, host_gen: bool = False):
    inp = make_inputs(c, host_gen=host_gen)
    G1, G2 = scales_for(inp, tokens)
    layer, y = run_gpu(inp, G1, G2)
    prepared = {}
    ref = oracle.forward(oracle_layer(c), inp.x_np, inp.logits_np, inp.bias_np,
                         lambda e: (inp.w1_np[e], inp.w2_np[e]), G1=G1, G2=G2, tokens=tokens, prepared=prepared)
    ror = check_routing(layer, ref)
    if c.mode != synth.MODE_W4A16:
        check_x_quant(layer, ref, ror)
    frac, slack = check_fc2_input(layer, ref, ror, G2, prepared)
    rel = check_y(y, ref, slack)
    return dict(code_match=frac, y_rel_err=rel, layer=layer, y=y, ref=ref, inp=inp,
                flipped_tokens=int(np.sum(slack > 0)))


# ---------------------------------------------------------------------------
# full-size workloads: everything that is cheap for the oracle on all tokens,
# the expert MLPs on a seeded token sample
# ---------------------------------------------------------------------------

def routed_parity(c: synth.MoEConfig, ids: np.ndarray, w: np.ndarray, tokens=None):
    """moe_nvfp4_forward_routed on caller-supplied ids / weights against the
    oracle's forward on the same routing (ids sanitized by its stated rule)."""
    inp = make_inputs(c)
    routing = (ids, w)
    wf = lambda e: (inp.w1_np[e], inp.w2_np[e])
    G1 = G2 = None
    if c.mode == synth.MODE_PER_TENSOR:
        G1 = np.float32(oracle.tensor_global_scale(oracle.bf16_bits_to_f64(inp.x_np).astype(np.float32)))
        G2 = np.float32(oracle.fc2_input_scale(oracle_layer(c), inp.x_np, None, None, wf, G1, tokens=tokens,
                                               routing=routing))
    layer = api.MoELayer.create(c.T, c.H, c.I, c.E, c.K, c.flags())
    layer.prepare(inp.w1, inp.w2)
    g1 = None if G1 is None else torch.tensor([G1], dtype=torch.float32, device="cuda")
    g2 = None if G2 is None else torch.tensor([G2], dtype=torch.float32, device="cuda")
    ids_t = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    w_t = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).cuda()
    y = layer.forward_routed(inp.x, ids_t, w_t, g1, g2)
    torch.cuda.synchronize()
    status = api.moe_nvfp4_last_device_status(layer.workspace)
    prepared = {}
    ref = oracle.forward(oracle_layer(c), inp.x_np, None, None, wf, G1=G1, G2=G2, tokens=tokens,
                         prepared=prepared, routing=routing)
    want_status = api.MOE_ERR_INVALID_ARG if (ref.ids < 0).any() else api.MOE_OK
    assert status == want_status, f"device status {status}, expected {want_status}"
    ror = check_routing(layer, ref)
    if c.mode != synth.MODE_W4A16:
        check_x_quant(layer, ref, ror)
    frac, slack = check_fc2_input(layer, ref, ror, G2, prepared)
    rel = check_y(y, ref, slack)
    return dict(code_match=frac, y_rel_err=rel, layer=layer, y=y, ref=ref, inp=inp)


def random_routing(T: int, E: int, K: int, seed: int, bad_frac: float = 0.0):
    """Distinct ids per token and positive weights; with bad_frac > 0 some
    slots get -1, an id >= E or a repeat of the token's slot 0."""
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    w = rng.uniform(0.05, 1.0, size=(T, K)).astype(np.float32)
    if bad_frac > 0:
        bad = rng.random((T, K)) < bad_frac
        kind = rng.integers(0, 3, size=(T, K))
        for t, k in zip(*np.nonzero(bad)):
            ids[t, k] = [-1, E + int(rng.integers(0, 5)), ids[t, 0] if k > 0 else -7][kind[t, k]]
    return ids, w


def check_x_quant_all(layer: api.MoELayer, x_np: np.ndarray, G1, ror: np.ndarray):
    """NVFP4 codes and scales of x for every token and every one of its K
    permuted rows, bit for bit."""
    T, K, H = layer.T, layer.K, layer.H
    x32 = oracle.bf16_bits_to_f64(x_np).astype(np.float32)
    cap = layer.layout()["rows_cap"]
    if is_mx(layer):
        codes_ref, sf_ref = oracle.quant_rows_mx(x32)
        cb, sf_of, per_sf = H, sf_rowmajor_mx, 32
    else:
        four_six = bool(layer.flags & api.MOE_QUANT_4OVER6)
        div = oracle.SCALE_DIV_4OVER6 if four_six else oracle.SCALE_DIV
        G = oracle.row_global_scale(x32, div) if is_per_token(layer) else np.float32(G1)
        codes_ref, sf_ref = oracle.quant_rows(x32, G, four_six)
        cb, sf_of, per_sf = H // 2, sf_rowmajor, 16
    codes = layer.view("xq_codes", torch.uint8, cap * cb).view(cap, cb)
    sfbuf = layer.view("xq_sf", torch.uint8, cap * H // per_sf).cpu().numpy()
    rr = ror.reshape(T, K)
    for k in range(K):
        rows = rr[:, k]
        got = codes[torch.as_tensor(rows, device=codes.device, dtype=torch.long)].cpu().numpy()
        assert np.array_equal(got, codes_ref), f"x codes differ (slot {k})"
        assert np.array_equal(sf_of(sfbuf, rows, H), sf_ref), f"x scales differ (slot {k})"


def fullsize_parity(c: synth.MoEConfig, n_tokens: int):
    dev = "cuda"
    x = synth.gen_x(c, dev)
    logits = synth.gen_logits(c, dev, x)
    bias = synth.gen_bias(c, dev)
    x_np, logits_np = bits(x), logits.cpu().numpy()
    bias_np = None if bias is None else bias.cpu().numpy()
    layer = api.MoELayer.create(c.T, c.H, c.I, c.E, c.K, c.flags())
    w1 = synth.gen_w1(c, dev)
    w2 = synth.gen_w2(c, dev)
    layer.prepare(w1, w2)
    torch.cuda.synchronize()
    del w1, w2

    def weights(e):
        return (bits(synth.gen_w1_expert(c, e, dev)), bits(synth.gen_w2_expert(c, e, dev)))

    tokens = synth.sample_tokens(c, n_tokens)
    L = oracle_layer(c)
    G1 = G2 = None
    if c.mode == synth.MODE_PER_TENSOR:
        G1 = np.float32(oracle.tensor_global_scale(oracle.bf16_bits_to_f64(x_np).astype(np.float32)))
        G2 = np.float32(oracle.fc2_input_scale(L, x_np, logits_np, bias_np, weights, G1, tokens=tokens))
    g1 = None if G1 is None else torch.tensor([G1], device=dev)
    g2 = None if G2 is None else torch.tensor([G2], device=dev)
    y = layer.forward(x, logits, bias, g1, g2)
    torch.cuda.synchronize()
    assert api.moe_nvfp4_last_device_status(layer.workspace) == api.MOE_OK
    ref = oracle.forward(L, x_np, logits_np, bias_np, weights, G1=G1, G2=G2, tokens=tokens)
    ror = check_routing(layer, ref)
    if c.mode != synth.MODE_W4A16:
        check_x_quant_all(layer, x_np, G1, ror)
    frac, slack = check_fc2_input(layer, ref, ror, G2, W2Colmax(None, weights, mx=is_mx(layer)))
    rel = check_y(y, ref, slack)
    return dict(code_match=frac, y_rel_err=rel, flipped_tokens=int(np.sum(slack > 0)))
