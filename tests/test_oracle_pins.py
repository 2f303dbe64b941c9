"""Pins for the CPU oracle: checks against things other than the oracle itself.

* number formats: brute-force nearest search over the decode tables (a
  different algorithm from the oracle's bit manipulation), a library routine
  (torch.float8_e4m3fn), hand-derived values in tests/golden/;
* NVFP4 rows: exact round trip of representable blocks, the rounding-error
  bound, a brute-force quantizer built on the nearest-search converters;
* router / grouping: full stable sorts;
* layer: identities the pages state or that follow from the mathematics —
  K = E top-K equals the dense softmax mixture, one expert equals a plain
  gated MLP, input-side and output-side router-weight placement agree in
  exact arithmetic (FlashInfer PR #4366, "Motivation"), input-side ReLU2
  scales p * ReLU(z)^2 and not p^2 * ReLU(z)^2 (same page, "Existing SM120
  status"), and an independent per-token brute-force forward on tiny shapes.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from nvfp4_mixture_experts_router_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# ---------------------------------------------------------------------------
# independent brute-force converters (nearest value in the decode table,
# exact midpoint comparison, ties to the even code, saturation)
# ---------------------------------------------------------------------------

E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e4m3_table():
    vals = []
    for code in range(0x7F):          # 0x7F is NaN; 0..0x7E finite non-negative
        e, m = code >> 3, code & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


E4M3_MAG = _e4m3_table()


def brute_nearest(v, table, sign_bit):
    """Code of the table entry nearest |v| (ties -> even code), |v| above
    the largest entry saturates; sign from the sign bit of v."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    hi = np.searchsorted(table, a, side="left")            # table[hi] >= a
    hi = np.clip(hi, 0, len(table) - 1)
    lo = np.clip(hi - 1, 0, len(table) - 1)
    exact_hit = table[hi] == a
    # midpoint comparison 2a vs (lo + hi): exact in float64 for these ranges
    two_a = 2.0 * a
    mid = table[lo] + table[hi]
    pick_hi = np.where(two_a > mid, True, np.where(two_a < mid, False, (hi % 2) == 0))
    code = np.where(exact_hit, hi, np.where(pick_hi, hi, lo))
    code = np.where(a >= table[-1], len(table) - 1, code)
    code = np.where(a <= table[0], 0, code)
    neg = np.signbit(v)
    return (code | np.where(neg, sign_bit, 0)).astype(np.uint8)


def float_sweep(chunk=1 << 21):
    """float32 patterns in chunks: every sign/exponent, top 15 mantissa bits
    exhaustive, low 8 bits in {0x00, 0x01, 0xFF} (exact midpoints have few
    significant bits and sit at low bits 0; their one-ulp neighbours at
    0x01 / 0xFF)."""
    for start in range(0, 1 << 24, chunk):
        hi = np.arange(start, start + chunk, dtype=np.uint32) << 8
        pats = np.concatenate([hi, hi | 0x01, hi | 0xFF])
        f = pats.view(np.float32)
        yield f[np.isfinite(f)]


def test_e2m1_matches_bruteforce_sweep():
    for f in float_sweep():
        got = oracle.f32_to_e2m1(f)
        want = brute_nearest(f, E2M1_MAG, 8)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (f[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_e4m3_matches_bruteforce_sweep():
    for f in float_sweep():
        got = oracle.f32_to_e4m3(f)
        want = brute_nearest(f, E4M3_MAG, 0x80)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (f[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_e4m3_matches_torch_float8_in_range():
    for f in float_sweep():
        f = f[np.abs(f) < 464.0]          # torch's cast does not saturate
        got = oracle.f32_to_e4m3(f)
        want = torch.from_numpy(f).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (f[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_decode_tables():
    assert np.array_equal(oracle.e2m1_to_f32(np.arange(8)), E2M1_MAG.astype(np.float32))
    assert np.array_equal(oracle.e2m1_to_f32(np.arange(8, 16)), -E2M1_MAG.astype(np.float32))
    dec = oracle.e4m3_to_f32(np.arange(0x7F))
    assert np.array_equal(dec.astype(np.float64), E4M3_MAG)
    lib_dec = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    ours = oracle.e4m3_to_f32(np.arange(256))
    same = (lib_dec == ours) | (np.isnan(lib_dec) & np.isnan(ours))
    assert same.all()


def test_bf16_conversions():
    for f in float_sweep():
        got = oracle.f32_to_bf16_bits(f)
        want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, want)
    # FP64 -> BF16 with a single rounding: nearest of the two bracketing
    # BF16 values, exact midpoint test, ties to the even pattern
    rng = np.random.default_rng(7)
    v = rng.standard_normal(200000) * np.exp2(rng.integers(-130, 120, 200000))
    v = np.concatenate([v, [1 + 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -40, 1 + 3 * 2.0 ** -8,
                            -(1 + 2.0 ** -8), 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135]])
    got = oracle.f64_to_bf16_bits(v)
    a = np.abs(v)
    lo_bits = (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint32)
    # fix float32 rounding up past a: step down until lo <= a
    lo_val = (lo_bits << 16).view(np.float32).astype(np.float64)
    lo_bits = np.where(lo_val > a, lo_bits - 1, lo_bits)
    lo_val = (lo_bits << 16).view(np.float32).astype(np.float64)
    hi_bits = lo_bits + 1
    hi_val = (hi_bits << 16).view(np.float32).astype(np.float64)
    two_a, mid = 2 * a, lo_val + hi_val
    pick = np.where(lo_val == a, lo_bits,
                    np.where(two_a < mid, lo_bits,
                             np.where(two_a > mid, hi_bits,
                                      np.where(lo_bits % 2 == 0, lo_bits, hi_bits))))
    want = (pick | np.where(np.signbit(v), 0x8000, 0)).astype(np.uint16)
    assert np.array_equal(got, want)


def test_golden_format_values():
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_formats.json")))
    for val, code in g["e2m1_encode"]:
        assert int(oracle.f32_to_e2m1(np.array([val], np.float32))[0]) == code, val
    for val, code in g["e4m3_encode"]:
        assert int(oracle.f32_to_e4m3(np.array([val], np.float32))[0]) == code, val
    for case in g["blocks"]:
        x = np.array(case["x"], np.float32)[None]
        codes, sf = oracle.quant_rows(x, np.float32(case["G"]))
        assert sf.tolist()[0] == case["sf"], case["name"]
        assert codes.tolist()[0] == case["codes"], case["name"]
    for case in g["row_scale"]:
        got = oracle.row_global_scale(np.array(case["x"], np.float32)[None])[0]
        assert got == np.float32(case["G"]), case


# ---------------------------------------------------------------------------
# NVFP4 rows
# ---------------------------------------------------------------------------

def brute_quant_rows(x, G, M=6.0):
    """Row quantization spelled out with numpy float32 steps and the
    brute-force converters above; M = the E2M1 value the block maximum maps
    to (6, or 4 for the 4-over-6 alternative)."""
    x = x.astype(np.float32)
    rows, n = x.shape
    G = np.broadcast_to(np.asarray(G, np.float32), (rows,)).astype(np.float32)
    xb = x.reshape(rows, n // 16, 16)
    amax = np.abs(xb).max(axis=2)
    t = (amax / G[:, None]).astype(np.float32)
    s = brute_nearest((t / np.float32(M)).astype(np.float32), E4M3_MAG, 0x80)
    sv = E4M3_MAG[s & 0x7F].astype(np.float32)
    den = (sv * G[:, None]).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(sv == 0, np.float32(0), (np.float32(1.0) / den)).astype(np.float32)
    scaled = (xb * inv[:, :, None]).astype(np.float32)
    q = brute_nearest(scaled, E2M1_MAG, 8).reshape(rows, n)
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return codes, s.astype(np.uint8)


@pytest.mark.parametrize("scale_kind", ["tensor", "token"])
def test_quant_rows_matches_bruteforce(scale_kind):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((64, 512)) * np.exp2(rng.integers(-8, 8, (64, 1)))).astype(np.float32)
    x[3, :16] = 0.0                                      # zero block
    x[5, 16:32] = -0.0                                   # negative zeros
    x[7, 40] = 1e6                                       # one huge element
    if scale_kind == "tensor":
        G = oracle.tensor_global_scale(x)
    else:
        G = oracle.row_global_scale(x)
    c1, s1 = oracle.quant_rows(x, G)
    c2, s2 = brute_quant_rows(x, G)
    assert np.array_equal(s1, s2)
    assert np.array_equal(c1, c2)


def test_quant_roundtrip_exact_blocks():
    """Blocks made of exact NVFP4 values q*s*G with max |q| = 6 quantize to
    themselves (scale and every code recovered)."""
    rng = np.random.default_rng(5)
    rows, n = 32, 256
    for G in [np.float32(1.0), np.float32(0.375), np.float32(2.0 ** -12 * 1.5), np.float32(96.0)]:
        s_codes = rng.integers(8, 0x7F, (rows, n // 16)).astype(np.uint8)      # normal scales
        q = rng.integers(0, 16, (rows, n)).astype(np.uint8)
        q[:, ::16] = np.where(rng.random((rows, n // 16)) < 0.5, 7, 15)        # one |q| = 6 per block
        vals = E2M1_MAG[q & 7] * np.where(q & 8, -1, 1)
        x = (vals * E4M3_MAG[np.repeat(s_codes, 16, axis=1)] * np.float64(G)).astype(np.float32)
        assert np.array_equal(x.astype(np.float64), vals * E4M3_MAG[np.repeat(s_codes, 16, axis=1)] * float(G))
        codes, sf = oracle.quant_rows(x, G)
        assert np.array_equal(sf, s_codes)
        want = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
        # zero codes may carry either sign only if the input was -0: inputs here are +-q*s*G
        assert np.array_equal(codes, want)


def test_quant_error_bound():
    """|x - q s G| <= halfgap(|v|) s G + max(0, |v| - 6) s G, v = x/(s G):
    round-to-nearest on the E2M1 grid plus saturation."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((128, 1024)) * np.exp2(rng.integers(-20, 20, (128, 64)).repeat(16, 1))).astype(np.float32)
    G = oracle.row_global_scale(x)
    codes, sf = oracle.quant_rows(x, G)
    deq = oracle.dequant_rows(codes, sf) * G[:, None].astype(np.float64)
    s = oracle.e4m3_to_f32(sf).astype(np.float64).repeat(16, axis=1) * G[:, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        v = np.where(s > 0, np.abs(x) / s, 0.0)
    halfgap = np.where(v < 2, 0.25, np.where(v < 4, 0.5, 1.0))
    bound = (halfgap * (1 + 1e-6) + np.maximum(0, v - 6)) * s
    # a block whose scale underflowed to 0 (amax/(6G) <= 2^-10) encodes 0
    bound = np.where(s == 0, 6.0 * G[:, None].astype(np.float64) * 2.0 ** -10 * (1 + 1e-6), bound)
    err = np.abs(x.astype(np.float64) - deq)
    assert (err <= bound).all()
    assert (np.sign(deq) * np.sign(x) >= 0).all()


# ---------------------------------------------------------------------------
# MXFP8 rows (E4M3 elements, E8M0 scale per 32)
# ---------------------------------------------------------------------------

def brute_quant_rows_mx(x):
    """OCP MX quantization spelled out: shared exponent from frexp of the
    block amax, elements by the brute-force nearest E4M3 search."""
    x = x.astype(np.float32)
    rows, n = x.shape
    xb = x.reshape(rows, n // 32, 32).astype(np.float64)
    amax = np.abs(xb).max(axis=2)
    _, ex = np.frexp(amax)
    e = np.where(amax > 0, ex - 1 - 8, -127).clip(-127, 127)
    scaled = xb / np.exp2(e)[:, :, None]
    codes = brute_nearest(scaled, E4M3_MAG, 0x80).reshape(rows, n)
    return codes.astype(np.uint8), (e + 127).astype(np.uint8)


def test_mx_quant_matches_bruteforce():
    rng = np.random.default_rng(31)
    x = (rng.standard_normal((64, 512)) * np.exp2(rng.integers(-30, 30, (64, 16)).repeat(32, 1))).astype(np.float32)
    x[2, :32] = 0.0                                   # zero block -> scale 2^-127
    x[4, 32:64] = -0.0
    x[6, 64:96] = np.float32(511.0 * 2.0 ** 10)       # saturates: |v / X| = 511 > 448
    x[8, 96] = np.float32(2.0 ** -140)                # subnormal float32 amax
    c1, s1 = oracle.quant_rows_mx(x)
    c2, s2 = brute_quant_rows_mx(x)
    assert np.array_equal(s1, s2) and np.array_equal(c1, c2)
    assert s1[2, 0] == 0 and (c1[2, :32] == 0).all()
    assert (c1[6, 64:96] == 0x7E).all()               # 448
    assert oracle.mx_block_exp(448.0) == 0 and oracle.mx_block_exp(256.0) == 0 and oracle.mx_block_exp(255.9) == -1


def test_mx_roundtrip_exact_blocks():
    """Blocks of exact values P * 2^e with max |P| in [256, 448] quantize to
    themselves (scale exponent e and every E4M3 code recovered)."""
    rng = np.random.default_rng(32)
    rows, n = 32, 256
    e = rng.integers(-100, 100, (rows, n // 32))
    P = rng.integers(0, 0x7F, (rows, n)).astype(np.uint8) | ((rng.random((rows, n)) < 0.5).astype(np.uint8) << 7)
    big = rng.integers(0x78, 0x7F, (rows, n // 32)).astype(np.uint8)       # 256 .. 448
    P[:, ::32] = big | (P[:, ::32] & 0x80)
    P[:, 1::32] = np.minimum(P[:, 1::32] & 0x7F, big) | (P[:, 1::32] & 0x80)
    P = np.where((P & 0x7F) > np.repeat(big, 32, axis=1), (P & 0x80) | 0x30, P).astype(np.uint8)
    vals = E4M3_MAG[P & 0x7F] * np.where(P & 0x80, -1.0, 1.0) * np.exp2(np.repeat(e, 32, axis=1))
    x = vals.astype(np.float32)
    assert np.array_equal(x.astype(np.float64), vals)
    codes, sf = oracle.quant_rows_mx(x)
    assert np.array_equal(sf.astype(int) - 127, e)
    assert np.array_equal(codes & 0x7F, P & 0x7F)
    nz = (P & 0x7F) != 0
    assert np.array_equal(codes[nz], P[nz])
    assert np.array_equal(oracle.dequant_rows_mx(codes, sf), vals)


def test_mx_error_bound():
    """|x - q X| <= ulp_E4M3(|x| / X) / 2 * X plus the excess above 448."""
    rng = np.random.default_rng(33)
    x = (rng.standard_normal((64, 1024)) * np.exp2(rng.integers(-20, 20, (64, 32)).repeat(32, 1))).astype(np.float32)
    codes, sf = oracle.quant_rows_mx(x)
    deq = oracle.dequant_rows_mx(codes, sf)
    X = np.exp2(sf.astype(np.float64) - 127).repeat(32, axis=1)
    v = np.abs(x.astype(np.float64)) / X
    k = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
    ulp = np.exp2(k - 3)                                # E4M3: 3 mantissa bits, subnormal step 2^-9
    bound = (ulp / 2 + np.maximum(0, v - 448)) * X
    assert (np.abs(x - deq) <= bound * (1 + 1e-12)).all()
    assert (np.abs(x).reshape(64, 32, 32).max(axis=2) / np.exp2(sf.astype(np.float64) - 127) >= 256).all()


# ---------------------------------------------------------------------------
# 4-over-6 block quantization
# ---------------------------------------------------------------------------

def _exact_blocks(rng, rows, n, top, must, G):
    """Rows of exact NVFP4 values q*s*G (G a power of two, so every product
    is exact): every block holds +-`top` and +-`must` and other grid values
    no larger than `top`."""
    s_codes = rng.integers(16, 0x70, (rows, n // 16)).astype(np.uint8)
    allowed = [c for c in range(8) if E2M1_MAG[c] <= top]
    q = rng.choice(allowed, (rows, n)).astype(np.uint8)
    q[:, 0::16] = int(np.nonzero(E2M1_MAG == top)[0][0])
    q[:, 1::16] = int(np.nonzero(E2M1_MAG == must)[0][0])
    q |= (rng.random((rows, n)) < 0.5).astype(np.uint8) << 3
    vals = E2M1_MAG[q & 7] * np.where(q & 8, -1, 1)
    x64 = vals * E4M3_MAG[np.repeat(s_codes, 16, axis=1)] * float(G)
    x = x64.astype(np.float32)
    assert np.array_equal(x.astype(np.float64), x64)
    return x, q, s_codes


@pytest.mark.parametrize("G", [1.0, 2.0 ** -7, 2.0 ** 5])
def test_4over6_picks_max4_for_exact_max4_blocks(G):
    """Blocks of exact values with max |q| = 4 that contain a 3: the max-4
    candidate reproduces them (zero error) while the max-6 one cannot (3 s
    is off the grid scaled by 6/4), so 4-over-6 returns exactly q and s."""
    rng = np.random.default_rng(21)
    x, q, s_codes = _exact_blocks(rng, 24, 256, 4.0, 3.0, np.float32(G))
    codes, sf = oracle.quant_rows(x, np.float32(G), four_over_six=True)
    assert np.array_equal(sf, s_codes)
    assert np.array_equal(codes, (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8))
    c6, s6 = oracle.quant_rows(x, np.float32(G))
    assert not np.array_equal(oracle.dequant_rows(c6, s6), oracle.dequant_rows(codes, sf))


@pytest.mark.parametrize("G", [1.0, 2.0 ** -9])
def test_4over6_keeps_max6_for_exact_max6_blocks(G):
    """Blocks of exact values with max |q| = 6 that contain a 4 (off the
    grid when scaled by 4/6): the max-6 candidate is exact and is kept."""
    rng = np.random.default_rng(22)
    x, q, s_codes = _exact_blocks(rng, 24, 256, 6.0, 4.0, np.float32(G))
    codes, sf = oracle.quant_rows(x, np.float32(G), four_over_six=True)
    assert np.array_equal(sf, s_codes)
    assert np.array_equal(codes, (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8))


def test_4over6_choice_matches_fp64_error():
    """On random data each block gets the candidate with the smaller squared
    error, computed here in float64 from the brute-force candidates; blocks
    whose two errors are within float32 noise of each other may go either
    way but must then equal one of the two candidates."""
    rng = np.random.default_rng(23)
    x = (rng.standard_normal((96, 512)) * np.exp2(rng.integers(-6, 6, (96, 32)).repeat(16, 1))).astype(np.float32)
    G = oracle.row_global_scale(x, oracle.SCALE_DIV_4OVER6)
    codes, sf = oracle.quant_rows(x, G, four_over_six=True)
    cand = {}
    for M in (6.0, 4.0):
        c, s_ = brute_quant_rows(x, G, M)
        deq = oracle.dequant_rows(c, s_) * G[:, None].astype(np.float64)
        err = ((x.astype(np.float64) - deq) ** 2).reshape(96, 32, 16).sum(axis=2)
        cand[M] = (c.reshape(96, 32, 8), s_.reshape(96, 32), err)
    got_c, got_s = codes.reshape(96, 32, 8), sf.reshape(96, 32)
    is6 = (got_s == cand[6.0][1]) & (got_c == cand[6.0][0]).all(axis=2)
    is4 = (got_s == cand[4.0][1]) & (got_c == cand[4.0][0]).all(axis=2)
    assert (is6 | is4).all()
    e6, e4 = cand[6.0][2], cand[4.0][2]
    clear = np.abs(e4 - e6) > 1e-4 * np.maximum(e4, e6)
    assert (is4[clear & (e4 < e6)]).all() and (is6[clear & (e6 < e4)]).all()
    assert (clear & (e4 < e6)).sum() > 100 and (clear & (e6 < e4)).sum() > 100   # both choices exercised


def test_4over6_global_scale_bound():
    """E4M3_USE_256: G = amax/1536, so the max-4 block scale stays <= 384
    (E4M3 code 0x7C) and never saturates at 448."""
    assert oracle.row_global_scale(np.full((1, 16), 1536.0, np.float32), oracle.SCALE_DIV_4OVER6)[0] == 1.0
    rng = np.random.default_rng(24)
    x = (rng.standard_normal((64, 1024)) * np.exp2(rng.integers(-30, 30, (64, 1)))).astype(np.float32)
    G = oracle.row_global_scale(x, oracle.SCALE_DIV_4OVER6)
    _, s4 = brute_quant_rows(x, G, 4.0)
    assert (s4 & 0x7F).max() == 0x7C


# ---------------------------------------------------------------------------
# router and grouping
# ---------------------------------------------------------------------------

def _f32_nearest(q) -> np.float32:
    """The float32 nearest to the rational q, ties to the even significand
    (exact comparisons of rationals; no intermediate rounding)."""
    from fractions import Fraction
    c = np.float32(float(q))
    cands = [c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(-np.inf))]
    dist = [abs(Fraction(float(v)) - q) for v in cands]
    best = min(dist)
    tied = [v for v, d in zip(cands, dist) if d == best]
    if len(tied) > 1:
        tied = [v for v in tied if (np.array(v, np.float32).view(np.uint32) & 1) == 0]
    return tied[0]


def test_router_logits_exact_rational_bruteforce():
    """x . W_g^T against sums of exact rationals rounded once to float32, on
    random BF16 data (the products and sums carry no rounding at all)."""
    from fractions import Fraction
    rng = np.random.default_rng(5)
    T, E, H = 5, 7, 48
    x = oracle.f64_to_bf16_bits(rng.standard_normal((T, H)))
    wg = oracle.f64_to_bf16_bits(rng.standard_normal((E, H)) / np.sqrt(H))
    got = oracle.router_logits(x, wg)
    assert got.shape == (T, E) and got.dtype == np.float32
    xf = oracle.bf16_bits_to_f64(x)
    wf = oracle.bf16_bits_to_f64(wg)
    for t in range(T):
        for e in range(E):
            q = sum(Fraction(float(xf[t, h])) * Fraction(float(wf[e, h])) for h in range(H))
            assert got[t, e] == _f32_nearest(q), (t, e)


def test_router_logits_closed_forms():
    """Ones times a power of two is H * 2^-k exactly; a row that cancels
    leaves exactly its last product; rows and columns follow x and W_g."""
    H = 64
    one = oracle.f64_to_bf16_bits(np.ones((2, H)))
    wg = oracle.f64_to_bf16_bits(np.stack([np.full(H, 2.0 ** -k) for k in range(3)]))
    got = oracle.router_logits(one, wg)
    np.testing.assert_array_equal(got, np.tile(np.float32([H, H / 2, H / 4]), (2, 1)))
    v = np.zeros(H)
    v[0], v[1], v[2] = 3.0, -3.0, 0.375
    got = oracle.router_logits(oracle.f64_to_bf16_bits(v[None, :]), oracle.f64_to_bf16_bits(np.ones((1, H))))
    assert got[0, 0] == np.float32(0.375)
    rng = np.random.default_rng(6)
    x = oracle.f64_to_bf16_bits(rng.standard_normal((4, H)))
    w = oracle.f64_to_bf16_bits(rng.standard_normal((5, H)))
    base = oracle.router_logits(x, w)
    np.testing.assert_array_equal(oracle.router_logits(x[::-1].copy(), w), base[::-1])
    np.testing.assert_array_equal(oracle.router_logits(x, w[[4, 0, 2, 1, 3]].copy()), base[:, [4, 0, 2, 1, 3]])


@pytest.mark.parametrize("renorm", [True, False])
def test_router_matches_stable_sort(renorm):
    rng = np.random.default_rng(1)
    T, E, K = 200, 37, 5
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[0, :] = 0.5                          # all tied: picks 0..K-1
    logits[1, 10] = logits[1, 3] = 9.0           # tie at the top: 3 before 10
    bias = rng.standard_normal(E).astype(np.float32)
    ids, w = oracle.router(logits, bias, K, renorm)
    l = (logits + bias).astype(np.float32)
    l[0, :] = (np.float32(0.5) + bias)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(l[t, e]), e))[:K]
        assert ids[t].tolist() == order
        p = np.exp(l[t].astype(np.float64) - l[t].max())
        den = p[order].sum() if renorm else p.sum()
        np.testing.assert_allclose(w[t], p[order] / den, rtol=1e-14)
    # bias-free tie case
    ids0, _ = oracle.router(np.full((1, E), 0.5, np.float32), None, K, True)
    assert ids0[0].tolist() == list(range(K))


def test_grouping_is_stable_counting_sort():
    rng = np.random.default_rng(2)
    T, E, K = 300, 16, 3
    allowed = [e for e in range(E) if e != 5]        # expert 5 stays empty
    ids = np.stack([rng.choice(allowed, K, replace=False) for _ in range(T)]).astype(np.int32)
    g = oracle.group(ids, E)
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")       # routes by expert, token order kept
    assert np.array_equal(g.count, np.bincount(flat, minlength=E))
    assert g.count[5] == 0
    assert np.array_equal(g.offsets, np.concatenate([[0], np.cumsum(g.count)]))
    pad = np.ceil(g.count / 128).astype(int) * 128
    assert np.array_equal(g.padded_offsets, np.concatenate([[0], np.cumsum(pad)]))
    rows = []
    for e in range(E):
        rows += list(range(g.padded_offsets[e], g.padded_offsets[e] + g.count[e]))
    assert np.array_equal(g.row_of_route[order], np.array(rows))
    valid = np.zeros(g.route_of_row.size, bool)
    valid[rows] = True
    assert (g.route_of_row[~valid] == -1).all()
    assert np.array_equal(g.route_of_row[g.row_of_route], np.arange(T * K))


# ---------------------------------------------------------------------------
# layer identities (exact mode: FP64, no quantization)
# ---------------------------------------------------------------------------

def _tiny(T=6, H=32, I=16, E=4, K=2, act=0, seed=0, on_input=False, exact=True, mode=0):
    c = synth.MoEConfig("pin", T, H, I, E, K, act=act, mode=mode, router_on_input=on_input,
                        seed=seed, logits="normal", w_std=0.3)
    x = synth.gen_x(c).view(torch.int16).numpy().view(np.uint16)
    logits = synth.gen_logits(c).numpy()
    w1 = synth.gen_w1(c).view(torch.int16).numpy().view(np.uint16)
    w2 = synth.gen_w2(c).view(torch.int16).numpy().view(np.uint16)
    layer = oracle.Layer(H, I, E, K, act=act, mode=mode, router_on_input=on_input, exact=exact)
    return c, layer, x, logits, w1, w2


def _act(z, I, act):
    if act == 0:
        g, u = z[..., :I], z[..., I:]
        return g / (1 + np.exp(-g)) * u
    return np.maximum(z, 0) ** 2


@pytest.mark.parametrize("act", [0, 1])
def test_topk_all_experts_equals_dense_mixture(act):
    c, layer, x, logits, w1, w2 = _tiny(E=5, K=5, act=act)
    res = oracle.forward(layer, x, logits, None, lambda e: (w1[e], w2[e]))
    xv = oracle.bf16_bits_to_f64(x)
    W1 = oracle.bf16_bits_to_f64(w1)
    W2 = oracle.bf16_bits_to_f64(w2)
    p = np.exp(logits.astype(np.float64) - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    y = np.zeros((c.T, c.H))
    for e in range(c.E):
        y += p[:, e:e + 1] * (_act(xv @ W1[e].T, c.I, act) @ W2[e].T)
    np.testing.assert_allclose(res.y64, y, rtol=1e-12, atol=1e-12 * np.abs(y).max())


def test_single_expert_equals_gated_mlp():
    c, layer, x, logits, w1, w2 = _tiny(E=1, K=1, act=0)
    res = oracle.forward(layer, x, logits, None, lambda e: (w1[e], w2[e]))
    xv = oracle.bf16_bits_to_f64(x)
    Wg = oracle.bf16_bits_to_f64(w1[0, :c.I])
    Wu = oracle.bf16_bits_to_f64(w1[0, c.I:])
    Wd = oracle.bf16_bits_to_f64(w2[0])
    g = xv @ Wg.T
    y = ((g * (1 / (1 + np.exp(-g)))) * (xv @ Wu.T)) @ Wd.T
    np.testing.assert_allclose(res.y64, y, rtol=1e-12, atol=1e-13 * np.abs(y).max())
    assert np.all(res.w == 1.0)


@pytest.mark.parametrize("act", [0, 1])
def test_placement_equal_in_exact_arithmetic(act):
    """sum_r p_r W2(a_r) == sum_r W2(p_r a_r) when nothing is rounded
    (FlashInfer PR #4366, "Motivation")."""
    c, lo, x, logits, w1, w2 = _tiny(T=9, E=6, K=3, act=act, on_input=False)
    li = oracle.Layer(lo.H, lo.I, lo.E, lo.K, act=act, router_on_input=True, exact=True)
    wf = lambda e: (w1[e], w2[e])
    yo = oracle.forward(lo, x, logits, None, wf).y64
    yi = oracle.forward(li, x, logits, None, wf).y64
    np.testing.assert_allclose(yi, yo, rtol=1e-12, atol=1e-12 * np.abs(yo).max())


def test_input_side_relu2_is_post_activation():
    """Input-side placement scales the post-activation FC2 input:
    p*ReLU(z)^2, not ReLU(p*z)^2 = p^2*ReLU(z)^2
    (FlashInfer PR #4366, "Existing SM120 status")."""
    c, li, x, logits, w1, w2 = _tiny(T=5, E=4, K=2, act=1, on_input=True)
    res = oracle.forward(li, x, logits, None, lambda e: (w1[e], w2[e]))
    xv = oracle.bf16_bits_to_f64(x)
    W1 = oracle.bf16_bits_to_f64(w1)
    checked = 0
    for t in range(c.T):
        for k in range(c.K):
            e, p = res.ids[t, k], res.w[t, k]
            relu2 = np.maximum(xv[t] @ W1[e].T, 0) ** 2
            h = res.h[t * c.K + k]
            np.testing.assert_allclose(h, p * relu2, rtol=1e-13, atol=1e-300)
            if relu2.max() > 0 and p < 0.999:
                assert not np.allclose(h, p * p * relu2, rtol=1e-6)
                checked += 1
    assert checked > 0


# ---------------------------------------------------------------------------
# quantized layer vs an independent per-token brute-force forward
# ---------------------------------------------------------------------------

def brute_forward(c, x, logits, bias, w1, w2, G1, G2, mode, on_input, act, routing=None):
    T, H, I, E, K = c.T, c.H, c.I, c.E, c.K
    y = np.zeros((T, H))
    xv = oracle.bf16_bits_to_f64(x)
    if routing is None:
        l = logits if bias is None else (logits + bias).astype(np.float32)
    for t in range(T):
        if routing is None:
            order = sorted(range(E), key=lambda e: (-float(l[t, e]), e))[:K]
            p = np.exp(l[t, order].astype(np.float64) - float(l[t, order[0]]))
            p /= p.sum()
        else:
            # caller-supplied: walk the slots, keep in-range ids not seen before
            order, p = [], []
            for k in range(K):
                e = int(routing[0][t, k])
                if 0 <= e < E and e not in order:
                    order.append(e)
                    p.append(float(np.float32(routing[1][t, k])))
        if mode == 2:
            a = xv[t][None]
            g1 = np.float32(1.0)
        elif mode == 3:
            xc, xs = brute_quant_rows_mx(xv[t][None].astype(np.float32))
            a = _dq_mx(xc, xs)
            g1 = np.float32(1.0)
        else:
            g1 = np.float32(G1) if mode == 0 else (np.float32(np.abs(xv[t]).max()) / np.float32(2688.0))
            xc, xs = brute_quant_rows(xv[t][None].astype(np.float32), g1)
            a = _dq(xc, xs)
        for k, e in enumerate(order):
            if mode == 3:
                wq1 = _dq_mx(*brute_quant_rows_mx(oracle.bf16_bits_to_f64(w1[e]).astype(np.float32)))
                wq2 = _dq_mx(*brute_quant_rows_mx(oracle.bf16_bits_to_f64(w2[e]).astype(np.float32)))
                h = _act(a @ wq1.T, I, act)
                if on_input:
                    h = h * p[k]
                hc, hs = brute_quant_rows_mx(h.astype(np.float32))
                o = _dq_mx(hc, hs) @ wq2.T
                y[t] += (1.0 if on_input else p[k]) * o[0]
                continue
            q1c, q1s, gw1 = _bprep(w1[e])
            q2c, q2s, gw2 = _bprep(w2[e])
            if mode == 2:
                z = (a @ _dq(q1c, q1s).T) * np.float64(gw1)
            else:
                z = (a @ _dq(q1c, q1s).T) * (np.float64(g1) * np.float64(gw1))
            h = _act(z, I, act)
            if on_input:
                h = h * p[k]
            if mode == 2:
                hb = torch.from_numpy(h.astype(np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)
                o = (hb @ _dq(q2c, q2s).T) * np.float64(gw2)
            else:
                h32 = h.astype(np.float32)
                g2 = np.float32(G2) if mode == 0 else (np.float32(np.abs(h32).max()) / np.float32(2688.0))
                hc, hs = brute_quant_rows(h32, g2)
                o = (_dq(hc, hs) @ _dq(q2c, q2s).T) * (np.float64(g2) * np.float64(gw2))
            y[t] += (1.0 if on_input else p[k]) * o[0]
    return y


def _dq_mx(codes, sf):
    v = E4M3_MAG[codes & 0x7F] * np.where(codes & 0x80, -1.0, 1.0)
    return v * np.exp2(np.repeat(sf.astype(np.float64) - 127, 32, axis=1))


def _dq(codes, sf):
    q = np.stack([codes & 15, codes >> 4], axis=-1).reshape(codes.shape[0], -1)
    v = E2M1_MAG[q & 7] * np.where(q & 8, -1.0, 1.0)
    return v * E4M3_MAG[np.repeat(sf & 0x7F, 16, axis=1)]


def _bprep(wbits):
    w = oracle.bf16_bits_to_f64(wbits).astype(np.float32)
    G = np.float32(np.abs(w).max()) / np.float32(2688.0)
    c, s = brute_quant_rows(w, G)
    return c, s, G


@pytest.mark.parametrize("mode,on_input,act", [(0, False, 0), (1, True, 0), (1, False, 1),
                                               (2, False, 1), (2, True, 0), (0, True, 1), (3, False, 0),
                                               (3, True, 1)])
def test_tiny_forward_matches_bruteforce(mode, on_input, act):
    c, layer, x, logits, w1, w2 = _tiny(T=4, H=32, I=32 if mode == 3 else 16, E=4, K=2, act=act, exact=False,
                                        mode=mode, on_input=on_input, seed=mode * 7 + act)
    bias = np.array([0.1, -0.2, 0.05, 0.0], np.float32)
    xv = oracle.bf16_bits_to_f64(x).astype(np.float32)
    G1 = np.float32(np.abs(xv).max()) / np.float32(2688.0)
    G2 = np.float32(0.02) / np.float32(2688.0) * np.float32(400.0)
    res = oracle.forward(layer, x, logits, bias, lambda e: (w1[e], w2[e]), G1=G1, G2=G2)
    yb = brute_forward(c, x, logits, bias, w1, w2, G1, G2, mode, on_input, act)
    np.testing.assert_allclose(res.y64, yb, rtol=1e-9, atol=1e-12 * np.abs(yb).max())
    if mode in (0, 1):
        G1v = G1 if mode == 0 else oracle.row_global_scale(xv)
        xc, xs = brute_quant_rows(xv, G1v)
        assert np.array_equal(res.x_codes, xc) and np.array_equal(res.x_sf, xs)
    if mode == 3:
        xc, xs = brute_quant_rows_mx(xv)
        assert np.array_equal(res.x_codes, xc) and np.array_equal(res.x_sf, xs)


def test_sanitize_routes_rule():
    """Caller-supplied routing: per token the kept ids are distinct, in
    range, each in-range id of the input is kept exactly once, at its first
    slot; every other slot is dropped (-1)."""
    rng = np.random.default_rng(11)
    T, E, K = 300, 6, 4
    ids = rng.integers(-3, E + 3, size=(T, K))
    s = oracle.sanitize_routes(ids, E)
    for t in range(T):
        kept = [int(e) for e in s[t] if e >= 0]
        assert len(kept) == len(set(kept))
        assert set(kept) == {int(e) for e in ids[t] if 0 <= e < E}
        for k in range(K):
            first = 0 <= ids[t, k] < E and ids[t, k] not in ids[t, :k]
            assert (s[t, k] == ids[t, k]) if first else (s[t, k] == -1)


@pytest.mark.parametrize("mode,on_input,act", [(0, False, 0), (1, True, 0), (1, False, 1), (2, False, 1)])
def test_routed_forward_matches_bruteforce(mode, on_input, act):
    """Forward on caller-supplied ids and weights (with a repeated, an
    out-of-range and a -1 id) against the per-token brute force."""
    c, layer, x, logits, w1, w2 = _tiny(T=5, H=32, I=16, E=4, K=3, act=act, exact=False, mode=mode,
                                        on_input=on_input, seed=40 + mode * 3 + act)
    rng = np.random.default_rng(mode * 3 + act)
    ids = np.stack([rng.permutation(4)[:3] for _ in range(5)]).astype(np.int32)
    ids[1, 2] = ids[1, 0]
    ids[3, 1] = 7
    ids[4, 0] = -1
    w = rng.uniform(0.05, 1.0, size=(5, 3)).astype(np.float32)
    xv = oracle.bf16_bits_to_f64(x).astype(np.float32)
    G1 = np.float32(np.abs(xv).max()) / np.float32(2688.0)
    G2 = np.float32(0.02) / np.float32(2688.0) * np.float32(400.0)
    res = oracle.forward(layer, x, None, None, lambda e: (w1[e], w2[e]), G1=G1, G2=G2, routing=(ids, w))
    yb = brute_forward(c, x, None, None, w1, w2, G1, G2, mode, on_input, act, routing=(ids, w))
    np.testing.assert_allclose(res.y64, yb, rtol=1e-9, atol=1e-12 * np.abs(yb).max())
    assert (res.ids == -1).sum() == 3
    flat = res.ids.reshape(-1)
    assert np.array_equal(res.grouping.count, np.bincount(flat[flat >= 0], minlength=4))
    assert (res.grouping.row_of_route[flat < 0] == -1).all()


@pytest.mark.parametrize("on_input", [False, True])
def test_dropped_route_equals_zero_weight_route(on_input):
    """A dropped route contributes exactly what a route of weight 0 does."""
    c, layer, x, logits, w1, w2 = _tiny(T=6, E=5, K=2, exact=False, mode=1, on_input=on_input, seed=9)
    wf = lambda e: (w1[e], w2[e])
    ids = np.array([[0, 1], [2, 3], [4, 0], [1, 2], [3, 4], [0, 2]], np.int32)
    w = np.full((6, 2), 0.5, np.float32)
    drop = ids.copy()
    drop[[1, 4], 1] = drop[[1, 4], 0]
    zw = w.copy()
    zw[[1, 4], 1] = 0.0
    a = oracle.forward(layer, x, None, None, wf, routing=(drop, w))
    b = oracle.forward(layer, x, None, None, wf, routing=(ids, zw))
    assert np.array_equal(a.y64, b.y64)
    assert np.array_equal(a.y_bf16, b.y_bf16)


def test_subset_forward_equals_full_forward():
    """Computing only some tokens gives those tokens' full-forward rows."""
    c, layer, x, logits, w1, w2 = _tiny(T=12, E=5, K=2, exact=False, mode=1)
    wf = lambda e: (w1[e], w2[e])
    full = oracle.forward(layer, x, logits, None, wf)
    sub = oracle.forward(layer, x, logits, None, wf, tokens=[0, 5, 11])
    assert np.array_equal(sub.y_bf16, full.y_bf16[[0, 5, 11]])
    assert np.array_equal(sub.y64, full.y64[[0, 5, 11]])


def test_thread_count_does_not_change_results():
    """The single-thread timing of the oracle computes what the all-core
    one does: every parallel loop writes disjoint outputs in a fixed order."""
    c, layer, x, logits, w1, w2 = _tiny(T=40, E=6, K=3, exact=False, mode=1)
    wf = lambda e: (w1[e], w2[e])
    full = oracle.forward(layer, x, logits, None, wf)
    try:
        oracle.set_threads(1)
        assert oracle.max_threads() == 1
        one = oracle.forward(layer, x, logits, None, wf)
    finally:
        oracle.set_threads(0)
    assert np.array_equal(one.y_bf16, full.y_bf16)
    assert np.array_equal(one.y64, full.y64)
