"""CPU oracle for the NVFP4 MoE layer forward — TEST INFRASTRUCTURE ONLY.

Loaded only by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py``.  The arithmetic lives in ``moe_oracle.cpp`` (plain C++,
FP64 accumulation, bit-exact NVFP4 emulation); this module builds it with
gcc, loads it with ctypes and composes its steps into the layer forward:

    router -> grouping -> NVFP4 x -> FC1 + activation (+ input-side weight)
           -> FC2-input quantization -> FC2 -> finalize

Readings of points the pages leave open are listed in ``moe_oracle.cpp``
beside the step they concern.  No value here ever comes from the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import Callable, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ACT_SWIGLU, ACT_RELU2 = 0, 1
MODE_PER_TENSOR, MODE_PER_TOKEN, MODE_W4A16, MODE_MXFP8 = 0, 1, 2, 3
PAD_ROWS = 128          # expert segments are padded to whole 128-row tiles
SCALE_DIV = 2688.0      # 6 (largest E2M1) * 448 (largest E4M3)


def build(force: bool = False) -> str:
    """Compile liboracle.so from moe_oracle.cpp (gcc; no CUDA)."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                               os.path.getmtime(os.path.join(_HERE, "moe_oracle.h"))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
            sig = {
                "orc_f32_to_e4m3": (ctypes.c_uint8, [f32]),
                "orc_e4m3_to_f32": (f32, [ctypes.c_uint8]),
                "orc_f32_to_e2m1": (ctypes.c_uint8, [f32]),
                "orc_e2m1_to_f32": (f32, [ctypes.c_uint8]),
                "orc_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
                "orc_f32_to_bf16": (ctypes.c_uint16, [f32]),
                "orc_bf16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
                "orc_f32_to_e4m3_n": (None, [P, P, i64]),
                "orc_f32_to_e2m1_n": (None, [P, P, i64]),
                "orc_f64_to_bf16_n": (None, [P, P, i64]),
                "orc_f32_to_bf16_n": (None, [P, P, i64]),
                "orc_row_global_scale": (f32, [P, i64]),
                "orc_quant_rows": (None, [P, i64, i64, P, P, P]),
                "orc_quant_rows_4over6": (None, [P, i64, i64, P, P, P]),
                "orc_mx_block_exp": (i32, [f32]),
                "orc_quant_rows_mx": (None, [P, i64, i64, P, P]),
                "orc_dequant_rows_mx": (None, [P, P, i64, i64, P]),
                "orc_prepare_matrix_mx": (None, [P, i64, i64, P, P]),
                "orc_row_global_scale_div": (f32, [P, i64, f32]),
                "orc_dequant_rows": (None, [P, P, i64, i64, P]),
                "orc_router": (None, [i64, i32, i32, P, P, i32, P, P]),
                "orc_group": (i64, [i64, i32, i32, P, i32, P, P, P, P, P, i64]),
                "orc_prepare_matrix": (f32, [P, i64, i64, P, P]),
                "orc_fc1": (None, [P, P, i64, i64, P, i64, i32, P, P]),
                "orc_fc2": (None, [P, P, i64, i64, P, i64, P]),
                "orc_finalize": (None, [i64, i32, i64, P, P, P, P]),
                "orc_set_threads": (None, [i32]),
                "orc_max_threads": (i32, []),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def set_threads(n: int) -> None:
    """Host threads of the C steps' parallel loops (n < 1: the default).
    For timing only: the results do not depend on it."""
    lib().orc_set_threads(int(n))


def max_threads() -> int:
    return int(lib().orc_max_threads())


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def f32_to_e4m3(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().orc_f32_to_e4m3_n(_p(v), _p(out), v.size)
    return out


def f32_to_e2m1(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().orc_f32_to_e2m1_n(_p(v), _p(out), v.size)
    return out


def e4m3_to_f32(b) -> np.ndarray:
    return np.array([lib().orc_e4m3_to_f32(int(x)) for x in np.ravel(b)],
                    dtype=np.float32).reshape(np.shape(b))


def e2m1_to_f32(c) -> np.ndarray:
    return np.array([lib().orc_e2m1_to_f32(int(x)) for x in np.ravel(c)],
                    dtype=np.float32).reshape(np.shape(c))


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) -> exact float64 values."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """FP64 -> BF16 bits, one round-to-nearest-even step."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().orc_f64_to_bf16_n(_p(v), _p(out), v.size)
    return out


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bits, round-to-nearest-even."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16_n(_p(v), _p(out), v.size)
    return out


# ---------------------------------------------------------------------------
# NVFP4 rows
# ---------------------------------------------------------------------------

SCALE_DIV_4OVER6 = 1536.0     # 6 * 256: global scale under 4-over-6 with the 256 E4M3 bound


def row_global_scale(x: np.ndarray, div: float = 2688.0) -> np.ndarray:
    """Per-row amax/div (1 if the row is all zero), float32; div = 2688
    (6 * 448) by default, 1536 (6 * 256) for 4-over-6 quantization."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    x2 = x.reshape(-1, x.shape[-1])
    if div == 2688.0:
        return np.array([lib().orc_row_global_scale(_p(np.ascontiguousarray(r)), r.size) for r in x2],
                        dtype=np.float32)
    return np.array([lib().orc_row_global_scale_div(_p(np.ascontiguousarray(r)), r.size, div) for r in x2],
                    dtype=np.float32)


def tensor_global_scale(x: np.ndarray) -> np.float32:
    """amax over the whole tensor / 2688 (per-tensor calibration)."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(1, -1)
    return row_global_scale(x)[0]


def quant_rows(x: np.ndarray, G, four_over_six: bool = False) -> tuple:
    """NVFP4-quantize rows of x (float32 [rows, n]) with per-row global scale
    G (scalar or [rows]); four_over_six picks, per block, the better of the
    max-6 and max-4 scalings.  Returns (codes [rows, n/2] u8, sf [rows, n/16]
    u8)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, n = x.shape
    assert n % 16 == 0
    G = np.ascontiguousarray(np.broadcast_to(np.asarray(G, dtype=np.float32), (rows,)))
    codes = np.empty((rows, n // 2), dtype=np.uint8)
    sf = np.empty((rows, n // 16), dtype=np.uint8)
    fn = lib().orc_quant_rows_4over6 if four_over_six else lib().orc_quant_rows
    fn(_p(x), rows, n, _p(G), _p(codes), _p(sf))
    return codes, sf


def quant_rows_mx(x: np.ndarray) -> tuple:
    """MXFP8-quantize rows of x (float32 [rows, n], n % 32 == 0): E4M3 codes
    [rows, n] and E8M0 scales [rows, n/32]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, n = x.shape
    assert n % 32 == 0
    codes = np.empty((rows, n), dtype=np.uint8)
    sf = np.empty((rows, n // 32), dtype=np.uint8)
    lib().orc_quant_rows_mx(_p(x), rows, n, _p(codes), _p(sf))
    return codes, sf


def dequant_rows_mx(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """e4m3(code) * 2^(sf - 127) as float64 [rows, n]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    rows, n = codes.shape
    out = np.empty((rows, n), np.float64)
    lib().orc_dequant_rows_mx(_p(codes), _p(sf), rows, n, _p(out))
    return out


def mx_block_exp(amax: float) -> int:
    return int(lib().orc_mx_block_exp(float(amax)))


def dequant_rows(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """q*s as float64 [rows, n] (without the global scale)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    rows = codes.shape[0]
    n = codes.shape[1] * 2
    out = np.empty((rows, n), dtype=np.float64)
    lib().orc_dequant_rows(_p(codes), _p(sf), rows, n, _p(out))
    return out


# ---------------------------------------------------------------------------
# router and grouping
# ---------------------------------------------------------------------------

def router_logits(x_bf16: np.ndarray, wg_bf16: np.ndarray) -> np.ndarray:
    """Router logits of the optional first stage, logits = x . W_g^T
    [FlashInfer PR #4366, "Motivation": the MoE wrapper is handed routing
    computed upstream from the gate projection; here that projection is the
    layer's own first step].  Reading: BF16 x [T, H] and W_g [E, H] taken
    exactly, products summed in FP64 (a library matmul), the sum rounded once
    to FP32 (round to nearest even) -- the FP32 logits the router consumes."""
    x = bf16_bits_to_f64(np.ascontiguousarray(x_bf16, dtype=np.uint16))
    w = bf16_bits_to_f64(np.ascontiguousarray(wg_bf16, dtype=np.uint16))
    return (x @ w.T).astype(np.float32)


def router(logits: np.ndarray, bias: Optional[np.ndarray], K: int, renorm: bool = True):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    lib().orc_router(T, E, K, _p(logits), _p(b), int(bool(renorm)), _p(ids), _p(w))
    return ids, w


def rows_capacity(T: int, K: int, E: int) -> int:
    """Upper bound of the padded row total: every expert with at least one
    route may add up to PAD_ROWS-1 pad rows."""
    R = T * K
    cap = R + min(E, R) * (PAD_ROWS - 1)
    return (cap + PAD_ROWS - 1) // PAD_ROWS * PAD_ROWS


@dataclass
class Grouping:
    count: np.ndarray
    offsets: np.ndarray
    padded_offsets: np.ndarray
    row_of_route: np.ndarray    # [T*K] padded row of each route
    route_of_row: np.ndarray    # [rows_cap] route of each row, -1 in pad rows
    rows: int                   # padded row total


def group(ids: np.ndarray, E: int, rows_cap: Optional[int] = None) -> Grouping:
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, K = ids.shape
    cap = rows_capacity(T, K, E) if rows_cap is None else rows_cap
    count = np.empty(E, np.int32)
    off = np.empty(E + 1, np.int32)
    poff = np.empty(E + 1, np.int32)
    ror = np.empty(T * K, np.int32)
    rrow = np.empty(max(cap, 1), np.int32)
    total = lib().orc_group(T, E, K, _p(ids), PAD_ROWS, _p(count), _p(off), _p(poff),
                            _p(ror), _p(rrow), cap)
    if total < 0:
        raise ValueError(f"grouping failed ({total})")
    return Grouping(count, off, poff, ror, rrow[:cap], int(total))


# ---------------------------------------------------------------------------
# weights
# ---------------------------------------------------------------------------

@dataclass
class PreparedMatrix:
    codes: np.ndarray   # [N, Kd/2]
    sf: np.ndarray      # [N, Kd/16] E4M3, row-major
    G: np.float32       # global scale

    def operand(self) -> np.ndarray:
        return dequant_rows(self.codes, self.sf)


@dataclass
class PreparedMatrixMX:
    codes: np.ndarray   # [N, Kd] E4M3
    sf: np.ndarray      # [N, Kd/32] E8M0
    G: np.float32 = np.float32(1.0)

    def operand(self) -> np.ndarray:
        return dequant_rows_mx(self.codes, self.sf)


def prepare_matrix_mx(w_bf16_bits: np.ndarray) -> PreparedMatrixMX:
    w = np.ascontiguousarray(w_bf16_bits, dtype=np.uint16)
    N, Kd = w.shape
    codes = np.empty((N, Kd), np.uint8)
    sf = np.empty((N, Kd // 32), np.uint8)
    lib().orc_prepare_matrix_mx(_p(w), N, Kd, _p(codes), _p(sf))
    return PreparedMatrixMX(codes, sf)


def prepare_matrix(w_bf16_bits: np.ndarray) -> PreparedMatrix:
    w = np.ascontiguousarray(w_bf16_bits, dtype=np.uint16)
    N, Kd = w.shape
    codes = np.empty((N, Kd // 2), np.uint8)
    sf = np.empty((N, Kd // 16), np.uint8)
    G = lib().orc_prepare_matrix(_p(w), N, Kd, _p(codes), _p(sf))
    return PreparedMatrix(codes, sf, np.float32(G))


# ---------------------------------------------------------------------------
# expert MLP steps
# ---------------------------------------------------------------------------

def fc1(a: np.ndarray, alpha: np.ndarray, w1: np.ndarray, I: int, act: int,
        p: Optional[np.ndarray] = None) -> np.ndarray:
    a = np.ascontiguousarray(a, np.float64)
    rows, H = a.shape
    alpha = np.ascontiguousarray(np.broadcast_to(np.asarray(alpha, np.float64), (rows,)))
    w1 = np.ascontiguousarray(w1, np.float64)
    pp = None if p is None else np.ascontiguousarray(p, np.float64)
    h = np.empty((rows, I), np.float64)
    if rows:
        lib().orc_fc1(_p(a), _p(alpha), rows, H, _p(w1), I, act, _p(pp), _p(h))
    return h


def fc2(a: np.ndarray, alpha: np.ndarray, w2: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, np.float64)
    rows, I = a.shape
    H = w2.shape[0]
    alpha = np.ascontiguousarray(np.broadcast_to(np.asarray(alpha, np.float64), (rows,)))
    w2 = np.ascontiguousarray(w2, np.float64)
    o = np.empty((rows, H), np.float64)
    if rows:
        lib().orc_fc2(_p(a), _p(alpha), rows, I, _p(w2), H, _p(o))
    return o


def finalize(o: np.ndarray, o_index: np.ndarray, wk: Optional[np.ndarray], K: int) -> np.ndarray:
    o = np.ascontiguousarray(o, np.float64)
    o_index = np.ascontiguousarray(o_index, np.int64)
    n_tok = o_index.size // K
    H = o.shape[1]
    y = np.empty((n_tok, H), np.float64)
    wkk = None if wk is None else np.ascontiguousarray(wk, np.float64)
    lib().orc_finalize(n_tok, K, H, _p(o_index), _p(wkk), _p(o), _p(y))
    return y


# ---------------------------------------------------------------------------
# the layer forward, composed from the steps above
# ---------------------------------------------------------------------------

@dataclass
class Layer:
    """Shapes and flags of one MoE layer."""
    H: int
    I: int
    E: int
    K: int
    act: int = ACT_SWIGLU
    mode: int = MODE_PER_TENSOR
    router_on_input: bool = False
    renorm: bool = True
    exact: bool = False    # FP64 with no quantization anywhere (pins only)
    four_over_six: bool = False   # per-token W4A4: 4-over-6 activation quantization


@dataclass
class Result:
    ids: np.ndarray            # [T, K]
    w: np.ndarray              # [T, K] float64
    grouping: Grouping
    tokens: np.ndarray         # tokens whose outputs were computed
    G1: np.ndarray             # [n_tok] global scale of each computed token's x
    x_codes: np.ndarray        # [n_tok, H/2]
    x_sf: np.ndarray           # [n_tok, H/16]
    h: dict                    # route -> FP64 FC2-input row before rounding
    h_codes: dict              # route -> codes [I/2]     (W4A4)
    h_sf: dict                 # route -> scales [I/16]   (W4A4)
    G2: dict                   # route -> FC2-input global scale (W4A4)
    h_bf16: dict               # route -> BF16 bits [I]   (W4A16)
    y64: np.ndarray            # [n_tok, H] FP64 sums
    y_bf16: np.ndarray         # [n_tok, H] BF16 bits


WeightFn = Callable[[int], tuple]   # e -> (w1 bf16 bits [N1,H], w2 bf16 bits [H,I])


def prepare_expert(layer: Layer, weights: WeightFn, e: int):
    """Oracle-prepared (canonical) FC1 and FC2 operands of expert e."""
    w1, w2 = weights(e)
    if layer.exact:
        return (bf16_bits_to_f64(w1), 1.0, bf16_bits_to_f64(w2), 1.0)
    prep = prepare_matrix_mx if layer.mode == MODE_MXFP8 else prepare_matrix
    p1 = prep(w1)
    p2 = prep(w2)
    return (p1.operand(), float(p1.G), p2.operand(), float(p2.G))


def sanitize_routes(ids: np.ndarray, E: int) -> np.ndarray:
    """Caller-supplied routing (FlashInfer PR #4366, "Motivation": the
    wrapper takes precomputed top-K ids and weights).  Reading: a slot whose
    id is outside [0, E) or repeats the id of an earlier kept slot of the same
    token is dropped (id -1): it has no row and contributes nothing."""
    ids = np.asarray(ids, dtype=np.int64)
    T, K = ids.shape
    out = np.full((T, K), -1, np.int32)
    for t in range(T):
        kept = set()
        for k in range(K):
            e = int(ids[t, k])
            if 0 <= e < E and e not in kept:
                kept.add(e)
                out[t, k] = e
    return out


def forward(layer: Layer, x_bf16: np.ndarray, logits: Optional[np.ndarray], bias: Optional[np.ndarray],
            weights: WeightFn, G1: Optional[float] = None, G2: Optional[float] = None,
            tokens: Optional[Sequence[int]] = None, x_rows: Optional[np.ndarray] = None,
            prepared: Optional[dict] = None, routing=None) -> Result:
    """Layer forward.

    x_bf16   BF16 bits [T, H] (or None when ``x_rows`` gives the rows of
             ``tokens`` only)
    logits   float32 [T, E]; bias float32 [E] or None (unused with ``routing``)
    weights  e -> (w1 bits [N1, H], w2 bits [H, I]) in checkpoint order
    G1, G2   per-tensor global scales (per-tensor W4A4 only)
    tokens   compute outputs for these tokens only (routing and grouping are
             always computed for all T)
    prepared optional cache dict e -> prepare_expert(...) result
    routing  optional caller-supplied (ids int [T, K], weights float32
             [T, K]) in place of the router: ids sanitized by
             sanitize_routes, weights used as given
    """
    L = layer
    if routing is None:
        T, E = logits.shape
        assert E == L.E
        ids, w = router(logits, bias, L.K, L.renorm)
    else:
        E = L.E
        ids = sanitize_routes(routing[0], E)
        w = np.asarray(routing[1], dtype=np.float32).astype(np.float64)
        T = ids.shape[0]
        assert ids.shape == (T, L.K) and w.shape == (T, L.K)
    grp = group(ids, E)
    toks = np.arange(T) if tokens is None else np.asarray(sorted(set(int(t) for t in tokens)))
    n_tok = len(toks)
    if x_rows is None:
        x_rows = np.ascontiguousarray(x_bf16[toks])
    xv = bf16_bits_to_f64(x_rows)               # exact BF16 values
    x32 = xv.astype(np.float32)

    # activation operand of FC1 and its accumulator factor
    if L.exact or L.mode == MODE_W4A16:
        G1_tok = np.ones(n_tok, np.float32)
        x_codes = np.zeros((n_tok, L.H // 2), np.uint8)
        x_sf = np.zeros((n_tok, L.H // 16), np.uint8)
        a_tok = xv
    elif L.mode == MODE_MXFP8:
        G1_tok = np.ones(n_tok, np.float32)          # no global scale
        x_codes, x_sf = quant_rows_mx(x32)
        a_tok = dequant_rows_mx(x_codes, x_sf)
    else:
        if L.mode == MODE_PER_TENSOR:
            assert G1 is not None, "per-tensor mode needs the FC1 activation scale"
            G1_tok = np.full(n_tok, np.float32(G1), np.float32)
        else:
            G1_tok = row_global_scale(x32, SCALE_DIV_4OVER6 if L.four_over_six else SCALE_DIV)
        x_codes, x_sf = quant_rows(x32, G1_tok, L.four_over_six)
        a_tok = dequant_rows(x_codes, x_sf)

    # routes of the selected tokens, grouped by expert
    tok_pos = {int(t): i for i, t in enumerate(toks)}
    by_expert: dict = {}
    for t in toks:
        for k in range(L.K):
            if ids[t, k] >= 0:
                by_expert.setdefault(int(ids[t, k]), []).append((int(t), k))

    o_rows = np.zeros((n_tok * L.K, L.H), np.float64)
    h_out, hc_out, hs_out, g2_out, hb_out = {}, {}, {}, {}, {}
    for e in sorted(by_expert):
        routes = by_expert[e]
        if prepared is not None and e in prepared:
            w1op, gw1, w2op, gw2 = prepared[e]
        else:
            w1op, gw1, w2op, gw2 = prepare_expert(L, weights, e)
            if prepared is not None:
                prepared[e] = (w1op, gw1, w2op, gw2)
        rows = np.array([tok_pos[t] for t, _ in routes])
        a = a_tok[rows]
        alpha1 = G1_tok[rows].astype(np.float64) * gw1
        p = np.array([w[t, k] for t, k in routes]) if L.router_on_input else None
        h = fc1(a, alpha1, w1op, L.I, L.act, p)
        # FC2 input: quantization boundary (W4A4) or BF16 store (W4A16)
        if L.exact:
            a2 = h
            alpha2 = np.ones(len(routes))
        elif L.mode == MODE_W4A16:
            hb = f32_to_bf16_bits(h.astype(np.float32))
            a2 = bf16_bits_to_f64(hb)
            alpha2 = np.full(len(routes), gw2)
        elif L.mode == MODE_MXFP8:
            g2 = np.ones(len(routes), np.float32)
            hc, hs = quant_rows_mx(h.astype(np.float32))
            a2 = dequant_rows_mx(hc, hs)
            alpha2 = np.ones(len(routes))
        else:
            h32 = h.astype(np.float32)
            if L.mode == MODE_PER_TENSOR:
                assert G2 is not None, "per-tensor mode needs the FC2 activation scale"
                g2 = np.full(len(routes), np.float32(G2), np.float32)
            else:
                g2 = row_global_scale(h32, SCALE_DIV_4OVER6 if L.four_over_six else SCALE_DIV)
            hc, hs = quant_rows(h32, g2, L.four_over_six)
            a2 = dequant_rows(hc, hs)
            alpha2 = g2.astype(np.float64) * gw2
        o = fc2(a2, alpha2, w2op)
        for i, (t, k) in enumerate(routes):
            r = t * L.K + k
            o_rows[tok_pos[t] * L.K + k] = o[i]
            h_out[r] = h[i]
            if not L.exact and L.mode != MODE_W4A16:
                hc_out[r], hs_out[r], g2_out[r] = hc[i], hs[i], g2[i]
            if not L.exact and L.mode == MODE_W4A16:
                hb_out[r] = hb[i]

    o_index = np.arange(n_tok * L.K, dtype=np.int64)
    wk = None if L.router_on_input else np.ascontiguousarray(w[toks].reshape(-1))
    y64 = finalize(o_rows, o_index, wk, L.K)
    y_bf16 = np.zeros((n_tok, L.H), np.uint16) if L.exact else f64_to_bf16_bits(y64)
    return Result(ids, w, grp, toks, G1_tok, x_codes, x_sf, h_out, hc_out, hs_out, g2_out,
                  hb_out, y64, y_bf16)


def fc2_input_scale(layer: Layer, x_bf16, logits, bias, weights: WeightFn, G1: float,
                    tokens: Optional[Sequence[int]] = None, prepared=None, routing=None) -> np.float32:
    """Per-tensor FC2-input calibration: amax of the float32 FC2 input over
    the given tokens' routes, divided by 2688."""
    res = forward(layer, x_bf16, logits, bias, weights, G1=G1, G2=1.0, tokens=tokens,
                  prepared=prepared, routing=routing)
    amax = np.float32(0.0)
    for h in res.h.values():
        amax = max(amax, np.float32(np.max(np.abs(h.astype(np.float32)))) if h.size else 0)
    return np.float32(1.0) if amax == 0 else np.float32(amax) / np.float32(SCALE_DIV)
