"""Python binding of libmoe_nvfp4.so (ctypes).  Argument marshalling only:
every step of the layer runs in the library's CUDA kernels.  PyTorch
supplies device memory and streams.

The functions carry the C names (moe_nvfp4_*); ``MoELayer`` bundles the
buffers of one layer for convenience.  There is no CPU fallback: loading
fails loudly if the library is missing or the device is not sm_103a.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_nvfp4.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT = range(6)
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
                4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT"}

MOE_ACT_SWIGLU = 0
MOE_ACT_RELU2 = 1
MOE_W4A4_PER_TENSOR = 0 << 2
MOE_W4A4_PER_TOKEN = 1 << 2
MOE_W4A16 = 2 << 2
MOE_ROUTER_W_ON_INPUT = 1 << 4
MOE_FINALIZE_DETERMINISTIC = 1 << 5
MOE_ROUTE_NO_RENORM = 1 << 6
MOE_GEMM_PAIRS_NEVER = 1 << 7
MOE_GEMM_PAIRS_ALWAYS = 1 << 8
MOE_QUANT_4OVER6 = 1 << 9
MOE_FUSED_LAYER = 1 << 10
MOE_GEMM_SWAP_NEVER = 1 << 11
MOE_GEMM_SWAP_ALWAYS = 1 << 12
MOE_DEBUG_FC1_SKIP_STAGE = 1 << 13
MOE_ROUTER_GEMM = 1 << 14
MOE_W8A8_MXFP8 = 3 << 2


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(code, code)}")
        self.code = code


class moe_shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int),
                ("K", ctypes.c_int)]


_LAYOUT_FIELDS = ["rows_cap", "status", "topk_ids", "topk_w", "count", "offsets", "padded_offsets", "meta",
                  "unit_base", "unit_mask", "row_of_route", "route_of_row", "tile_expert", "tile_pair", "tile_half", "g1",
                  "xq_codes", "xq_sf", "h_f32", "g2", "hq_codes", "hq_sf", "x_bf16_perm", "h_bf16", "o_bf16",
                  "y_acc", "logits", "total"]


class moe_workspace_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in _LAYOUT_FIELDS]


_lib = None


def lib():
    """Load libmoe_nvfp4.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m nvfp4_mixture_experts_router_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        P, S = ctypes.c_void_p, moe_shape
        u32, i64, sz = ctypes.c_uint32, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "moe_nvfp4_version": (ctypes.c_char_p, []),
            "moe_nvfp4_prepared_bytes": (sz, [S, u32]),
            "moe_nvfp4_prepare_weights": (ctypes.c_int, [S, u32, P, P, P, sz, P]),
            "moe_nvfp4_workspace_bytes": (sz, [S, u32]),
            "moe_nvfp4_workspace_layout": (ctypes.c_int, [S, u32, ctypes.POINTER(moe_workspace_layout)]),
            "moe_nvfp4_forward": (ctypes.c_int, [S, u32, P, P, P, P, P, P, P, sz, P, P]),
            "moe_nvfp4_forward_routed": (ctypes.c_int, [S, u32, P, P, P, P, P, P, P, sz, P, P]),
            "moe_nvfp4_forward_staged": (ctypes.c_int, [S, u32, P, P, P, P, P, P, P, sz, P, P,
                                                        ctypes.POINTER(ctypes.c_void_p)]),
            "moe_nvfp4_forward_launches": (ctypes.c_int, [S, u32]),
            "moe_nvfp4_last_device_status": (ctypes.c_int, [P, P]),
            "moe_nvfp4_debug_convert": (ctypes.c_int, [P, i64, P, P, P]),
            "moe_nvfp4_route_noalloc": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, u32, P, P,
                                                       P, P, P, P, P, P, P, P]),
            "moe_nvfp4_router_logits": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P]),
            "moe_nvfp4_forward_gate": (ctypes.c_int, [S, u32, P, P, P, P, P, P, P, sz, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


EXPORTED = ["moe_nvfp4_version", "moe_nvfp4_prepared_bytes", "moe_nvfp4_prepare_weights",
            "moe_nvfp4_workspace_bytes", "moe_nvfp4_workspace_layout", "moe_nvfp4_forward",
            "moe_nvfp4_forward_routed",
            "moe_nvfp4_forward_staged", "moe_nvfp4_forward_launches",
            "moe_nvfp4_last_device_status", "moe_nvfp4_debug_convert", "moe_nvfp4_route_noalloc",
            "moe_nvfp4_router_logits", "moe_nvfp4_forward_gate"]
EXPORTED.sort()
NUM_STAGE_EVENTS = 8
STAGES = ["router", "permute", "quantize_x", "fc1", "quantize_h", "fc2", "finalize"]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, code: int):
    if code != MOE_OK:
        raise MoEError(fn, code)


def shape(T: int, H: int, I: int, E: int, K: int) -> moe_shape:
    return moe_shape(T, H, I, E, K)


# ---- C entry points ---------------------------------------------------------

def moe_nvfp4_version() -> str:
    return lib().moe_nvfp4_version().decode()


def moe_nvfp4_prepared_bytes(s: moe_shape, flags: int) -> int:
    return int(lib().moe_nvfp4_prepared_bytes(s, flags))


def moe_nvfp4_workspace_bytes(s: moe_shape, flags: int) -> int:
    return int(lib().moe_nvfp4_workspace_bytes(s, flags))


def moe_nvfp4_workspace_layout(s: moe_shape, flags: int) -> dict:
    out = moe_workspace_layout()
    _check("moe_nvfp4_workspace_layout", lib().moe_nvfp4_workspace_layout(s, flags, ctypes.byref(out)))
    return {n: int(getattr(out, n)) for n in _LAYOUT_FIELDS}


def moe_nvfp4_prepare_weights(s: moe_shape, flags: int, w1_bf16: torch.Tensor, w2_bf16: torch.Tensor,
                              prepared: torch.Tensor, stream=None) -> None:
    code = lib().moe_nvfp4_prepare_weights(s, flags, _ptr(w1_bf16), _ptr(w2_bf16), _ptr(prepared),
                                           prepared.numel() * prepared.element_size(), _stream(stream))
    _check("moe_nvfp4_prepare_weights", code)


def moe_nvfp4_forward(s: moe_shape, flags: int, x_bf16: torch.Tensor, router_logits: torch.Tensor,
                      router_bias: Optional[torch.Tensor], act_scale_fc1: Optional[torch.Tensor],
                      act_scale_fc2: Optional[torch.Tensor], prepared: torch.Tensor, workspace: torch.Tensor,
                      y_bf16: torch.Tensor, stream=None) -> None:
    code = lib().moe_nvfp4_forward(s, flags, _ptr(x_bf16), _ptr(router_logits), _ptr(router_bias),
                                   _ptr(act_scale_fc1), _ptr(act_scale_fc2), _ptr(prepared), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _ptr(y_bf16), _stream(stream))
    _check("moe_nvfp4_forward", code)


def moe_nvfp4_forward_routed(s: moe_shape, flags: int, x_bf16: torch.Tensor, topk_ids: torch.Tensor,
                             topk_weights: torch.Tensor, act_scale_fc1: Optional[torch.Tensor],
                             act_scale_fc2: Optional[torch.Tensor], prepared: torch.Tensor, workspace: torch.Tensor,
                             y_bf16: torch.Tensor, stream=None) -> None:
    """Forward on caller-supplied routing: topk_ids int32 [T, K], topk_weights
    float32 [T, K] (CUDA, contiguous)."""
    if topk_ids.dtype != torch.int32 or topk_weights.dtype != torch.float32:
        raise TypeError("topk_ids must be int32 and topk_weights float32")
    if not (topk_ids.is_contiguous() and topk_weights.is_contiguous()):
        raise ValueError("topk_ids and topk_weights must be contiguous")
    if tuple(topk_ids.shape) != (s.T, s.K) or tuple(topk_weights.shape) != (s.T, s.K):
        raise ValueError(f"routing arrays must be [{s.T}, {s.K}]")
    code = lib().moe_nvfp4_forward_routed(s, flags, _ptr(x_bf16), _ptr(topk_ids), _ptr(topk_weights),
                                          _ptr(act_scale_fc1), _ptr(act_scale_fc2), _ptr(prepared),
                                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _ptr(y_bf16), _stream(stream))
    _check("moe_nvfp4_forward_routed", code)


def moe_nvfp4_router_logits(x_bf16: torch.Tensor, gate_w_bf16: torch.Tensor, logits: torch.Tensor,
                            stream=None) -> None:
    """logits [T, E] float32 = x [T, H] . gate_w [E, H]^T (BF16, CUDA, contiguous)."""
    T, H = x_bf16.shape
    E = gate_w_bf16.shape[0]
    if x_bf16.dtype != torch.bfloat16 or gate_w_bf16.dtype != torch.bfloat16 or logits.dtype != torch.float32:
        raise TypeError("x and gate_w must be bfloat16, logits float32")
    if tuple(gate_w_bf16.shape) != (E, H) or tuple(logits.shape) != (T, E):
        raise ValueError("shapes must be x [T, H], gate_w [E, H], logits [T, E]")
    if not (x_bf16.is_contiguous() and gate_w_bf16.is_contiguous() and logits.is_contiguous()):
        raise ValueError("x, gate_w and logits must be contiguous")
    code = lib().moe_nvfp4_router_logits(T, E, H, _ptr(x_bf16), _ptr(gate_w_bf16), _ptr(logits), _stream(stream))
    _check("moe_nvfp4_router_logits", code)


def moe_nvfp4_forward_gate(s: moe_shape, flags: int, x_bf16: torch.Tensor, gate_w_bf16: torch.Tensor,
                           router_bias: Optional[torch.Tensor], act_scale_fc1: Optional[torch.Tensor],
                           act_scale_fc2: Optional[torch.Tensor], prepared: torch.Tensor, workspace: torch.Tensor,
                           y_bf16: torch.Tensor, stream=None) -> None:
    """Forward from the gate projection: flags must include MOE_ROUTER_GEMM;
    gate_w_bf16 is W_g [E, H] (CUDA, contiguous)."""
    if gate_w_bf16.dtype != torch.bfloat16 or tuple(gate_w_bf16.shape) != (s.E, s.H):
        raise ValueError(f"gate_w must be bfloat16 [{s.E}, {s.H}]")
    code = lib().moe_nvfp4_forward_gate(s, flags, _ptr(x_bf16), _ptr(gate_w_bf16), _ptr(router_bias),
                                        _ptr(act_scale_fc1), _ptr(act_scale_fc2), _ptr(prepared), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _ptr(y_bf16), _stream(stream))
    _check("moe_nvfp4_forward_gate", code)


def moe_nvfp4_forward_staged(s: moe_shape, flags: int, x_bf16, router_logits, router_bias, act_scale_fc1,
                             act_scale_fc2, prepared, workspace, y_bf16, events, stream=None) -> None:
    """Forward that records the torch.cuda.Event objects ``events``
    (NUM_STAGE_EVENTS, timing enabled) at the stage boundaries."""
    for ev in events:
        if not ev.cuda_event:       # torch creates the CUDA event lazily, on its first record
            ev.record(stream)
    arr = (ctypes.c_void_p * NUM_STAGE_EVENTS)(*[ctypes.c_void_p(ev.cuda_event) for ev in events])
    code = lib().moe_nvfp4_forward_staged(s, flags, _ptr(x_bf16), _ptr(router_logits), _ptr(router_bias),
                                          _ptr(act_scale_fc1), _ptr(act_scale_fc2), _ptr(prepared),
                                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _ptr(y_bf16), _stream(stream), arr)
    _check("moe_nvfp4_forward_staged", code)


def moe_nvfp4_forward_launches(s: moe_shape, flags: int) -> int:
    return int(lib().moe_nvfp4_forward_launches(s, flags))


def moe_nvfp4_last_device_status(workspace: torch.Tensor, stream=None) -> int:
    return int(lib().moe_nvfp4_last_device_status(_ptr(workspace), _stream(stream)))


def moe_nvfp4_debug_convert(x: torch.Tensor, stream=None):
    """Device E4M3 and E2M1 codes of the float32 CUDA tensor x."""
    x = x.contiguous()
    e4 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    e2 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check("moe_nvfp4_debug_convert",
           lib().moe_nvfp4_debug_convert(_ptr(x), x.numel(), _ptr(e4), _ptr(e2), _stream(stream)))
    return e4, e2


def moe_nvfp4_route_noalloc(T: int, E: int, K: int, flags: int, router_logits: torch.Tensor,
                            router_bias: Optional[torch.Tensor], out: dict, stream=None) -> None:
    """Routing + permutation into the caller's buffers, with the library's
    fixed device scratch instead of a workspace (for callers that cannot
    allocate device memory).  ``out`` holds int32/float32 CUDA tensors
    topk_ids, topk_w, count, offsets, padded_offsets, row_of_route,
    route_of_row (sizes as in include/moe_nvfp4.h)."""
    code = lib().moe_nvfp4_route_noalloc(T, E, K, flags, _ptr(router_logits), _ptr(router_bias),
                                         _ptr(out["topk_ids"]), _ptr(out["topk_w"]), _ptr(out["count"]),
                                         _ptr(out["offsets"]), _ptr(out["padded_offsets"]),
                                         _ptr(out["row_of_route"]), _ptr(out["route_of_row"]), _stream(stream))
    _check("moe_nvfp4_route_noalloc", code)


# ---- convenience ---------------------------------------------------------------

@dataclass
class MoELayer:
    """Buffers of one MoE layer on one device: prepared weights + workspace."""
    T: int
    H: int
    I: int
    E: int
    K: int
    flags: int
    prepared: torch.Tensor
    workspace: torch.Tensor

    @property
    def shape(self) -> moe_shape:
        return moe_shape(self.T, self.H, self.I, self.E, self.K)

    @classmethod
    def create(cls, T, H, I, E, K, flags, device="cuda") -> "MoELayer":
        s = moe_shape(T, H, I, E, K)
        pb = moe_nvfp4_prepared_bytes(s, flags)
        wb = moe_nvfp4_workspace_bytes(s, flags)
        if pb == 0 or wb == 0:
            raise MoEError("moe_nvfp4_*_bytes", MOE_ERR_INVALID_ARG)
        prepared = torch.empty(pb, dtype=torch.uint8, device=device)
        workspace = torch.empty(wb, dtype=torch.uint8, device=device)
        return cls(T, H, I, E, K, flags, prepared, workspace)

    def prepare(self, w1_bf16: torch.Tensor, w2_bf16: torch.Tensor, stream=None):
        moe_nvfp4_prepare_weights(self.shape, self.flags, w1_bf16, w2_bf16, self.prepared, stream)

    def forward(self, x_bf16, logits, bias=None, g1=None, g2=None, y=None, stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty(self.T, self.H, dtype=torch.bfloat16, device=x_bf16.device)
        moe_nvfp4_forward(self.shape, self.flags, x_bf16, logits, bias, g1, g2, self.prepared, self.workspace,
                          y, stream)
        return y

    def forward_gate(self, x_bf16, gate_w_bf16, bias=None, g1=None, g2=None, y=None, stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty(self.T, self.H, dtype=torch.bfloat16, device=x_bf16.device)
        moe_nvfp4_forward_gate(self.shape, self.flags, x_bf16, gate_w_bf16, bias, g1, g2, self.prepared,
                               self.workspace, y, stream)
        return y

    def forward_routed(self, x_bf16, topk_ids, topk_weights, g1=None, g2=None, y=None, stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty(self.T, self.H, dtype=torch.bfloat16, device=x_bf16.device)
        moe_nvfp4_forward_routed(self.shape, self.flags, x_bf16, topk_ids, topk_weights, g1, g2, self.prepared,
                                 self.workspace, y, stream)
        return y

    # -- views of the intermediates (tests / debugging) --
    def layout(self) -> dict:
        return moe_nvfp4_workspace_layout(self.shape, self.flags)

    def view(self, name: str, dtype: torch.dtype, numel: int) -> torch.Tensor:
        off = self.layout()[name]
        if off == 2 ** 64 - 1:
            raise KeyError(f"workspace region {name} is not used in this mode")
        nbytes = numel * torch.empty((), dtype=dtype).element_size()
        return self.workspace[off:off + nbytes].view(dtype)

    def prepared_regions(self) -> dict:
        """Byte offsets of the prepared-weight regions (same rule as the library)."""
        def up(v):
            return (v + 255) // 256 * 256
        N1 = 2 * self.I if (self.flags & 3) == MOE_ACT_SWIGLU else self.I
        E, H, I = self.E, self.H, self.I
        mx = (self.flags & (3 << 2)) == MOE_W8A8_MXFP8
        cd, sd = (1, 32) if mx else (2, 16)        # MXFP8: a byte per element, a scale per 32
        o = 0
        r = {}
        for name, nbytes in [("gw1", 4 * E), ("gw2", 4 * E), ("w1_codes", E * N1 * H // cd),
                             ("w1_sf", E * N1 * H // sd), ("w2_codes", E * H * I // cd), ("w2_sf", E * H * I // sd)]:
            r[name] = (o, nbytes)
            o = up(o + nbytes)
        r["total"] = (o, 0)
        return r
