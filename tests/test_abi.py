"""C-ABI checks that need no GPU: the library loads, exports every entry
point include/moe_nvfp4.h declares, sizes its buffers consistently and
rejects invalid arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from nvfp4_mixture_experts_router_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_nvfp4.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return api.lib()


def declared_entry_points():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[^;(]*?\b(moe_nvfp4_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_entry_points()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n
    assert sorted(api.EXPORTED) == names


def test_version(L):
    assert "sm_103a" in api.moe_nvfp4_version()


def test_sizes_and_layout_consistent(L):
    s = api.shape(512, 2048, 768, 64, 6)
    for flags in [0, api.MOE_W4A4_PER_TOKEN | api.MOE_ROUTER_W_ON_INPUT, api.MOE_W4A16 | api.MOE_ACT_RELU2,
                  api.MOE_FINALIZE_DETERMINISTIC]:
        wb = api.moe_nvfp4_workspace_bytes(s, flags)
        lay = api.moe_nvfp4_workspace_layout(s, flags)
        assert lay["total"] == wb > 0
        assert lay["status"] == 0 and lay["rows_cap"] % 128 == 0
        used = [v for k, v in lay.items() if k not in ("rows_cap", "total") and v != 2 ** 64 - 1]
        assert all(v % 256 == 0 for v in used) and len(set(used)) == len(used)
        pb = api.moe_nvfp4_prepared_bytes(s, flags)
        layer = api.MoELayer(512, 2048, 768, 64, 6, flags, None, None)
        assert layer.prepared_regions()["total"][0] == pb
    # rows capacity bound: T*K + min(E, T*K) * 127, rounded to 128
    assert api.moe_nvfp4_workspace_layout(api.shape(1, 256, 128, 8, 2), 0)["rows_cap"] == 256
    assert api.moe_nvfp4_workspace_layout(api.shape(512, 2048, 768, 64, 6), 0)["rows_cap"] == \
        (3072 + 64 * 127 + 127) // 128 * 128


@pytest.mark.parametrize("bad", [
    dict(T=0), dict(H=100), dict(H=64), dict(I=96), dict(E=0), dict(E=2000), dict(K=0), dict(K=9, E=8),
    dict(K=33, E=64)])
def test_invalid_shapes_rejected(L, bad):
    d = dict(T=16, H=256, I=128, E=8, K=2)
    d.update(bad)
    s = api.shape(d["T"], d["H"], d["I"], d["E"], d["K"])
    assert api.moe_nvfp4_workspace_bytes(s, 0) == 0
    assert api.moe_nvfp4_prepared_bytes(s, 0) == 0
    fake = ctypes.c_void_p(1 << 20)
    code = L.moe_nvfp4_forward(s, 0, fake, fake, None, fake, fake, fake, fake, 1 << 40, fake, None)
    assert code == api.MOE_ERR_INVALID_ARG


def test_invalid_arguments_rejected_before_cuda(L):
    s = api.shape(16, 256, 128, 8, 2)
    wb = api.moe_nvfp4_workspace_bytes(s, 0)
    A = ctypes.c_void_p(1 << 20)          # aligned fake pointers: never dereferenced
    B = ctypes.c_void_p(1 << 30)
    Y = ctypes.c_void_p(1 << 34)
    W = ctypes.c_void_p(1 << 36)
    f = L.moe_nvfp4_forward
    # unknown flag bits, bad mode, bad activation
    assert f(s, 1 << 15, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    # the router-GEMM flag belongs to moe_nvfp4_forward_gate only
    assert f(s, api.MOE_ROUTER_GEMM, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert api.moe_nvfp4_workspace_bytes(s, api.MOE_ROUTER_GEMM) >= wb + 16 * 8 * 4   # room for the logits
    # the bounded-wait test hook: launch sequence, W4A4, standard orientation only
    dbg, sn = api.MOE_DEBUG_FC1_SKIP_STAGE, api.MOE_GEMM_SWAP_NEVER
    assert f(s, dbg, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, dbg | sn | api.MOE_FUSED_LAYER, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, dbg | sn | api.MOE_GEMM_PAIRS_ALWAYS, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, dbg | sn | api.MOE_W4A16, A, B, None, None, None, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert api.moe_nvfp4_workspace_bytes(s, dbg | sn) == wb
    # GEMM orientation hints: not both, and the swapped one only for W4A4 / W4A16 on the launch sequence
    sw, sn = api.MOE_GEMM_SWAP_ALWAYS, api.MOE_GEMM_SWAP_NEVER
    assert f(s, sw | sn, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, sw | api.MOE_GEMM_PAIRS_ALWAYS, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, sw | api.MOE_FUSED_LAYER, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, sw | api.MOE_W8A8_MXFP8, A, B, None, None, None, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert api.moe_nvfp4_workspace_bytes(s, sw) == wb and api.moe_nvfp4_workspace_bytes(s, sn | api.MOE_W4A16) > 0
    # the single-kernel layer: NVFP4 activation modes, E <= 256, single-CTA tiles
    fu = api.MOE_FUSED_LAYER
    assert f(s, fu | api.MOE_W4A16, A, B, None, None, None, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, fu | api.MOE_W8A8_MXFP8, A, B, None, None, None, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, fu | api.MOE_GEMM_PAIRS_ALWAYS, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    big = api.shape(16, 256, 128, 257, 2)
    assert api.moe_nvfp4_workspace_bytes(big, fu) == 0 and api.moe_nvfp4_workspace_bytes(big, 0) > 0
    assert api.moe_nvfp4_forward_launches(s, fu) == 1
    assert api.moe_nvfp4_forward_launches(s, fu | api.MOE_W4A4_PER_TOKEN | api.MOE_QUANT_4OVER6) == 1
    # 4-over-6 quantization only with per-token W4A4
    assert f(s, api.MOE_QUANT_4OVER6, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, api.MOE_QUANT_4OVER6 | api.MOE_W4A16, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, 3 << 2, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, 2, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    # caller-supplied routing: ids and weights required, no router options
    fr = L.moe_nvfp4_forward_routed
    assert fr(s, 0, A, None, B, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert fr(s, 0, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert fr(s, api.MOE_ROUTE_NO_RENORM, A, B, B, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert fr(s, 0, A, ctypes.c_void_p((1 << 30) + 2), B, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert fr(s, 0, A, W, B, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG   # ids inside the workspace
    # contradictory GEMM scheduling hints
    both = api.MOE_GEMM_PAIRS_NEVER | api.MOE_GEMM_PAIRS_ALWAYS
    assert f(s, both, A, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    # null pointers
    assert f(s, 0, None, B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, 0, A, B, None, A, A, A, W, wb, None, None) == api.MOE_ERR_INVALID_ARG
    # per-tensor mode needs both activation scales
    assert f(s, 0, A, B, None, None, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, 0, A, B, None, A, None, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    # misaligned
    assert f(s, 0, ctypes.c_void_p((1 << 20) + 8), B, None, A, A, A, W, wb, Y, None) == api.MOE_ERR_INVALID_ARG
    assert f(s, 0, A, B, None, A, A, A, ctypes.c_void_p((1 << 36) + 16), wb, Y, None) == api.MOE_ERR_INVALID_ARG
    # workspace too small
    assert f(s, 0, A, B, None, A, A, A, W, wb - 1, Y, None) == api.MOE_ERR_WORKSPACE
    # output aliasing the workspace
    assert f(s, 0, A, B, None, A, A, A, W, wb, W, None) == api.MOE_ERR_INVALID_ARG
    # prepare: too small a buffer
    pb = api.moe_nvfp4_prepared_bytes(s, 0)
    assert L.moe_nvfp4_prepare_weights(s, 0, A, B, W, pb - 1, None) == api.MOE_ERR_WORKSPACE
    assert L.moe_nvfp4_prepare_weights(s, 0, None, B, W, pb, None) == api.MOE_ERR_INVALID_ARG


def test_valid_call_without_gpu_reports_cuda_error(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    s = api.shape(16, 256, 128, 8, 2)
    wb = api.moe_nvfp4_workspace_bytes(s, api.MOE_W4A4_PER_TOKEN)
    A, W, Y = ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 36), ctypes.c_void_p(1 << 34)
    code = L.moe_nvfp4_forward(s, api.MOE_W4A4_PER_TOKEN, A, A, None, None, None, A, W, wb, Y, None)
    assert code in (api.MOE_ERR_CUDA, api.MOE_ERR_UNSUPPORTED)
