"""Parity at the workloads' full sizes, through the same entry point and
launch configuration the benchmark times: routing, permutation and the x
quantization checked bit for bit on every token, the expert MLPs (FC2-input
codes, scales, per-token G2 and y) on a seeded sample of tokens the oracle
computes one by one: 256 tokens ({0, 1, T-1} and 253 more) at the DSV3 shape
with 4096 tokens and at prefill scale, fewer where a case only adds a
variant of a path those two already cover."""
import pytest

from nvfp4_mixture_experts_router_gb300 import api, build, synth

from gpu_parity import fullsize_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    api.lib()


def test_dsv3_shape_T4096_deterministic():
    """DeepSeek-V3-like expert shape: T=4096, H=7168, I=2048, E=256, top-8,
    per-tensor scales, deterministic finalize."""
    r = fullsize_parity(synth.config(2, 4096), n_tokens=256)
    assert r["code_match"] >= 0.999


def test_dsv3_shape_T8192_on_cta_pairs():
    """T=8192 at DSV3 shape (about 2.5 M tiles per expert) with both GEMMs
    forced onto CTA pairs."""
    r = fullsize_parity(synth.config(2, 8192).with_(gemm_pairs="always"), n_tokens=16)
    assert r["code_match"] >= 0.999


def test_dsv3_shape_T4096_mxfp8():
    """The DSV3-like shape at T=4096 in MXFP8 W8A8 (E4M3, E8M0 per 32)."""
    r = fullsize_parity(synth.config(2, 4096).with_(mode=synth.MODE_MXFP8), n_tokens=16)
    assert r["code_match"] >= 0.999


def test_w4a16_T4096():
    """W4A16: T=4096, H=4096, I=1536, E=128, top-8, ReLU2, fused finalize."""
    fullsize_parity(synth.config(3, 4096), n_tokens=24)


@pytest.mark.parametrize("finalize", ["deterministic", "fused"])
def test_prefill_T16384_zipf(finalize):
    """Prefill scale: T=16384, H=7168, I=2048, E=256, top-8, per-token
    scales, Zipf-skewed expert popularity (one expert takes most tokens,
    others none); both finalize modes (the workload's is deterministic)."""
    import numpy as np
    import oracle
    c = synth.config(4).with_(deterministic=finalize == "deterministic")
    ids, _ = oracle.router(synth.gen_logits(c).numpy(), synth.gen_bias(c).numpy(), c.K)
    count = np.bincount(ids.reshape(-1), minlength=c.E)
    assert count.max() >= 10 * count.mean() and (count == 0).any()
    r = fullsize_parity(c, n_tokens=256)
    assert r["code_match"] >= 0.999


def test_dsv3_shape_single_token():
    """T=1 at DSV3 shape: eight experts with one route each."""
    fullsize_parity(synth.config(2, 1), n_tokens=1)


@pytest.mark.parametrize("T", [1, 64])
def test_dsv3_shape_single_kernel(T):
    """The DSV3-like shape at decode token counts through the single
    persistent kernel (MOE_FUSED_LAYER), per-tensor scales, deterministic
    finalize."""
    r = fullsize_parity(synth.config(2, T).with_(fused=True), n_tokens=min(T, 16))
    assert r["code_match"] >= 0.999


def test_prefill_T16384_single_kernel():
    """The prefill workload (per-token scales, Zipf skew, deterministic
    finalize) through the single persistent kernel: the same kernel at
    16384 tokens."""
    r = fullsize_parity(synth.config(4).with_(fused=True), n_tokens=16)
    assert r["code_match"] >= 0.999


@pytest.mark.parametrize("T", [2560, 2000])
def test_fc2_output_slabs(T):
    """Fused finalize with an FP32 accumulator beyond 48 MB (T x H x 4 B =
    73 MB at T = 2560, 57 MB at T = 2000): FC2 walks its output width in
    slabs of at most 48 MiB of accumulator (38 + 18 and 49 + 7 of the 56
    128-wide N tiles, the last slab narrower) so that a token's reductions
    stay in L2; same results."""
    c = synth.MoEConfig("slab", T, 7168, 256, 8, 2, mode=synth.MODE_PER_TOKEN, seed=12, logits="normal")
    r = fullsize_parity(c, n_tokens=24)
    assert r["code_match"] >= 0.999
