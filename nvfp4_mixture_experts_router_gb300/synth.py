"""Seeded synthetic inputs for the NVFP4 MoE layer forward.

This module only draws numbers. It holds none of the layer's arithmetic
(no routing, no quantization, no GEMM), so both the CUDA path and the CPU
oracle can consume what it produces without sharing any method code.

Generator (counter based, index addressable, identical on CPU and GPU):

* ``lowbias32`` — the 32-bit integer hash published by C. Wellons
  ("Prospecting for Hash Functions", 2018): ``x ^= x>>16; x *= 0x7feb352d;
  x ^= x>>15; x *= 0x846ca68b; x ^= x>>16`` (all mod 2**32).  Implemented with
  int64 tensors and 16-bit limb multiplication so that no intermediate ever
  overflows a signed 64-bit integer.
* one value = two hashes of its 36-bit counter ``(seed, stream, index)``;
  the 64 hash bits give four 16-bit uniforms ``u_j = (b_j + 0.5) / 65536``.
* an approximately normal deviate is the Irwin-Hall sum of those four
  uniforms, centred and scaled to unit variance: ``(u0+u1+u2+u3-2)*sqrt(3)``.
  Every step up to the single float32 multiply by ``std*sqrt(3)`` is exact in
  float32, so CPU and GPU give bit-identical values; the BF16 inputs are the
  round-to-nearest-even conversion of that float32.

Streams: 0 x, 1 router weight W_g, 2 router bias, 3 W1, 4 W2, 5 logits,
6 expert-popularity permutation.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

MASK32 = 0xFFFFFFFF

STREAM_X = 0
STREAM_WG = 1
STREAM_BIAS = 2
STREAM_W1 = 3
STREAM_W2 = 4
STREAM_LOGITS = 5
STREAM_PERM = 6


def _mul32(a: torch.Tensor, c: int) -> torch.Tensor:
    """(a * c) mod 2**32 for 0 <= a < 2**32, using 16-bit limbs of c."""
    lo = a * (c & 0xFFFF)
    hi = (a * (c >> 16)) & 0xFFFF
    return (lo + (hi << 16)) & MASK32


def lowbias32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _key(seed: int, stream: int, hi: torch.Tensor) -> torch.Tensor:
    assert 0 <= seed < (1 << 20) and 0 <= stream < 64
    return lowbias32((hi & 63) | (stream << 6) | (seed << 12))


def hash_pair(seed: int, stream: int, index: torch.Tensor):
    """Two 32-bit hashes (as int64 tensors) of the counters in ``index``."""
    lo = index & MASK32
    hi = index >> 32
    k = _key(seed, stream, hi)
    h1 = lowbias32(lo ^ k)
    h2 = lowbias32(h1 ^ 0x9E3779B9)
    return h1, h2


def _counters(start: int, n: int, device) -> torch.Tensor:
    assert start + n < (1 << 38)
    return torch.arange(start, start + n, dtype=torch.int64, device=device)


def normal_f32(seed: int, stream: int, start: int, n: int, std: float,
               device="cpu") -> torch.Tensor:
    """``n`` Irwin-Hall(4) deviates with standard deviation ``std``, float32."""
    h1, h2 = hash_pair(seed, stream, _counters(start, n, device))
    inv = 1.0 / 65536.0
    u0 = ((h1 & 0xFFFF).to(torch.float32) + 0.5) * inv
    u1 = ((h1 >> 16).to(torch.float32) + 0.5) * inv
    u2 = ((h2 & 0xFFFF).to(torch.float32) + 0.5) * inv
    u3 = ((h2 >> 16).to(torch.float32) + 0.5) * inv
    s = ((u0 + u1) + u2) + u3 - 2.0
    scale = torch.tensor(std * math.sqrt(3.0), dtype=torch.float32, device=device)
    return s * scale


def uniform_f64(seed: int, stream: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """``n`` uniforms in (0, 1) with 32 random bits, float64."""
    h1, _ = hash_pair(seed, stream, _counters(start, n, device))
    return (h1.to(torch.float64) + 0.5) / 4294967296.0


def normal_bf16(seed, stream, start, n, std, device="cpu"):
    return normal_f32(seed, stream, start, n, std, device).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# Workload definitions (shapes, distributions and flags of the five layer
# configurations exercised by the tests and the benchmark).
# ---------------------------------------------------------------------------

ACT_SWIGLU, ACT_RELU2 = 0, 1
MODE_PER_TENSOR, MODE_PER_TOKEN, MODE_W4A16, MODE_MXFP8 = 0, 1, 2, 3


@dataclass
class MoEConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    K: int
    act: int = ACT_SWIGLU
    mode: int = MODE_PER_TENSOR
    router_on_input: bool = False
    deterministic: bool = False
    renorm: bool = True
    seed: int = 0
    logits: str = "gate"          # "gate": x @ W_g^T ; "normal": N(0,1)
    bias: str = "none"            # "none" | "normal" | "zipf"
    bias_std: float = 0.5
    zipf_s: float = 1.1
    zipf_beta: float = 2.0
    w_std: float = 0.02
    gemm_pairs: str = "auto"      # GEMM tile scheduling: "auto" | "never" | "always"
    four_over_six: bool = False   # per-token W4A4: 4-over-6 activation quantization
    fused: bool = False           # W4A4: the whole forward as one persistent kernel
    gemm_swap: str = "auto"       # W4A4 / W4A16 GEMM orientation: "auto" | "never" | "always"
    extra: dict = field(default_factory=dict)

    @property
    def N1(self) -> int:
        return 2 * self.I if self.act == ACT_SWIGLU else self.I

    def flags(self) -> int:
        f = self.act | (self.mode << 2)
        if self.router_on_input:
            f |= 1 << 4
        if self.deterministic:
            f |= 1 << 5
        if not self.renorm:
            f |= 1 << 6
        if self.gemm_pairs == "never":
            f |= 1 << 7
        elif self.gemm_pairs == "always":
            f |= 1 << 8
        if self.four_over_six:
            f |= 1 << 9
        if self.fused:
            f |= 1 << 10
        if self.gemm_swap == "never":
            f |= 1 << 11
        elif self.gemm_swap == "always":
            f |= 1 << 12
        return f

    def with_(self, **kw) -> "MoEConfig":
        d = dict(self.__dict__)
        d.update(kw)
        return MoEConfig(**d)


def config(idx: int, T: Optional[int] = None) -> MoEConfig:
    """The five workloads: 0 tiny, 1 mid, 2 DeepSeek-V3-like expert shape,
    3 W4A16 ReLU2, 4 prefill-scale with Zipf-skewed expert popularity."""
    if idx == 0:
        c = MoEConfig("tiny_w4a4_T16_H256_I128_E8_K2", 16, 256, 128, 8, 2,
                      seed=0, logits="gate")
    elif idx == 1:
        c = MoEConfig("mid_w4a4_T512_H2048_I768_E64_K6", 512, 2048, 768, 64, 6,
                      mode=MODE_PER_TOKEN, router_on_input=True, seed=1,
                      logits="gate", bias="normal")
    elif idx == 2:
        c = MoEConfig("dsv3_w4a4_H7168_I2048_E256_K8", 4096, 7168, 2048, 256, 8,
                      deterministic=True, seed=2, logits="normal")
    elif idx == 3:
        c = MoEConfig("w4a16_relu2_H4096_I1536_E128_K8", 4096, 4096, 1536, 128, 8,
                      act=ACT_RELU2, mode=MODE_W4A16, seed=3, logits="normal")
    elif idx == 4:
        c = MoEConfig("prefill_w4a4_T16384_H7168_I2048_E256_K8", 16384, 7168, 2048,
                      256, 8, mode=MODE_PER_TOKEN, deterministic=True, seed=4, logits="normal",
                      bias="zipf")
    else:
        raise ValueError(idx)
    if T is not None:
        c = c.with_(T=T, name=c.name + f"_T{T}")
    return c


def gen_x(c: MoEConfig, device="cpu") -> torch.Tensor:
    """x: BF16 [T, H], N(0, 1)."""
    return normal_bf16(c.seed, STREAM_X, 0, c.T * c.H, 1.0, device).view(c.T, c.H)


def gen_tokens_x(c: MoEConfig, tokens, device="cpu") -> torch.Tensor:
    """Rows ``tokens`` of x, without generating the rest."""
    rows = [normal_bf16(c.seed, STREAM_X, int(t) * c.H, c.H, 1.0, device) for t in tokens]
    return torch.stack(rows) if rows else torch.empty(0, c.H, dtype=torch.bfloat16)


def zipf_bias(c: MoEConfig) -> torch.Tensor:
    """Per-expert logit bias giving Zipf(s) expert popularity.

    Ranks come from a seeded Fisher-Yates permutation of the experts; expert
    of rank r (1-based) gets popularity p_r ~ r^-s, and its bias is
    beta * ln(E * p_r)."""
    E = c.E
    u = uniform_f64(c.seed, STREAM_PERM, 0, E).tolist()
    perm = list(range(E))
    for i in range(E - 1, 0, -1):
        j = min(int(u[i] * (i + 1)), i)
        perm[i], perm[j] = perm[j], perm[i]
    pr = [(r + 1) ** (-c.zipf_s) for r in range(E)]
    z = sum(pr)
    bias = [0.0] * E
    for r, e in enumerate(perm):
        bias[e] = c.zipf_beta * math.log(E * pr[r] / z)
    return torch.tensor(bias, dtype=torch.float64).to(torch.float32)


def gen_bias(c: MoEConfig, device="cpu") -> Optional[torch.Tensor]:
    if c.bias == "none":
        return None
    if c.bias == "normal":
        return normal_f32(c.seed, STREAM_BIAS, 0, c.E, c.bias_std, device)
    if c.bias == "zipf":
        return zipf_bias(c).to(device)
    raise ValueError(c.bias)


def gen_logits(c: MoEConfig, device="cpu", x: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Router logits FP32 [T, E].

    "gate": x @ W_g^T with W_g ~ N(0, 1/H) (variance 1/H), product taken in
    float64 and rounded once to float32.  "normal": N(0, 1) directly."""
    if c.logits == "normal":
        return normal_f32(c.seed, STREAM_LOGITS, 0, c.T * c.E, 1.0, device).view(c.T, c.E)
    if x is None:
        x = gen_x(c, device)
    wg = gen_wg(c, device)
    return (x.double() @ wg.double().t()).to(torch.float32)


def gen_wg(c: MoEConfig, device="cpu") -> torch.Tensor:
    """Router (gate projection) weight W_g: BF16 [E, H], N(0, 1/H)."""
    return normal_f32(c.seed, STREAM_WG, 0, c.E * c.H, 1.0 / math.sqrt(c.H), device).view(c.E, c.H).to(torch.bfloat16)


def gen_w1_expert(c: MoEConfig, e: int, device="cpu") -> torch.Tensor:
    """FC1 weight of expert e, BF16 [N1, H] in checkpoint order: for SwiGLU
    rows 0..I-1 are the gate projection and rows I..2I-1 the up projection."""
    n = c.N1 * c.H
    return normal_bf16(c.seed, STREAM_W1, e * n, n, c.w_std, device).view(c.N1, c.H)


def gen_w2_expert(c: MoEConfig, e: int, device="cpu") -> torch.Tensor:
    """FC2 weight of expert e, BF16 [H, I]."""
    n = c.H * c.I
    return normal_bf16(c.seed, STREAM_W2, e * n, n, c.w_std, device).view(c.H, c.I)


def gen_w1(c: MoEConfig, device="cpu") -> torch.Tensor:
    out = torch.empty(c.E, c.N1, c.H, dtype=torch.bfloat16, device=device)
    for e in range(c.E):
        out[e] = gen_w1_expert(c, e, device)
    return out


def gen_w2(c: MoEConfig, device="cpu") -> torch.Tensor:
    out = torch.empty(c.E, c.H, c.I, dtype=torch.bfloat16, device=device)
    for e in range(c.E):
        out[e] = gen_w2_expert(c, e, device)
    return out


def sample_tokens(c: MoEConfig, n: int) -> list:
    """Seeded token subset: 0, 1, T-1 plus n-3 further distinct tokens."""
    T = c.T
    if n >= T:
        return list(range(T))
    picked = []
    for t in (0, 1, T - 1):
        if t not in picked:
            picked.append(t)
    u = uniform_f64(c.seed, STREAM_PERM, 1 << 20, 8 * n + 64).tolist()
    for v in u:
        if len(picked) >= n:
            break
        t = min(int(v * T), T - 1)
        if t not in picked:
            picked.append(t)
    return sorted(picked)
