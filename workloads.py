"""Seeded synthetic inputs for the MX / FP16 GEMM workloads.

Shared by the tests, the smoke check and the benchmark, so that the oracle
and the CUDA library always see identical bytes.  This module holds no part of
the method's arithmetic (no quantization, no matmul): it only draws numbers.

Every source is drawn on the CPU in float32 with ``torch.Generator`` seeded
per matrix, so the values do not depend on the device or on its RNG.

Workloads (sizes and value recipes):
  mx256      MXFP8, M=N=K=256, N(0,1) sources, fp32 output
  f16        FP16 / BF16 dense, M=N=K in {1024, 2048, 4096}, U[-1, 1]
             sources rounded to the 16-bit type, fp32 output (also 8192,
             the size the MX GEMMs are profiled at)
  mxfp8      MXFP8, M=N=K in {2048, 4096, 8192}, N(0,1) with 1 % of the
             entries (Bernoulli(0.01), drawn from the same generator)
             multiplied by 100, bf16 output
  mxfp4      MXFP4, M=N=K in {4096, 8192}, N(0,1), bf16 output
  mxfp8_e5m2 MXFP8 with E5M2 elements on both sides, M=N=K=8192, the
             mxfp8 recipe, bf16 output
  w4a8       mixed MX formats: E4M3 activations (A, the mxfp8 recipe) times
             E2M1 weights (B, N(0, 0.02)), M=N=K in {2048, 8192}, bf16 output
  w4a16      weight-only quantization: bf16 activations (A, N(0,1)) times
             int4 weights (B, N(0, 0.02), quantized by the MX rule),
             M=N=K=8192, a decode-shaped M=64, N=K=8192, and a single
             token M=1, N=K=8192; bf16 output
  w2a16      the same with int2 weights, M=N=K=8192
  attn       fused attention over image tokens: 2 images x 16 heads, 4096
             tokens each (a 64 x 64 patch grid, the image-segmentation model
             the FlashAttention chapter integrates into), d = 64 and 128,
             Q / K / V N(0,1) rounded to bf16
  proj       transformer projections of a 1B-parameter model at 32 x 512
             tokens (M=16384), hidden 2048, FFN 8192: qkv (K=2048, N=6144),
             out (K=2048, N=2048), up (K=2048, N=8192), down (K=8192,
             N=2048); activations N(0,1) as A, weights N(0, 0.02) as B
             (K x N), MXFP8, bf16 output
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


# Element formats (A, B) of the MX kinds, as the library's format codes:
# 1 = E4M3, 2 = E2M1, 3 = E5M2.
MX_FORMATS = {"mxfp8": (1, 1), "mxfp4": (2, 2), "mxfp8_e5m2": (3, 3),
              "w4a8": (1, 2)}
# Weight-only kinds: a bf16 A times an MX tensor B of this format (4 = int8,
# 5 = int4, 6 = int2), dequantized in the GEMM.
DEQUANT_FORMATS = {"w8a16": 4, "w4a16": 5, "w2a16": 6}


@dataclass(frozen=True)
class GemmCase:
    name: str
    kind: str          # an MX_FORMATS key | "f16" | "bf16"
    M: int
    N: int
    K: int
    out: str           # "f32" | "bf16"
    dist_a: str        # value recipe of A
    dist_b: str        # value recipe of B
    seed_a: int
    seed_b: int


def _seeds(group: int, tag: int):
    base = 1000 * group + 10 * tag
    return base + 1, base + 2


def mx256() -> GemmCase:
    sa, sb = _seeds(0, 8)
    return GemmCase("mx256", "mxfp8", 256, 256, 256, "f32", "normal",
                    "normal", sa, sb)


def f16_cases():
    out = []
    for kind in ("f16", "bf16"):
        for n in (1024, 2048, 4096, 8192):
            sa, sb = _seeds(1, int(math.log2(n)))
            out.append(GemmCase(f"{kind}_{n}", kind, n, n, n, "f32",
                                "uniform", "uniform", sa, sb))
    return out


def mxfp8_cases():
    out = []
    for n in (2048, 4096, 8192):
        sa, sb = _seeds(2, int(math.log2(n)))
        out.append(GemmCase(f"mxfp8_{n}", "mxfp8", n, n, n, "bf16",
                            "outlier", "outlier", sa, sb))
    return out


def mxfp4_cases():
    out = []
    for n in (4096, 8192):
        sa, sb = _seeds(3, int(math.log2(n)))
        out.append(GemmCase(f"mxfp4_{n}", "mxfp4", n, n, n, "bf16",
                            "normal", "normal", sa, sb))
    return out


def format_cases():
    sa, sb = _seeds(5, 13)
    out = [GemmCase("mxfp8_e5m2_8192", "mxfp8_e5m2", 8192, 8192, 8192, "bf16",
                    "outlier", "outlier", sa, sb)]
    for n in (2048, 8192):
        sa, sb = _seeds(6, int(math.log2(n)))
        out.append(GemmCase(f"w4a8_{n}", "w4a8", n, n, n, "bf16", "outlier",
                            "weight", sa, sb))
    return out


def dequant_cases():
    out = []
    for i, (name, kind, M) in enumerate((("w4a16_8192", "w4a16", 8192),
                                         ("w2a16_8192", "w2a16", 8192),
                                         ("w4a16_decode", "w4a16", 64),
                                         ("w4a16_decode_m1", "w4a16", 1))):
        sa, sb = _seeds(7, i)
        out.append(GemmCase(name, kind, M, 8192, 8192, "bf16", "normal",
                            "weight", sa, sb))
    return out


def is_mx(c: GemmCase) -> bool:
    return c.kind in MX_FORMATS


def is_dequant(c: GemmCase) -> bool:
    return c.kind in DEQUANT_FORMATS


def formats(c: GemmCase):
    """(format of A, format of B): an MX case's two formats; for a
    weight-only case (None, B's format), A being bf16."""
    if c.kind in DEQUANT_FORMATS:
        return None, DEQUANT_FORMATS[c.kind]
    return MX_FORMATS[c.kind]


PROJ_SHAPES = (("qkv", 2048, 6144), ("out", 2048, 2048), ("up", 2048, 8192),
               ("down", 8192, 2048))


def proj_cases():
    out = []
    for i, (name, K, N) in enumerate(PROJ_SHAPES):
        sa, sb = _seeds(4, i)
        out.append(GemmCase(f"proj_{name}", "mxfp8", 16384, N, K, "bf16",
                            "normal", "weight", sa, sb))
    return out


def all_cases():
    return [mx256()] + f16_cases() + mxfp8_cases() + mxfp4_cases() + \
        format_cases() + dequant_cases() + proj_cases()


def case(name: str) -> GemmCase:
    for c in all_cases():
        if c.name == name:
            return c
    raise KeyError(name)


def draw(shape, dist: str, seed: int) -> torch.Tensor:
    """float32 CPU tensor of the given recipe, from its own seeded stream."""
    g = torch.Generator().manual_seed(int(seed))
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32)
    if dist == "weight":
        return torch.randn(shape, generator=g, dtype=torch.float32) * 0.02
    if dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2 - 1
    if dist == "outlier":
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        mask = torch.rand(shape, generator=g, dtype=torch.float32) < 0.01
        return torch.where(mask, x * 100.0, x)
    raise ValueError(dist)


def sources(c: GemmCase, M: int | None = None, N: int | None = None,
            K: int | None = None):
    """(A, B) float32 sources: A is M x K row-major, B is K x N row-major.
    Sizes may be overridden to draw a smaller problem of the same recipe."""
    M = c.M if M is None else M
    N = c.N if N is None else N
    K = c.K if K is None else K
    A = draw((M, K), c.dist_a, c.seed_a)
    B = draw((K, N), c.dist_b, c.seed_b)
    if c.kind in ("f16", "bf16"):
        dt = torch.float16 if c.kind == "f16" else torch.bfloat16
        A, B = A.to(dt), B.to(dt)
    elif c.kind in DEQUANT_FORMATS:
        A = A.to(torch.bfloat16)            # B stays fp32: it gets quantized
    return A, B


@dataclass(frozen=True)
class AttnCase:
    name: str
    BH: int            # batch x heads
    Lq: int
    Lk: int
    d: int
    dtype: str         # "bf16" | "f16"
    seed: int


def attn_cases():
    # 32 heads x 4096 tokens (self-attention, d 64 / 128); 8 heads of 256
    # queries against a 32768-token context (long-context prefill chunk:
    # fewer (head, 256-query) units than SMs)
    return [AttnCase(f"attn_sam_d{d}", 32, 4096, 4096, d, "bf16", 8000 + d)
            for d in (64, 128)] + [
        AttnCase("attn_long_d128", 8, 256, 32768, 128, "bf16", 8300)]


def attn_case(name: str) -> AttnCase:
    for c in attn_cases():
        if c.name == name:
            return c
    raise KeyError(name)


def attn_sources(c: AttnCase, BH: int | None = None, Lq: int | None = None,
                 Lk: int | None = None):
    """(Q, K, V): BH x Lq x d and BH x Lk x d, N(0,1) rounded to c.dtype,
    each from its own seeded stream."""
    BH = c.BH if BH is None else BH
    Lq = c.Lq if Lq is None else Lq
    Lk = c.Lk if Lk is None else Lk
    dt = torch.bfloat16 if c.dtype == "bf16" else torch.float16
    Q = draw((BH, Lq, c.d), "normal", c.seed + 1).to(dt)
    K = draw((BH, Lk, c.d), "normal", c.seed + 2).to(dt)
    V = draw((BH, Lk, c.d), "normal", c.seed + 3).to(dt)
    return Q, K, V


def random_codes(shape, fmt: int, seed: int, scale_lo: int = 112,
                 scale_hi: int = 142):
    """Random MX planes for GEMM-only tests: finite element codes (uint8,
    one per byte, unpacked) and UE8M0 scale codes drawn uniformly from
    [scale_lo, scale_hi].  Returns (codes outer x K, scales outer x K/32)."""
    outer, K = shape
    g = torch.Generator().manual_seed(int(seed))
    if fmt in (1, 3):
        codes = torch.randint(0, 256, (outer, K), generator=g,
                              dtype=torch.int32)
        # redraw the non-finite codes as zeros: 0x7F / 0xFF in E4M3,
        # 0x7C-0x7F / 0xFC-0xFF in E5M2
        bad = (codes & 0x7F) >= (0x7F if fmt == 1 else 0x7C)
        codes = torch.where(bad, torch.zeros_like(codes), codes)
    else:
        # E2M1 and the integer formats: every code of their width is finite
        ncodes = {2: 16, 4: 256, 5: 16, 6: 4}[fmt]
        codes = torch.randint(0, ncodes, (outer, K), generator=g,
                              dtype=torch.int32)
    scales = torch.randint(scale_lo, scale_hi + 1, (outer, K // 32),
                           generator=g, dtype=torch.int32)
    return (codes.to(torch.uint8).numpy(), scales.to(torch.uint8).numpy())
