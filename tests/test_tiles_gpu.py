"""The GEMM's tile configurations, each forced in turn (mx_set_tile_width),
against the float64 oracle.

Configurations: CTA pairs (256-row tiles, M > 128) or single CTAs (M <= 128)
times 256- or 128-column tiles.  A tile's width does not change the order in
which any element of C is summed (the K stages run in order inside one tile),
so an unsplit product must come out bit for bit the same in every
configuration; each is also checked element by element against the oracle
with the usual bound |C - C_ref| <= 1e-4 * S (plus one bf16 ulp of C_ref for
bf16 output).  The shapes have ragged edges in M, N and K, and the last tile
of every CTA is written by the epilogue's TMA stores (the tiles before it by
register stores), so both store paths are covered in every configuration."""
import numpy as np
import pytest
import torch

import block_scaled_quantized_mx_gb300 as mx
import oracle
import workloads
from tests._parity import (check_close, check_epilogue_close, f16_bits,
                           nan_like, planes_from_codes)

pytestmark = pytest.mark.gpu

WIDTHS = [0, 128, 256]


@pytest.fixture(scope="module", autouse=True)
def _built():
    mx.build()
    mx.lib()
    yield
    mx.set_tile_width(0)


@pytest.fixture(autouse=True)
def _reset_width():
    yield
    mx.set_tile_width(0)


def _codes(fmt, M, N, K, seed):
    ca, sa = workloads.random_codes((M, K), fmt, seed=seed)
    cb, sb = workloads.random_codes((N, K), fmt, seed=seed + 1)
    return ca, sa, cb, sb


# (M, N, K): pairs with several tiles and ragged edges; single CTAs (M <= 128)
SHAPES = [(640, 1000, 544), (1024, 1024, 1024), (96, 1800, 640), (128, 384, 256)]


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E2M1])
@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_mx_every_width(fmt, M, N, K, out):
    ca, sa, cb, sb = _codes(fmt, M, N, K, seed=M + N + K)
    a, b = planes_from_codes(ca, sa, fmt), planes_from_codes(cb, sb, fmt)
    odt = torch.bfloat16 if out == "bf16" else torch.float32
    Cr, S = oracle.gemm_mx(ca, sa, cb, sb, fmt)
    results = []
    for w in WIDTHS:
        mx.set_tile_width(w)
        C = nan_like((M, N), odt)
        mx.mx_gemm(a, b, out_dtype=odt, out=C)
        assert mx.mx_last_error() == 0
        check_close(C.float().cpu().numpy(), Cr, S, out, f"width {w}")
        results.append(C)
    for C in results[1:]:
        assert torch.equal(C.view(torch.uint8), results[0].view(torch.uint8))


@pytest.mark.parametrize("M,N,K", [(520, 776, 512), (1024, 1024, 1024),
                                   (64, 1280, 384)])
@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_f16_every_width(M, N, K, dt):
    g = torch.Generator().manual_seed(M * 3 + N)
    A = (torch.rand(M, K, generator=g) * 2 - 1).to(dt)
    B = (torch.rand(K, N, generator=g) * 2 - 1).to(dt)
    Cr, S = oracle.gemm_f16(f16_bits(A), f16_bits(B),
                            oracle.F16 if dt == torch.float16 else oracle.BF16)
    results = []
    for w in WIDTHS:
        mx.set_tile_width(w)
        C = nan_like((M, N), torch.float32)
        mx.gemm_f16(A.cuda(), B.cuda(), out=C)
        assert mx.mx_last_error() == 0
        check_close(C.cpu().numpy(), Cr, S, "f32", f"width {w}")
        results.append(C)
    for C in results[1:]:
        assert torch.equal(C, results[0])


@pytest.mark.parametrize("w", [128, 256])
def test_mixed_pair_and_fused_epilogue_narrow(w):
    """A mixed E4M3 x E2M1 pair and the fused bias + GELU epilogue in each
    width (the 128-wide tiles hold 64 columns per epilogue thread)."""
    M, N, K = 768, 640, 512
    ca, sa = workloads.random_codes((M, K), oracle.E4M3, seed=11)
    cb, sb = workloads.random_codes((N, K), oracle.E2M1, seed=12)
    a = planes_from_codes(ca, sa, oracle.E4M3)
    b = planes_from_codes(cb, sb, oracle.E2M1)
    mx.set_tile_width(w)
    C = nan_like((M, N), torch.float32)
    mx.mx_gemm(a, b, out_dtype=torch.float32, out=C)
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_mx(ca, sa, cb, sb, oracle.E4M3, fmt_b=oracle.E2M1)
    check_close(C.cpu().numpy(), Cr, S, "f32", f"mixed width {w}")

    bias = torch.randn(N, generator=torch.Generator().manual_seed(5)) * 0.5
    Cf = nan_like((M, N), torch.bfloat16)
    mx.mx_gemm_fused(a, b, bias.cuda(), mx.ACT_GELU, out_dtype=torch.bfloat16, out=Cf)
    assert mx.mx_last_error() == 0
    check_epilogue_close(Cf.float().cpu().numpy(), Cr, S, bias.numpy().astype(np.float64),
                         mx.ACT_GELU, "bf16", f"fused width {w}")


def test_set_tile_width_rejects_other_values():
    L = mx.lib()
    for bad in (1, 64, 192, 512, -1):
        assert L.mx_set_tile_width(bad) == 1
    assert L.mx_set_tile_width(0) == 0
