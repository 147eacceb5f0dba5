"""gemm_dequant on the GPU vs the oracle: a 16-bit A times an MX tensor B of
every element format (the integer formats int8 / int4 / int2 included),
B dequantized in shared memory and multiplied on the 16-bit tensor cores.

Checks: exact integer products; random codes with ragged M / N tails for
both CTA-group shapes (M <= 128 runs one CTA per tile, larger M a CTA pair);
the fused bias + GELU epilogue; a full-size weight-only workload (sampled
rows); determinism.  Every output starts as NaN, so a tile the kernel missed
fails."""
import numpy as np
import pytest
import torch

import block_scaled_quantized_mx_gb300 as mx
import oracle
import workloads
from tests._parity import (check_close, check_epilogue_close, f16_bits,
                           nan_like, planes_from_codes, sample_rows)

pytestmark = pytest.mark.gpu

ALL_FMTS = [oracle.E4M3, oracle.E5M2, oracle.E2M1, oracle.INT8, oracle.INT4,
            oracle.INT2]


@pytest.fixture(scope="module", autouse=True)
def _built():
    mx.build()
    mx.lib()


def _tdt(a):
    return torch.float16 if a == "f16" else torch.bfloat16


def _odt(out):
    return torch.bfloat16 if out == "bf16" else torch.float32


def _ocode(a):
    return oracle.F16 if a == "f16" else oracle.BF16


@pytest.mark.parametrize("fmt,vmax", [(oracle.INT8, 127), (oracle.INT4, 7),
                                      (oracle.INT2, 1), (oracle.E4M3, 14),
                                      (oracle.E2M1, 4)])
@pytest.mark.parametrize("a", ["bf16", "f16"])
def test_dequant_integer_exact(fmt, vmax, a):
    """Integer A and integer B values that quantize without loss (the
    oracle's own quantization of B): C is the exact integer product."""
    g = np.random.default_rng(fmt * 7 + len(a))
    M, N, K = 256, 384, 512
    vals = np.arange(-vmax, vmax + 1)
    if fmt == oracle.E2M1:
        vals = np.array([-4, -3, -2, -1, 0, 1, 2, 3, 4])
    A = torch.from_numpy(g.integers(-60, 61, (M, K)).astype(np.float32))
    B = g.choice(vals, (K, N)).astype(np.float32)
    cb, sb = oracle.quantize(B, fmt, k_axis=0)
    b = planes_from_codes(cb, sb, fmt)
    C = nan_like((M, N), torch.float32)
    mx.gemm_dequant(A.to(_tdt(a)).cuda(), b, out=C)
    assert mx.mx_last_error() == 0
    want = A.numpy().astype(np.int64) @ B.astype(np.int64)
    assert np.array_equal(C.cpu().numpy(), want.astype(np.float32))


@pytest.mark.parametrize("fmt", ALL_FMTS)
@pytest.mark.parametrize("a", ["bf16", "f16"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (100, 296, 192),
                                   (200, 264, 128), (384, 520, 1088),
                                   (1000, 136, 2048)])
def test_dequant_random_codes(fmt, a, out, M, N, K):
    g = torch.Generator().manual_seed(M + 3 * N + K + fmt)
    A = torch.randn(M, K, generator=g).to(_tdt(a))
    # scales that keep every dequantized value inside f16's range too
    cb, sb = workloads.random_codes((N, K), fmt, seed=N + K + fmt,
                                    scale_lo=116, scale_hi=127)
    b = planes_from_codes(cb, sb, fmt)
    C = nan_like((M, N), _odt(out))
    mx.gemm_dequant(A.cuda(), b, out_dtype=_odt(out), out=C)
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), _ocode(a), cb, sb, fmt)
    check_close(C.float().cpu().numpy(), Cr, S, out,
                f"{a} x fmt{fmt} {M}x{N}x{K}")


@pytest.mark.parametrize("out,ld,off,split", [("bf16", 264, 8, False),
                                              ("f32", 260, 4, False),
                                              ("bf16", 264, 8, True)])
def test_dequant_padded_ldc(out, ld, off, split):
    """C inside a wider buffer whose row starts are 16- but not always
    32-byte aligned (see test_padded_ldc in the GEMM tests); nothing outside
    C is written, with and without the K-split."""
    fmt = oracle.INT4
    M, N, K = (200, 256, 4096) if split else (200, 256, 256)
    g = torch.Generator().manual_seed(ld + off)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    cb, sb = workloads.random_codes((N, K), fmt, seed=ld, scale_lo=116,
                                    scale_hi=127)
    b = planes_from_codes(cb, sb, fmt)
    ws = None
    if split:
        nbytes = mx.gemm_dequant_workspace_bytes(M, N, K)
        assert nbytes > 0, "expected a split for this shape"
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    big = nan_like((M, ld), _odt(out))
    mx.gemm_dequant(A.cuda(), b, out_dtype=_odt(out), out=big[:, off:off + N],
                    workspace=ws)
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    check_close(big[:, off:off + N].float().cpu().numpy(), Cr, S, out,
                f"ldc {ld} offset {off}")
    assert torch.isnan(big[:, :off].float()).all()
    assert torch.isnan(big[:, off + N:].float()).all()


@pytest.mark.parametrize("M", [256, 64])
@pytest.mark.parametrize("fmt", [oracle.INT8, oracle.INT4, oracle.INT2, oracle.E5M2])
def test_dequant_wide_scales_bf16(fmt, M):
    """bf16 A: scales across a wide range are still exact after the
    dequantization to bf16 (M = 64: the decode kernel, whose quads take a
    shorter conversion loop when every scale code is at most 231, or 247 for
    4- and 2-bit codes, and the general one otherwise)."""
    N, K = 256, 256
    g = torch.Generator().manual_seed(90 + fmt)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    cb, sb = workloads.random_codes((N, K), fmt, seed=91 + fmt, scale_lo=40,
                                    scale_hi=200)
    b = planes_from_codes(cb, sb, fmt)
    C = mx.gemm_dequant(A.cuda(), b, out_dtype=torch.float32)
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    ok = (S < 1e37) & (S > 1e-30)
    check_close(np.where(ok, C.cpu().numpy(), Cr), Cr, S, "f32", "wide scales")


@pytest.mark.parametrize("fmt", [oracle.INT8, oracle.INT4, oracle.INT2])
def test_dequant_extreme_scales_bf16(fmt):
    """Scale codes from 226 up to the largest whose every q X fits bf16
    (int8: -128 X, so X <= 2^120, code 247; int4 / int2: code 248), against
    a bf16 A of magnitude 2^-100 so that every product stays in range: the
    integer paths must stay exact where their multiply-add constants would
    overflow (fp32 beyond X = 2^104, bf16 beyond X = 2^120)."""
    M, N, K = 128, 256, 256
    g = torch.Generator().manual_seed(70 + fmt)
    A = (torch.randn(M, K, generator=g) * 2.0 ** -100).to(torch.bfloat16)
    hi = 247 if fmt == oracle.INT8 else 248
    cb, sb = workloads.random_codes((N, K), fmt, seed=71 + fmt, scale_lo=226,
                                    scale_hi=hi)
    b = planes_from_codes(cb, sb, fmt)
    C = nan_like((M, N), torch.float32)
    mx.gemm_dequant(A.cuda(), b, out_dtype=torch.float32, out=C)
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    assert (S < 1e37).all() and sb.max() == hi and sb.min() <= 231
    check_close(C.cpu().numpy(), Cr, S, "f32", f"extreme scales fmt{fmt}")


@pytest.mark.parametrize("fmt", [oracle.INT4, oracle.E2M1])
@pytest.mark.parametrize("act", [oracle.ACT_GELU, oracle.ACT_GELU_TANH])
def test_dequant_fused_epilogue(fmt, act):
    M, N, K = 200, 296, 512
    g = torch.Generator().manual_seed(5 + fmt + act)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = torch.randn(K, N, generator=g) * 0.05
    bias = torch.randn(N, generator=g) * 0.5
    b = mx.mx_quantize(W.cuda(), fmt, k_strided=True)
    C = nan_like((M, N), torch.float32)
    mx.gemm_dequant(A.cuda(), b, bias.cuda(), act, out=C)
    assert mx.mx_last_error() == 0
    cb, sb = oracle.quantize(W.numpy(), fmt, k_axis=0)
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    check_epilogue_close(C.cpu().numpy(), Cr, S, bias.numpy(), act, "f32",
                         f"fmt{fmt} act{act}")


@pytest.mark.parametrize("name", ["w4a16_8192", "w2a16_8192", "w4a16_decode"])
def test_dequant_workload_sampled(name):
    """Full-size weight-only workloads: the library quantizes the weights
    (checked bit for bit against the oracle elsewhere), the oracle
    recomputes sampled rows from its own quantization of them."""
    c = workloads.case(name)
    fb = workloads.formats(c)[1]
    A, B = workloads.sources(c)
    b = mx.mx_quantize(B.cuda(), fb, k_strided=True)
    C = nan_like((c.M, c.N), _odt(c.out))
    mx.gemm_dequant(A.cuda(), b, out_dtype=_odt(c.out), out=C)
    assert mx.mx_last_error() == 0
    rows = sample_rows(c.M, n_random=12, seed=c.seed_a)
    cb, sb = oracle.quantize(B.float().numpy(), fb, k_axis=0)
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fb,
                                rows=rows)
    check_close(C.float().cpu().numpy()[rows], Cr, S, c.out, name)


def test_dequant_deterministic():
    g = torch.Generator().manual_seed(3)
    A = torch.randn(512, 1024, generator=g).to(torch.bfloat16).cuda()
    b = mx.mx_quantize(torch.randn(1024, 768, generator=g).cuda(), mx.INT4,
                       k_strided=True)
    C1 = mx.gemm_dequant(A, b)
    C2 = mx.gemm_dequant(A, b)
    assert torch.equal(C1, C2)


@pytest.mark.parametrize("fmt", [oracle.INT4, oracle.INT2, oracle.E4M3])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(1, 2048, 4096), (16, 1024, 8192),
                                   (64, 2048, 2048), (128, 512, 4096),
                                   (200, 768, 4096)])
def test_dequant_splitk(fmt, out, M, N, K):
    """Decode-like shapes: few output tiles, K split over the idle SMs.  Over
    128 tokens the parts go to the workspace and are summed in a fixed order
    by the reduction kernel; up to 128 tokens the decode kernel splits each
    weight block's K range inside a thread-block cluster and needs no
    workspace.  Either way a repeat gives the same bits."""
    g = torch.Generator().manual_seed(M + N + K + fmt)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    cb, sb = workloads.random_codes((N, K), fmt, seed=N + fmt, scale_lo=116,
                                    scale_hi=127)
    b = planes_from_codes(cb, sb, fmt)
    nbytes = mx.gemm_dequant_workspace_bytes(M, N, K)
    if M > 128:
        assert nbytes > 0, "expected a split for this shape"
    else:
        assert nbytes == 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
    C = nan_like((M, N), _odt(out))
    mx.gemm_dequant(A.cuda(), b, out_dtype=_odt(out), out=C, workspace=ws)
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    check_close(C.float().cpu().numpy(), Cr, S, out, f"split {M}x{N}x{K}")
    C2 = mx.gemm_dequant(A.cuda(), b, out_dtype=_odt(out), workspace=ws)
    assert torch.equal(C.view(torch.uint8), C2.view(torch.uint8))


def test_dequant_splitk_fused_epilogue():
    M, N, K = 200, 1024, 4096
    g = torch.Generator().manual_seed(44)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = torch.randn(K, N, generator=g) * 0.02
    bias = torch.randn(N, generator=g) * 0.5
    b = mx.mx_quantize(W.cuda(), mx.INT4, k_strided=True)
    ws = torch.empty(mx.gemm_dequant_workspace_bytes(M, N, K),
                     dtype=torch.uint8, device="cuda")
    C = mx.gemm_dequant(A.cuda(), b, bias.cuda(), mx.ACT_GELU, workspace=ws)
    assert mx.mx_last_error() == 0
    cb, sb = oracle.quantize(W.numpy(), oracle.INT4, k_axis=0)
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, oracle.INT4)
    check_epilogue_close(C.cpu().numpy(), Cr, S, bias.numpy(), oracle.ACT_GELU,
                         "f32", "split + GELU")


def test_dequant_workspace_only_for_idle_sms():
    assert mx.gemm_dequant_workspace_bytes(8192, 8192, 8192) == 0
    assert mx.gemm_dequant_workspace_bytes(200, 768, 4096) > 0
    assert mx.gemm_dequant_workspace_bytes(200, 768, 100) == 0      # K % 64
    # up to 128 tokens: the decode kernel splits K inside clusters
    assert mx.gemm_dequant_workspace_bytes(64, 8192, 8192) == 0
