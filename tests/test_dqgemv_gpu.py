"""gemm_dequant for a few rows of A, against the oracle: one bf16 token with
4- or 2-bit weights takes the CUDA-core kernel that streams B once
(dqgemv.cu); two to four tokens, 8-bit weights or an f16 A take the
tensor-core decode kernel (dqdec.cu).  The same checks hold for both.

Checks: every element format with ragged N and K tails and 1, 2, 3 and 4
tokens; fp32 and bf16 output; the fused bias + GELU epilogue; C inside a
wider buffer and A inside a wider buffer; scales at both ends of the range;
the full-size single-token workload (sampled columns); determinism.  Every
output starts as NaN, so a column a kernel missed fails."""
import numpy as np
import pytest
import torch

import block_scaled_quantized_mx_gb300 as mx
import oracle
import workloads
from tests._parity import (check_close, check_epilogue_close, f16_bits,
                           nan_like, planes_from_codes)

pytestmark = pytest.mark.gpu

ALL_FMTS = [oracle.E4M3, oracle.E5M2, oracle.E2M1, oracle.INT8, oracle.INT4,
            oracle.INT2]


@pytest.fixture(scope="module", autouse=True)
def _built():
    mx.build()
    mx.lib()


def _odt(out):
    return torch.bfloat16 if out == "bf16" else torch.float32


def _case(M, N, K, fmt, seed, scale_lo=116, scale_hi=127, a_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    A = (torch.randn(M, K, generator=g) * a_scale).to(torch.bfloat16)
    cb, sb = workloads.random_codes((N, K), fmt, seed=seed + 1,
                                    scale_lo=scale_lo, scale_hi=scale_hi)
    return A, cb, sb, planes_from_codes(cb, sb, fmt)


@pytest.mark.parametrize("fmt", ALL_FMTS)
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", [(1000, 640), (8, 4160), (129, 64),
                                 (263, 2048)])
def test_gemv_formats(fmt, M, N, K):
    """N not a multiple of a CTA's eight rows for some shapes: C is a view of
    a buffer padded to a multiple of 8 columns (the row pitch must be a
    multiple of 16 bytes), whose padding must stay untouched."""
    A, cb, sb, b = _case(M, N, K, fmt, 11 * M + N + K + fmt)
    ld = (N + 7) // 8 * 8
    big = nan_like((M, ld), torch.float32)
    mx.gemm_dequant(A.cuda(), b, out_dtype=torch.float32, out=big[:, :N])
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    check_close(big[:, :N].cpu().numpy(), Cr, S, "f32",
                f"gemv fmt{fmt} {M}x{N}x{K}")
    assert torch.isnan(big[:, N:]).all()


@pytest.mark.parametrize("M", [1, 4])
def test_gemv_bf16_output(M):
    fmt, N, K = oracle.INT4, 520, 1024
    A, cb, sb, b = _case(M, N, K, fmt, 40 + M)
    C = nan_like((M, N), torch.bfloat16)
    mx.gemm_dequant(A.cuda(), b, out_dtype=torch.bfloat16, out=C)
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    check_close(C.float().cpu().numpy(), Cr, S, "bf16", f"gemv bf16 out M={M}")


@pytest.mark.parametrize("act", [oracle.ACT_NONE, oracle.ACT_GELU,
                                 oracle.ACT_GELU_TANH])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_gemv_fused_epilogue(act, out):
    M, N, K, fmt = 1, 296, 512, oracle.E2M1
    g = torch.Generator().manual_seed(7 + act)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = torch.randn(K, N, generator=g) * 0.05
    bias = torch.randn(N, generator=g) * 0.5
    b = mx.mx_quantize(W.cuda(), fmt, k_strided=True)
    C = nan_like((M, N), _odt(out))
    mx.gemm_dequant(A.cuda(), b, bias.cuda(), act, out_dtype=_odt(out), out=C)
    assert mx.mx_last_error() == 0
    cb, sb = oracle.quantize(W.numpy(), fmt, k_axis=0)
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    check_epilogue_close(C.float().cpu().numpy(), Cr, S, bias.numpy(), act,
                         out, f"gemv epilogue act{act} {out}")


@pytest.mark.parametrize("out,ld,off", [("bf16", 264, 8), ("f32", 260, 4)])
def test_gemv_padded_lda_ldc(out, ld, off):
    """A rows inside a wider buffer (lda > K) and C inside a wider buffer
    whose row starts are 16- but not always 32-byte aligned: nothing outside
    C is written."""
    M, N, K, fmt = 1, 256, 512, oracle.INT4
    g = torch.Generator().manual_seed(ld)
    Abig = torch.randn(M, K + 64, generator=g).to(torch.bfloat16)
    A = Abig[:, 16:16 + K]
    cb, sb = workloads.random_codes((N, K), fmt, seed=ld + 1, scale_lo=116,
                                    scale_hi=127)
    b = planes_from_codes(cb, sb, fmt)
    big = nan_like((M, ld), _odt(out))
    Ad = Abig.cuda()[:, 16:16 + K]
    mx.gemm_dequant(Ad, b, out_dtype=_odt(out), out=big[:, off:off + N])
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    check_close(big[:, off:off + N].float().cpu().numpy(), Cr, S, out,
                f"gemv lda {K + 64} ldc {ld} offset {off}")
    assert torch.isnan(big[:, :off].float()).all()
    assert torch.isnan(big[:, off + N:].float()).all()


@pytest.mark.parametrize("fmt", [oracle.INT8, oracle.INT4, oracle.INT2,
                                 oracle.E4M3])
@pytest.mark.parametrize("lo,hi,a_scale", [(226, 247, 2.0 ** -100),
                                           (12, 40, 2.0 ** 60)])
def test_gemv_scales_at_the_ends(fmt, lo, hi, a_scale):
    """Scale codes near both ends of the range (products kept in range by
    A's magnitude): the kernel multiplies exact fp32 codes by the power of
    two, so nothing overflows or underflows on the way."""
    M, N, K = 1, 256, 256
    if fmt == oracle.E4M3 and hi > 240:
        hi = 240            # 448 x 2^(hi - 127) must stay below fp32's maximum
    A, cb, sb, b = _case(M, N, K, fmt, 60 + fmt + lo, scale_lo=lo,
                         scale_hi=hi, a_scale=a_scale)
    C = nan_like((M, N), torch.float32)
    mx.gemm_dequant(A.cuda(), b, out_dtype=torch.float32, out=C)
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    assert (S < 1e37).all() and (S[S > 0] > 1e-30).all()
    check_close(C.cpu().numpy(), Cr, S, "f32", f"gemv scales {lo}..{hi}")


def test_gemv_workload_sampled():
    """The full-size single-token workload (1 x 8192 x 8192, int4 weights):
    the library quantizes the weights, the oracle recomputes sampled columns
    of C from its own quantization of them."""
    c = workloads.case("w4a16_decode_m1")
    fb = workloads.formats(c)[1]
    A, B = workloads.sources(c)
    b = mx.mx_quantize(B.cuda(), fb, k_strided=True)
    C = nan_like((c.M, c.N), torch.bfloat16)
    mx.gemm_dequant(A.cuda(), b, out_dtype=torch.bfloat16, out=C)
    assert mx.mx_last_error() == 0
    assert not torch.isnan(C.float()).any()
    cols = np.sort(np.random.default_rng(c.seed_b).choice(c.N, 48, replace=False))
    cb, sb = oracle.quantize(B[:, cols].float().numpy(), fb, k_axis=0)
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fb)
    check_close(C.float().cpu().numpy()[:, cols], Cr, S, "bf16",
                "w4a16_decode_m1 sampled columns")


def test_gemv_deterministic():
    g = torch.Generator().manual_seed(5)
    A = torch.randn(1, 4096, generator=g).to(torch.bfloat16).cuda()
    b = mx.mx_quantize(torch.randn(4096, 1536, generator=g).cuda(), mx.INT4,
                       k_strided=True)
    C1 = mx.gemm_dequant(A, b)
    C2 = mx.gemm_dequant(A, b)
    assert torch.equal(C1, C2)


def test_f16_tokens_take_the_decode_kernel():
    """An f16 A is not the single-token kernel's case (it dequantizes to
    bf16); the tensor-core decode kernel takes it, and still matches the
    oracle."""
    M, N, K, fmt = 2, 384, 1024, oracle.INT4
    g = torch.Generator().manual_seed(9)
    A = torch.randn(M, K, generator=g).to(torch.float16)
    cb, sb = workloads.random_codes((N, K), fmt, seed=10, scale_lo=116,
                                    scale_hi=127)
    b = planes_from_codes(cb, sb, fmt)
    C = nan_like((M, N), torch.float32)
    mx.gemm_dequant(A.cuda(), b, out_dtype=torch.float32, out=C)
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.F16, cb, sb, fmt)
    check_close(C.cpu().numpy(), Cr, S, "f32", "f16 tokens")
