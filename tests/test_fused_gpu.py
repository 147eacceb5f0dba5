"""The fused epilogue on the GPU vs the oracle: bias and GELU on the fp32
accumulator (mx_gemm_fused, gemm_f16_fused), and C quantized to an MX tensor
in the same epilogue (mx_gemm_fused_quantize).

fp32 / bf16 outputs are compared element by element with the oracle's
act(C + bias) within the bound of tests/_parity.py.  The quantized output is
checked three ways: exactly against the oracle where the product is exact
(integer matrices, no activation); against the oracle's allowed code
intervals everywhere else; and bit for bit against the library's own
two-step path (fp32 output of the fused call, then mx_quantize), which must
agree because both quantize the same fp32 values with the same rule."""
import numpy as np
import pytest
import torch

import block_scaled_quantized_mx_gb300 as mx
import oracle
import workloads
from oracle import layout
from tests._parity import (check_epilogue_close, check_mx_output,
                           epilogue_tolerance, lib_quantize_to_oracle_form,
                           mx_quantize_both, nan_like, oracle_mx_product,
                           sample_rows, f16_bits)

pytestmark = pytest.mark.gpu

ACTS = [oracle.ACT_NONE, oracle.ACT_GELU, oracle.ACT_GELU_TANH]
PAIRS = [(oracle.E4M3, oracle.E4M3), (oracle.E2M1, oracle.E2M1),
         (oracle.E4M3, oracle.E2M1), (oracle.E5M2, oracle.E5M2)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    mx.build()
    mx.lib()


def _sources(M, N, K, seed):
    """Activations N(0,1) and weights N(0, 0.02^2 * 256 / K), so that the
    product is O(1) and GELU works in its curved region; bias N(0, 0.5^2)."""
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=g)
    B = torch.randn(K, N, generator=g) * (0.32 / np.sqrt(K))
    bias = torch.randn(N, generator=g) * 0.5
    return A, B, bias


def _odt(out):
    return torch.bfloat16 if out == "bf16" else torch.float32


@pytest.mark.parametrize("fa,fb", PAIRS)
@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("use_bias", [False, True])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(200, 296, 256), (384, 520, 1152)])
def test_fused_bias_act(fa, fb, act, use_bias, out, M, N, K):
    A, B, bias = _sources(M, N, K, seed=M + N + K + 10 * fa + fb)
    a, b = mx_quantize_both(A, B, fa, fb)
    C = nan_like((M, N), _odt(out))
    mx.mx_gemm_fused(a, b, bias.cuda() if use_bias else None, act,
                     out_dtype=_odt(out), out=C)
    assert mx.mx_last_error() == 0
    Cr, S = oracle_mx_product(A, B, fa, fb)
    check_epilogue_close(C.float().cpu().numpy(), Cr, S,
                         bias.numpy() if use_bias else None, act, out,
                         f"{fa}x{fb} act {act} bias {use_bias}")


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("act", ACTS)
def test_gemm_f16_fused(dt, act):
    M, N, K = 200, 264, 520
    tdt = torch.float16 if dt == "f16" else torch.bfloat16
    A, B, bias = _sources(M, N, K, seed=7 + act)
    A, B = A.to(tdt), B.to(tdt)
    C = nan_like((M, N), torch.float32)
    mx.gemm_f16_fused(A.cuda(), B.cuda(), bias.cuda(), act, out=C)
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_f16(f16_bits(A), f16_bits(B),
                            oracle.F16 if dt == "f16" else oracle.BF16)
    check_epilogue_close(C.cpu().numpy(), Cr, S, bias.numpy(), act, "f32",
                         f"{dt} act {act}")


def _quantized_pair(fa, fb, fq, act, M, N, K, seed, use_bias=True):
    A, B, bias = _sources(M, N, K, seed)
    a, b = mx_quantize_both(A, B, fa, fb)
    db = bias.cuda() if use_bias else None
    q = mx.mx_gemm_fused_quantize(a, b, fq, db, act)
    y = mx.mx_gemm_fused(a, b, db, act, out_dtype=torch.float32)
    assert mx.mx_last_error() == 0
    return A, B, bias, q, y


@pytest.mark.parametrize("fa,fb", PAIRS)
@pytest.mark.parametrize("fq", [oracle.E4M3, oracle.E5M2, oracle.E2M1])
@pytest.mark.parametrize("act", [oracle.ACT_NONE, oracle.ACT_GELU])
@pytest.mark.parametrize("M,N,K", [(200, 160, 256), (256, 512, 1024),
                                   (130, 288, 128)])
def test_fused_quantize_vs_oracle(fa, fb, fq, act, M, N, K):
    """Quantized output: allowed code intervals of the oracle, padding of
    the scale plane zero, and bit-identical to mx_quantize of the fused
    fp32 output."""
    A, B, bias, q, y = _quantized_pair(fa, fb, fq, act, M, N, K,
                                       seed=3 * M + N + K + fq)
    codes, scales = lib_quantize_to_oracle_form(q)
    Cr, S = oracle_mx_product(A, B, fa, fb)
    Y_ref = oracle.epilogue(Cr, bias.numpy(), act)
    tol = epilogue_tolerance(Cr, S, bias.numpy(), act, Y_ref)
    frac = check_mx_output(codes, scales, Y_ref, tol, fq,
                           f"{fa}x{fb} -> {fq} act {act}")
    assert frac > 0.5, f"only {frac:.2%} of the codes were decided"
    pad = layout.pad_positions(M, N)
    assert not q.scales.cpu().numpy()[pad].any(), "scale padding not zero"
    q2 = mx.mx_quantize(y, fq)
    assert torch.equal(q.data, q2.data), "data plane differs from two-step"
    assert torch.equal(q.scales, q2.scales), "scales differ from two-step"


@pytest.mark.parametrize("fq", [oracle.E4M3, oracle.E5M2, oracle.E2M1])
def test_fused_quantize_integers_exact(fq):
    """Integer operands and bias, no activation: y is an exact integer in
    fp32 on both sides, so the quantized planes must equal the oracle's
    quantization of the exact product, bit for bit."""
    g = np.random.default_rng(31)
    M, N, K = 256, 384, 512
    A = torch.from_numpy(g.integers(-14, 15, (M, K)).astype(np.float32))
    B = torch.from_numpy(g.integers(-14, 15, (K, N)).astype(np.float32))
    bias = torch.from_numpy(g.integers(-1000, 1000, N).astype(np.float32))
    a, b = mx_quantize_both(A, B, oracle.E4M3, oracle.E4M3)
    q = mx.mx_gemm_fused_quantize(a, b, fq, bias.cuda(), mx.ACT_NONE)
    assert mx.mx_last_error() == 0
    Y = (A.numpy().astype(np.int64) @ B.numpy().astype(np.int64)
         + bias.numpy().astype(np.int64)[None, :])
    assert np.abs(Y).max() < 2 ** 24
    cq, sq = oracle.quantize(Y.astype(np.float32), fq)
    codes, scales = lib_quantize_to_oracle_form(q)
    assert np.array_equal(scales, sq)
    assert np.array_equal(codes, cq)


@pytest.mark.parametrize("fq", [oracle.E4M3, oracle.E5M2])
def test_fused_quantize_into_16_byte_aligned_plane(fq):
    """An output data plane that starts 16 bytes past a 32-byte boundary:
    the epilogue's 32-byte store of each row's block falls back to two
    16-byte stores and writes the same bytes (integer operands, so the
    planes are exact), and nothing outside the plane."""
    g = np.random.default_rng(37 + fq)
    M, N, K = 256, 384, 512
    A = torch.from_numpy(g.integers(-14, 15, (M, K)).astype(np.float32))
    B = torch.from_numpy(g.integers(-14, 15, (K, N)).astype(np.float32))
    a, b = mx_quantize_both(A, B, oracle.E4M3, oracle.E4M3)
    nd, ns = mx.data_bytes(fq, M, N), mx.scale_bytes(M, N)
    buf = torch.zeros(nd + 32, dtype=torch.uint8, device="cuda")
    q = mx.MXTensor(buf[16:16 + nd],
                    torch.zeros(ns, dtype=torch.uint8, device="cuda"), fq,
                    M, N)
    assert q.data.data_ptr() % 32 == 16
    mx.mx_gemm_fused_quantize(a, b, fq, None, mx.ACT_NONE, out=q)
    assert mx.mx_last_error() == 0
    Y = A.numpy().astype(np.int64) @ B.numpy().astype(np.int64)
    assert np.abs(Y).max() < 2 ** 24
    cq, sq = oracle.quantize(Y.astype(np.float32), fq)
    codes, scales = lib_quantize_to_oracle_form(q)
    assert np.array_equal(scales, sq)
    assert np.array_equal(codes, cq)
    assert not buf[:16].any() and not buf[16 + nd:].any()


@pytest.mark.parametrize("name", ["proj_up", "w4a8_8192"])
def test_fused_workload_sampled(name):
    """Full-size workload, bias + GELU, quantized to E4M3 for the next
    layer: sampled rows vs the oracle, the whole output vs the two-step
    path."""
    c = workloads.case(name)
    fa, fb = workloads.formats(c)
    A, B = workloads.sources(c)
    bias = torch.randn(c.N, generator=torch.Generator().manual_seed(9)) * 0.5
    a, b = mx_quantize_both(A, B, fa, fb)
    db = bias.cuda()
    q = mx.mx_gemm_fused_quantize(a, b, oracle.E4M3, db, mx.ACT_GELU)
    y = mx.mx_gemm_fused(a, b, db, mx.ACT_GELU, out_dtype=torch.float32)
    assert mx.mx_last_error() == 0
    q2 = mx.mx_quantize(y, oracle.E4M3)
    assert torch.equal(q.data, q2.data) and torch.equal(q.scales, q2.scales)
    rows = sample_rows(c.M, n_random=8, seed=c.seed_a)
    Cr, S = oracle_mx_product(A, B, fa, fb, rows=rows)
    Y_ref = check_epilogue_close(y.cpu().numpy()[rows], Cr, S, bias.numpy(),
                                 oracle.ACT_GELU, "f32", name)[0]
    tol = epilogue_tolerance(Cr, S, bias.numpy(), oracle.ACT_GELU, Y_ref)
    codes, scales = lib_quantize_to_oracle_form(q)
    check_mx_output(codes[rows], scales[rows], Y_ref, tol, oracle.E4M3, name)


def test_fused_deterministic():
    A, B, bias = _sources(512, 512, 1024, seed=77)
    a, b = mx_quantize_both(A, B, oracle.E4M3, oracle.E2M1)
    db = bias.cuda()
    q1 = mx.mx_gemm_fused_quantize(a, b, oracle.E4M3, db, mx.ACT_GELU_TANH)
    q2 = mx.mx_gemm_fused_quantize(a, b, oracle.E4M3, db, mx.ACT_GELU_TANH)
    assert torch.equal(q1.data, q2.data) and torch.equal(q1.scales, q2.scales)
