"""gemm_dequant for decode shapes (M <= 128 tokens) on the GPU vs the oracle.

These products run the weights-as-M kernel: C^T = dequant(B) A^T with the
128-row weight blocks as the MMA's M, the tokens (padded to 64 or 128) as
its N, the weights dequantized into tensor memory 256 K at a time.  Checked
against the float64 oracle (oracle.gemm_a16_bmx) element by element with
the bound every GEMM test uses, |C - C_ref| <= 1e-4 * S (+ one bf16 ulp of
C_ref for bf16 output): every element format; token counts at the padding
edges (1, 17, 64, 65, 128); ragged N; K from one 64-K step to many, with
and without a partial last 256-K quad; each cluster size the kernel picks
(a weight block's K range split over S = 2, 4 or 8 CTAs whose partial
accumulators are summed in rank order through distributed shared memory,
or S = 1 with whole blocks per CTA, several per CTA when there are more
blocks than SMs); the fused bias + GELU epilogue; padded ldc; and run-to-run
bitwise determinism.  The kernel takes no workspace: a workspace passed in
is ignored.  Every output starts as NaN."""
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


def _inputs(M, N, K, fmt, a_dt, seed):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=g).to(a_dt)
    cb, sb = workloads.random_codes((N, K), fmt, seed=seed + 1, scale_lo=116,
                                    scale_hi=127)
    return A, cb, sb, planes_from_codes(cb, sb, fmt)


def _ws(M, N, K):
    """A workspace of garbage, as a caller of the split entry point would
    pass one; the decode kernel needs none (0 bytes) and must not touch it."""
    assert mx.gemm_dequant_workspace_bytes(M, N, K) == 0
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    ws.fill_(0xA5)
    return ws


@pytest.mark.parametrize("fmt", ALL_FMTS)
@pytest.mark.parametrize("M,N,K", [(1, 1000, 1024), (17, 384, 4160),
                                   (64, 2048, 2048), (65, 520, 640),
                                   (128, 256, 64)])
@pytest.mark.parametrize("split", [True, False])
def test_decode_formats(fmt, M, N, K, split):
    A, cb, sb, b = _inputs(M, N, K, fmt, torch.bfloat16, M * 7 + N + K + fmt)
    C = nan_like((M, N), torch.float32)
    mx.gemm_dequant(A.cuda(), b, out_dtype=torch.float32, out=C,
                    workspace=_ws(M, N, K) if split else None)
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    check_close(C.cpu().numpy(), Cr, S, "f32",
                f"decode fmt{fmt} {M}x{N}x{K} split={split}")


@pytest.mark.parametrize("a,out", [("f16", "bf16"), ("bf16", "bf16"),
                                   ("f16", "f32")])
def test_decode_dtypes(a, out):
    M, N, K, fmt = 48, 768, 2048, oracle.INT4
    adt = torch.float16 if a == "f16" else torch.bfloat16
    odt = torch.bfloat16 if out == "bf16" else torch.float32
    A, cb, sb, b = _inputs(M, N, K, fmt, adt, 99)
    C = nan_like((M, N), odt)
    mx.gemm_dequant(A.cuda(), b, out_dtype=odt, out=C, workspace=_ws(M, N, K))
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.F16 if a == "f16" else oracle.BF16,
                                cb, sb, fmt)
    check_close(C.float().cpu().numpy(), Cr, S, out, f"decode {a} -> {out}")


@pytest.mark.parametrize("act", [mx.ACT_GELU, mx.ACT_GELU_TANH])
@pytest.mark.parametrize("split", [True, False])
def test_decode_fused_epilogue(act, split):
    M, N, K, fmt = 32, 1280, 2048, oracle.INT4
    A, cb, sb, b = _inputs(M, N, K, fmt, torch.bfloat16, 7 + act)
    bias = torch.randn(N, generator=torch.Generator().manual_seed(3)) * 0.5
    C = nan_like((M, N), torch.bfloat16)
    mx.gemm_dequant(A.cuda(), b, bias=bias.cuda(), act=act,
                    out_dtype=torch.bfloat16, out=C,
                    workspace=_ws(M, N, K) if split else None)
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    check_epilogue_close(C.float().cpu().numpy(), Cr, S,
                         bias.numpy().astype(np.float64), act, "bf16",
                         f"decode act {act} split={split}")


def test_decode_padded_ldc_and_determinism():
    """C inside a wider buffer (nothing outside it written); two runs give
    the same bits (a cluster's parts are summed in rank order)."""
    M, N, K, fmt = 64, 1000, 4096, oracle.INT4
    A, cb, sb, b = _inputs(M, N, K, fmt, torch.bfloat16, 5)
    ws = _ws(M, N, K)
    big = nan_like((M, 1032), torch.float32)
    C = big[:, 8:8 + N]
    mx.gemm_dequant(A.cuda(), b, out_dtype=torch.float32, out=C, workspace=ws)
    first = C.clone()
    mx.gemm_dequant(A.cuda(), b, out_dtype=torch.float32, out=C, workspace=ws)
    assert mx.mx_last_error() == 0
    assert torch.equal(first, C)
    assert torch.isnan(big[:, :8]).all() and torch.isnan(big[:, 8 + N:]).all()
    Cr, S = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    check_close(C.cpu().numpy(), Cr, S, "f32", "decode padded ldc")


def _cluster_size(N, K, sms):
    """The cluster size the kernel picks (mirrors dqd_cluster): the largest
    power of two up to 8 with nbk * S <= SMs and S <= quads per block; 1
    once the weight blocks alone fill half the SMs."""
    nbk, kq = -(-N // 128), -(-(K // 64) // 4)
    if 2 * nbk > sms:
        return 1
    S = 1
    while 2 * S <= 8 and nbk * 2 * S <= sms and 2 * S <= kq:
        S *= 2
    return S


@pytest.mark.parametrize("M,N,K,S", [(1, 128 * 9, 2048, 8),      # 9 blocks
                                     (33, 128 * 30, 1024, 4),    # 30 blocks
                                     (64, 128 * 64, 1216, 2),    # 64 blocks, last quad 3 steps
                                     (128, 128 * 50, 768, 2),    # NT = 128
                                     (5, 128 * 200, 512, 1),     # 200 blocks: some CTAs take two
                                     (100, 128 * 200, 256, 1),   # the same with NT = 128
                                     (128, 128 * 100, 512, 1),   # NT = 128, one block per CTA
                                     (64, 128 * 20, 256, 1)])    # one quad: no split
def test_decode_cluster_sizes(M, N, K, S):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert _cluster_size(N, K, sms) == S or sms != 152
    fmt = oracle.INT4
    A, cb, sb, b = _inputs(M, N, K, fmt, torch.bfloat16, N + K)
    C = nan_like((M, N), torch.bfloat16)
    mx.gemm_dequant(A.cuda(), b, out_dtype=torch.bfloat16, out=C)
    assert mx.mx_last_error() == 0
    Cr, Sc = oracle.gemm_a16_bmx(f16_bits(A), oracle.BF16, cb, sb, fmt)
    check_close(C.float().cpu().numpy(), Cr, Sc, "bf16", f"decode S={S} {M}x{N}x{K}")
