"""mx_gemm_splitk_noalloc: the K-split MX GEMM whose scratch is a fixed
array inside the library, for callers that cannot allocate device memory
(operator interfaces that pass only operand and result pointers, processes
whose memory is all reserved by a framework allocator).

Called through the C ABI (ctypes), twice in a row on the same problems, its
output must
  * agree with the oracle's C element by element: |C - C_ref| <= 1e-4 * S,
    S = sum_k |a_ik b_kj| (plus one bf16 ulp of C_ref for bf16 output), the
    bound every GEMM test uses;
  * equal, bit for bit, mx_gemm_splitk's output given a caller workspace:
    the two run the same kernels with the same split and the same fixed
    reduction order, so any difference is a fault, not rounding.
This file is collected last on purpose."""
import ctypes

import pytest
import torch

import block_scaled_quantized_mx_gb300 as mx
import oracle
from tests._parity import check_close, nan_like

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,M,N,K,out", [
    (oracle.E4M3, 1024, 1024, 1024, torch.float32),
    (oracle.E2M1, 1000, 520, 1056, torch.bfloat16),
    (oracle.E4M3, 2304, 2304, 1024, torch.bfloat16)])
def test_noalloc_matches_workspace_entry_point(fmt, M, N, K, out):
    mx.build()
    L = mx.lib()
    # 128-wide tiles: the split applies to every shape with a partial wave
    mx.set_tile_width(128)
    try:
        _check(L, fmt, M, N, K, out)
    finally:
        mx.set_tile_width(0)


def _check(L, fmt, M, N, K, out):
    assert mx.mx_gemm_workspace_bytes(fmt, M, N, K) > 0   # the split applies
    g = torch.Generator().manual_seed(M + N + K)
    A = torch.randn(M, K, generator=g)
    B = torch.randn(K, N, generator=g)
    a = mx.mx_quantize(A.cuda(), fmt)
    b = mx.mx_quantize(B.cuda(), fmt, k_strided=True)

    ws = torch.empty(mx.mx_gemm_workspace_bytes(fmt, M, N, K),
                     dtype=torch.uint8, device="cuda")
    C_ws = mx.mx_gemm(a, b, out_dtype=out, workspace=ws)   # mx_gemm_splitk
    torch.cuda.synchronize()
    ca, sa = oracle.quantize(A.numpy(), fmt, k_axis=1)
    cb, sb = oracle.quantize(B.numpy(), fmt, k_axis=0)
    ref, S = oracle.gemm_mx(ca, sa, cb, sb, fmt)
    kind = "bf16" if out == torch.bfloat16 else "f32"
    check_close(C_ws.float().cpu().numpy(), ref, S, kind, "workspace entry point")

    ta, tb = a.c(), b.c()
    dt = mx.DT_BF16 if out == torch.bfloat16 else mx.DT_F32
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        C = nan_like((M, N), out)
        st = L.mx_gemm_splitk_noalloc(ctypes.byref(ta), ctypes.byref(tb),
                                      C.data_ptr(), dt, C.stride(0), stream)
        assert st == 0, mx.STATUS.get(st, st)
        torch.cuda.synchronize()
        assert mx.mx_last_error() == 0
        check_close(C.float().cpu().numpy(), ref, S, kind,
                    f"no-alloc call {call}")
        assert torch.equal(C.view(torch.int16) if out == torch.bfloat16
                           else C.view(torch.int32),
                           C_ws.view(torch.int16) if out == torch.bfloat16
                           else C_ws.view(torch.int32)), \
            f"no-alloc call {call} differs in bits from mx_gemm_splitk"


def test_noalloc_rejects_bad_arguments():
    L = mx.lib()
    assert L.mx_gemm_splitk_noalloc(None, None, None, 0, 0, None) == 1
