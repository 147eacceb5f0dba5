"""Failure detection on the GPU without faulting it: a kernel whose bounded
wait runs out (an mbarrier nothing arrives at) must return cleanly and report
MX_ERR_TIMEOUT through mx_last_error, after which the context is still usable
and the status is clear again."""
import pytest
import torch

import block_scaled_quantized_mx_gb300 as mx

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    mx.build()
    assert mx.mx_last_error() == 0
    # about half a millisecond of SM clock
    assert mx.mx_selftest_wait_timeout(1_000_000) == 0
    assert mx.mx_last_error() == 6          # MX_ERR_TIMEOUT
    assert mx.mx_last_error() == 0          # cleared by the read
    x = torch.randn(128, 128, device="cuda")
    q = mx.mx_quantize(x, mx.E4M3)
    C = mx.mx_gemm(q, mx.mx_quantize(x, mx.E4M3, k_strided=True),
                   out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert mx.mx_last_error() == 0
    assert torch.isfinite(C).all()


def test_errors_raise_in_binding():
    x = torch.randn(128, 100, device="cuda")       # K not a multiple of 32
    with pytest.raises(mx.MXError) as e:
        mx.mx_quantize(x, mx.E4M3)
    assert e.value.status == 2
