"""The C ABI without a GPU: the library loads, exports every function that
include/mx.h declares, rejects bad arguments on the host before any launch,
and its host-side helpers agree with the oracle's independent restatement of
the memory layouts."""
import ctypes
import os
import re

import numpy as np
import pytest

import block_scaled_quantized_mx_gb300 as mx
from oracle import layout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mx.h")


@pytest.fixture(scope="module")
def L():
    mx.build()
    return mx.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:[\w\s\*]+?)\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_exports_every_declared_function(L):
    names = _declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(mx.EXPORTS)


def test_status_strings_and_version(L):
    for code, name in mx.STATUS.items():
        assert L.mx_status_string(code).decode() == name
    assert L.mx_status_string(99).decode() == "MX_ERR_UNKNOWN"
    assert L.mx_version() >= 100


@pytest.mark.parametrize("outer,K", [(0, 0), (1, 32), (128, 128), (300, 160),
                                     (8192, 8192), (16384, 2048)])
def test_plane_sizes(L, outer, K):
    assert mx.data_bytes(mx.E4M3, outer, K) == outer * K
    assert mx.data_bytes(mx.E5M2, outer, K) == outer * K
    assert mx.data_bytes(mx.INT8, outer, K) == outer * K
    assert mx.data_bytes(mx.INT4, outer, K) == outer * K // 2
    assert mx.data_bytes(mx.INT2, outer, K) == outer * K // 4
    for f in (mx.E4M3, mx.E5M2, mx.E2M1, mx.INT8, mx.INT4, mx.INT2):
        assert mx.data_bytes(f, outer, K) == layout.data_plane_bytes(f, outer, K)
    assert mx.data_bytes(mx.E2M1, outer, K) == outer * K // 2
    assert mx.scale_bytes(outer, K) == layout.scale_plane_bytes(outer, K)


def test_plane_sizes_reject_bad(L):
    assert mx.data_bytes(mx.E4M3, 4, 33) == 0
    assert mx.data_bytes(7, 4, 32) == 0
    assert mx.scale_bytes(-1, 32) == 0


@pytest.mark.parametrize("outer,K", [(128, 128), (200, 96), (1, 32),
                                     (300, 544)])
def test_scales_to_rowmajor_matches_oracle_layout(L, outer, K):
    g = np.random.default_rng(outer * 7 + K)
    s = g.integers(0, 255, (outer, K // 32)).astype(np.uint8)
    tiled = layout.tile_scales(s, K)
    assert np.array_equal(mx.scales_to_rowmajor(tiled, outer, K), s)


def _t(fmt=mx.E4M3, outer=128, K=128, data=0x1000, scales=0x2000):
    return mx.CMXTensor(data, scales, fmt, outer, K)


def test_host_validation_without_launch(L):
    P = 0x10000            # never dereferenced: every call fails its checks
    byref = ctypes.byref
    ep = lambda bias=None, act=0: byref(mx.CEpilogue(bias, act))  # noqa
    # mx_quantize
    assert L.mx_quantize(P, 128, 0, None, None) == 1
    assert L.mx_quantize(P, 128, 0, byref(_t(fmt=7)), None) == 1
    assert L.mx_quantize(P, 128, 0, byref(_t(fmt=0)), None) == 1
    assert L.mx_quantize(P, 128, 5, byref(_t()), None) == 1
    assert L.mx_quantize(None, 128, 0, byref(_t()), None) == 1
    assert L.mx_quantize(P, 128, 0, byref(_t(K=100)), None) == 2
    assert L.mx_quantize(P, 64, 0, byref(_t()), None) == 2       # ld < K
    assert L.mx_quantize(P, 130, 0, byref(_t()), None) == 2      # ld % 4
    assert L.mx_quantize(P + 4, 128, 0, byref(_t()), None) == 3
    assert L.mx_quantize(P, 128, 0, byref(_t(data=0x1001)), None) == 3
    assert L.mx_quantize(P, 128, 0, byref(_t(scales=None)), None) == 1
    assert L.mx_quantize(P, 128, 0, byref(_t(outer=-1)), None) == 2
    # empty problems are a no-op success, with no launch
    assert L.mx_quantize(None, 0, 0, byref(_t(outer=0)), None) == 0
    assert L.mx_quantize(None, 0, 0, byref(_t(K=0, data=None,
                                                 scales=None)), None) == 0
    # mx_gemm
    a, b = _t(), _t(outer=256)
    assert L.mx_gemm(None, byref(b), P, 1, 256, None) == 1
    # an E2M1 operand beside an 8-bit one: K % 128 and a 32-byte aligned
    # E2M1 plane (TMA unpacks it); either order, E4M3 or E5M2
    for f8 in (mx.E4M3, mx.E5M2):
        for fa, fb in ((f8, mx.E2M1), (mx.E2M1, f8)):
            assert L.mx_gemm(byref(_t(fmt=fa, K=96)),
                             byref(_t(fmt=fb, outer=256, K=96)), P, 1, 256,
                             None) == 2
            bad = dict(data=0x1010)
            ta = _t(fmt=fa, **(bad if fa == mx.E2M1 else {}))
            tb = _t(fmt=fb, outer=256, **(bad if fb == mx.E2M1 else {}))
            assert L.mx_gemm(byref(ta), byref(tb), P, 1, 256, None) == 3
            assert L.mx_gemm_splitk(byref(ta), byref(tb), P, 1, 256, None, 0,
                                    None) == 3
    assert L.mx_gemm(byref(_t(fmt=7)), byref(b), P, 1, 256, None) == 1
    # integer tensors are gemm_dequant's B operand only
    for fi in (mx.INT8, mx.INT4, mx.INT2):
        assert L.mx_gemm(byref(_t(fmt=fi)), byref(b), P, 1, 256, None) == 1
        assert L.mx_gemm(byref(a), byref(_t(fmt=fi, outer=256)), P, 1, 256,
                         None) == 1
        assert L.mx_gemm_fused_quantize(byref(a), byref(b), None,
                                        byref(_t(fmt=fi, outer=128, K=256)),
                                        None) == 1
    # gemm_dequant
    bq = _t(fmt=mx.INT4, outer=256, K=128)
    assert L.gemm_dequant(P, 0, 128, 128, byref(bq), None, P, 0, 256,
                          None) == 1                          # a_dtype f32
    assert L.gemm_dequant(P, 1, 128, 128, byref(bq), None, P, 2, 256,
                          None) == 1                          # c_dtype f16
    assert L.gemm_dequant(P, 1, 128, 128, byref(_t(fmt=7, outer=256)), None,
                          P, 0, 256, None) == 1
    assert L.gemm_dequant(P, 1, 128, 96, byref(_t(fmt=mx.INT4, outer=256,
                                                   K=96)), None, P, 0, 256,
                          None) == 2                          # K % 64
    assert L.gemm_dequant(P, 1, 128, 100, byref(bq), None, P, 0, 256,
                          None) == 2                          # lda % 8
    assert L.gemm_dequant(P, 1, 128, 64, byref(bq), None, P, 0, 256,
                          None) == 2                          # lda < K
    assert L.gemm_dequant(P, 1, 128, 128, byref(bq), None, P, 0, 200,
                          None) == 2                          # ldc < N
    assert L.gemm_dequant(P + 8, 1, 128, 128, byref(bq), None, P, 0, 256,
                          None) == 3
    assert L.gemm_dequant(P, 1, 128, 128, byref(bq), None, P + 4, 0, 256,
                          None) == 3
    assert L.gemm_dequant(None, 1, 128, 128, byref(bq), None, P, 0, 256,
                          None) == 1
    assert L.gemm_dequant(P, 1, -1, 128, byref(bq), None, P, 0, 256,
                          None) == 2
    assert L.gemm_dequant(None, 1, 0, 128, byref(bq), None, None, 0, 256,
                          None) == 0                          # M = 0
    assert L.gemm_dequant(P, 1, 128, 128, byref(bq), ep(act=9), P, 0, 256,
                          None) == 1
    assert L.mx_gemm(byref(a), byref(_t(outer=256, K=256)), P, 1, 256,
                     None) == 2
    assert L.mx_gemm(byref(a), byref(b), P, 2, 256, None) == 1   # f16 out
    assert L.mx_gemm(byref(a), byref(b), None, 1, 256, None) == 1
    assert L.mx_gemm(byref(a), byref(b), P, 1, 200, None) == 2   # ldc < N
    assert L.mx_gemm(byref(a), byref(b), P, 1, 260, None) == 2   # ldc*2 % 16
    assert L.mx_gemm(byref(a), byref(b), P + 8, 1, 256, None) == 3
    assert L.mx_gemm(byref(_t(outer=0)), byref(b), None, 1, 256, None) == 0
    # fused epilogue
    assert L.mx_gemm_fused(byref(a), byref(b), ep(act=3), P, 1, 256,
                           None) == 1
    assert L.mx_gemm_fused(byref(a), byref(b), ep(act=-1), P, 1, 256,
                           None) == 1
    assert L.mx_gemm_fused(byref(a), byref(b), ep(bias=P + 4), P, 1, 256,
                           None) == 3
    assert L.mx_gemm_fused(byref(_t(K=0, data=None, scales=None)),
                           byref(_t(outer=256, K=0, data=None, scales=None)),
                           ep(act=1), P, 1, 256, None) == 2
    cq = _t(outer=128, K=256)                       # M x N output tensor
    assert L.mx_gemm_fused_quantize(byref(a), byref(b), None, None,
                                    None) == 1
    assert L.mx_gemm_fused_quantize(byref(a), byref(b), None,
                                    byref(_t(outer=64, K=256)), None) == 2
    assert L.mx_gemm_fused_quantize(byref(a), byref(b), None,
                                    byref(_t(outer=128, K=224)), None) == 2
    assert L.mx_gemm_fused_quantize(byref(a), byref(b), None,
                                    byref(_t(fmt=9, outer=128, K=256)),
                                    None) == 1
    assert L.mx_gemm_fused_quantize(byref(a), byref(b), ep(act=4),
                                    byref(cq), None) == 1
    assert L.mx_gemm_fused_quantize(byref(a), byref(b), None,
                                    byref(_t(outer=128, K=256, data=0x1008)),
                                    None) == 3
    assert L.mx_gemm_fused_quantize(
        byref(_t(K=0, data=None, scales=None)),
        byref(_t(outer=256, K=0, data=None, scales=None)), None,
        byref(cq), None) == 2
    assert L.gemm_f16_fused(P, P, ep(act=7), P, 2, 128, 128, 128, 128, 128,
                            128, None) == 1
    assert L.gemm_f16_fused(P, P, ep(bias=P + 8), P, 2, 128, 128, 128, 128,
                            128, 128, None) == 3
    assert L.gemm_f16_fused(P, P, ep(act=1), P, 2, 128, 128, 0, 128, 128,
                            128, None) == 2
    # flash_attention
    fa = L.flash_attention
    assert fa(P, P, P, P, 0, 0, 2, 128, 128, 64, 0.125, None) == 1      # f32 in
    assert fa(P, P, P, P, 1, 5, 2, 128, 128, 64, 0.125, None) == 1      # o_dtype
    assert fa(P, P, P, P, 1, 0, 2, 128, 128, 96, 0.125, None) == 2      # d
    assert fa(P, P, P, P, 1, 0, 2, 128, 0, 64, 0.125, None) == 2        # Lk = 0
    assert fa(P, P, P, P, 1, 0, 70000, 128, 128, 64, 0.125, None) == 2  # BH
    assert fa(P, P, P, P, 1, 0, -1, 128, 128, 64, 0.125, None) == 2
    assert fa(P, P, P, P, 1, 0, 2, 128, 128, 64, float("nan"), None) == 1
    assert fa(P, P, P, P, 1, 0, 2, 128, 128, 64, float("inf"), None) == 1
    assert fa(P + 8, P, P, P, 1, 0, 2, 128, 128, 64, 0.125, None) == 3
    assert fa(P, P, P, P + 2, 1, 0, 2, 128, 128, 64, 0.125, None) == 3
    assert fa(None, P, P, P, 1, 0, 2, 128, 128, 64, 0.125, None) == 1
    assert fa(None, None, None, None, 1, 0, 0, 128, 128, 64, 0.125, None) == 0
    assert fa(None, None, None, None, 1, 0, 2, 0, 128, 64, 0.125, None) == 0
    # gemm_f16
    assert L.gemm_f16(P, P, P, 0, 128, 128, 128, 128, 128, 128, None) == 1
    assert L.gemm_f16(P, P, P, 2, -1, 128, 128, 128, 128, 128, None) == 2
    assert L.gemm_f16(P, P, P, 2, 128, 128, 128, 100, 128, 128, None) == 2
    assert L.gemm_f16(P, P, P, 2, 128, 128, 128, 132, 128, 128, None) == 2
    assert L.gemm_f16(P, P, P, 2, 128, 128, 128, 128, 128, 126, None) == 2
    assert L.gemm_f16(P + 2, P, P, 2, 128, 128, 128, 128, 128, 128,
                      None) == 3
    assert L.gemm_f16(None, P, P, 1, 128, 128, 128, 128, 128, 128,
                      None) == 1
    assert L.gemm_f16(None, None, None, 1, 0, 128, 128, 128, 128, 128,
                      None) == 0
    # self test bound
    assert L.mx_selftest_wait_timeout(0, None) == 1


def test_binding_checks_planes_before_any_launch(L):
    """The C ABI receives bare pointers, so the binding checks that an MX
    tensor's planes hold the bytes its format and shape need, and raises
    before any compute entry point is called (these tensors live on the
    host: a call that got through would fail in the library instead)."""
    import torch
    good = mx.empty_mx(mx.E4M3, 256, 256, device="cpu")
    short = mx.MXTensor(good.data[:-1], good.scales, mx.E4M3, 256, 256)
    few_scales = mx.MXTensor(good.data, good.scales[:-16], mx.E4M3, 256, 256)
    as_e2m1 = mx.empty_mx(mx.E2M1, 256, 256, device="cpu")
    as_e4m3 = mx.MXTensor(as_e2m1.data, as_e2m1.scales, mx.E4M3, 256, 256)
    strided = mx.MXTensor(torch.empty(2 * good.data.numel(), dtype=torch.uint8)[::2],
                          good.scales, mx.E4M3, 256, 256)
    for bad in (short, few_scales, as_e4m3, strided):
        with pytest.raises(ValueError):
            mx.mx_gemm(bad, good)
        with pytest.raises(ValueError):
            mx.mx_gemm(good, bad)
        with pytest.raises(ValueError):
            mx.mx_gemm_fused(bad, good)
        with pytest.raises(ValueError):
            mx.gemm_dequant(torch.empty(256, 256, dtype=torch.bfloat16), bad)
    # an output MX tensor of another format than asked for
    with pytest.raises(ValueError):
        mx.mx_gemm_fused_quantize(good, good, mx.E2M1, out=good)
    # an output type the call does not produce
    for call in (lambda: mx.mx_gemm(good, good, out_dtype=torch.float16),
                 lambda: mx.mx_gemm_fused(good, good, out_dtype=torch.int8),
                 lambda: mx.gemm_dequant(
                     torch.empty(256, 256, dtype=torch.bfloat16), good,
                     out_dtype=torch.float16)):
        with pytest.raises(ValueError):
            call()


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(mx, "_lib", None)
    monkeypatch.setattr(mx._build, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        mx.lib()
