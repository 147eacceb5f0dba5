"""The algorithmic work bench.py divides by (roofline `achieved`, GB/s and
TFLOP/s figures), against counts written out by hand from the shapes: a
miscount here would scale every reported fraction."""
import pytest

import bench
import workloads


def test_gemm_flops():
    assert bench.flops_of(workloads.case("mxfp8_8192")) == 2 * 8192 ** 3
    c = workloads.case("proj_up")
    assert bench.flops_of(c) == 2 * 16384 * 8192 * 2048


@pytest.mark.parametrize("fmt,per_elem", [(1, 5.03125), (3, 5.03125),
                                          (2, 4.53125)])
def test_quantize_bytes_per_element(fmt, per_elem):
    # fp32 read (4 B) + one code (1 B, or half a byte for E2M1) + one scale
    # byte per 32 elements
    assert bench.quant_bytes(fmt, 8192, 8192) == per_elem * 8192 * 8192


def test_dequant_bytes_decode_shapes():
    # 64 x 8192 x 8192, int4 weights, bf16 A and C:
    # A 2*64*8192 + codes 8192*8192/2 + scales 8192*8192/32 + C 2*64*8192
    c = workloads.case("w4a16_decode")
    assert bench.dequant_bytes(c) == (2 * 64 * 8192 + 8192 * 8192 // 2 +
                                      8192 * 8192 // 32 + 2 * 64 * 8192)
    assert bench.dequant_bytes(c) == 37748736
    # one token
    c1 = workloads.case("w4a16_decode_m1")
    assert (c1.M, c1.N, c1.K) == (1, 8192, 8192)
    assert bench.dequant_bytes(c1) == 35684352
    # int2 weights: a quarter byte per element
    c2 = workloads.case("w2a16_8192")
    assert bench.dequant_bytes(c2) == (2 * 8192 * 8192 + 8192 * 8192 // 4 +
                                       8192 * 8192 // 32 + 2 * 8192 * 8192)
