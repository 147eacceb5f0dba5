"""Pins for the CPU oracle (no GPU needed).

Each test ties the oracle to something other than its own formulas: a library
decoder (torch's float8 types, numpy's float16), hand-derived values, values
the pages print (tests/golden/), exact integer arithmetic, or brute force in
exact rationals.  Together they are meant to fail on a plausible mistake in
any part of the oracle: a wrong bias or field width, a rounding or saturation
slip, a wrong block or scale index, a dropped term, a transposed operand.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import layout

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()
            out[k] = float(v)
    return out


def _torch_e4m3_table():
    u = torch.arange(256, dtype=torch.uint8)
    return u.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_e5m2_table():
    u = torch.arange(256, dtype=torch.uint8)
    return u.view(torch.float8_e5m2).to(torch.float64).numpy()


def _e5m2_finite_code(c):
    return (c & 0x7F) < 0x7C


# Magnitudes of E2M1 codes 0..7 as listed in the OCP MX v1.0 format table.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# ---------------------------------------------------------------- decoding

def test_e4m3_decode_all_codes_match_torch():
    ref = _torch_e4m3_table()
    ours = oracle.decode_table(oracle.E4M3)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])
    # signs of zero agree too
    assert math.copysign(1.0, ours[0x80]) == -1.0
    assert math.copysign(1.0, ours[0x00]) == 1.0


def test_e4m3_landmarks():
    assert oracle.decode_e4m3(0x7E) == 448.0          # largest finite
    assert math.isnan(oracle.decode_e4m3(0x7F))
    assert math.isnan(oracle.decode_e4m3(0xFF))
    assert oracle.decode_e4m3(0x01) == 2.0 ** -9       # smallest subnormal
    assert oracle.decode_e4m3(0x08) == 2.0 ** -6       # smallest normal
    assert oracle.decode_e4m3(0x38) == 1.0
    assert oracle.decode_e4m3(0xB8) == -1.0
    finite = [oracle.decode_e4m3(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(finite, finite[1:]))   # monotone
    assert len(set(finite)) == 127


def test_e5m2_decode_all_codes_match_torch():
    ref = _torch_e5m2_table()
    ours = oracle.decode_table(oracle.E5M2)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])        # +-Inf included
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_e5m2_landmarks():
    assert oracle.decode_e5m2(0x7B) == 57344.0         # 1.75 * 2^15
    assert oracle.decode_e5m2(0x7C) == math.inf
    assert oracle.decode_e5m2(0xFC) == -math.inf
    for c in (0x7D, 0x7E, 0x7F, 0xFF):
        assert math.isnan(oracle.decode_e5m2(c))
    assert oracle.decode_e5m2(0x01) == 2.0 ** -16      # smallest subnormal
    assert oracle.decode_e5m2(0x03) == 0.75 * 2.0 ** -14
    assert oracle.decode_e5m2(0x04) == 2.0 ** -14      # smallest normal
    assert oracle.decode_e5m2(0x3C) == 1.0
    assert oracle.decode_e5m2(0xBE) == -1.5


def test_e2m1_decode_table():
    for c in range(16):
        mag = E2M1_MAGNITUDES[c & 7]
        v = oracle.decode_e2m1(c)
        assert abs(v) == mag
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)


def test_ue8m0_decode_all_codes_match_torch():
    u = torch.arange(256, dtype=torch.uint8)
    ref = u.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.decode_ue8m0(c)
        if c == 255:
            assert math.isnan(v) and math.isnan(ref[c])
        else:
            assert v == ref[c] == 2.0 ** (c - 127)


def test_f16_bf16_decode_match_libraries():
    bits = np.arange(65536, dtype=np.uint16)
    f16 = bits.view(np.float16).astype(np.float64)
    bf16 = torch.from_numpy(bits.view(np.int16).copy()).view(
        torch.bfloat16).to(torch.float64).numpy()
    rng = np.random.default_rng(5)
    for b in np.concatenate([rng.integers(0, 65536, 3000),
                             [0, 1, 0x3C00, 0x7BFF, 0x8000, 0x0400, 0x7F7F,
                              0x0080, 0x3F80, 0xFF7F]]):
        b = int(b)
        for ours, ref in ((oracle.decode_f16(b), f16[b]),
                          (oracle.decode_bf16(b), bf16[b])):
            if math.isnan(ref):
                assert math.isnan(ours)
            else:
                assert ours == ref


# ---------------------------------------------------------------- encoding

def test_encode_e4m3_matches_torch_inside_range():
    table = _torch_e4m3_table()
    finite = np.sort(table[:0x7F])
    mids = (finite[:-1] + finite[1:]) / 2          # exact ties
    rng = np.random.default_rng(11)
    rand = rng.uniform(-460, 460, 20000)
    small = rng.uniform(-0.02, 0.02, 5000)
    vals = np.concatenate([finite, -finite, mids, -mids, rand, small,
                           mids * (1 + 2 ** -40), mids * (1 - 2 ** -40)])
    vals = vals[np.abs(vals) < 464]                # torch turns >= 464 to NaN
    vals = vals.astype(np.float32)                 # both sides see fp32
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()
    ours = np.array([oracle.encode_e4m3(float(v)) for v in vals],
                    dtype=np.uint8)
    assert np.array_equal(ours, ref)


def test_encode_e4m3_saturates_golden():
    with open(os.path.join(GOLDEN, "e4m3_saturation.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and ln[0] != "#"]
    for v, code in rows:
        assert oracle.encode_e4m3(float(v)) == int(code, 16), v


def test_encode_e4m3_roundtrip_and_signed_zero():
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert oracle.encode_e4m3(oracle.decode_e4m3(c)) == c
    assert oracle.encode_e4m3(-1e-30) == 0x80
    assert oracle.encode_e4m3(1e-30) == 0x00
    # half of the smallest subnormal is a tie between 0 and 2^-9 -> even (0)
    assert oracle.encode_e4m3(2.0 ** -10) == 0x00
    assert oracle.encode_e4m3(3 * 2.0 ** -10) == 0x02   # tie 1 vs 2 -> 2


def test_encode_e5m2_matches_torch_inside_range():
    table = _torch_e5m2_table()
    finite = np.sort(table[:0x7C])
    mids = (finite[:-1] + finite[1:]) / 2
    rng = np.random.default_rng(12)
    vals = np.concatenate([finite, -finite, mids, -mids,
                           rng.uniform(-61000, 61000, 20000),
                           rng.uniform(-2e-4, 2e-4, 5000),
                           mids * (1 + 2 ** -40), mids * (1 - 2 ** -40)])
    vals = vals[np.abs(vals) < 61440]              # torch turns >= 61440 to Inf
    vals = vals.astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e5m2).view(
        torch.uint8).numpy()
    ours = np.array([oracle.encode_e5m2(float(v)) for v in vals],
                    dtype=np.uint8)
    assert np.array_equal(ours, ref)


def test_encode_e5m2_saturates_and_roundtrips():
    # Beyond the range an MX element saturates instead of becoming Inf.
    for v, code in ((61440.0, 0x7B), (1e9, 0x7B), (math.inf, 0x7B),
                    (-65536.0, 0xFB), (57344.0, 0x7B),
                    (53248.0, 0x7A),                 # tie 1.5|1.75 -> even
                    (55296.0, 0x7B), (50000.0, 0x7A)):
        assert oracle.encode_e5m2(v) == code, v
    for c in range(256):
        if _e5m2_finite_code(c):
            assert oracle.encode_e5m2(oracle.decode_e5m2(c)) == c
    assert oracle.encode_e5m2(2.0 ** -17) == 0x00    # tie 0 | 2^-16 -> even
    assert oracle.encode_e5m2(3 * 2.0 ** -17) == 0x02


def test_encode_array_matches_scalar_encoders():
    g = np.random.default_rng(13)
    v = np.concatenate([g.standard_normal(3000) * 100, [0.0, -0.0, 1e9,
                                                          -1e9, 2.0 ** -20]])
    for fmt, enc in ((oracle.E4M3, oracle.encode_e4m3),
                     (oracle.E5M2, oracle.encode_e5m2),
                     (oracle.E2M1, oracle.encode_e2m1)):
        got = oracle.encode_array(v.reshape(-1, 5), fmt)
        assert got.shape == (len(v) // 5, 5)
        assert np.array_equal(got.reshape(-1),
                              np.array([enc(x) for x in v], dtype=np.uint8))


def test_encode_e2m1_hand_values():
    cases = {6.9: 0x7, 100.0: 0x7, 0.25: 0x0, 0.75: 0x2, 2.5: 0x4,
             5.0: 0x6, 1.25: 0x2, 1.75: 0x4, 3.5: 0x6, 0.2: 0x0,
             0.3: 0x1, 4.9: 0x6, 5.1: 0x7, -0.1: 0x8, -6.0: 0xF,
             -2.6: 0xD}
    for v, code in cases.items():
        assert oracle.encode_e2m1(v) == code, v


def test_encode_nearest_by_brute_force():
    """Chosen code is the nearest representable value (ties to even code),
    checked by scanning every code through the torch / hand tables."""
    rng = np.random.default_rng(3)
    t8 = _torch_e4m3_table()[:0x7F]
    t5 = _torch_e5m2_table()[:0x7C]
    t4 = np.array(E2M1_MAGNITUDES)
    for table, enc, vmax in ((t8, oracle.encode_e4m3, 448.0),
                             (t5, oracle.encode_e5m2, 57344.0),
                             (t4, oracle.encode_e2m1, 6.0)):
        for v in np.concatenate([rng.uniform(0, vmax * 1.1, 3000),
                                 rng.uniform(0, vmax / 64, 1000)]):
            d = np.abs(table - v)
            best = np.flatnonzero(d == d.min())
            want = best[0] if len(best) == 1 else [b for b in best
                                                    if b % 2 == 0][0]
            if v > vmax:
                want = len(table) - 1
            assert enc(float(v)) == want, v


# ---------------------------------------------------------------- scale rule

def _qblock(vals, fmt):
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, :len(vals)] = vals
    codes, scales = oracle.quantize(x, fmt)
    return codes[0], int(scales[0, 0])


def test_scale_rule_hand_values():
    assert _qblock([1.0], oracle.E4M3)[1] == 119       # 2^(0-8)
    assert _qblock([1.0], oracle.E2M1)[1] == 125       # 2^(0-2)
    assert _qblock([-1.0, 0.5], oracle.E4M3)[1] == 119
    just_below = float(np.float32(256.0) - np.float32(2.0 ** -16))
    assert _qblock([just_below], oracle.E4M3)[1] == 126  # floor(log2) = 7
    assert _qblock([256.0], oracle.E4M3)[1] == 127
    codes, s = _qblock([0.0], oracle.E4M3)
    assert s == 0 and not codes.any()                   # all-zero block
    codes, s = _qblock([-0.0, 0.0], oracle.E4M3)
    assert s == 0 and codes[0] == 0x80 and codes[1] == 0
    # the block's own maximum saturates when its significand exceeds 1.75
    codes, s = _qblock([500.0], oracle.E4M3)
    assert s == 127 and codes[0] == 0x7E
    codes, s = _qblock([15.0, 1.0], oracle.E4M3)        # 15 * 2^5 = 480
    assert s == 122 and codes[0] == 0x7E
    # clamping: huge and subnormal maxima
    assert _qblock([3.0e38], oracle.E4M3)[1] == 127 + 127 - 8
    tiny = float(np.float32(2.0 ** -130))
    codes, s = _qblock([tiny], oracle.E4M3)
    assert s == 0 and oracle.decode_e4m3(codes[0]) == 2.0 ** -3
    # non-finite blocks get the NaN scale
    assert _qblock([1.0, float("nan")], oracle.E4M3)[1] == 0xFF
    assert _qblock([float("inf")], oracle.E2M1)[1] == 0xFF


def test_scale_rule_hand_values_e5m2():
    assert _qblock([1.0], oracle.E5M2)[1] == 112       # 2^(0-15)
    codes, s = _qblock([1.0, 0.25], oracle.E5M2)
    assert codes[0] == 0x78 and codes[1] == 0x70       # 2^15, 2^13
    codes, s = _qblock([1.9], oracle.E5M2)             # 1.9 * 2^15 > 57344
    assert s == 112 and codes[0] == 0x7B
    codes, s = _qblock([-3.0e38], oracle.E5M2)
    # 3e38 = 1.763 * 2^127: significand above 1.75, so it saturates
    assert s == 127 + 127 - 15 and codes[0] == 0xFB
    assert _qblock([float("-inf")], oracle.E5M2)[1] == 0xFF


def test_floor_log2_from_bits():
    assert oracle.floor_log2_f32(1.0) == 0
    assert oracle.floor_log2_f32(float(np.nextafter(np.float32(2), 0))) == 0
    assert oracle.floor_log2_f32(2.0) == 1
    assert oracle.floor_log2_f32(float(np.float32(2.0 ** -149))) == -149
    assert oracle.floor_log2_f32(float(np.float32(3 * 2.0 ** -140))) == -139


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2, oracle.E2M1])
def test_quantize_properties(fmt):
    """Per block: X * 2^emax <= amax < X * 2^(emax+1) unless clamped, and
    every element code is the nearest representable value of x / X."""
    g = torch.Generator().manual_seed(77)
    x = torch.randn(24, 256, generator=g)
    x[torch.rand(24, 256, generator=g) < 0.02] *= 100
    x[3, 32:64] = 0
    x[5, 64:96] *= 2.0 ** -120
    x = x.numpy()
    codes, scales = oracle.quantize(x, fmt)
    emax = {oracle.E4M3: 8, oracle.E5M2: 15, oracle.E2M1: 2}[fmt]
    if fmt == oracle.E4M3:
        table = _torch_e4m3_table()
    elif fmt == oracle.E5M2:
        table = _torch_e5m2_table()
        table[0x7C:0x80] = np.nan                       # no Inf in an MX block
        table[0xFC:] = np.nan
    else:
        table = np.array(E2M1_MAGNITUDES + [-m for m in E2M1_MAGNITUDES])
    for r in range(x.shape[0]):
        for b in range(x.shape[1] // 32):
            blk = x[r, b * 32:(b + 1) * 32].astype(np.float64)
            X = 2.0 ** (int(scales[r, b]) - 127)
            amax = np.abs(blk).max()
            if amax == 0:
                assert scales[r, b] == 0
                continue
            if 0 < scales[r, b] < 254:
                assert X * 2 ** emax <= amax < X * 2 ** (emax + 1)
            for i, v in enumerate(blk / X):
                got = table[codes[r, b * 32 + i]] * 1.0
                dist = np.abs(np.nan_to_num(table, nan=np.inf) - v).min()
                if abs(v) <= table[~np.isnan(table)].max():
                    assert abs(got - v) == dist


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2, oracle.E2M1])
def test_quantize_k_axis_layouts_agree(fmt):
    g = torch.Generator().manual_seed(8)
    src = torch.randn(64, 96, generator=g).numpy()       # K=64 x outer=96
    c0, s0 = oracle.quantize(src, fmt, k_axis=0)
    c1, s1 = oracle.quantize(np.ascontiguousarray(src.T), fmt, k_axis=1)
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1)
    assert c0.shape == (96, 64) and s0.shape == (96, 2)


# ---------------------------------------------------------------- GEMMs

def _int_matrix(shape, values, seed):
    g = np.random.default_rng(seed)
    return g.choice(values, size=shape).astype(np.float32)


E5M2_INTS = np.array([0, 1, 2, 3, 4, 5, 6, 7, 8, 10, 12, 14, 16])
E5M2_INTS = np.concatenate([E5M2_INTS, -E5M2_INTS[1:]])


@pytest.mark.parametrize("fmt,fmt_b,values,values_b", [
    (oracle.E4M3, None, np.arange(-14, 15), None),
    (oracle.E5M2, None, E5M2_INTS, None),
    (oracle.E4M3, oracle.E5M2, np.arange(-14, 15), E5M2_INTS),
    (oracle.E5M2, oracle.E4M3, E5M2_INTS, np.arange(-14, 15)),
    (oracle.E2M1, None, np.array([0, 1, 2, 3, 4, 6, -1, -2, -3, -4, -6]),
     None)])
def test_gemm_mx_integer_matrices_exact(fmt, fmt_b, values, values_b):
    """Integer-valued sources whose blocks quantize without loss must give
    exactly the integer product (numpy int64 matmul), for a non-square
    problem so that a transposed operand would show.  E5M2 holds 3
    significant bits, so its integers are those of the form m * 2^e with
    m <= 7 (any block maximum up to 16 scales without loss)."""
    M, N, K = 40, 24, 96
    A = _int_matrix((M, K), values, 1)
    B = _int_matrix((K, N), values if values_b is None else values_b, 2)
    fb = fmt if fmt_b is None else fmt_b
    ca, sa = oracle.quantize(A, fmt, k_axis=1)
    cb, sb = oracle.quantize(B, fb, k_axis=0)
    C, S = oracle.gemm_mx(ca, sa, cb, sb, fmt, fmt_b=fb)
    want = A.astype(np.int64) @ B.astype(np.int64)
    assert np.array_equal(C, want.astype(np.float64))
    assert np.array_equal(S, (np.abs(A).astype(np.int64)
                              @ np.abs(B).astype(np.int64)).astype(float))
    # rows subset evaluates the same rows
    rows = [0, 7, 39]
    C2, S2 = oracle.gemm_mx(ca, sa, cb, sb, fmt, rows=rows, fmt_b=fb)
    assert np.array_equal(C2, C[rows]) and np.array_equal(S2, S[rows])


def test_gemm_mx_identity():
    """B = identity: every 1.0 lands in a block whose maximum is 1, so it is
    code 1 * 2^8 = 256 with scale 2^-8, exactly; C must reproduce A's
    dequantized values."""
    K = 128
    g = torch.Generator().manual_seed(4)
    A = torch.randn(16, K, generator=g).numpy()
    ca, sa = oracle.quantize(A, oracle.E4M3)
    cb, sb = oracle.quantize(np.eye(K, dtype=np.float32), oracle.E4M3,
                             k_axis=0)
    C, _ = oracle.gemm_mx(ca, sa, cb, sb, oracle.E4M3)
    t = _torch_e4m3_table()
    deq = t[ca] * np.repeat(2.0 ** (sa.astype(np.int64) - 127), 32, axis=1)
    assert np.array_equal(C, deq)


def _random_finite_codes(fmt, shape, g):
    """Random finite codes of a format and the torch / hand value table."""
    if fmt == oracle.E4M3:
        vals = _torch_e4m3_table()
        c = g.integers(0, 256, shape)
        c[(c & 0x7F) == 0x7F] = 0x3F
    elif fmt == oracle.E5M2:
        vals = _torch_e5m2_table()
        c = g.integers(0, 256, shape)
        c[(c & 0x7F) >= 0x7C] = 0x3D
    else:
        vals = np.array(E2M1_MAGNITUDES + [-m for m in E2M1_MAGNITUDES])
        c = g.integers(0, 16, shape)
    return c, vals


@pytest.mark.parametrize("fmt,fmt_b", [
    (oracle.E4M3, oracle.E4M3), (oracle.E5M2, oracle.E5M2),
    (oracle.E4M3, oracle.E5M2), (oracle.E5M2, oracle.E4M3),
    (oracle.E2M1, oracle.E2M1)])
def test_gemm_mx_brute_force_rationals(fmt, fmt_b):
    """4 x 4 x 64 random codes with extreme scales: float64 oracle vs the
    exact rational sum (element values from torch / the hand table)."""
    g = np.random.default_rng(21)
    M, N, K = 4, 4, 64
    codes_a, vals = _random_finite_codes(fmt, (M, K), g)
    codes_b, vals_b = _random_finite_codes(fmt_b, (N, K), g)
    sa = g.integers(0, 255, (M, K // 32))
    sb = g.integers(0, 255, (N, K // 32))
    sa[0, 0], sb[1, 1], sa[2, 1], sb[3, 0] = 0, 254, 1, 253
    C, S = oracle.gemm_mx(codes_a.astype(np.uint8), sa.astype(np.uint8),
                          codes_b.astype(np.uint8), sb.astype(np.uint8), fmt,
                          fmt_b=fmt_b)
    for i in range(M):
        for j in range(N):
            exact = Fraction(0)
            eabs = Fraction(0)
            for k in range(K):
                a = Fraction(float(vals[codes_a[i, k]])) * \
                    Fraction(2) ** (int(sa[i, k // 32]) - 127)
                b = Fraction(float(vals_b[codes_b[j, k]])) * \
                    Fraction(2) ** (int(sb[j, k // 32]) - 127)
                exact += a * b
                eabs += abs(a * b)
            tol = float(eabs) * K * 2.0 ** -52
            assert abs(Fraction(C[i, j]) - exact) <= Fraction(tol)
            assert abs(Fraction(S[i, j]) - eabs) <= Fraction(tol)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_gemm_f16_matches_numpy_float64(dtype):
    g = torch.Generator().manual_seed(9)
    M, N, K = 33, 20, 70
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    A = (torch.rand(M, K, generator=g) * 2 - 1).to(tdt)
    B = (torch.rand(K, N, generator=g) * 2 - 1).to(tdt)
    ab = A.view(torch.int16).numpy().view(np.uint16)
    bb = B.view(torch.int16).numpy().view(np.uint16)
    code = oracle.F16 if dtype == "f16" else oracle.BF16
    C, S = oracle.gemm_f16(ab, bb, code)
    A64 = A.to(torch.float64).numpy()
    B64 = B.to(torch.float64).numpy()
    assert np.allclose(C, A64 @ B64, rtol=0, atol=1e-12)
    assert np.allclose(S, np.abs(A64) @ np.abs(B64), rtol=0, atol=1e-12)
    C2, _ = oracle.gemm_f16(ab, bb, code, rows=[3, 32])
    assert np.array_equal(C2, C[[3, 32]])


def test_hostile_accumulator_golden():
    gold = _golden_kv("hostile_accumulator.txt")
    K = 1 + int(gold["small_count"])
    a = np.full((1, K), gold["small"], dtype=np.float32)
    a[0, 0] = gold["large"]
    b = np.ones((K, 1), dtype=np.float32)
    ca, sa = oracle.quantize(a, oracle.E4M3)
    cb, sb = oracle.quantize(b, oracle.E4M3, k_axis=0)
    C, _ = oracle.gemm_mx(ca, sa, cb, sb, oracle.E4M3)
    assert C[0, 0] == gold["expected"]
    # the same terms in fp16 through the 16-bit path
    ah = torch.from_numpy(a).to(torch.float16).view(torch.int16).numpy()
    bh = torch.from_numpy(b).to(torch.float16).view(torch.int16).numpy()
    C16, _ = oracle.gemm_f16(ah.view(np.uint16), bh.view(np.uint16),
                             oracle.F16)
    assert C16[0, 0] == gold["expected"]
    # and the stall the page describes for a 16-bit accumulator
    acc = np.float16(0)
    for v in a[0]:
        acc = np.float16(acc + np.float16(v))
    assert float(acc) == gold["fp16_accumulator_stall"]


# ---------------------------------------------------------------- layouts

@pytest.mark.parametrize("outer,K", [(128, 128), (256, 512), (200, 96),
                                     (1, 32), (130, 160)])
def test_scale_tiling_roundtrip(outer, K):
    g = np.random.default_rng(outer + K)
    s = g.integers(0, 255, (outer, K // 32)).astype(np.uint8)
    t = layout.tile_scales(s, K)
    assert t.size == layout.scale_plane_bytes(outer, K)
    assert np.array_equal(layout.untile_scales(t, outer, K), s)
    pad = layout.pad_positions(outer, K)
    assert pad.sum() == t.size - s.size
    assert not t[pad].any()


def test_scale_tiling_atom_positions():
    # first atom: row r, block j at 16*(r%32) + 4*(r//32) + j
    s = np.zeros((256, 8), dtype=np.uint8)
    s[33, 2] = 7          # -> 16*1 + 4*1 + 2 = 22 in atom 0
    s[0, 5] = 9           # block 5 -> atom 1 (second K chunk), byte 1
    s[130, 0] = 11        # row 130 -> atom 2 (second row group), byte 32
    t = layout.tile_scales(s, 256)
    assert t[22] == 7 and t[512 + 1] == 9 and t[2 * 512 + 32] == 11
    assert np.count_nonzero(t) == 3


def test_e2m1_pack_roundtrip():
    g = np.random.default_rng(2)
    c = g.integers(0, 16, (5, 64)).astype(np.uint8)
    p = layout.pack_e2m1(c)
    assert p.shape == (5, 32)
    assert p[0, 0] == (c[0, 0] | (c[0, 1] << 4))
    assert np.array_equal(layout.unpack_e2m1(p), c)


# ---------------------------------------------------------------- epilogue

def test_gelu_textbook_values_and_identity():
    # GELU(x) = x * Phi(x); Phi(1) = 0.8413447460685429 and
    # Phi(-1) = 0.15865525393145707 (standard normal table)
    assert oracle.gelu(1.0) == pytest.approx(0.8413447460685429, rel=1e-15)
    assert oracle.gelu(-1.0) == pytest.approx(-0.15865525393145707, rel=1e-15)
    assert oracle.gelu(0.0) == 0.0
    for x in (0.3, 1.7, 4.0, 9.0, 30.0):
        # x Phi(x) - (-x) Phi(-x) = x (Phi(x) + Phi(-x)) = x
        assert oracle.gelu(x) - oracle.gelu(-x) == pytest.approx(x, rel=1e-15)
    assert oracle.gelu(40.0) == 40.0
    # deep negative tail: -x Phi(-x) keeps its relative accuracy
    assert oracle.gelu(-10.0) == pytest.approx(-10.0 * 7.61985302416047e-24,
                                               rel=1e-12)


def test_gelu_matches_scipy_and_torch():
    sp = pytest.importorskip("scipy.special")
    x = np.concatenate([np.linspace(-12, 12, 4001),
                        np.random.default_rng(5).standard_normal(2000) * 3])
    ours = np.array([oracle.gelu(v) for v in x])
    ref = x * sp.ndtr(x)
    assert np.allclose(ours, ref, rtol=1e-13, atol=1e-300)
    tx = torch.from_numpy(x)
    ref_t = torch.nn.functional.gelu(tx).numpy()
    assert np.allclose(ours, ref_t, rtol=1e-13, atol=1e-15)
    ours_t = np.array([oracle.gelu_tanh(v) for v in x])
    ref_tt = torch.nn.functional.gelu(tx, approximate="tanh").numpy()
    assert np.allclose(ours_t, ref_tt, rtol=1e-13, atol=1e-15)
    # the two forms differ (by up to ~1e-3 near |x| ~ 2), so a swapped
    # activation code would show
    assert np.abs(ours - ours_t).max() > 1e-4


def test_epilogue_bias_runs_along_columns():
    g = np.random.default_rng(8)
    C = g.standard_normal((7, 5))
    bias = np.array([1.0, -2.0, 0.5, 3.0, -0.25])
    Y = oracle.epilogue(C, bias, oracle.ACT_NONE)
    assert np.array_equal(Y, C + bias[None, :])
    assert np.array_equal(oracle.epilogue(C, None, oracle.ACT_NONE), C)
    sp = pytest.importorskip("scipy.special")
    Yg = oracle.epilogue(C, bias, oracle.ACT_GELU)
    x = C + bias[None, :]
    assert np.allclose(Yg, x * sp.ndtr(x), rtol=1e-13, atol=1e-300)
    with pytest.raises(ValueError):
        oracle.epilogue(C, bias[:4], oracle.ACT_GELU)


# ---------------------------------------------------------------- integer formats

INT_FMTS = [oracle.INT8, oracle.INT4, oracle.INT2]


def test_int_decode_matches_twos_complement():
    ref8 = np.arange(256, dtype=np.int64).astype(np.uint8).view(np.int8)
    assert np.array_equal(oracle.decode_table(oracle.INT8), ref8.astype(float))
    assert list(oracle.decode_table(oracle.INT4)) == \
        [0, 1, 2, 3, 4, 5, 6, 7, -8, -7, -6, -5, -4, -3, -2, -1]
    assert list(oracle.decode_table(oracle.INT2)) == [0, 1, -2, -1]


@pytest.mark.parametrize("fmt", INT_FMTS)
def test_int_encode_matches_numpy_round_half_even(fmt):
    bits = oracle.INT_BITS[fmt]
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1)) - 1
    g = np.random.default_rng(bits)
    v = np.concatenate([g.uniform(lo - 3, hi + 3, 4000),
                        np.arange(lo - 2, hi + 3) + 0.5,          # ties
                        np.arange(lo - 2, hi + 3).astype(float)])
    want = np.clip(np.round(v), lo, hi).astype(np.int64) & ((1 << bits) - 1)
    got = np.array([oracle.encode_int(x, bits) for x in v])
    assert np.array_equal(got, want)


def test_int_scale_rule_hand_values():
    c, s = _qblock([1.0, -1.0], oracle.INT8)
    assert s == 121 and c[0] == 64 and c[1] == 0xC0      # 2^(0-6); +-64
    c, s = _qblock([1.999], oracle.INT8)                  # 127.9 -> 127
    assert s == 121 and c[0] == 127
    c, s = _qblock([100.0, 3.0], oracle.INT8)             # X = 2^(6-6) = 1
    assert s == 127 and c[0] == 100 and c[1] == 3
    c, s = _qblock([1.0, 0.3], oracle.INT4)               # X = 2^-2
    assert s == 125 and c[0] == 4 and c[1] == 1           # 1.2 -> 1
    c, s = _qblock([1.5, -1.5], oracle.INT2)              # X = 1
    assert s == 127 and c[0] == 1 and c[1] == 2           # 2 -> 1; -2
    c, s = _qblock([-0.5, 0.5, 1.0], oracle.INT2)         # ties to even 0
    assert c[0] == 0 and c[1] == 0


@pytest.mark.parametrize("fmt", INT_FMTS)
def test_int_quantize_properties(fmt):
    bits = oracle.INT_BITS[fmt]
    emax = bits - 2
    g = torch.Generator().manual_seed(40 + bits)
    x = (torch.randn(16, 256, generator=g) *
         torch.exp(torch.randn(16, 1, generator=g) * 3)).numpy()
    codes, scales = oracle.quantize(x, fmt)
    tab = oracle.decode_table(fmt)
    lo, hi = tab.min(), tab.max()
    for r in range(x.shape[0]):
        for b in range(x.shape[1] // 32):
            blk = x[r, b * 32:(b + 1) * 32].astype(np.float64)
            X = 2.0 ** (int(scales[r, b]) - 127)
            assert X * 2 ** emax <= np.abs(blk).max() < X * 2 ** (emax + 1)
            q = tab[codes[r, b * 32:(b + 1) * 32]]
            assert np.array_equal(q, np.clip(np.round(blk / X), lo, hi))


@pytest.mark.parametrize("fmt,vmax", [(oracle.INT8, 127), (oracle.INT4, 7),
                                      (oracle.INT2, 1)])
@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.F16])
def test_gemm_a16_bmx_integer_exact(fmt, vmax, dtype):
    """Integer sources within the format's range quantize without loss, so
    the product is the integer product (numpy int64), non-square so that a
    transposed operand shows."""
    g = np.random.default_rng(fmt + 10 * dtype)
    M, N, K = 24, 40, 96
    A = g.integers(-50, 51, (M, K))
    B = g.integers(-vmax, vmax + 1, (K, N))
    tdt = torch.bfloat16 if dtype == oracle.BF16 else torch.float16
    A_bits = torch.from_numpy(A.astype(np.float32)).to(tdt).view(
        torch.int16).numpy().view(np.uint16)
    cb, sb = oracle.quantize(B.astype(np.float32), fmt, k_axis=0)
    C, S = oracle.gemm_a16_bmx(A_bits, dtype, cb, sb, fmt)
    assert np.array_equal(C, (A @ B).astype(float))
    assert np.array_equal(S, (np.abs(A) @ np.abs(B)).astype(float))
    C2, _ = oracle.gemm_a16_bmx(A_bits, dtype, cb, sb, fmt, rows=[3, 0, 23])
    assert np.array_equal(C2, C[[3, 0, 23]])


@pytest.mark.parametrize("fmt", INT_FMTS + [oracle.E4M3, oracle.E2M1])
def test_gemm_a16_bmx_brute_force_rationals(fmt):
    g = np.random.default_rng(77 + fmt)
    M, N, K = 3, 4, 64
    A = torch.from_numpy(g.standard_normal((M, K)).astype(np.float32) * 8)
    A_bits = A.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    a_vals = A.to(torch.bfloat16).to(torch.float64).numpy()
    ncodes = 16 if fmt == oracle.E2M1 else 1 << layout.CODE_BITS[fmt]
    cb = g.integers(0, ncodes, (N, K))
    if fmt == oracle.E4M3:
        cb[(cb & 0x7F) == 0x7F] = 0x11
    sb = g.integers(60, 190, (N, K // 32))
    C, S = oracle.gemm_a16_bmx(A_bits, oracle.BF16, cb.astype(np.uint8),
                               sb.astype(np.uint8), fmt)
    tab = (_torch_e4m3_table() if fmt == oracle.E4M3 else
           np.array(E2M1_MAGNITUDES + [-m for m in E2M1_MAGNITUDES])
           if fmt == oracle.E2M1 else oracle.decode_table(fmt))
    for i in range(M):
        for j in range(N):
            exact = sum(Fraction(float(a_vals[i, k])) *
                        Fraction(float(tab[cb[j, k]])) *
                        Fraction(2) ** (int(sb[j, k // 32]) - 127)
                        for k in range(K))
            tol = Fraction(float(S[i, j]) * K * 2.0 ** -52)
            assert abs(Fraction(C[i, j]) - exact) <= tol


def test_int2_packing_roundtrip():
    g = np.random.default_rng(4)
    codes = g.integers(0, 4, (5, 64)).astype(np.uint8)
    packed = layout.pack_codes(codes, oracle.INT2)
    assert packed.shape == (5, 16)
    assert packed[0, 0] == codes[0, 0] | (codes[0, 1] << 2) | \
        (codes[0, 2] << 4) | (codes[0, 3] << 6)
    assert np.array_equal(layout.unpack_codes(packed, oracle.INT2, 64), codes)
    assert layout.data_plane_bytes(oracle.INT2, 5, 64) == 80
    assert layout.data_plane_bytes(oracle.E5M2, 5, 64) == 320


# ---------------------------------------------------------------- attention

def _bits16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dt,code", [(torch.bfloat16, oracle.BF16),
                                     (torch.float16, oracle.F16)])
def test_attention_matches_torch_sdpa(dt, code):
    g = torch.Generator().manual_seed(21)
    q = torch.randn(3, 9, 16, generator=g).to(dt)
    k = torch.randn(3, 13, 16, generator=g).to(dt)
    v = torch.randn(3, 13, 16, generator=g).to(dt)
    for scale in (None, 0.3):
        O, Sv = oracle.attention(_bits16(q), _bits16(k), _bits16(v), code,
                                 scale=scale)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.double(), k.double(), v.double(), scale=scale).numpy()
        assert np.allclose(O, ref, rtol=1e-12, atol=1e-12)
        assert (Sv >= np.abs(O) - 1e-12).all()


def test_attention_closed_forms():
    g = torch.Generator().manual_seed(5)
    v = torch.randn(2, 11, 8, generator=g).to(torch.bfloat16)
    k = torch.randn(2, 11, 8, generator=g).to(torch.bfloat16)
    q0 = torch.zeros(2, 4, 8, dtype=torch.bfloat16)
    # Q = 0: every score is 0, the weights uniform: O is the mean of V's rows
    O, Sv = oracle.attention(_bits16(q0), _bits16(k), _bits16(v), oracle.BF16)
    vd = v.double().numpy()
    assert np.allclose(O, vd.mean(axis=1, keepdims=True).repeat(4, axis=1),
                       rtol=1e-13, atol=1e-15)
    assert np.allclose(Sv, np.abs(vd).mean(axis=1, keepdims=True).repeat(4, 1))
    # one key aligned with the query and far larger than the rest: O picks
    # that key's value row
    q = torch.zeros(1, 1, 8, dtype=torch.bfloat16)
    q[0, 0, 3] = 4.0
    kk = torch.zeros(1, 6, 8, dtype=torch.bfloat16)
    kk[0, 4, 3] = 64.0                                   # score 256 / sqrt(8)
    vv = torch.arange(48, dtype=torch.float32).reshape(1, 6, 8).to(torch.bfloat16)
    O, _ = oracle.attention(_bits16(q), _bits16(kk), _bits16(vv), oracle.BF16)
    assert np.allclose(O[0, 0], vv[0, 4].double().numpy(), rtol=1e-15)


def test_attention_permutation_and_rows():
    g = torch.Generator().manual_seed(9)
    q = torch.randn(2, 6, 8, generator=g).to(torch.float16)
    k = torch.randn(2, 10, 8, generator=g).to(torch.float16)
    v = torch.randn(2, 10, 8, generator=g).to(torch.float16)
    O, _ = oracle.attention(_bits16(q), _bits16(k), _bits16(v), oracle.F16)
    perm = torch.randperm(10, generator=g)
    Op, _ = oracle.attention(_bits16(q), _bits16(k[:, perm]),
                             _bits16(v[:, perm]), oracle.F16)
    assert np.allclose(O, Op, rtol=1e-12, atol=1e-14)     # keys are a set
    Ok, _ = oracle.attention(_bits16(q), _bits16(k[:, perm]), _bits16(v),
                             oracle.F16)
    assert not np.allclose(O, Ok, atol=1e-3)               # K and V paired
    O2, _ = oracle.attention(_bits16(q), _bits16(k), _bits16(v), oracle.F16,
                             rows=[5, 0])
    assert np.array_equal(O2, O[:, [5, 0]])


def test_results_do_not_depend_on_thread_count():
    """The benchmark times the oracle on one core and on all cores; its
    parallel loops split rows only, so every result is bit-identical."""
    g = np.random.default_rng(21)
    x = (g.standard_normal((96, 256)) * 3).astype(np.float32)
    y = (g.standard_normal((256, 64)) * 3).astype(np.float32)
    outs = []
    for n in (1, 3, 0):
        oracle.set_num_threads(n)
        try:
            ca, sa = oracle.quantize(x, oracle.E4M3, k_axis=1)
            cb, sb = oracle.quantize(y, oracle.E4M3, k_axis=0)
            C, S = oracle.gemm_mx(ca, sa, cb, sb, oracle.E4M3)
        finally:
            oracle.set_num_threads(0)
        outs.append((ca, sa, cb, sb, C, S))
    assert oracle.num_threads() >= 1
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert np.array_equal(a, b)
