"""Helpers shared by the GPU parity tests: run the library, run the oracle on
the same seeded inputs, compare.

Tolerances (per element, S = sum_k |a_ik * b_kj| from the oracle):
  fp32 output:  |C - C_ref| <= 1e-4 * S
  bf16 output:  |C - C_ref| <= 1e-4 * S + ulp_bf16(|C_ref|)
The 1e-4 * S bound is the per-element accumulation bound the method is held
to; a bf16 store adds its own round-to-nearest (half an ulp), and an
accumulator error that crosses a rounding boundary can move the stored value
by one more half ulp, hence one bf16 ulp of C_ref on top.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import block_scaled_quantized_mx_gb300 as mx
import oracle
from oracle import layout

REL_TOL = 1e-4


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126)
    return np.where(ax > 0, 2.0 ** (e - 7), 2.0 ** -133)


def check_close(C_gpu: np.ndarray, C_ref: np.ndarray, S: np.ndarray,
                out: str, what: str = ""):
    C_gpu = np.asarray(C_gpu, dtype=np.float64)
    assert C_gpu.shape == C_ref.shape, (C_gpu.shape, C_ref.shape)
    assert np.isfinite(C_gpu).all(), f"{what}: non-finite output"
    bound = REL_TOL * S
    if out == "bf16":
        bound = bound + ulp_bf16(C_ref)
    err = np.abs(C_gpu - C_ref)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
            f"first at {tuple(i)}: gpu {C_gpu[tuple(i)]!r} ref "
            f"{C_ref[tuple(i)]!r} S {S[tuple(i)]!r}")
    return float((err / np.maximum(S, 1e-300)).max()) if err.size else 0.0


def sample_rows(M: int, n_random: int = 24, seed: int = 0):
    fixed = {0, 1, 31, 32, 127, 128, 129, M // 2, M - 129, M - 128, M - 1}
    g = np.random.default_rng(seed)
    rnd = set(g.integers(0, M, n_random).tolist()) if M > 0 else set()
    return sorted(r for r in fixed | rnd if 0 <= r < M)


def mx_quantize_both(A32: torch.Tensor, B32: torch.Tensor, fa: int, fb: int):
    """Library quantization of A (M x K) and of B (K x N, K-strided)."""
    a = mx.mx_quantize(A32.cuda(), fa)
    b = mx.mx_quantize(B32.cuda(), fb, k_strided=True)
    return a, b


def oracle_mx_product(A32: torch.Tensor, B32: torch.Tensor, fa: int, fb: int,
                      rows=None):
    """Oracle quantization of both sources and the float64 product."""
    ca, sa = oracle.quantize(A32.numpy(), fa, k_axis=1)
    cb, sb = oracle.quantize(B32.numpy(), fb, k_axis=0)
    return oracle.gemm_mx(ca, sa, cb, sb, fa, rows=rows, fmt_b=fb)


def lib_quantize_to_oracle_form(q: mx.MXTensor):
    """Library planes (device) -> (codes outer x K, scales outer x K/32) in
    the oracle's plain form, using the oracle's own layout restatement."""
    data = q.data.cpu().numpy()
    sc = q.scales.cpu().numpy()
    codes = layout.unpack_codes(data.reshape(q.outer, -1), q.fmt, q.K)
    return codes, layout.untile_scales(sc, q.outer, q.K)


def planes_from_codes(codes: np.ndarray, scales: np.ndarray, fmt: int,
                      device="cuda") -> mx.MXTensor:
    """Build library-format device planes from oracle-form codes."""
    outer, K = codes.shape
    data = layout.pack_codes(codes, fmt).reshape(-1)
    tiled = layout.tile_scales(scales, K)
    return mx.MXTensor(torch.from_numpy(np.ascontiguousarray(data)).to(device),
                       torch.from_numpy(tiled).to(device), fmt, outer, K)


def nan_like(shape, dtype, device="cuda"):
    return torch.full(shape, float("nan"), dtype=dtype, device=device)


def f16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def is_pow2(x: int) -> bool:
    return x > 0 and (x & (x - 1)) == 0 and math.log2(x) == int(math.log2(x))


# ---------------------------------------------------------------- epilogue

# max |d/dx GELU(x)| = 1.1289 (at x ~ 1.41); the tanh form's is the same to
# three digits
GELU_SLOPE = 1.13


def epilogue_tolerance(C_ref, S, bias, act, Y_ref):
    """Bound on |y_gpu - y_ref| for y = act(acc + bias).

    The accumulator is within REL_TOL * S of C_ref; the fp32 bias add rounds
    by at most 2^-24 |pre| (pre = C_ref + bias); the activation moves the
    error by at most its slope and adds a few ulp of its own: 2^-21 |y|
    covers erff / tanhf and the products around them; where 1 + erf or
    1 + tanh cancels in fp32 (the negative tail) the absolute error stays
    near 2^-24 |pre|, inside the slope * 2^-23 |pre| term."""
    pre = C_ref + (0.0 if bias is None else np.asarray(bias, np.float64)[None, :])
    slope = 1.0 if act == oracle.ACT_NONE else GELU_SLOPE
    return slope * (REL_TOL * S + 2.0 ** -23 * np.abs(pre)) + \
        2.0 ** -21 * np.abs(Y_ref)


def check_epilogue_close(Y_gpu, C_ref, S, bias, act, out, what=""):
    """Y_gpu (fp32 or bf16 output of a fused call) vs the oracle's
    act(C_ref + bias)."""
    Y_gpu = np.asarray(Y_gpu, dtype=np.float64)
    Y_ref = oracle.epilogue(C_ref, bias, act)
    assert Y_gpu.shape == Y_ref.shape
    assert np.isfinite(Y_gpu).all(), f"{what}: non-finite output"
    bound = epilogue_tolerance(C_ref, S, bias, act, Y_ref)
    if out == "bf16":
        bound = bound + ulp_bf16(Y_ref)
    err = np.abs(Y_gpu - Y_ref)
    bad = err > bound
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} out of "
                             f"tolerance; first at {i}: gpu {Y_gpu[i]!r} ref "
                             f"{Y_ref[i]!r} bound {bound[i]!r}")
    return Y_ref, bound


EMAX = {oracle.E4M3: 8, oracle.E5M2: 15, oracle.E2M1: 2}


def _scale_codes(amax, emax):
    """UE8M0 code of the OCP rule for float64 block maxima (0 for 0)."""
    a = np.asarray(amax, dtype=np.float64)
    _, e = np.frexp(np.where(a > 0, a, 1.0))     # a = m 2^e, m in [0.5, 1)
    es = np.clip(e - 1 - emax, -127, 127)
    return np.where(a > 0, es + 127, 0).astype(np.int64)


def check_mx_output(codes, scales, Y_ref, tol, fmt, what=""):
    """The GPU quantized y = act(acc + bias) itself, and its fp32 y is known
    only to lie within Y_ref +- tol.  Checks, from the oracle's side only:
    every block's scale code is one the OCP rule gives for some block
    maximum in the allowed interval, and, under that scale, every element
    code is the oracle's encoding of some value in its allowed interval
    (encoding is monotone, so the codes between those of the interval's
    ends).  Returns the fraction of elements whose code the interval fixes
    uniquely (compared exactly)."""
    rows, N = Y_ref.shape
    nb = N // 32
    lo_abs = np.maximum(np.abs(Y_ref) - tol, 0.0).reshape(rows, nb, 32)
    hi_abs = (np.abs(Y_ref) + tol).reshape(rows, nb, 32)
    s_lo = _scale_codes(lo_abs.max(axis=2), EMAX[fmt])
    s_hi = _scale_codes(hi_abs.max(axis=2), EMAX[fmt])
    sc = scales.astype(np.int64)
    bad = (sc < s_lo) | (sc > s_hi)
    assert not bad.any(), (f"{what}: scale code outside the allowed range at "
                           f"{np.argwhere(bad)[:3].tolist()}")
    X = np.repeat(2.0 ** (sc - 127).astype(np.float64), 32, axis=1)
    c_lo = oracle.encode_array((Y_ref - tol) / X, fmt)
    c_hi = oracle.encode_array((Y_ref + tol) / X, fmt)
    tab = oracle.decode_table(fmt)
    v_lo, v_hi, v = tab[c_lo], tab[c_hi], tab[codes]
    bad = ~((v >= v_lo) & (v <= v_hi))
    assert not bad.any(), (
        f"{what}: {bad.sum()} codes outside the allowed interval; first at "
        f"{tuple(np.argwhere(bad)[0])}")
    unique = (c_lo == c_hi) & np.repeat(s_lo == s_hi, 32, axis=1)
    return float(unique.mean())
