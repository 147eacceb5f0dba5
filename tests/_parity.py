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
    if q.fmt != mx.E2M1:
        codes = data.reshape(q.outer, q.K)
    else:
        codes = layout.unpack_e2m1(data.reshape(q.outer, q.K // 2))
    return codes, layout.untile_scales(sc, q.outer, q.K)


def planes_from_codes(codes: np.ndarray, scales: np.ndarray, fmt: int,
                      device="cuda") -> mx.MXTensor:
    """Build library-format device planes from oracle-form codes."""
    outer, K = codes.shape
    if fmt != oracle.E2M1:
        data = codes.reshape(-1)
    else:
        data = layout.pack_e2m1(codes).reshape(-1)
    tiled = layout.tile_scales(scales, K)
    return mx.MXTensor(torch.from_numpy(np.ascontiguousarray(data)).to(device),
                       torch.from_numpy(tiled).to(device), fmt, outer, K)


def nan_like(shape, dtype, device="cuda"):
    return torch.full(shape, float("nan"), dtype=dtype, device=device)


def f16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def is_pow2(x: int) -> bool:
    return x > 0 and (x & (x - 1)) == 0 and math.log2(x) == int(math.log2(x))
