"""CPU oracle for the MX block-scaled and FP16/BF16 matrix multiply.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product library never imports it,
and it imports nothing from the product.

The arithmetic lives in ``mx_oracle.c`` (float64 throughout, formats decoded
from their bit fields, encoding by search over the representable values); this
module compiles it with gcc on first use and marshals numpy arrays in and out.

What each function follows:
  * ``quantize`` -- the OCP MX conversion rule on blocks of 32 consecutive
    K elements sharing one UE8M0 scale (WWDC26 session 330, "Multi-plane
    tensors" and its 4:48 listing: block factors {32, 1} on the innermost
    dimension; the MX scaling formats named in "Managing quantized data").
  * ``gemm_mx`` / ``gemm_f16`` -- the float64 reference over exactly the same
    quantized bytes (RIGEL technical summary, "Metodologia", checksum gate),
    returning C and S = sum_k |a_ik * b_kj| for the per-element tolerance
    |C_gpu - C| <= tol * S.
  * ``epilogue`` -- bias and GELU on the product, the fused GEMM + bias +
    GELU kernel of the RIGEL summary (Main findings section 4); GELU is
    x * Phi(x) (through erfc), or its tanh approximation.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3 = 1
E2M1 = 2
E5M2 = 3
INT8 = 4
INT4 = 5
INT2 = 6
INT_BITS = {INT8: 8, INT4: 4, INT2: 2}
F16 = 2
BF16 = 1
ACT_NONE = 0
ACT_GELU = 1
ACT_GELU_TANH = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``mx_oracle.c`` into ``liboracle.so`` (gcc, OpenMP)."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC",
               _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        u8, u16, i32, i64, dbl = (ctypes.c_uint8, ctypes.c_uint16,
                                  ctypes.c_int, ctypes.c_int64,
                                  ctypes.c_double)
        p = ctypes.c_void_p
        lib.mxo_decode_e4m3.restype = dbl
        lib.mxo_decode_e4m3.argtypes = [u8]
        lib.mxo_decode_e5m2.restype = dbl
        lib.mxo_decode_e5m2.argtypes = [u8]
        lib.mxo_encode_e5m2.restype = u8
        lib.mxo_encode_e5m2.argtypes = [dbl]
        lib.mxo_decode_int.restype = dbl
        lib.mxo_decode_int.argtypes = [u8, i32]
        lib.mxo_encode_int.restype = u8
        lib.mxo_encode_int.argtypes = [dbl, i32]
        lib.mxo_gemm_a16_bmx.restype = None
        lib.mxo_gemm_a16_bmx.argtypes = [p, i32, p, p, i32, i64, i64, i64, p,
                                         i64, p, p]
        lib.mxo_decode_e2m1.restype = dbl
        lib.mxo_decode_e2m1.argtypes = [u8]
        lib.mxo_decode_ue8m0.restype = dbl
        lib.mxo_decode_ue8m0.argtypes = [u8]
        lib.mxo_decode_f16.restype = dbl
        lib.mxo_decode_f16.argtypes = [u16]
        lib.mxo_decode_bf16.restype = dbl
        lib.mxo_decode_bf16.argtypes = [u16]
        lib.mxo_encode_e4m3.restype = u8
        lib.mxo_encode_e4m3.argtypes = [dbl]
        lib.mxo_encode_e2m1.restype = u8
        lib.mxo_encode_e2m1.argtypes = [dbl]
        lib.mxo_encode_array.restype = None
        lib.mxo_encode_array.argtypes = [p, i64, i32, p]
        lib.mxo_floor_log2_f32.restype = i32
        lib.mxo_floor_log2_f32.argtypes = [ctypes.c_float]
        lib.mxo_quantize.restype = None
        lib.mxo_quantize.argtypes = [p, i64, i64, i64, i64, i32, p, p]
        lib.mxo_gemm_mx.restype = None
        lib.mxo_gemm_mx.argtypes = [p, p, p, p, i64, i64, i64, i32, i32, p,
                                    i64, p, p]
        lib.mxo_gemm_f16.restype = None
        lib.mxo_gemm_f16.argtypes = [p, p, i64, i64, i64, i32, p, i64, p, p]
        lib.mxo_gelu.restype = dbl
        lib.mxo_gelu.argtypes = [dbl]
        lib.mxo_gelu_tanh.restype = dbl
        lib.mxo_gelu_tanh.argtypes = [dbl]
        lib.mxo_epilogue.restype = None
        lib.mxo_epilogue.argtypes = [p, i64, i64, p, i32]
        lib.mxo_attention.restype = None
        lib.mxo_attention.argtypes = [p, p, p, i32, i64, i64, i64, i64, dbl, p,
                                      i64, p, p]
        lib.mxo_num_threads.restype = i32
        lib.mxo_num_threads.argtypes = []
        lib.mxo_set_num_threads.restype = None
        lib.mxo_set_num_threads.argtypes = [i32]
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# --------------------------------------------------------------------------
# scalar codecs
# --------------------------------------------------------------------------

def decode_e4m3(code: int) -> float:
    return _load().mxo_decode_e4m3(int(code) & 0xFF)


def decode_e5m2(code: int) -> float:
    return _load().mxo_decode_e5m2(int(code) & 0xFF)


def encode_e5m2(v: float) -> int:
    return int(_load().mxo_encode_e5m2(float(v)))


def decode_int(code: int, bits: int) -> float:
    return _load().mxo_decode_int(int(code) & 0xFF, int(bits))


def encode_int(v: float, bits: int) -> int:
    return int(_load().mxo_encode_int(float(v), int(bits)))


def decode_e2m1(code: int) -> float:
    return _load().mxo_decode_e2m1(int(code) & 0xF)


def decode_ue8m0(code: int) -> float:
    return _load().mxo_decode_ue8m0(int(code) & 0xFF)


def decode_f16(bits: int) -> float:
    return _load().mxo_decode_f16(int(bits) & 0xFFFF)


def decode_bf16(bits: int) -> float:
    return _load().mxo_decode_bf16(int(bits) & 0xFFFF)


def encode_e4m3(v: float) -> int:
    return int(_load().mxo_encode_e4m3(float(v)))


def encode_e2m1(v: float) -> int:
    return int(_load().mxo_encode_e2m1(float(v)))


def encode_array(values, fmt: int) -> np.ndarray:
    """Codes (uint8, one per element, same shape) of float64 values:
    round to nearest, ties to even, saturating, as the scalar encoders."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().mxo_encode_array(_ptr(v), v.size, int(fmt), _ptr(out))
    return out


def floor_log2_f32(a: float) -> int:
    return int(_load().mxo_floor_log2_f32(float(a)))


def decode_table(fmt: int) -> np.ndarray:
    """float64 value of every code: 256 entries for E4M3 / E5M2, 16 for
    E2M1, 2^bits for the integer formats."""
    if fmt in INT_BITS:
        b = INT_BITS[fmt]
        return np.array([decode_int(c, b) for c in range(1 << b)])
    if fmt == E4M3:
        return np.array([decode_e4m3(c) for c in range(256)])
    if fmt == E5M2:
        return np.array([decode_e5m2(c) for c in range(256)])
    return np.array([decode_e2m1(c) for c in range(16)])


def gelu(x: float) -> float:
    return float(_load().mxo_gelu(float(x)))


def gelu_tanh(x: float) -> float:
    return float(_load().mxo_gelu_tanh(float(x)))


def epilogue(C, bias=None, act: int = ACT_NONE) -> np.ndarray:
    """float64 act(C + bias) of a float64 rows x N product (bias: N values
    added to every row, or None)."""
    Y = np.array(C, dtype=np.float64, order="C", copy=True)
    rows, N = Y.shape
    b = None
    if bias is not None:
        b = np.ascontiguousarray(bias, dtype=np.float64)
        if b.shape != (N,):
            raise ValueError("bias must hold N values")
    _load().mxo_epilogue(_ptr(Y), rows, N, None if b is None else _ptr(b),
                         int(act))
    return Y


def attention(Q_bits, K_bits, V_bits, dtype: int, scale: float | None = None,
              rows=None):
    """float64 O = softmax(Q K^T * scale) V per head, and Sv = sum_j w_j |v_j|.

    Q is BH x Lq x d, K and V BH x Lk x d, as uint16 fp16 / bf16 bit
    patterns; scale defaults to 1/sqrt(d); rows selects query rows (the same
    rows of every head).  Returns O, Sv of shape BH x len(rows) x d."""
    Q = np.ascontiguousarray(Q_bits, dtype=np.uint16)
    K = np.ascontiguousarray(K_bits, dtype=np.uint16)
    V = np.ascontiguousarray(V_bits, dtype=np.uint16)
    BH, Lq, d = Q.shape
    if K.shape != V.shape or K.shape[0] != BH or K.shape[2] != d:
        raise ValueError("shape mismatch")
    Lk = K.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    r, nr = _rows_arg(rows, Lq)
    O = np.empty((BH, nr, d), dtype=np.float64)
    Sv = np.empty((BH, nr, d), dtype=np.float64)
    _load().mxo_attention(_ptr(Q), _ptr(K), _ptr(V), dtype, BH, Lq, Lk, d,
                          float(scale), None if r is None else _ptr(r), nr,
                          _ptr(O), _ptr(Sv))
    return O, Sv


def num_threads() -> int:
    return int(_load().mxo_num_threads())


def set_num_threads(n: int) -> None:
    """Threads for the oracle's parallel loops (n <= 0: one per host core).
    For timing only: every result is the same for any thread count."""
    _load().mxo_set_num_threads(int(n))


# --------------------------------------------------------------------------
# array operations
# --------------------------------------------------------------------------

def quantize(src: np.ndarray, fmt: int, k_axis: int = 1):
    """OCP MX quantization of a 2-D float32 matrix.

    ``k_axis=1``: src is outer x K (K contiguous; the A operand).
    ``k_axis=0``: src is K x outer (the row-major K x N B operand); blocks of
    32 still run along K, i.e. down the columns.

    Returns ``(codes, scales)``: codes outer x K uint8, one code per byte
    (E2M1 codes in the low nibble), and scales outer x K/32 UE8M0 codes.
    """
    lib = _load()
    src = np.ascontiguousarray(src, dtype=np.float32)
    if k_axis == 1:
        outer, K = src.shape
        s_row, s_k = K, 1
    else:
        K, outer = src.shape
        s_row, s_k = 1, outer
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    codes = np.empty((outer, K), dtype=np.uint8)
    scales = np.empty((outer, K // 32), dtype=np.uint8)
    lib.mxo_quantize(_ptr(src), outer, K, s_row, s_k, fmt, _ptr(codes),
                     _ptr(scales))
    return codes, scales


def _rows_arg(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if r.size and (r.min() < 0 or r.max() >= M):
        raise IndexError("row index out of range")
    return r, int(r.size)


def gemm_mx(codesA, scalesA, codesB, scalesB, fmt: int, rows=None,
            fmt_b: int | None = None):
    """float64 C = A_mx * B_mx^T and S = sum |products|.

    codesA M x K, scalesA M x K/32, codesB N x K, scalesB N x K/32 (both
    operands K-major, as returned by ``quantize``).  ``fmt`` is A's element
    format and B's too unless ``fmt_b`` is given.  ``rows`` restricts the
    evaluation to those rows of A (C and S then have len(rows) rows).
    """
    lib = _load()
    cA = np.ascontiguousarray(codesA, dtype=np.uint8)
    sA = np.ascontiguousarray(scalesA, dtype=np.uint8)
    cB = np.ascontiguousarray(codesB, dtype=np.uint8)
    sB = np.ascontiguousarray(scalesB, dtype=np.uint8)
    M, K = cA.shape
    N, K2 = cB.shape
    if K != K2 or sA.shape != (M, K // 32) or sB.shape != (N, K // 32):
        raise ValueError("shape mismatch")
    r, nr = _rows_arg(rows, M)
    C = np.empty((nr, N), dtype=np.float64)
    S = np.empty((nr, N), dtype=np.float64)
    lib.mxo_gemm_mx(_ptr(cA), _ptr(sA), _ptr(cB), _ptr(sB), M, N, K, fmt,
                    fmt if fmt_b is None else fmt_b,
                    None if r is None else _ptr(r), nr, _ptr(C), _ptr(S))
    return C, S


def gemm_a16_bmx(A_bits, dtype: int, codesB, scalesB, fmt_b: int, rows=None):
    """float64 C = A * B_mx^T for a row-major fp16 / bf16 A (uint16 bit
    patterns, M x K) and an MX tensor B (codes N x K, scales N x K/32) of
    any element format; also S = sum |products|."""
    lib = _load()
    A = np.ascontiguousarray(A_bits, dtype=np.uint16)
    cB = np.ascontiguousarray(codesB, dtype=np.uint8)
    sB = np.ascontiguousarray(scalesB, dtype=np.uint8)
    M, K = A.shape
    N, K2 = cB.shape
    if K != K2 or sB.shape != (N, K // 32):
        raise ValueError("shape mismatch")
    r, nr = _rows_arg(rows, M)
    C = np.empty((nr, N), dtype=np.float64)
    S = np.empty((nr, N), dtype=np.float64)
    lib.mxo_gemm_a16_bmx(_ptr(A), dtype, _ptr(cB), _ptr(sB), fmt_b, M, N, K,
                         None if r is None else _ptr(r), nr, _ptr(C), _ptr(S))
    return C, S


def gemm_f16(A_bits, B_bits, dtype: int, rows=None):
    """float64 C = A * B for row-major fp16/bf16 bit patterns (uint16)
    A (M x K) and B (K x N); also S = sum |products|."""
    lib = _load()
    A = np.ascontiguousarray(A_bits, dtype=np.uint16)
    B = np.ascontiguousarray(B_bits, dtype=np.uint16)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("shape mismatch")
    r, nr = _rows_arg(rows, M)
    C = np.empty((nr, N), dtype=np.float64)
    S = np.empty((nr, N), dtype=np.float64)
    lib.mxo_gemm_f16(_ptr(A), _ptr(B), M, N, K, dtype,
                     None if r is None else _ptr(r), nr, _ptr(C), _ptr(S))
    return C, S
