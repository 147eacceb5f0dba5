"""Python binding of libmx_gb300.so (the C ABI in include/mx.h).

Argument marshalling only: every step of quantization and matrix multiply runs
in the library's CUDA kernels.  PyTorch supplies device memory and the current
stream.  There is no fallback: if the shared library is missing or fails to
load, every call raises.

    from block_scaled_quantized_mx_gb300 import mx_quantize, mx_gemm, gemm_f16
    a = mx_quantize(A_fp32, E4M3)                      # A: M x K, K contiguous
    b = mx_quantize(B_fp32, E4M3, k_strided=True)      # B: K x N row-major
    C = mx_gemm(a, b, out_dtype=torch.bfloat16)        # C = A @ B
"""
from __future__ import annotations

import ctypes
import functools
import os
from dataclasses import dataclass

import torch

from . import _build

E4M3 = 1
E2M1 = 2
E5M2 = 3
INT8 = 4
INT4 = 5
INT2 = 6
DT_F32, DT_BF16, DT_F16 = 0, 1, 2
SRC_K_CONTIGUOUS, SRC_K_STRIDED = 0, 1
ACT_NONE, ACT_GELU, ACT_GELU_TANH = 0, 1, 2

STATUS = {0: "MX_OK", 1: "MX_ERR_INVALID_ARG", 2: "MX_ERR_SHAPE",
          3: "MX_ERR_ALIGN", 4: "MX_ERR_UNSUPPORTED", 5: "MX_ERR_CUDA",
          6: "MX_ERR_TIMEOUT"}

EXPORTS = ("mx_data_bytes", "mx_scale_bytes", "mx_quantize", "mx_gemm",
           "gemm_f16", "mx_gemm_fused", "mx_gemm_fused_quantize",
           "gemm_f16_fused", "gemm_dequant", "gemm_dequant_splitk",
           "gemm_dequant_workspace_bytes", "flash_attention",
           "flash_attention_workspace_bytes", "flash_attention_splitkv",
           "mx_gemm_workspace_bytes",
           "mx_gemm_splitk",
           "gemm_f16_workspace_bytes", "gemm_f16_splitk",
           "mx_gemm_splitk_noalloc", "mx_last_error",
           "mx_selftest_wait_timeout", "mx_scales_to_rowmajor",
           "mx_status_string", "mx_version", "mx_set_tile_width")


class MXError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed: %s" % (what, STATUS.get(status, status)))
        self.status = status


class CMXTensor(ctypes.Structure):
    """Mirror of struct mx_tensor."""
    _fields_ = [("data", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("fmt", ctypes.c_int32), ("outer", ctypes.c_int64),
                ("K", ctypes.c_int64)]


class CEpilogue(ctypes.Structure):
    """Mirror of struct mx_epilogue."""
    _fields_ = [("bias", ctypes.c_void_p), ("act", ctypes.c_int32)]


_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA sources for sm_103a into the in-tree shared library."""
    return _build.build(force=force, verbose=verbose)


def lib_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB_PATH):
        raise RuntimeError("%s is not built: call "
                           "block_scaled_quantized_mx_gb300.build() first"
                           % _build.LIB_PATH)
    L = ctypes.CDLL(_build.LIB_PATH)
    i32, i64, p, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, \
        ctypes.c_size_t
    pt = ctypes.POINTER(CMXTensor)
    L.mx_data_bytes.restype = sz
    L.mx_data_bytes.argtypes = [i32, i64, i64]
    L.mx_scale_bytes.restype = sz
    L.mx_scale_bytes.argtypes = [i64, i64]
    L.mx_quantize.restype = i32
    L.mx_quantize.argtypes = [p, i64, i32, pt, p]
    L.mx_gemm.restype = i32
    L.mx_gemm.argtypes = [pt, pt, p, i32, i64, p]
    L.gemm_f16.restype = i32
    L.gemm_f16.argtypes = [p, p, p, i32, i64, i64, i64, i64, i64, i64, p]
    pe = ctypes.POINTER(CEpilogue)
    L.mx_gemm_fused.restype = i32
    L.mx_gemm_fused.argtypes = [pt, pt, pe, p, i32, i64, p]
    L.mx_gemm_fused_quantize.restype = i32
    L.mx_gemm_fused_quantize.argtypes = [pt, pt, pe, pt, p]
    L.gemm_f16_fused.restype = i32
    L.gemm_f16_fused.argtypes = [p, p, pe, p, i32, i64, i64, i64, i64, i64,
                                 i64, p]
    L.gemm_dequant.restype = i32
    L.gemm_dequant.argtypes = [p, i32, i64, i64, pt, pe, p, i32, i64, p]
    L.gemm_dequant_splitk.restype = i32
    L.gemm_dequant_splitk.argtypes = [p, i32, i64, i64, pt, pe, p, i32, i64, p,
                                      sz, p]
    L.gemm_dequant_workspace_bytes.restype = sz
    L.gemm_dequant_workspace_bytes.argtypes = [i64, i64, i64]
    L.flash_attention.restype = i32
    L.flash_attention.argtypes = [p, p, p, p, i32, i32, i64, i64, i64, i64,
                                  ctypes.c_float, p]
    L.flash_attention_workspace_bytes.restype = sz
    L.flash_attention_workspace_bytes.argtypes = [i64, i64, i64, i64]
    L.flash_attention_splitkv.restype = i32
    L.flash_attention_splitkv.argtypes = [p, p, p, p, i32, i32, i64, i64, i64,
                                          i64, ctypes.c_float, p, sz, p]
    L.mx_gemm_workspace_bytes.restype = sz
    L.mx_gemm_workspace_bytes.argtypes = [i32, i64, i64, i64]
    L.mx_gemm_splitk.restype = i32
    L.mx_gemm_splitk.argtypes = [pt, pt, p, i32, i64, p, sz, p]
    L.gemm_f16_workspace_bytes.restype = sz
    L.gemm_f16_workspace_bytes.argtypes = [i64, i64, i64]
    L.gemm_f16_splitk.restype = i32
    L.gemm_f16_splitk.argtypes = [p, p, p, i32, i64, i64, i64, i64, i64, i64,
                                  p, sz, p]
    L.mx_gemm_splitk_noalloc.restype = i32
    L.mx_gemm_splitk_noalloc.argtypes = [pt, pt, p, i32, i64, p]
    L.mx_last_error.restype = i32
    L.mx_last_error.argtypes = [p]
    L.mx_selftest_wait_timeout.restype = i32
    L.mx_selftest_wait_timeout.argtypes = [i64, p]
    L.mx_scales_to_rowmajor.restype = i32
    L.mx_scales_to_rowmajor.argtypes = [p, p, i64, i64]
    L.mx_status_string.restype = ctypes.c_char_p
    L.mx_status_string.argtypes = [i32]
    L.mx_version.restype = i32
    L.mx_version.argtypes = []
    L.mx_set_tile_width.restype = i32
    L.mx_set_tile_width.argtypes = [i32]
    _lib = L
    return L


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != 0:
        raise MXError(status, what)


@dataclass
class MXTensor:
    """An MX tensor: data plane and scale plane (device uint8 tensors) of an
    outer x K matrix, K being the contraction axis."""
    data: torch.Tensor
    scales: torch.Tensor
    fmt: int
    outer: int
    K: int

    def c(self) -> CMXTensor:
        return CMXTensor(self.data.data_ptr() if self.data.numel() else None,
                         self.scales.data_ptr() if self.scales.numel() else None,
                         self.fmt, self.outer, self.K)


@functools.lru_cache(maxsize=1024)
def data_bytes(fmt: int, outer: int, K: int) -> int:
    return int(lib().mx_data_bytes(fmt, outer, K))


@functools.lru_cache(maxsize=1024)
def scale_bytes(outer: int, K: int) -> int:
    return int(lib().mx_scale_bytes(outer, K))


def empty_mx(fmt: int, outer: int, K: int, device="cuda") -> MXTensor:
    nd = data_bytes(fmt, outer, K)
    ns = scale_bytes(outer, K)
    return MXTensor(torch.empty(nd, dtype=torch.uint8, device=device),
                    torch.empty(ns, dtype=torch.uint8, device=device),
                    fmt, outer, K)


def _check_mx(t: MXTensor, name: str, fmt=None, outer=None, K=None):
    """An MX tensor's planes are contiguous buffers holding at least the
    bytes the library reads or writes for its format and shape (the C ABI
    receives bare pointers and cannot check their extent)."""
    if ((fmt is not None and t.fmt != fmt) or
            (outer is not None and t.outer != outer) or
            (K is not None and t.K != K)):
        raise ValueError(f"{name} must be format {fmt}, {outer} x {K}")
    for plane, need in ((t.data, data_bytes(t.fmt, t.outer, t.K)),
                        (t.scales, scale_bytes(t.outer, t.K))):
        if not plane.is_contiguous():
            raise ValueError(f"{name}: planes must be contiguous")
        if plane.numel() * plane.element_size() < need:
            raise ValueError(f"{name}: a plane holds fewer than the {need} "
                             "bytes its format and shape need")


def _check_out(out: torch.Tensor, rows: int, cols: int, dtype):
    """A caller-supplied output matrix: of the requested dtype, on the GPU,
    rows x cols with a unit inner stride (its row stride becomes ldc)."""
    if out.dtype != dtype or not out.is_cuda:
        raise ValueError(f"out must be a {dtype} CUDA tensor")
    if out.dim() != 2 or tuple(out.shape) != (rows, cols):
        raise ValueError(f"out must be {rows} x {cols}")
    if cols > 1 and out.stride(1) != 1:
        raise ValueError("out must have a unit inner stride")


def _out_code(dtype, allowed) -> int:
    """The C ABI's code for an output dtype among those a call supports."""
    if dtype not in allowed:
        raise ValueError("out_dtype must be one of %s, not %s"
                         % (", ".join(str(a) for a in allowed), dtype))
    return {torch.float32: DT_F32, torch.bfloat16: DT_BF16,
            torch.float16: DT_F16}[dtype]


def _nbytes(t: torch.Tensor | None) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def mx_quantize(src: torch.Tensor, fmt: int, k_strided: bool = False,
                out: MXTensor | None = None, stream=None) -> MXTensor:
    """Quantize a 2-D fp32 CUDA tensor.  ``k_strided=False``: src is
    outer x K; ``k_strided=True``: src is K x outer (e.g. a row-major K x N
    B operand).  The row stride may exceed the width."""
    if src.dtype != torch.float32 or src.dim() != 2 or not src.is_cuda:
        raise ValueError("src must be a 2-D float32 CUDA tensor")
    if src.stride(1) != 1:
        raise ValueError("src must have a unit inner stride")
    if k_strided:
        K, outer = src.shape
    else:
        outer, K = src.shape
    if out is None:
        out = empty_mx(fmt, outer, K, src.device)
    _check_mx(out, "out", fmt, outer, K)
    ct = out.c()
    _check(lib().mx_quantize(src.data_ptr(), src.stride(0),
                             SRC_K_STRIDED if k_strided else SRC_K_CONTIGUOUS,
                             ctypes.byref(ct), _stream(stream)), "mx_quantize")
    return out


def mx_gemm_workspace_bytes(fmt: int, M: int, N: int, K: int) -> int:
    return int(lib().mx_gemm_workspace_bytes(fmt, M, N, K))


def gemm_f16_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().gemm_f16_workspace_bytes(M, N, K))


def mx_gemm(A: MXTensor, B: MXTensor, out_dtype=torch.bfloat16,
            out: torch.Tensor | None = None, stream=None,
            workspace: torch.Tensor | None = None) -> torch.Tensor:
    """C = A * B for MX tensors A (M x K) and B (quantized from K x N); the
    two may hold different element formats.  With a workspace (a CUDA tensor of at least mx_gemm_workspace_bytes()
    bytes) the K-split entry point is used."""
    dt = _out_code(out_dtype, (torch.float32, torch.bfloat16))
    _check_mx(A, "A")
    _check_mx(B, "B")
    if out is None:
        out = torch.empty((A.outer, B.outer), dtype=out_dtype,
                          device=A.data.device)
    _check_out(out, A.outer, B.outer, out_dtype)
    ca, cb = A.c(), B.c()
    cptr = out.data_ptr() if out.numel() else None
    ldc = out.stride(0)
    if workspace is None:
        _check(lib().mx_gemm(ctypes.byref(ca), ctypes.byref(cb), cptr, dt, ldc,
                             _stream(stream)), "mx_gemm")
    else:
        _check(lib().mx_gemm_splitk(
            ctypes.byref(ca), ctypes.byref(cb), cptr, dt, ldc,
            workspace.data_ptr() if workspace.numel() else None,
            _nbytes(workspace), _stream(stream)),
            "mx_gemm_splitk")
    return out


def gemm_f16(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor | None = None,
             stream=None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """C (fp32) = A * B for row-major fp16 or bf16 CUDA tensors."""
    if A.dtype != B.dtype or A.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("A and B must both be fp16 or both bf16")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check_out(out, M, N, torch.float32)
    dt = DT_F16 if A.dtype == torch.float16 else DT_BF16
    args = (A.data_ptr() if A.numel() else None,
            B.data_ptr() if B.numel() else None,
            out.data_ptr() if out.numel() else None, dt, M, N, K,
            A.stride(0), B.stride(0), out.stride(0))
    if workspace is None:
        _check(lib().gemm_f16(*args, _stream(stream)), "gemm_f16")
    else:
        _check(lib().gemm_f16_splitk(
            *args, workspace.data_ptr() if workspace.numel() else None,
            _nbytes(workspace), _stream(stream)),
            "gemm_f16_splitk")
    return out


def _epilogue(bias, act) -> CEpilogue:
    if bias is not None:
        if (bias.dtype != torch.float32 or bias.dim() != 1 or not bias.is_cuda
                or not bias.is_contiguous()):
            raise ValueError("bias must be a contiguous 1-D float32 CUDA tensor")
    return CEpilogue(bias.data_ptr() if bias is not None and bias.numel() else
                     None, int(act))


def _check_bias(bias, N):
    if bias is not None and bias.numel() != N:
        raise ValueError("bias must hold N values")


def mx_gemm_fused(A: MXTensor, B: MXTensor, bias: torch.Tensor | None = None,
                  act: int = ACT_NONE, out_dtype=torch.bfloat16,
                  out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """C = act(A * B + bias) with the bias and activation applied to the
    fp32 accumulator inside the GEMM epilogue."""
    _check_bias(bias, B.outer)
    dt = _out_code(out_dtype, (torch.float32, torch.bfloat16))
    _check_mx(A, "A")
    _check_mx(B, "B")
    if out is None:
        out = torch.empty((A.outer, B.outer), dtype=out_dtype,
                          device=A.data.device)
    _check_out(out, A.outer, B.outer, out_dtype)
    ca, cb, ep = A.c(), B.c(), _epilogue(bias, act)
    ldc = out.stride(0)
    _check(lib().mx_gemm_fused(ctypes.byref(ca), ctypes.byref(cb),
                               ctypes.byref(ep),
                               out.data_ptr() if out.numel() else None, dt,
                               ldc, _stream(stream)), "mx_gemm_fused")
    return out


def mx_gemm_fused_quantize(A: MXTensor, B: MXTensor, fmt: int,
                           bias: torch.Tensor | None = None,
                           act: int = ACT_NONE, out: MXTensor | None = None,
                           stream=None) -> MXTensor:
    """act(A * B + bias) quantized in the GEMM epilogue to an M x N MX
    tensor (blocks of 32 along N) of element format fmt."""
    _check_bias(bias, B.outer)
    _check_mx(A, "A")
    _check_mx(B, "B")
    if out is None:
        out = empty_mx(fmt, A.outer, B.outer, A.data.device)
    _check_mx(out, "out", fmt, A.outer, B.outer)
    ca, cb, cc, ep = A.c(), B.c(), out.c(), _epilogue(bias, act)
    _check(lib().mx_gemm_fused_quantize(ctypes.byref(ca), ctypes.byref(cb),
                                        ctypes.byref(ep), ctypes.byref(cc),
                                        _stream(stream)),
           "mx_gemm_fused_quantize")
    return out


def gemm_f16_fused(A: torch.Tensor, B: torch.Tensor,
                   bias: torch.Tensor | None = None, act: int = ACT_NONE,
                   out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """C (fp32) = act(A * B + bias) for row-major fp16 or bf16 tensors."""
    if A.dtype != B.dtype or A.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("A and B must both be fp16 or both bf16")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    _check_bias(bias, N)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check_out(out, M, N, torch.float32)
    dt = DT_F16 if A.dtype == torch.float16 else DT_BF16
    ep = _epilogue(bias, act)
    _check(lib().gemm_f16_fused(
        A.data_ptr() if A.numel() else None,
        B.data_ptr() if B.numel() else None, ctypes.byref(ep),
        out.data_ptr() if out.numel() else None, dt, M, N, K, A.stride(0),
        B.stride(0), out.stride(0), _stream(stream)), "gemm_f16_fused")
    return out


def gemm_dequant_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().gemm_dequant_workspace_bytes(M, N, K))


def gemm_dequant(A: torch.Tensor, B: MXTensor, bias: torch.Tensor | None = None,
                 act: int = ACT_NONE, out_dtype=torch.float32,
                 out: torch.Tensor | None = None, stream=None,
                 workspace: torch.Tensor | None = None) -> torch.Tensor:
    """C = act(A * dequant(B)^T + bias) for a row-major fp16 / bf16 A
    (M x K) and an MX tensor B of any format (N x K, quantized from a K x N
    matrix): B is dequantized to A's type in shared or tensor memory, or in
    registers for a single bf16 row with 4- or 2-bit codes.  With a
    workspace (gemm_dequant_workspace_bytes) the K-split entry point runs."""
    if A.dtype not in (torch.float16, torch.bfloat16) or A.dim() != 2:
        raise ValueError("A must be a 2-D fp16 or bf16 tensor")
    if A.stride(1) != 1:
        raise ValueError("A must have a unit inner stride")
    M, K = A.shape
    if K != B.K:
        raise ValueError("inner dimensions differ")
    _check_bias(bias, B.outer)
    dt = _out_code(out_dtype, (torch.float32, torch.bfloat16))
    _check_mx(B, "B")
    if out is None:
        out = torch.empty((M, B.outer), dtype=out_dtype, device=A.device)
    _check_out(out, M, B.outer, out_dtype)
    cb, ep = B.c(), _epilogue(bias, act)
    args = (A.data_ptr() if A.numel() else None,
            DT_F16 if A.dtype == torch.float16 else DT_BF16, M, A.stride(0),
            ctypes.byref(cb), ctypes.byref(ep),
            out.data_ptr() if out.numel() else None, dt,
            out.stride(0))
    if workspace is None:
        _check(lib().gemm_dequant(*args, _stream(stream)), "gemm_dequant")
    else:
        _check(lib().gemm_dequant_splitk(
            *args, workspace.data_ptr() if workspace.numel() else None,
            _nbytes(workspace), _stream(stream)),
            "gemm_dequant_splitk")
    return out


def flash_attention(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor,
                    scale: float | None = None, out_dtype=torch.float32,
                    out: torch.Tensor | None = None, stream=None,
                    workspace: torch.Tensor | None = None) -> torch.Tensor:
    """O = softmax(Q K^T * scale) V per head.  Q is (..., Lq, d), K and V
    (..., Lk, d), contiguous fp16 or bf16 CUDA tensors with the same leading
    dimensions (flattened into heads); scale defaults to 1/sqrt(d).  With a
    device `workspace` (uint8, flash_attention_workspace_bytes() long) the
    key axis is split over SMs that would otherwise idle."""
    if Q.dtype not in (torch.float16, torch.bfloat16) or K.dtype != Q.dtype \
            or V.dtype != Q.dtype:
        raise ValueError("Q, K, V must share an fp16 or bf16 dtype")
    if not (Q.is_contiguous() and K.is_contiguous() and V.is_contiguous()):
        raise ValueError("Q, K, V must be contiguous")
    if K.shape != V.shape or Q.shape[:-2] != K.shape[:-2] or \
            Q.shape[-1] != K.shape[-1]:
        raise ValueError("shape mismatch")
    Lq, d = Q.shape[-2], Q.shape[-1]
    Lk = K.shape[-2]
    BH = Q.numel() // max(1, Lq * d)
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    odt = _out_code(out_dtype, (torch.float32, torch.bfloat16, torch.float16))
    if out is None:
        out = torch.empty(Q.shape, dtype=out_dtype, device=Q.device)
    if (out.dtype != out_dtype or not out.is_cuda or out.shape != Q.shape
            or not out.is_contiguous()):
        raise ValueError("out must be a contiguous CUDA tensor of Q's shape "
                         "and type out_dtype")
    ptr = lambda t: t.data_ptr() if t.numel() else None  # noqa
    dt = DT_F16 if Q.dtype == torch.float16 else DT_BF16
    if workspace is None:
        _check(lib().flash_attention(
            ptr(Q), ptr(K), ptr(V), ptr(out), dt, odt, BH, Lq, Lk, d,
            float(scale), _stream(stream)), "flash_attention")
    else:
        _check(lib().flash_attention_splitkv(
            ptr(Q), ptr(K), ptr(V), ptr(out), dt, odt, BH, Lq, Lk, d,
            float(scale), ptr(workspace), _nbytes(workspace), _stream(stream)),
            "flash_attention_splitkv")
    return out


def flash_attention_workspace_bytes(BH: int, Lq: int, Lk: int, d: int) -> int:
    """Bytes of workspace flash_attention splits into (0: no split)."""
    return int(lib().flash_attention_workspace_bytes(BH, Lq, Lk, d))


def mx_last_error(stream=None) -> int:
    """Synchronize the stream and return (and clear) the library's device
    status (0 = MX_OK, 6 = MX_ERR_TIMEOUT)."""
    return int(lib().mx_last_error(_stream(stream)))


def mx_selftest_wait_timeout(limit_cycles: int, stream=None) -> int:
    return int(lib().mx_selftest_wait_timeout(limit_cycles, _stream(stream)))


def scales_to_rowmajor(tiled, outer: int, K: int):
    """Host helper: tiled scale plane (numpy uint8) -> outer x K/32 array."""
    import numpy as np
    t = np.ascontiguousarray(tiled, dtype=np.uint8)
    out = np.empty((outer, K // 32), dtype=np.uint8)
    _check(lib().mx_scales_to_rowmajor(t.ctypes.data, out.ctypes.data, outer,
                                       K), "mx_scales_to_rowmajor")
    return out


def set_tile_width(tbn: int) -> None:
    """Fix the GEMMs' output-tile width (128 or 256) for later calls, or let
    the library pick it per shape (0, the default)."""
    _check(lib().mx_set_tile_width(int(tbn)), "mx_set_tile_width")
