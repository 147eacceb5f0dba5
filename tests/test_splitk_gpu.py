"""K-split GEMM entry points (mx_gemm_splitk, gemm_f16_splitk) vs the oracle.

Most tests fix the tile width at 128 (the split's tiles), which makes every
shape with a partial wave split; test_auto_plan_splits_long_k leaves the
choice to the library.

The split path applies to problems whose last wave of tiles would leave
clusters idle: those tiles are cut along K, partials go to the workspace and
the last part of each tile to finish adds them in part order, inside the same
launch.  Checked: the workspace size
query, parity against the float64 oracle within the usual tolerance for
shapes that split 2-way and 4-way (ragged edges included), run-to-run bitwise
determinism, and that a missing or too small workspace falls back to the
unsplit path."""
import numpy as np
import pytest
import torch

import block_scaled_quantized_mx_gb300 as mx
import oracle
import workloads
from tests._parity import (check_close, f16_bits, mx_quantize_both, nan_like,
                           oracle_mx_product, planes_from_codes, sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    mx.build()
    mx.lib()


@pytest.fixture(autouse=True)
def _split_tiles():
    """The K-split runs on 128-wide tiles; fixing that width makes the split
    calls split whenever the tiles leave part of a wave idle, so these
    shapes exercise it whatever the library's cost model would pick."""
    mx.set_tile_width(128)
    yield
    mx.set_tile_width(0)


def _ws(nbytes):
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E2M1])
@pytest.mark.parametrize("M,N,K", [(1024, 1024, 1024), (1000, 520, 1056),
                                   (256, 256, 4096), (2304, 2304, 1024)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_mx_splitk_random_codes(fmt, M, N, K, out):
    nbytes = mx.mx_gemm_workspace_bytes(fmt, M, N, K)
    assert nbytes > 0, "this shape is expected to split"
    ca, sa = workloads.random_codes((M, K), fmt, seed=M + 3 * K)
    cb, sb = workloads.random_codes((N, K), fmt, seed=N + 5 * K + 1)
    a, b = planes_from_codes(ca, sa, fmt), planes_from_codes(cb, sb, fmt)
    odt = torch.bfloat16 if out == "bf16" else torch.float32
    C = nan_like((M, N), odt)
    ws = _ws(nbytes)
    ws.fill_(0xFF)                         # garbage in, must not matter
    mx.mx_gemm(a, b, out_dtype=odt, out=C, workspace=ws)
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_mx(ca, sa, cb, sb, fmt)
    check_close(C.float().cpu().numpy(), Cr, S, out, f"split {M}x{N}x{K}")
    C2 = nan_like((M, N), odt)
    mx.mx_gemm(a, b, out_dtype=odt, out=C2, workspace=ws)
    assert torch.equal(C.view(torch.uint8), C2.view(torch.uint8))


def test_mx_splitk_small_workspace_falls_back():
    fmt, M, N, K = oracle.E4M3, 1024, 1024, 1024
    nbytes = mx.mx_gemm_workspace_bytes(fmt, M, N, K)
    ca, sa = workloads.random_codes((M, K), fmt, 1)
    cb, sb = workloads.random_codes((N, K), fmt, 2)
    a, b = planes_from_codes(ca, sa, fmt), planes_from_codes(cb, sb, fmt)
    C_unsplit = mx.mx_gemm(a, b, out_dtype=torch.float32)
    C_small = mx.mx_gemm(a, b, out_dtype=torch.float32,
                         workspace=_ws(nbytes - 16))
    assert torch.equal(C_unsplit, C_small)        # same (unsplit) kernel path
    C_split = mx.mx_gemm(a, b, out_dtype=torch.float32, workspace=_ws(nbytes))
    Cr, S = oracle.gemm_mx(ca, sa, cb, sb, fmt)
    for Cg in (C_unsplit, C_split):
        check_close(Cg.cpu().numpy(), Cr, S, "f32", "fallback")


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", [(1024, 1024, 1024), (2304, 2304, 1024),
                                   (520, 776, 2048)])
def test_f16_splitk(dt, M, N, K):
    nbytes = mx.gemm_f16_workspace_bytes(M, N, K)
    assert nbytes > 0
    g = torch.Generator().manual_seed(M * 7 + N)
    A = (torch.rand(M, K, generator=g) * 2 - 1).to(dt)
    B = (torch.rand(K, N, generator=g) * 2 - 1).to(dt)
    C = nan_like((M, N), torch.float32)
    mx.gemm_f16(A.cuda(), B.cuda(), out=C, workspace=_ws(nbytes))
    assert mx.mx_last_error() == 0
    rows = sample_rows(M, seed=3) if M > 1024 else None
    Cr, S = oracle.gemm_f16(f16_bits(A), f16_bits(B),
                            oracle.F16 if dt == torch.float16 else oracle.BF16,
                            rows=rows)
    Cg = C.cpu().numpy()
    check_close(Cg if rows is None else Cg[rows], Cr, S, "f32", "f16 split")


@pytest.mark.parametrize("name", ["mxfp8_8192", "mxfp4_4096", "bf16_4096",
                                  "proj_out", "w4a8_2048"])
def test_workloads_splitk_sampled(name):
    c = workloads.case(name)
    A, B = workloads.sources(c)
    rows = sample_rows(c.M, seed=c.seed_b)
    if c.kind in ("f16", "bf16"):
        nbytes = mx.gemm_f16_workspace_bytes(c.M, c.N, c.K)
        C = nan_like((c.M, c.N), torch.float32)
        mx.gemm_f16(A.cuda(), B.cuda(), out=C, workspace=_ws(nbytes))
        Cr, S = oracle.gemm_f16(f16_bits(A), f16_bits(B),
                                oracle.F16 if c.kind == "f16" else oracle.BF16,
                                rows=rows)
    else:
        fa, fb = workloads.formats(c)
        # both E2M1: the FP4-rate kernel; any other pair: the FP8-rate one
        wfmt = fa if fa == fb else oracle.E4M3
        nbytes = mx.mx_gemm_workspace_bytes(wfmt, c.M, c.N, c.K)
        a, b = mx_quantize_both(A, B, fa, fb)
        odt = torch.bfloat16 if c.out == "bf16" else torch.float32
        C = nan_like((c.M, c.N), odt)
        mx.mx_gemm(a, b, out_dtype=odt, out=C, workspace=_ws(nbytes))
        Cr, S = oracle_mx_product(A, B, fa, fb, rows=rows)
    assert mx.mx_last_error() == 0
    check_close(C.float().cpu().numpy()[rows], Cr, S, c.out, name)


def test_mx_splitk_graph_replay():
    """A split call captured in a CUDA graph replays with the same counter
    tag; the completing arrival of each tile returns its counter to zero, so
    every replay reduces correctly and gives the eager call's bits."""
    fmt, M, N, K = oracle.E4M3, 1024, 1024, 2048
    nbytes = mx.mx_gemm_workspace_bytes(fmt, M, N, K)
    assert nbytes > 0
    ca, sa = workloads.random_codes((M, K), fmt, 21)
    cb, sb = workloads.random_codes((N, K), fmt, 22)
    a, b = planes_from_codes(ca, sa, fmt), planes_from_codes(cb, sb, fmt)
    ws = _ws(nbytes)
    ws.fill_(0x5A)
    C_eager = mx.mx_gemm(a, b, out_dtype=torch.float32, workspace=ws)
    torch.cuda.synchronize()
    C = nan_like((M, N), torch.float32)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        mx.mx_gemm(a, b, out_dtype=torch.float32, out=C, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mx.mx_gemm(a, b, out_dtype=torch.float32, out=C, workspace=ws, stream=s)
    for _ in range(3):
        C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert mx.mx_last_error() == 0
        assert torch.equal(C, C_eager)
    Cr, S = oracle.gemm_mx(ca, sa, cb, sb, fmt)
    check_close(C.cpu().numpy(), Cr, S, "f32", "graph replay")


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E2M1])
@pytest.mark.parametrize("M,N,K", [(256, 256, 16384), (128, 1024, 16384)])
def test_auto_plan_splits_long_k(fmt, M, N, K):
    """Few tiles and a long K: the library's own plan splits."""
    mx.set_tile_width(0)
    nbytes = mx.mx_gemm_workspace_bytes(fmt, M, N, K)
    assert nbytes > 0
    ca, sa = workloads.random_codes((M, K), fmt, 31)
    cb, sb = workloads.random_codes((N, K), fmt, 32)
    a, b = planes_from_codes(ca, sa, fmt), planes_from_codes(cb, sb, fmt)
    C = nan_like((M, N), torch.float32)
    mx.mx_gemm(a, b, out_dtype=torch.float32, out=C, workspace=_ws(nbytes))
    assert mx.mx_last_error() == 0
    Cr, S = oracle.gemm_mx(ca, sa, cb, sb, fmt)
    check_close(C.cpu().numpy(), Cr, S, "f32", "auto split")
