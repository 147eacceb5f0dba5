"""flash_attention on the GPU vs the float64 oracle.

Tolerance (per element, Sv = sum_j w_j |v_jc| from the oracle): the kernel
rounds each probability p_j to the operand type (relative error at most the
unit roundoff u = 2^-8 for bf16, 2^-11 for f16) before the product with V
and divides by the fp32 sum of the unrounded p, so each weight differs from
softmax by at most u relative and each output by at most u Sv; the bound
used allows twice that (2^-7 Sv / 2^-10 Sv), plus one ulp of a 16-bit
output.  The fp32 scores, the sum and the hardware 2^x add far less.

Covered: d = 64 and 128, both operand types, fp32 / bf16 / f16 outputs,
ragged query and key counts (a partial last key block, a single key, a
single query), a long key sequence whose maximum grows by more than 2^8
many times (the path that moves the exponentials' reference point and
rescales O), the closed form Q = 0, determinism, and sampled rows of the
full-size workloads.  The key-split entry point (flash_attention_splitkv):
decode-like shapes with fewer units than SMs, a last partial wave beside
whole waves, ranges whose maxima differ widely (the merge's reweighting),
16-bit outputs, determinism, and the workspace rule."""
import numpy as np
import pytest
import torch

import block_scaled_quantized_mx_gb300 as mx
import oracle
import workloads
from tests._parity import nan_like, ulp_bf16

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 2.0 ** -7, torch.float16: 2.0 ** -10}


@pytest.fixture(scope="module", autouse=True)
def _built():
    mx.build()
    mx.lib()


def _bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _ulp_f16(x):
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (np.maximum(e, -14) - 10), 2.0 ** -24)


def _check(O, Q, K, V, scale=None, rows=None, what=""):
    code = oracle.BF16 if Q.dtype == torch.bfloat16 else oracle.F16
    Oref, Sv = oracle.attention(_bits(Q), _bits(K), _bits(V), code,
                                scale=scale, rows=rows)
    Og = O.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        Og = Og[:, rows]
    assert np.isfinite(Og).all(), f"{what}: non-finite output"
    bound = TOL[Q.dtype] * Sv
    if O.dtype == torch.bfloat16:
        bound = bound + ulp_bf16(Oref)
    elif O.dtype == torch.float16:
        bound = bound + _ulp_f16(Oref)
    err = np.abs(Og - Oref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} out of "
                           f"tolerance; worst ratio {(err / bound).max():.3g}")
    return float((err / np.maximum(Sv, 1e-30)).max())


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("BH,Lq,Lk", [(2, 256, 256), (3, 200, 300),
                                      (1, 1, 77), (2, 130, 1),
                                      (1, 384, 1000)])
def test_attention_shapes(dt, d, BH, Lq, Lk):
    g = torch.Generator().manual_seed(BH + Lq + 7 * Lk + d)
    Q = torch.randn(BH, Lq, d, generator=g).to(dt)
    K = torch.randn(BH, Lk, d, generator=g).to(dt)
    V = torch.randn(BH, Lk, d, generator=g).to(dt)
    O = nan_like((BH, Lq, d), torch.float32)
    mx.flash_attention(Q.cuda(), K.cuda(), V.cuda(), out=O)
    assert mx.mx_last_error() == 0
    _check(O, Q, K, V, what=f"{dt} d{d} {BH}x{Lq}x{Lk}")


@pytest.mark.parametrize("odt", [torch.bfloat16, torch.float16])
def test_attention_16bit_output(odt):
    g = torch.Generator().manual_seed(3)
    Q, K, V = (torch.randn(2, 256, 128, generator=g).to(torch.bfloat16)
               for _ in range(3))
    O = mx.flash_attention(Q.cuda(), K.cuda(), V.cuda(), out_dtype=odt)
    assert mx.mx_last_error() == 0
    _check(O, Q, K, V, what=str(odt))


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_attention_growing_maximum(dt):
    """Keys whose norm grows along the sequence, with a large scale: the row
    maximum increases in every key block, so every block rescales O."""
    g = torch.Generator().manual_seed(11)
    Lk = 1536
    Q = torch.randn(2, 256, 64, generator=g).to(dt)
    grow = torch.linspace(0.2, 3.0, Lk).reshape(1, Lk, 1)
    K = (torch.randn(2, Lk, 64, generator=g).abs() * grow).to(dt)
    Q = Q.abs()
    V = torch.randn(2, Lk, 64, generator=g).to(dt)
    O = mx.flash_attention(Q.cuda(), K.cuda(), V.cuda(), scale=0.5)
    assert mx.mx_last_error() == 0
    _check(O, Q, K, V, scale=0.5, what="growing maximum")


def test_attention_zero_queries_average_values():
    g = torch.Generator().manual_seed(2)
    Q = torch.zeros(2, 130, 128, dtype=torch.bfloat16)
    K = torch.randn(2, 700, 128, generator=g).to(torch.bfloat16)
    V = torch.randn(2, 700, 128, generator=g).to(torch.bfloat16)
    O = mx.flash_attention(Q.cuda(), K.cuda(), V.cuda()).cpu().numpy()
    assert mx.mx_last_error() == 0
    mean = V.double().numpy().mean(axis=1, keepdims=True)
    # equal weights, each exactly representable: only fp32 sums remain
    assert np.allclose(O, np.repeat(mean, 130, axis=1), rtol=0, atol=1e-4)


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("name", ["attn_sam_d64", "attn_sam_d128",
                                  "attn_long_d128"])
def test_attention_workload_sampled(name, split):
    """The benchmark's attention workloads at full size, through both entry
    points (the split one as the benchmark launches it)."""
    c = workloads.attn_case(name)
    Q, K, V = workloads.attn_sources(c)
    O = nan_like((c.BH, c.Lq, c.d), torch.float32)
    nbytes = mx.flash_attention_workspace_bytes(c.BH, c.Lq, c.Lk, c.d)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") \
        if split else None
    mx.flash_attention(Q.cuda(), K.cuda(), V.cuda(), out=O, workspace=ws)
    assert mx.mx_last_error() == 0
    g = np.random.default_rng(c.seed)
    rows = sorted(set([0, 127, 128, c.Lq - 1] +
                      g.integers(0, c.Lq, 8).tolist()))
    _check(O, Q, K, V, rows=rows, what=name)


@pytest.mark.parametrize("Lk", [256, 300])
def test_attention_zero_scale_averages_values(Lk):
    """scale = 0: every key gets the same weight, so each output row is the
    mean of V's rows (full key blocks fold the scale into the exponent,
    the partial last block of Lk = 300 scales and masks)."""
    g = torch.Generator().manual_seed(17)
    Q, K = (torch.randn(2, 200, 64, generator=g).to(torch.bfloat16)
            for _ in range(2))
    K = torch.randn(2, Lk, 64, generator=g).to(torch.bfloat16)
    V = torch.randn(2, Lk, 64, generator=g).to(torch.bfloat16)
    O = mx.flash_attention(Q.cuda(), K.cuda(), V.cuda(), scale=0.0)
    assert mx.mx_last_error() == 0
    mean = V.double().numpy().mean(axis=1, keepdims=True)
    assert np.allclose(O.cpu().numpy(), np.repeat(mean, 200, axis=1), rtol=0,
                       atol=1e-4)


def test_attention_deterministic():
    g = torch.Generator().manual_seed(6)
    Q, K, V = (torch.randn(4, 512, 128, generator=g).to(torch.bfloat16).cuda()
               for _ in range(3))
    O1 = mx.flash_attention(Q, K, V)
    O2 = mx.flash_attention(Q, K, V)
    assert torch.equal(O1, O2)


def test_attention_negative_scale():
    """A negative scale turns the largest dot product into the smallest
    score: the maximum must be taken over the scaled scores."""
    g = torch.Generator().manual_seed(13)
    Q, K, V = (torch.randn(2, 200, 64, generator=g).to(torch.bfloat16)
               for _ in range(3))
    O = mx.flash_attention(Q.cuda(), K.cuda(), V.cuda(), scale=-0.3)
    assert mx.mx_last_error() == 0
    _check(O, Q, K, V, scale=-0.3, what="negative scale")


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _split_call(Q, K, V, **kw):
    BH = Q.numel() // (Q.shape[-2] * Q.shape[-1])
    nbytes = mx.flash_attention_workspace_bytes(BH, Q.shape[-2], K.shape[-2],
                                                Q.shape[-1])
    assert nbytes > 0, "expected a split for this shape"
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    return mx.flash_attention(Q, K, V, workspace=ws, **kw), ws


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("BH,Lq,Lk", [(2, 128, 4096), (3, 300, 1000),
                                      (1, 1, 777), (8, 256, 2048),
                                      (1, 513, 600)])
def test_attention_splitkv_shapes(dt, d, BH, Lq, Lk):
    """Fewer (head, 256-query) units than SMs: every unit is split along the
    keys (ragged ranges, a partial last key block in the last range)."""
    g = torch.Generator().manual_seed(BH * 3 + Lq + Lk + d)
    Q = torch.randn(BH, Lq, d, generator=g).to(dt)
    K = torch.randn(BH, Lk, d, generator=g).to(dt)
    V = torch.randn(BH, Lk, d, generator=g).to(dt)
    O = nan_like((BH, Lq, d), torch.float32)
    _split_call(Q.cuda(), K.cuda(), V.cuda(), out=O)
    assert mx.mx_last_error() == 0
    _check(O, Q, K, V, what=f"split {dt} d{d} {BH}x{Lq}x{Lk}")


@pytest.mark.parametrize("odt", [torch.bfloat16, torch.float16])
def test_attention_splitkv_16bit_output(odt):
    g = torch.Generator().manual_seed(21)
    Q, K, V = (torch.randn(2, 256, 128, generator=g).to(torch.bfloat16)
               for _ in range(3))
    K = torch.randn(2, 2048, 128, generator=g).to(torch.bfloat16)
    V = torch.randn(2, 2048, 128, generator=g).to(torch.bfloat16)
    O, _ = _split_call(Q.cuda(), K.cuda(), V.cuda(), out_dtype=odt)
    assert mx.mx_last_error() == 0
    _check(O, Q, K, V, what=f"split {odt}")


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_attention_splitkv_growing_maximum(dt):
    """Ranges of keys whose maxima differ by tens of powers of two: the
    merge must weight each range by 2^(m_p - M)."""
    g = torch.Generator().manual_seed(12)
    Lk = 1536
    Q = torch.randn(2, 256, 64, generator=g).abs().to(dt)
    grow = torch.linspace(0.2, 3.0, Lk).reshape(1, Lk, 1)
    K = (torch.randn(2, Lk, 64, generator=g).abs() * grow).to(dt)
    V = torch.randn(2, Lk, 64, generator=g).to(dt)
    O, _ = _split_call(Q.cuda(), K.cuda(), V.cuda(), scale=0.5)
    assert mx.mx_last_error() == 0
    _check(O, Q, K, V, scale=0.5, what="split growing maximum")


def test_attention_splitkv_tail_beside_whole_waves():
    """Five units more than one per SM: a whole wave of units runs unsplit,
    the five left over are split; sampled rows of every head against the
    oracle."""
    sms = _sms()
    BH, Lq, Lk, d = sms + 5, 256, 1024, 64
    g = torch.Generator().manual_seed(31)
    Q = torch.randn(BH, Lq, d, generator=g).to(torch.bfloat16)
    K = torch.randn(BH, Lk, d, generator=g).to(torch.bfloat16)
    V = torch.randn(BH, Lk, d, generator=g).to(torch.bfloat16)
    O = nan_like((BH, Lq, d), torch.float32)
    _split_call(Q.cuda(), K.cuda(), V.cuda(), out=O)
    assert mx.mx_last_error() == 0
    _check(O, Q, K, V, rows=[0, 77, 128, 255], what="tail beside whole waves")


def test_attention_splitkv_deterministic_and_close_to_unsplit():
    g = torch.Generator().manual_seed(8)
    Q = torch.randn(4, 256, 128, generator=g).to(torch.bfloat16).cuda()
    K = torch.randn(4, 4096, 128, generator=g).to(torch.bfloat16).cuda()
    V = torch.randn(4, 4096, 128, generator=g).to(torch.bfloat16).cuda()
    O1, ws = _split_call(Q, K, V)
    O2 = mx.flash_attention(Q, K, V, workspace=ws)
    assert torch.equal(O1, O2)
    O0 = mx.flash_attention(Q, K, V)
    assert mx.mx_last_error() == 0
    # both are within the same bound of the exact result; they differ only
    # in how the sums are grouped
    assert (O1 - O0).abs().max().item() < 1e-3


def test_attention_splitkv_small_workspace_runs_unsplit():
    g = torch.Generator().manual_seed(9)
    Q = torch.randn(2, 256, 64, generator=g).to(torch.bfloat16).cuda()
    K = torch.randn(2, 1024, 64, generator=g).to(torch.bfloat16).cuda()
    V = torch.randn(2, 1024, 64, generator=g).to(torch.bfloat16).cuda()
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    O1 = mx.flash_attention(Q, K, V, workspace=ws)
    O0 = mx.flash_attention(Q, K, V)
    assert mx.mx_last_error() == 0
    assert torch.equal(O1, O0)


def test_attention_workspace_rule():
    sms = _sms()
    assert mx.flash_attention_workspace_bytes(sms, 256, 4096, 128) == 0  # whole wave
    assert mx.flash_attention_workspace_bytes(2, 256, 128, 128) == 0     # one key block
    assert mx.flash_attention_workspace_bytes(2, 256, 4096, 128) > 0
    n = mx.flash_attention_workspace_bytes(sms + 1, 256, 4096, 64)
    # one tail unit, 16 parts of 256 rows x (64 + 2) floats
    assert n == 16 * 256 * 66 * 4
