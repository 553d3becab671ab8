"""GPU parity of the scale layouts for GEMM consumers (SGQ_F_SCALE_SWIZZLED
for MXFP8, SGQ_F_SCALE_COL_MAJOR for 1x128): the kernels' rearranged scales
equal the oracle's rearrangement of the row-major scales, byte for byte and
padding included; the E4M3 values do not change with the layout; nothing is
written past the scale buffer. A block-scaled GEMM from a library (cuBLASLt
through torch._scaled_mm) then consumes swizzled scales, from the oracle and
from the kernels, and must reproduce the fp64 product of the dequantised
operands: the layout is the one such consumers read.
"""
import numpy as np
import pytest
import torch

import oracle
from swiglu_fp8_activation_gb300 import (inputs, quantize_fp8, rmsnorm_add_quant, scale_shape, swiglu_quant)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GUARD = 256


def _bits(t):
    return inputs.bf16_bits(t.cpu())


def _guarded_scale(fmt, M, W, layout):
    """A scale tensor of the layout's shape inside a larger buffer filled with
    0xFF bytes (an E8M0 NaN, a float32 NaN), so that unwritten padding and
    writes past the end both show."""
    shape = scale_shape(fmt, M, W, layout)
    n = int(np.prod(shape))
    esz = 1 if fmt == "mxfp8" else 4
    raw = torch.full(((n + GUARD) * esz,), 0xFF, dtype=torch.uint8, device=DEV)
    view = raw[:n * esz] if esz == 1 else raw[:n * esz].view(torch.float32)
    return raw, view.view(shape), n * esz


def _check_guard(raw, nbytes):
    assert (raw[nbytes:] == 0xFF).all(), "bytes written past the scale buffer"


def _rearranged(fmt, row_scale, layout):
    return oracle.scale_layout(fmt, row_scale.cpu().numpy(), layout)


MX_SHAPES = [(1, 6144), (8, 4160), (200, 4160), (256, 6144), (129, 96)]


@pytest.mark.parametrize("M,W", MX_SHAPES)
def test_swizzled_mx_quantize(M, W):
    src = (torch.randn(M, W, generator=torch.Generator().manual_seed(M + W)) * 4).to(torch.bfloat16).to(DEV)
    q_r, s_r = quantize_fp8(src, fmt="mxfp8")
    raw, s_view, nb = _guarded_scale("mxfp8", M, W, "swizzled")
    q_s, s_s = quantize_fp8(src, fmt="mxfp8", scale_out=s_view, scale_layout="swizzled")
    torch.cuda.synchronize()
    assert torch.equal(q_r, q_s)
    np.testing.assert_array_equal(s_s.cpu().numpy(), _rearranged("mxfp8", s_r, "swizzled"))
    # and against the oracle's own scales
    ref = oracle.quantize("mxfp8", _bits(src))
    np.testing.assert_array_equal(s_s.cpu().numpy(), oracle.scale_layout("mxfp8", ref["scale"], "swizzled"))
    _check_guard(raw, nb)


@pytest.mark.parametrize("M,H", [(1, 6144), (37, 4160), (256, 6144)])
def test_swizzled_mx_norm(M, H):
    t = inputs.norm_inputs(M, H, seed=M, x_std=3.0, r_std=1.0, w_mean=0.0, w_std=0.1)
    x, r, w = t["x"].to(DEV), t["r"].to(DEV), t["w"].to(DEV)
    q_r, s_r, n_r, ro_r = rmsnorm_add_quant(x, w, residual_in=r, residual_out=torch.empty_like(r), normed=True)
    raw, s_view, nb = _guarded_scale("mxfp8", M, H, "swizzled")
    q_s, s_s, n_s, ro_s = rmsnorm_add_quant(x, w, residual_in=r, residual_out=torch.empty_like(r), normed=True,
                                            scale_out=s_view, scale_layout="swizzled")
    torch.cuda.synchronize()
    assert torch.equal(q_r, q_s) and torch.equal(n_r, n_s) and torch.equal(ro_r, ro_s)
    np.testing.assert_array_equal(s_s.cpu().numpy(), _rearranged("mxfp8", s_r, "swizzled"))
    _check_guard(raw, nb)


def test_swizzled_mx_norm_zero_eps_padding_rows():
    # eps = 0: the padding rows of the layout must still come out as code 0
    M, H = 3, 2048
    t = inputs.norm_inputs(M, H, seed=5, x_std=1.0, r_std=None, w_mean=1.0, w_std=0.1)
    raw, s_view, nb = _guarded_scale("mxfp8", M, H, "swizzled")
    _, s_s, _, _ = rmsnorm_add_quant(t["x"].to(DEV), t["w"].to(DEV), eps=0.0, gemma=False, scale_out=s_view,
                                     scale_layout="swizzled")
    _, s_r, _, _ = rmsnorm_add_quant(t["x"].to(DEV), t["w"].to(DEV), eps=0.0, gemma=False)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(s_s.cpu().numpy(), _rearranged("mxfp8", s_r, "swizzled"))
    _check_guard(raw, nb)


@pytest.mark.parametrize("M,I", [(8, 768), (200, 3072), (128, 96 * 8)])
def test_swizzled_mx_swiglu(M, I):
    gu = inputs.swiglu_inputs(M, I, seed=M + I, std=2.0).to(DEV)
    q_r, s_r = swiglu_quant(gu)
    raw, s_view, nb = _guarded_scale("mxfp8", M, I, "swizzled")
    q_s, s_s = swiglu_quant(gu, scale_out=s_view, scale_layout="swizzled")
    torch.cuda.synchronize()
    assert torch.equal(q_r, q_s)
    np.testing.assert_array_equal(s_s.cpu().numpy(), _rearranged("mxfp8", s_r, "swizzled"))
    _check_guard(raw, nb)


@pytest.mark.parametrize("M", [1, 5, 37, 256])
def test_col_major_block128(M):
    t = inputs.norm_inputs(M, 4096, seed=M, x_std=1.0, r_std=None, w_mean=1.0, w_std=0.1)
    x, w = t["x"].to(DEV), t["w"].to(DEV)
    q_r, s_r, _, _ = rmsnorm_add_quant(x, w, fmt="block128", gemma=False, quant_from_fp32=True)
    raw, s_view, nb = _guarded_scale("block128", M, 4096, "col_major")
    q_c, s_c, _, _ = rmsnorm_add_quant(x, w, fmt="block128", gemma=False, quant_from_fp32=True, scale_out=s_view,
                                       scale_layout="col_major")
    torch.cuda.synchronize()
    assert torch.equal(q_r, q_c)
    np.testing.assert_array_equal(s_c.cpu().numpy(), _rearranged("block128", s_r, "col_major"))
    _check_guard(raw, nb)

    gu = inputs.swiglu_inputs(M, 12288, seed=M, std=1.0).to(DEV)
    q_r, s_r = swiglu_quant(gu, fmt="block128", act="silu_mul", quant_from_fp32=False, round_act_bf16=True)
    raw, s_view, nb = _guarded_scale("block128", M, 12288, "col_major")
    q_c, s_c = swiglu_quant(gu, fmt="block128", act="silu_mul", quant_from_fp32=False, round_act_bf16=True,
                            scale_out=s_view, scale_layout="col_major")
    src = gu[:, :2048].contiguous()
    q_q, s_q = quantize_fp8(src, fmt="block128")
    raw2, s_view2, nb2 = _guarded_scale("block128", M, 2048, "col_major")
    q_q2, s_q2 = quantize_fp8(src, fmt="block128", scale_out=s_view2, scale_layout="col_major")
    torch.cuda.synchronize()
    assert torch.equal(q_r, q_c) and torch.equal(q_q, q_q2)
    np.testing.assert_array_equal(s_c.cpu().numpy(), _rearranged("block128", s_r, "col_major"))
    np.testing.assert_array_equal(s_q2.cpu().numpy(), _rearranged("block128", s_q, "col_major"))
    _check_guard(raw, nb)
    _check_guard(raw2, nb2)


# ------------------------------------------------------- a library consumer

_E4M3 = None


def _deq_mx(q, scale_rows):
    global _E4M3
    if _E4M3 is None:
        _E4M3 = np.array([oracle.e4m3_decode(c) for c in range(256)])
    return _E4M3[q] * np.repeat(2.0 ** (scale_rows.astype(np.int64) - 127), 32, axis=1)


def _scaled_mm(qa, sa_swz, qb, sb_swz):
    """cuBLASLt MXFP8 GEMM: A [M,K] E4M3, B [N,K] E4M3, swizzled E8M0 scales."""
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("this torch has no float8_e8m0fnu dtype")
    a = qa.view(torch.float8_e4m3fn)
    b = qb.view(torch.float8_e4m3fn).t()
    try:
        return torch._scaled_mm(a, b, sa_swz.view(torch.float8_e8m0fnu), sb_swz.view(torch.float8_e8m0fnu),
                                out_dtype=torch.bfloat16)
    except (RuntimeError, NotImplementedError) as e:   # capability, not a layout mismatch
        pytest.skip(f"block-scaled MXFP8 GEMM not available here: {str(e).splitlines()[0]}")


def _close(out, ref):
    out = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(out - ref)
    # bf16 output rounding (2^-9 relative) plus fp32 accumulation; a scale
    # read from the wrong place is off by powers of two
    assert err.max() <= 2.0 ** -6 * np.abs(ref).max(), err.max() / np.abs(ref).max()
    assert np.median(err / np.maximum(np.abs(ref), 1e-30)) <= 2.0 ** -7


@pytest.mark.parametrize("M,N,K", [(200, 256, 4096), (64, 128, 4160)])
def test_library_gemm_reads_the_oracle_swizzled_scales(M, N, K):
    g = torch.Generator().manual_seed(M + K)
    a = (torch.randn(M, K, generator=g) * 3).to(torch.bfloat16)
    b = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    ra, rb = oracle.quantize("mxfp8", _bits(a)), oracle.quantize("mxfp8", _bits(b))
    sa = torch.from_numpy(oracle.scale_layout("mxfp8", ra["scale"], "swizzled")).to(DEV)
    sb = torch.from_numpy(oracle.scale_layout("mxfp8", rb["scale"], "swizzled")).to(DEV)
    out = _scaled_mm(torch.from_numpy(ra["q"]).to(DEV), sa, torch.from_numpy(rb["q"]).to(DEV), sb)
    ref = _deq_mx(ra["q"], ra["scale"]) @ _deq_mx(rb["q"], rb["scale"]).T
    _close(out, ref)


@pytest.mark.parametrize("M,N,H", [(200, 256, 4096), (8, 128, 6144)])
def test_library_gemm_reads_the_kernels_swizzled_scales(M, N, H):
    t = inputs.norm_inputs(M, H, seed=M, x_std=3.0, r_std=1.0, w_mean=0.0, w_std=0.1)
    x, r, w = t["x"].to(DEV), t["r"].to(DEV), t["w"].to(DEV)
    wb = (torch.randn(N, H, generator=torch.Generator().manual_seed(N)) * 0.05).to(torch.bfloat16).to(DEV)
    qa, sa, _, _ = rmsnorm_add_quant(x, w, residual_in=r, residual_out=torch.empty_like(r), scale_layout="swizzled")
    qb, sb = quantize_fp8(wb, scale_layout="swizzled")
    _, sa_r, _, _ = rmsnorm_add_quant(x, w, residual_in=r, residual_out=torch.empty_like(r))
    _, sb_r = quantize_fp8(wb)
    out = _scaled_mm(qa, sa, qb, sb)
    torch.cuda.synchronize()
    ref = _deq_mx(qa.cpu().numpy(), sa_r.cpu().numpy()) @ _deq_mx(qb.cpu().numpy(), sb_r.cpu().numpy()).T
    _close(out, ref)
