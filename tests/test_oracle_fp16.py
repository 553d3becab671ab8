"""Pins of the oracle's fp16 activation type (the SGQ_F_FP16 path of the
norm and the standalone quant), independent of its code:

  * decoding of all 65,536 binary16 patterns and rounding of doubles (random
    over every binade, subnormals, exact ties, the overflow threshold) agree
    with numpy's float16, a correctly rounded library conversion;
  * a constant row normalises to (1 + w) up to eps, rounded to fp16 by numpy;
  * the standalone quantiser on fp16 rows gives the MX and FP8 closed forms
    (scale exponent from frexp, amax/448 by numpy fp32 division, codes by
    PyTorch's float8 cast).
"""
import numpy as np
import pytest
import torch

import oracle


def f16_bits(vals):
    return np.asarray(vals, dtype=np.float64).astype(np.float16).view(np.uint16)


def test_decode_all_patterns():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_decode(int(b)) for b in pats])
    nan = np.isnan(want)
    assert (np.isnan(got) == nan).all()
    np.testing.assert_array_equal(got[~nan], want[~nan])


def test_round_matches_numpy():
    rng = np.random.default_rng(0)
    e = rng.integers(-30, 17, size=20000)
    vals = rng.uniform(1.0, 2.0, size=e.size) * 2.0 ** e * np.where(rng.random(e.size) < 0.5, -1, 1)
    # exact ties between adjacent fp16 values, in normal and subnormal binades
    lo = np.arange(0, 65504, 7, dtype=np.float64)
    f = np.unique(lo.astype(np.float16).astype(np.float64))
    ties = (f[:-1] + f[1:]) / 2
    sub = (np.arange(0, 1024) + 0.5) * 2.0 ** -24
    edges = np.array([65504.0, 65519.99, 65520.0, 65535.0, 65536.0, 1e6, 2.0 ** -25, 2.0 ** -25 * 1.0001,
                      2.0 ** -14 * (1 - 2.0 ** -12), 0.0, -0.0])
    for v in (vals, ties, sub, edges):
        with np.errstate(over="ignore"):
            want = v.astype(np.float16).view(np.uint16)
        got = np.array([oracle.f16_round(x) for x in v], dtype=np.uint16)
        np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("c", [1.0, -3.0, 0.25])
@pytest.mark.parametrize("gemma", [True, False])
def test_constant_row_fp16(c, gemma):
    H, eps = 256, 1e-6
    rng = np.random.default_rng(2)
    w = f16_bits(rng.standard_normal(H) * 0.1 + (0.0 if gemma else 1.0))
    x = f16_bits(np.full((3, H), c))
    out = oracle.rmsnorm_add_quant("per_token", x, None, w, eps=eps, gemma=gemma, from_fp32=False, fp16=True)
    wd = w.view(np.float16).astype(np.float64)
    factor = c / np.sqrt(c * c + eps)
    want = (factor * ((1.0 + wd) if gemma else wd)).astype(np.float16).view(np.uint16)
    for i in range(3):
        np.testing.assert_array_equal(out["normed"][i], want)


def test_residual_written_in_fp16():
    rng = np.random.default_rng(3)
    x = f16_bits(rng.standard_normal((2, 64)) * 100)
    r = f16_bits(rng.standard_normal((2, 64)) * 100)
    w = f16_bits(np.ones(64))
    out = oracle.rmsnorm_add_quant("mxfp8", x, r, w, eps=1e-6, gemma=False, from_fp32=False, fp16=True)
    want = (x.view(np.float16).astype(np.float64) + r.view(np.float16).astype(np.float64)).astype(np.float16)
    np.testing.assert_array_equal(out["residual"], want.view(np.uint16))


def _e4m3(t):
    return torch.from_numpy(np.clip(t, -448, 448).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_standalone_quant_fp16_closed_forms():
    rng = np.random.default_rng(4)
    v = (rng.standard_normal((4, 256)) * 2.0 ** rng.integers(-12, 12, size=(4, 1))).astype(np.float16)
    vb, vd = v.view(np.uint16), v.astype(np.float64)
    # MX: exponent floor(log2 amax) - 8, exact power-of-two scaling
    mx = oracle.quantize("mxfp8", vb, fp16=True)
    g = vd.reshape(4, 8, 32)
    amax = np.abs(g).max(axis=2)
    e = np.frexp(amax)[1] - 1 - 8
    np.testing.assert_array_equal(mx["scale"], (e + 127).astype(np.uint8))
    np.testing.assert_array_equal(mx["q"], _e4m3((g * 2.0 ** -e[..., None]).reshape(4, 256)))
    # 1x128 and per-token: s = fp32(amax / 448), codes of the fp32 quotient
    for fmt, gs in (("block128", 128), ("per_token", 256)):
        out = oracle.quantize(fmt, vb, fp16=True)
        g = vd.reshape(4, 256 // gs, gs).astype(np.float32)
        s = np.abs(g).max(axis=2) / np.float32(448.0)
        np.testing.assert_array_equal(out["scale"].reshape(s.shape), s)
        np.testing.assert_array_equal(out["q"], _e4m3((g / s[..., None]).reshape(4, 256)))
