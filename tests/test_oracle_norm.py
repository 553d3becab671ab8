"""Pins of the oracle's residual add + RMSNorm + FP8 quantisation.

Closed forms: a constant row normalises to (1 + w) up to eps; a two-level row
has mean square (a^2 + b^2)/2. A plain RMSNorm of an all-ones row with eps = 0
returns w exactly, which turns the fused op into a standalone quantiser of a
chosen vector; its scales and codes are then checked against the MX / FP8
closed forms and PyTorch's float8 conversion. The page's own statements pin
the rest: the fused bf16-source norm is bit-identical to norm followed by a
standalone quant, and the fp32-source 1x128 norm differs on about 2.2% of
values by one step.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from swiglu_fp8_activation_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(vals):
    return inputs.bf16_bits(inputs.to_bf16(np.asarray(vals, dtype=np.float64)))


def dec(b):
    """bf16 bit patterns -> float64, through PyTorch's bfloat16 dtype."""
    return torch.from_numpy(np.asarray(b, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def quantize_vector(fmt, v_bits, from_fp32=False):
    """Standalone quantisation of a bf16 vector through the fused norm:
    plain weights, all-ones row, eps = 0 -> y = w exactly."""
    v_bits = np.asarray(v_bits, dtype=np.uint16).reshape(1, -1)
    n = v_bits.shape[1]
    ones = np.full((1, n), 0x3F80, dtype=np.uint16)
    out = oracle.rmsnorm_add_quant(fmt, ones, None, v_bits[0], eps=0.0, gemma=False,
                                   from_fp32=from_fp32, normed=True)
    np.testing.assert_array_equal(out["y"][0], dec(v_bits[0]))
    return out


def e4m3_expected(t):
    """E4M3 codes for fp32-exact arguments t: torch's RNE cast, saturated to
    +-448 past the largest finite value (the cast itself returns NaN there)."""
    t = np.asarray(t, dtype=np.float64)
    codes = torch.from_numpy(np.clip(t, -448, 448).astype(np.float32)).to(torch.float8_e4m3fn)
    return codes.view(torch.uint8).numpy()


@pytest.mark.parametrize("c", [1.0, 3.0, -0.5, 100.0, 2.0 ** -10])
@pytest.mark.parametrize("gemma", [True, False])
def test_constant_row_closed_form(c, gemma):
    H, eps = 256, 1e-6
    rng = np.random.default_rng(1)
    w = bits(rng.standard_normal(H) * 0.1)
    for sign_pattern in (np.ones(H), np.where(np.arange(H) % 3 == 0, -1.0, 1.0)):
        x = bits(c * sign_pattern).reshape(1, H)
        out = oracle.rmsnorm_add_quant("mxfp8", x, None, w, eps=eps, gemma=gemma, from_fp32=True)
        cb = dec(x[0])
        wv = dec(w)
        inv = 1.0 / math.sqrt(cb[0] ** 2 + float(np.float32(eps)))
        want = cb * inv * ((1.0 + wv) if gemma else wv)
        np.testing.assert_allclose(out["y"][0], want, rtol=1e-14, atol=0)


def test_two_level_row_mean_square():
    H = 512
    a, b = 3.0, -0.25
    x = bits(np.r_[np.full(H // 2, a), np.full(H // 2, b)]).reshape(1, H)
    w = bits(np.zeros(H))
    out = oracle.rmsnorm_add_quant("block128", x, None, w, eps=0.0, gemma=True, from_fp32=True)
    inv = 1.0 / math.sqrt((a * a + b * b) / 2.0)
    np.testing.assert_allclose(out["y"][0, : H // 2], a * inv, rtol=1e-15)
    np.testing.assert_allclose(out["y"][0, H // 2:], b * inv, rtol=1e-15)


def test_residual_is_added_before_the_norm():
    # x = 3 - r with r = +-1: h = 3 everywhere only if r is added.
    H = 128
    r = np.where(np.arange(H) % 2 == 0, 1.0, -1.0)
    x = bits(3.0 - r).reshape(1, H)
    rb = bits(r).reshape(1, H)
    w = bits(np.zeros(H))
    out = oracle.rmsnorm_add_quant("mxfp8", x, rb, w, eps=0.0, gemma=True, from_fp32=False)
    np.testing.assert_array_equal(out["residual"], np.full((1, H), bits([3.0])[0]))
    np.testing.assert_array_equal(out["y"], np.ones((1, H)))


def test_residual_out_matches_torch_add():
    case = inputs.norm_case_gemma_mx(16, 1024)
    t = inputs.make_norm(case)
    x, r, w = (inputs.bf16_bits(t[k]) for k in ("x", "r", "w"))
    out = oracle.rmsnorm_add_quant("mxfp8", x, r, w, eps=case.eps, gemma=True, from_fp32=False)
    want = inputs.bf16_bits((t["x"].float() + t["r"].float()).bfloat16())
    np.testing.assert_array_equal(out["residual"], want)


def test_unit_row_scales_and_codes():
    # h = 1, w = 0 (Gemma), eps = 1e-6: y = 1/sqrt(1 + eps) -> bf16 1.0.
    H = 256
    x = bits(np.ones(H)).reshape(1, H)
    w = bits(np.zeros(H))
    mx = oracle.rmsnorm_add_quant("mxfp8", x, None, w, eps=1e-6, gemma=True, from_fp32=False)
    assert (mx["normed"] == 0x3F80).all()
    assert (mx["scale"] == 127 - 8).all()         # E8M0 code of 2^-8
    assert (mx["q"] == 0x78).all()                # 1.0 * 2^8 = 256
    # from fp32: amax = 0.9999995 < 1 -> exponent -9 and 511.9997 saturates to 448
    mx32 = oracle.rmsnorm_add_quant("mxfp8", x, None, w, eps=1e-6, gemma=True, from_fp32=True)
    assert (mx32["scale"] == 127 - 9).all()
    assert (mx32["q"] == 0x7E).all()
    b = oracle.rmsnorm_add_quant("block128", x, None, w, eps=1e-6, gemma=True, from_fp32=False)
    assert (b["scale"] == np.float32(1.0) / np.float32(448.0)).all()
    assert (b["q"] == 0x7E).all()


def test_mx_block_scale_at_power_of_two_and_saturation():
    # group 0: amax exactly 2^3; group 1: amax 1.8984375 * 2^3 (saturates to 448)
    v = np.r_[np.linspace(-7.5, 8.0, 32), np.linspace(-3, 1.8984375 * 8, 32)]
    out = quantize_vector("mxfp8", bits(v))
    assert list(out["scale"][0]) == [127 + 3 - 8, 127 + 3 - 8]
    vv = dec(bits(v))
    np.testing.assert_array_equal(out["q"][0], e4m3_expected(vv * 2.0 ** -(3 - 8)))
    assert out["q"][0, 63] == 0x7E   # 486 -> 448


def test_mx_scale_per_group_index():
    # each 32-block has its own binade; scales must come out in block order
    n = 32 * 12
    ks = np.arange(12) * 3 - 17
    v = np.concatenate([(1.0 + np.arange(32) / 40.0) * 2.0 ** k * (-1) ** np.arange(32) for k in ks])
    out = quantize_vector("mxfp8", bits(v))
    np.testing.assert_array_equal(out["scale"][0], (ks + 0 - 8 + 127).astype(np.uint8))
    vv = dec(bits(v))
    e = np.repeat(ks - 8, 32)
    np.testing.assert_array_equal(out["q"][0], e4m3_expected(vv * 2.0 ** -e))
    assert out["q"].shape == (1, n)


@pytest.mark.parametrize("fmt", ["block128", "per_token"])
def test_fp8_scale_is_amax_over_448(fmt):
    rng = np.random.default_rng(5)
    v = rng.standard_normal(512) * np.repeat([0.01, 1.0, 37.0, 1e-3], 128)
    vb = bits(v)
    vv = dec(vb)
    out = quantize_vector(fmt, vb)
    gs = 128 if fmt == "block128" else 512
    amax = np.abs(vv).reshape(-1, gs).max(axis=1).astype(np.float32)
    want_s = amax / np.float32(448.0)
    np.testing.assert_array_equal(out["scale"][0], want_s)
    # the element that equals amax encodes to +-448
    for g in range(512 // gs):
        j = g * gs + int(np.argmax(np.abs(vv[g * gs:(g + 1) * gs])))
        assert out["q"][0, j] & 0x7F == 0x7E
    # codes: the IEEE fp32 quotient (numpy float32 division) rounded to E4M3
    s = np.repeat(want_s, gs)
    t = vv.astype(np.float32) / s
    want = e4m3_expected(t.astype(np.float64))
    np.testing.assert_array_equal(out["q"][0], want)


def test_dequant_within_half_step():
    rng = np.random.default_rng(9)
    v = rng.standard_normal(32 * 64) * 2.0 ** rng.integers(-6, 6, 32 * 64)
    vb = bits(v)
    vv = dec(vb)
    for fmt in ("mxfp8", "block128", "per_token"):
        out = quantize_vector(fmt, vb)
        gs = {"mxfp8": 32, "block128": 128, "per_token": vv.size}[fmt]
        if fmt == "mxfp8":
            scale = 2.0 ** (np.repeat(out["scale"][0].astype(np.int64), gs) - 127)
        else:
            scale = np.repeat(out["scale"][0].astype(np.float64), gs)
        deq = np.array([oracle.e4m3_decode(c) for c in out["q"][0]]) * scale
        t = vv / scale
        # half the E4M3 spacing at |t|: 2^(floor(log2|t|) - 3) / 2 for normals, 2^-10 below 2^-6
        e = np.floor(np.log2(np.maximum(np.abs(t), 2.0 ** -6)))
        half_step = 2.0 ** (e - 4) * scale
        ok = np.abs(t) <= 448
        assert ok.mean() > 0.9
        # FP8 formats: plus half an fp32 ulp of t, since t is the fp32 quotient
        slack = 0.0 if fmt == "mxfp8" else np.abs(vv) * 2.0 ** -24
        assert (np.abs(deq - vv)[ok] <= (half_step * (1 + 1e-12) + slack)[ok]).all(), fmt


def test_zero_and_tiny_groups():
    v = np.r_[np.zeros(32), np.full(32, 2.0 ** -130), np.linspace(1, 2, 64)]
    out = quantize_vector("mxfp8", bits(v))
    assert out["scale"][0, 0] == 0 and (out["q"][0, :32] & 0x7F == 0).all()
    assert out["scale"][0, 1] == 0                        # exponent clamped at -127
    assert (out["q"][0, 32:64] == 0x20).all()            # 2^-130 * 2^127 = 2^-3
    z = quantize_vector("block128", bits(np.r_[np.zeros(128), np.ones(128)]))
    assert z["scale"][0, 0] == 0.0 and (z["q"][0, :128] & 0x7F == 0).all()
    p = quantize_vector("per_token", bits(np.zeros(64)))
    assert p["scale"][0, 0] == 0.0 and (p["q"][0] & 0x7F == 0).all()


@pytest.mark.parametrize("fmt", ["mxfp8", "block128", "per_token"])
def test_bf16_source_equals_norm_then_standalone_quant(fmt):
    # The fused bf16-source norm is bit-identical to rounding the normed rows
    # to bf16 and quantising them separately.
    case = inputs.norm_case_gemma_mx(8, 1024)
    t = inputs.make_norm(case)
    x, r, w = (inputs.bf16_bits(t[k]) for k in ("x", "r", "w"))
    fused = oracle.rmsnorm_add_quant(fmt, x, r, w, eps=case.eps, gemma=True, from_fp32=False)
    for i in range(case.M):
        alone = quantize_vector(fmt, fused["normed"][i])
        np.testing.assert_array_equal(fused["q"][i], alone["q"][0])
        np.testing.assert_array_equal(fused["scale"][i], alone["scale"][0])


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                out[k] = float(v)
    return out


def test_fp32_source_block128_differs_from_bf16_source_like_the_page():
    g = _golden("rmsnorm_block128_fp32_vs_bf16.txt")
    case = inputs.norm_case_block128(64, 4096)
    t = inputs.make_norm(case)
    x, w = inputs.bf16_bits(t["x"]), inputs.bf16_bits(t["w"])
    a = oracle.rmsnorm_add_quant("block128", x, None, w, eps=case.eps, gemma=False, from_fp32=True)
    b = oracle.rmsnorm_add_quant("block128", x, None, w, eps=case.eps, gemma=False, from_fp32=False)
    sm = lambda q: np.where(q & 0x80, -(q & 0x7F).astype(np.int64), (q & 0x7F).astype(np.int64))
    step = np.abs(sm(a["q"]) - sm(b["q"]))
    frac = (step != 0).mean()
    assert step.max() <= g["max_step"]
    assert frac <= g["max_mismatch_fraction"]
    assert 0.5 * g["typical_mismatch_fraction"] <= frac <= 2.0 * g["typical_mismatch_fraction"], frac
    # scales differ only within the bf16 rounding of the group amax (half a bf16
    # ulp: at most 2^-8 relative)
    rel = np.abs(a["scale"].astype(np.float64) / b["scale"].astype(np.float64) - 1.0)
    assert rel.max() <= 2.0 ** -8 * (1 + 1e-6)


@pytest.mark.parametrize("fmt", ["mxfp8", "block128", "per_token"])
def test_standalone_quantize_matches_the_fused_norm_route(fmt):
    # The standalone quant of bf16 rows equals the quantiser reached through a
    # plain RMSNorm of an all-ones row with eps = 0 (which returns w), and the
    # unfused chain norm -> bf16 -> standalone quant equals the fused
    # bf16-source norm, bit for bit.
    rng = np.random.default_rng(12)
    v = bits(rng.standard_normal((3, 512)) * 2.0 ** rng.integers(-8, 8, (3, 1)))
    alone = oracle.quantize(fmt, v)
    for i in range(3):
        via_norm = quantize_vector(fmt, v[i])
        np.testing.assert_array_equal(alone["q"][i], via_norm["q"][0])
        np.testing.assert_array_equal(alone["scale"][i], via_norm["scale"][0])
    case = inputs.norm_case_gemma_mx(4, 1024)
    t = inputs.make_norm(case)
    x, r, w = (inputs.bf16_bits(t[k]) for k in ("x", "r", "w"))
    fused = oracle.rmsnorm_add_quant(fmt, x, r, w, eps=case.eps, gemma=True, from_fp32=False)
    chain = oracle.quantize(fmt, fused["normed"])
    np.testing.assert_array_equal(chain["q"], fused["q"])
    np.testing.assert_array_equal(chain["scale"], fused["scale"])
