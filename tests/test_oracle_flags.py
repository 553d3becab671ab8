"""Pins of the oracle's ambiguity flags, which the parity checker uses to
excuse decisions that sit on a rounding boundary (a group's scale, an
element's code). Each flag must be set where its definition says and stay
rare elsewhere, so that the checker is neither blind nor lax:

* an fp32-source MX group whose amax lies within 2^-20 of a power of two
  (a constant row normalises to 1 - 5.6e-8) is excused; the same row from a
  bf16 source (amax exactly 1) is not;
* an fp32-source FP8 element whose quotient y/s is an E4M3 midpoint up to
  the scale's fp32 rounding (448 * 3.625 / 7 = 232, between 224 and 240) is
  marked a tie;
* a bf16 quant source that is exactly a bf16 midpoint (a SiLU product
  1.0078125 * 1.5 = 1.51171875) is marked, and so is its group, whose
  largest element it is;
* on the workloads' random inputs the flags are rare (bounds a few times
  the measured rates). Runs on the CPU."""
import numpy as np
import torch

import oracle
from swiglu_fp8_activation_gb300 import inputs


def _bits(a):
    return inputs.bf16_bits(torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


def _bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


def test_mx_group_near_a_power_of_two_is_excused_only_from_fp32():
    x = _bits(np.full((1, 64), 3.0))
    w = _bits(np.zeros(64))
    f32 = oracle.rmsnorm_add_quant("mxfp8", x, None, w, eps=1e-6, gemma=True, from_fp32=True)
    b16 = oracle.rmsnorm_add_quant("mxfp8", x, None, w, eps=1e-6, gemma=True, from_fp32=False)
    assert f32["gamb"].all()
    assert not b16["gamb"].any() and (b16["scale"] == 119).all()


def test_fp8_quotient_on_an_e4m3_midpoint_is_a_tie():
    row = np.zeros((1, 128))
    row[0, 0], row[0, 1], row[0, 2] = 7.0, 3.625, 3.5     # 3.5 / 7 * 448 = 224, an E4M3 value
    ref = oracle.rmsnorm_add_quant("block128", _bits(row), None, _bits(np.ones(128)), eps=1e-6, gemma=False,
                                   from_fp32=True)
    tie = (ref["amb"][0] & oracle.AMB_TIE) != 0
    assert tie[1] and not tie[0] and not tie[2] and not tie[3:].any()
    assert abs(ref["t"][0, 1] - 232.0) <= 232.0 * 2.0 ** -22


def _silu_gate(target: float) -> float:
    """A bf16 gate g whose bf16(silu(g)) equals `target`."""
    g = np.arange(0x3F00, 0x4080, dtype=np.uint32)            # bf16 patterns over [0.5, 4)
    gv = (g << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    s = _bf16(gv / (1.0 + np.exp(-gv)))
    hit = np.flatnonzero(s == target)
    assert hit.size, "no gate found"
    return float(gv[hit[0]])


def test_bf16_source_on_a_bf16_midpoint_is_marked_with_its_group():
    g0 = _silu_gate(1.0078125)
    gate, up = np.zeros((1, 128)), np.zeros((1, 128))
    gate[0, 0], up[0, 0] = g0, 1.5                           # a = 1.0078125 * 1.5 = 1.51171875, a bf16 midpoint
    gate[0, 1], up[0, 1] = 1.0, 0.5                          # an ordinary element below it
    gu = _bits(np.concatenate([gate, up], axis=1))
    ref = oracle.swiglu_quant("block128", "silu_mul", gu, from_fp32=False, round_act_bf16=True)
    assert ref["a"][0, 0] == 1.51171875
    assert ref["amb"][0, 0] & oracle.AMB_SRC
    assert not ref["amb"][0, 1] & oracle.AMB_SRC
    assert ref["gamb"].reshape(-1)[0] == 1


def _rates(ref):
    amb = ref["amb"]
    return (float(ref["gamb"].mean()), float(((amb & oracle.AMB_SRC) != 0).mean()),
            float(((amb & oracle.AMB_TIE) != 0).mean()))


def test_flags_are_rare_on_random_rows():
    t = inputs.norm_inputs(64, 6144, seed=1, x_std=3.0, r_std=1.0, w_mean=0.0, w_std=0.1)
    x, r, w = (inputs.bf16_bits(t[k]) for k in ("x", "r", "w"))
    for fmt in ("mxfp8", "block128"):
        gamb, src, tie = _rates(oracle.rmsnorm_add_quant(fmt, x, r, w, eps=1e-6, gemma=True, from_fp32=False))
        assert gamb <= 4e-3 and src <= 2e-3 and tie == 0.0, (fmt, gamb, src, tie)
    gamb, src, tie = _rates(oracle.rmsnorm_add_quant("mxfp8", x, r, w, eps=1e-6, gemma=True, from_fp32=True))
    assert gamb <= 1e-3 and src == 0.0 and tie == 0.0, (gamb, src, tie)
    gamb, src, tie = _rates(oracle.rmsnorm_add_quant("block128", x, r, w, eps=1e-6, gemma=True, from_fp32=True))
    assert src == 0.0 and tie <= 1e-4, (src, tie)
