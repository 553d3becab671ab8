"""The two arithmetic shortcuts of the kernels, checked on the GPU:

* sigmoid8() (head/tail split exponent, hardware 2^x with a first-order
  tail correction, refined reciprocal) against fp64 over |z| <= 130, within
  2^-22 relative;
* activation8() (the OAI SwiGLU of the kernels, in its general and its
  pre-clamped form) against fp64, within 2^-21 relative, including an
  element whose exact value lies 3.1e-7 relative above an E4M3 rounding
  boundary;
* div_rn() and div2_rn() (one reciprocal per group + Markstein's FMA
  correction) against CUDA's correctly rounded __fdiv_rn, bit for bit, for
  the FP8 quotients the kernels form (|a| <= b * 448 * (1 + 2^-20), b
  normal), the FP8 scale amax / 448, quotients by integer widths, random
  pairs and signed zero numerators.
"""
import ctypes as C
import os
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def devlib():
    import __graft_entry__ as g
    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libdevice_math_check.so")
    cmd = [g._nvcc(), *g.ARCH, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-I", g.CSRC,
           "-o", so, os.path.join(ROOT, "tests", "cuda", "device_math_check.cu")]
    subprocess.run(cmd, check=True)
    L = C.CDLL(so)
    for f in (L.run_sigmoid, L.run_div, L.run_oai, L.run_oai_clamped):
        f.restype = C.c_int
    return L


def _p(t):
    return C.c_void_p(t.data_ptr())


def test_sigmoid_accuracy(devlib):
    z = np.concatenate([np.linspace(-130, 130, 2_000_001), np.array([0.0, -0.0, 1e-30, -1e-30, 87.3, -87.3, 1e30, -1e30]),
                        np.random.default_rng(0).standard_normal(200_000) * 8]).astype(np.float32)
    z = np.concatenate([z, np.zeros((-z.size) % 8, np.float32)])      # whole chunks of 8
    zt = torch.from_numpy(z).cuda()
    out = torch.empty_like(zt)
    assert devlib.run_sigmoid(_p(zt), _p(out), z.size) == 0
    got = out.cpu().numpy().astype(np.float64)
    zd = z.astype(np.float64)
    with np.errstate(over="ignore"):
        want = 1.0 / (1.0 + np.exp(-zd))
    tiny = want < 2.0 ** -126                       # below the fp32 normal range: absolute check
    rel = np.abs(got - want) / np.where(tiny, 1.0, want)
    assert rel[~tiny].max() <= 2.0 ** -22, rel[~tiny].max()
    assert np.abs(got - want)[tiny].max() <= 2.0 ** -126
    assert (got[z == 0] == 0.5).all()


@pytest.mark.parametrize("clamped", [False, True])
def test_oai_activation_accuracy(devlib, clamped):
    rng = np.random.default_rng(2)
    n = 2_000_000
    g = torch.from_numpy(rng.standard_normal(n) * 4.0).bfloat16().float().numpy()
    u = torch.from_numpy(rng.standard_normal(n) * 4.0).bfloat16().float().numpy()
    # the element that an error of 2.8e-7 pushed across an E4M3 boundary
    g[:2], u[:2] = -1.578125, -3.25
    # gates far below zero, where the sigmoid leaves the normal range and
    # the packed-bf16 kernels clamp from below
    g[8:8 + 4096] = torch.from_numpy(-np.geomspace(30.0, 3.0e4, 4096)).bfloat16().float().numpy()
    alpha, beta, limit = np.float32(1.702), 1.0, 7.0
    gt, ut = torch.from_numpy(g).cuda(), torch.from_numpy(u).cuda()
    out = torch.empty_like(gt)
    if clamped:      # the packed-bf16 kernels' lower gate bound: the bf16 value nearest -139 / alpha
        glo = float(torch.tensor(-139.0 / float(alpha)).bfloat16().float())
        assert devlib.run_oai_clamped(_p(gt), _p(ut), _p(out), n, C.c_float(alpha), C.c_float(beta),
                                      C.c_float(limit), C.c_float(glo)) == 0
    else:
        assert devlib.run_oai(_p(gt), _p(ut), _p(out), n, C.c_float(alpha), C.c_float(beta), C.c_float(limit)) == 0
    got = out.cpu().numpy().astype(np.float64)
    gc = np.minimum(g.astype(np.float64), limit)
    uc = np.clip(u.astype(np.float64), -limit, limit)
    with np.errstate(over="ignore"):            # exp overflows to inf far below zero: want = 0 there
        want = gc / (1.0 + np.exp(-float(alpha) * gc)) * (uc + beta)
    ok = np.abs(want) > 2.0 ** -100
    rel = np.abs(got - want)[ok] / np.abs(want)[ok]
    assert rel.max() <= 2.0 ** -21, rel.max()
    assert np.abs(got[~ok]).max(initial=0) <= 2.0 ** -100
    assert got[0] > 0.2265625          # exact value 0.22656257..., the boundary is 29/128


def test_div_rn_and_packed_form_match_ieee_division(devlib):
    rng = np.random.default_rng(1)
    n = 4_000_000
    # the kernels' case: b = amax / 448, |a| <= amax
    amax = (rng.standard_normal(n) * 2.0 ** rng.integers(-100, 100, n)).astype(np.float32)
    amax = np.abs(amax) + np.float32(2.0 ** -100)
    b = (amax / np.float32(448.0)).astype(np.float32)
    a = (amax * rng.uniform(-1, 1, n)).astype(np.float32)
    # bf16-valued numerators, where exact E4M3 midpoints are common
    a[: n // 4] = torch.from_numpy(a[: n // 4]).bfloat16().float().numpy()
    a[n // 4: n // 2] = amax[n // 4: n // 2] * rng.choice([-1, 1], n // 4)
    # unrelated random pairs
    a2 = (rng.standard_normal(n) * 2.0 ** rng.integers(-60, 60, n)).astype(np.float32)
    b2 = (np.abs(rng.standard_normal(n)) * 2.0 ** rng.integers(-60, 60, n) + 2.0 ** -100).astype(np.float32)
    # the FP8 scale itself: amax / 448 for amax >= 2^-100 (bf16 values and
    # arbitrary fp32 values), where the kernels use RN(1/448) = __frcp_rn(448)
    a3 = np.abs(rng.standard_normal(n) * 2.0 ** rng.integers(-100, 120, n)).astype(np.float32) + np.float32(2.0 ** -100)
    a3[: n // 2] = torch.from_numpy(a3[: n // 2]).bfloat16().float().numpy()
    b3 = np.full(n, 448.0, np.float32)
    # quotients by integer widths (multiples of 8 up to the maximum width)
    a4 = np.abs(rng.standard_normal(n) * 2.0 ** rng.integers(-90, 100, n)).astype(np.float32) + np.float32(2.0 ** -100)
    b4 = (8 * rng.integers(1, 2049, n)).astype(np.float32)
    for aa, bb in ((a, b), (a2, b2), (a3, b3), (a4, b4)):
        at, bt = torch.from_numpy(aa).cuda(), torch.from_numpy(bb).cuda()
        qf, qp, qi = torch.empty_like(at), torch.empty_like(at), torch.empty_like(at)
        assert devlib.run_div(_p(at), _p(bt), _p(qf), _p(qp), _p(qi), n) == 0
        qf, qp, qi = qf.cpu().numpy(), qp.cpu().numpy(), qi.cpu().numpy()
        normal = (np.abs(qi) >= 2.0 ** -126) & np.isfinite(qi)     # overflowing pairs never occur in the kernels
        np.testing.assert_array_equal(qf.view(np.uint32)[normal], qi.view(np.uint32)[normal])
        np.testing.assert_array_equal(qp.view(np.uint32)[normal], qi.view(np.uint32)[normal])
    # zero numerators keep their sign (-0 / b = -0), bit for bit (an FP8 code
    # of a -0 source is 0x80)
    az = np.zeros(1024, np.float32)
    az[1::2] = np.float32(-0.0)
    bz = np.abs(rng.standard_normal(1024) * 2.0 ** rng.integers(-60, 60, 1024)).astype(np.float32) + np.float32(1.0)
    at, bt = torch.from_numpy(az).cuda(), torch.from_numpy(bz).cuda()
    qf, qp, qi = torch.empty_like(at), torch.empty_like(at), torch.empty_like(at)
    assert devlib.run_div(_p(at), _p(bt), _p(qf), _p(qp), _p(qi), 1024) == 0
    qi = qi.cpu().numpy()
    assert (np.signbit(qi) == np.signbit(az)).all()
    np.testing.assert_array_equal(qf.cpu().numpy().view(np.uint32), qi.view(np.uint32))
    np.testing.assert_array_equal(qp.cpu().numpy().view(np.uint32), qi.view(np.uint32))
