"""GPU parity of the fp16 activation path (norm, unfused norm, standalone
quant) and of the two-segment q/kv norm against the oracle.

fp16: "[ROCm] Fuse per-token activation quant into RMSNorm for per-channel
quantized attention" (sglang PR 34502), "Change" (fp16 activations stay
fp16), and the review of "[ROCm][MiniMax-M3.1] Fuse MXFP8 quant into the
add+RMSNorm and SwiGLU epilogues" (vllm PR 65478), whose bitwise norm test
covers bf16 and fp16. q/kv norm: the same sglang page, "Change" (the decode
q_b_proj quant folded into the fused q/kv RMSNorm).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.parity import check_bf16, check_norm, check_quant
from swiglu_fp8_activation_gb300 import inputs, quantize_fp8, rmsnorm_add, rmsnorm_add_quant, rmsnorm_dual_quant

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _f16_norm_inputs(M, H, seed, r_std=1.0, x_std=3.0, w_mean=0.0):
    t = inputs.norm_inputs(M, H, seed=seed, x_std=x_std, r_std=r_std, w_mean=w_mean, w_std=0.1)
    return {k: (None if v is None else v.float().to(torch.float16)) for k, v in t.items()}


@pytest.mark.parametrize("fmt", ["mxfp8", "block128", "per_token"])
@pytest.mark.parametrize("from_fp32", [False, True])
@pytest.mark.parametrize("M,H,residual", [(37, 4096, "separate"), (8, 6144, "inplace"), (300, 8 * 160, None)])
def test_fp16_norm_matches_oracle(fmt, from_fp32, M, H, residual):
    if fmt != "per_token" and H % (32 if fmt == "mxfp8" else 128):
        pytest.skip("width not a multiple of the group")
    t = _f16_norm_inputs(M, H, seed=M + H, r_std=1.0 if residual else None, w_mean=0.0)
    x, w = t["x"].to(DEV), t["w"].to(DEV)
    r = t["r"].to(DEV) if residual else None
    r_out = None if r is None else (r if residual == "inplace" else torch.empty_like(r))
    q, s, n, ro = rmsnorm_add_quant(x, w, fmt=fmt, residual_in=r, residual_out=r_out, gemma=True,
                                    quant_from_fp32=from_fp32, normed=True)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm_add_quant(fmt, _bits(t["x"]), _bits(t["r"]) if residual else None, _bits(t["w"]), eps=1e-6,
                                   gemma=True, from_fp32=from_fp32, fp16=True)
    check_norm(fmt, ref, q.cpu().numpy(), s.cpu().numpy(), _bits(n), _bits(ro) if residual else None,
               from_fp32=from_fp32)


@pytest.mark.parametrize("fmt", ["mxfp8", "block128", "per_token"])
def test_fp16_quantize_exact(fmt):
    M, W = 37, 128 * 33
    g = torch.Generator().manual_seed(9)
    src = (torch.randn(M, W, generator=g) * 2.0 ** torch.randint(-8, 8, (M, 1), generator=g)).to(torch.float16)
    src[0] = 0
    q, s = quantize_fp8(src.to(DEV), fmt=fmt)
    torch.cuda.synchronize()
    ref = oracle.quantize(fmt, _bits(src), fp16=True)
    np.testing.assert_array_equal(q.cpu().numpy(), ref["q"])
    np.testing.assert_array_equal(s.cpu().numpy(), ref["scale"])


@pytest.mark.parametrize("fmt", ["mxfp8", "block128", "per_token"])
def test_fp16_norm_then_quant_equals_fused(fmt):
    M, H = 64, 4096
    t = _f16_norm_inputs(M, H, seed=3)
    x, r, w = t["x"].to(DEV), t["r"].to(DEV), t["w"].to(DEV)
    q_f, s_f, n_f, r_f = rmsnorm_add_quant(x, w, fmt=fmt, residual_in=r, residual_out=torch.empty_like(r), normed=True)
    n_u, r_u = rmsnorm_add(x, w, residual_in=r, residual_out=torch.empty_like(r))
    q_u, s_u = quantize_fp8(n_u, fmt=fmt)
    torch.cuda.synchronize()
    assert n_f.dtype == torch.float16 and torch.equal(n_f, n_u) and torch.equal(r_f, r_u)
    assert torch.equal(q_f, q_u) and torch.equal(s_f, s_u)


# ------------------------------------------------------------- q/kv norm


def _dual_case(M, Ha, Hb, dtype, seed, extra=64):
    """One projection output [M, Ha + Hb + extra] holding q, kv and a tail
    (as the fused q/kv-a projection of latent attention), with weights."""
    g = torch.Generator().manual_seed(seed)
    buf = (torch.randn(M, Ha + Hb + extra, generator=g) * 2).to(dtype)
    wa = (1 + 0.1 * torch.randn(Ha, generator=g)).to(dtype)
    wb = (1 + 0.1 * torch.randn(Hb, generator=g)).to(dtype)
    return buf, wa, wb


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("M", [1, 7, 64, 1000])
@pytest.mark.parametrize("Ha,Hb", [(1536, 512), (8 * 480, 4096), (256, 16384)])
def test_dual_norm_per_token_matches_oracle(dtype, M, Ha, Hb):
    buf, wa, wb = _dual_case(M, Ha, Hb, dtype, seed=M + Ha)
    d = buf.to(DEV)
    (qa, sa, na), (qb, sb, nb) = rmsnorm_dual_quant(d[:, :Ha], wa.to(DEV), d[:, Ha:Ha + Hb], wb.to(DEV),
                                                   fmt="per_token", quant_a=True, normed_a=True, quant_b=False,
                                                   normed_b=True)
    torch.cuda.synchronize()
    assert qb is None and sb is None
    fp16 = dtype == torch.float16
    ra, rb = oracle.rmsnorm_dual_quant("per_token", _bits(buf[:, :Ha]), _bits(wa), _bits(buf[:, Ha:Ha + Hb]), _bits(wb),
                                       eps=1e-6, gemma=False, from_fp32=False, fp16=fp16)
    check_norm("per_token", ra, qa.cpu().numpy(), sa.cpu().numpy(), _bits(na), None, from_fp32=False)
    check_bf16("normed_b", rb["normed"], _bits(nb))


@pytest.mark.parametrize("fmt", ["mxfp8", "block128"])
@pytest.mark.parametrize("from_fp32", [False, True])
def test_dual_norm_both_quantised(fmt, from_fp32):
    M, Ha, Hb = 33, 1536, 1024
    buf, wa, wb = _dual_case(M, Ha, Hb, torch.bfloat16, seed=5)
    d = buf.to(DEV)
    (qa, sa, na), (qb, sb, nb) = rmsnorm_dual_quant(d[:, :Ha], wa.to(DEV), d[:, Ha:Ha + Hb], wb.to(DEV), fmt=fmt,
                                                   gemma=True, quant_from_fp32=from_fp32, quant_a=True,
                                                   quant_b=True, normed_a=False, normed_b=False)
    torch.cuda.synchronize()
    assert na is None and nb is None
    ra, rb = oracle.rmsnorm_dual_quant(fmt, _bits(buf[:, :Ha]), _bits(wa), _bits(buf[:, Ha:Ha + Hb]), _bits(wb),
                                       eps=1e-6, gemma=True, from_fp32=from_fp32)
    check_quant(fmt, ra, qa.cpu().numpy(), sa.cpu().numpy(), from_fp32)
    check_quant(fmt, rb, qb.cpu().numpy(), sb.cpu().numpy(), from_fp32)


def test_dual_norm_leaves_the_input_tail_alone_and_writes_only_its_outputs():
    M, Ha, Hb = 9, 1536, 512
    buf, wa, wb = _dual_case(M, Ha, Hb, torch.bfloat16, seed=11)
    d = buf.to(DEV)
    before = d.clone()
    rmsnorm_dual_quant(d[:, :Ha], wa.to(DEV), d[:, Ha:Ha + Hb], wb.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(d, before)


# (fmt, M, Ha, Hb, gemma, from_fp32, dtype): each segment's outputs must equal
# a single rmsnorm_add_quant call on its rows bit for bit (the two-segment
# plan keeps each segment's single-norm threads per row). The M values cross
# the single norms' small-M plan boundaries of the latent widths (1536 / 512).
BITWISE = [("per_token", M, 1536, 512, False, False, torch.bfloat16) for M in (1, 64, 700, 1024, 2048, 4096)]
BITWISE += [("mxfp8", 300, 2048, 1024, True, False, torch.bfloat16),
            ("block128", 1500, 4096, 512, False, True, torch.float16),
            ("per_token", 2500, 7168, 512, False, True, torch.bfloat16)]


@pytest.mark.parametrize("c", BITWISE, ids=lambda c: "-".join(str(v) for v in c[:6]) + ("-f16" if c[6] == torch.float16 else ""))
def test_dual_norm_equals_single_calls_bitwise(c):
    fmt, M, Ha, Hb, gemma, from32, dtype = c
    buf, wa, wb = _dual_case(M, Ha, Hb, dtype, seed=M + Ha + Hb)
    d = buf.to(DEV)
    xa, xb = d[:, :Ha], d[:, Ha:Ha + Hb]
    wa, wb = wa.to(DEV), wb.to(DEV)
    (qa, sa, na), (qb, sb, nb) = rmsnorm_dual_quant(xa, wa, xb, wb, fmt=fmt, gemma=gemma, quant_from_fp32=from32,
                                                   quant_a=True, quant_b=True, normed_a=True, normed_b=True)
    kw = dict(fmt=fmt, gemma=gemma, quant_from_fp32=from32, normed=True)
    q1, s1, n1, _ = rmsnorm_add_quant(xa.contiguous(), wa, **kw)
    q2, s2, n2, _ = rmsnorm_add_quant(xb.contiguous(), wb, **kw)
    torch.cuda.synchronize()
    for got, want in ((qa, q1), (sa, s1), (na, n1), (qb, q2), (sb, s2), (nb, n2)):
        assert torch.equal(got, want)
