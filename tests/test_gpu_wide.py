"""GPU parity of rows wider than one CTA covers (16384 columns).

Norms of any format, per-token SwiGLU and the per-token standalone quant
split such a row over the CTAs of a thread block cluster, which combine
their partial sums of squares and amaxes through shared memory; MXFP8 and
1x128 SwiGLU and quant split it into independent column segments. Widths
cover two to eight CTAs a row, segments that do not fill their CTA's
threads, and the widest row; every result is checked against the oracle,
with guard bands around the outputs, and the in-place residual update must
equal the separate one bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.parity import check_norm, check_swiglu, check_quant
from swiglu_fp8_activation_gb300 import inputs, quantize_fp8, rmsnorm_add_quant, scale_shape, swiglu, swiglu_quant

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GUARD = 4096


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _guarded(shape, dtype):
    esz = torch.empty((), dtype=dtype).element_size()
    n = int(np.prod(shape)) * esz
    raw = torch.full((n + GUARD,), 0xFF, dtype=torch.uint8, device=DEV)
    return raw, raw[:n].view(dtype).view(shape), n


def _intact(raw, n):
    return bool((raw[n:] == 0xFF).all())


def _unlayout(fmt, s, M, W, layout):
    """Row-major scales read back out of a consumer layout (checked against
    the oracle's rearrangement of them)."""
    s = s.cpu().numpy()
    if layout == "row":
        return s
    G = W // (32 if fmt == "mxfp8" else 128)
    if layout == "col_major":
        row = np.ascontiguousarray(s[:, :M].T)
    else:
        flat, Gp = s.reshape(-1), -(-G // 4) * 4
        row = np.zeros((M, G), dtype=s.dtype)
        for r in range(M):
            for g in range(G):
                rr = r % 128
                row[r, g] = flat[((r // 128) * (Gp // 4) + g // 4) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + g % 4]
    np.testing.assert_array_equal(s, oracle.scale_layout(fmt, row, layout))
    return row


# (fmt, M, H, residual, normed, from_fp32, gemma, layout)
NORM_CASES = [
    ("mxfp8", 3, 18432, True, True, False, True, "row"),         # 2 CTAs a row
    ("mxfp8", 37, 24576, True, True, False, True, "swizzled"),    # 2 CTAs, padded layout
    ("mxfp8", 1, 16640, True, False, True, False, "row"),         # 2 CTAs, the second holds 32 chunks
    ("block128", 5, 24576, False, False, True, False, "col_major"),
    ("block128", 2, 40960, True, True, False, True, "row"),       # 3 CTAs
    ("per_token", 4, 20008, False, False, False, False, "row"),   # a width off every power of two
    ("per_token", 37, 24576, True, True, True, True, "row"),
    ("per_token", 2, 131072, False, False, False, False, "row"),  # the widest row: 8 CTAs
    ("mxfp8", 2, 131072, True, True, False, True, "row"),
]


@pytest.mark.parametrize("c", NORM_CASES, ids=lambda c: "-".join(map(str, c)))
def test_wide_norm(c):
    fmt, M, H, res, normed, from32, gemma, layout = c
    t = inputs.norm_inputs(M, H, seed=H + M, x_std=3.0, r_std=1.0 if res else None,
                           w_mean=0.0 if gemma else 1.0, w_std=0.1)
    x, w = t["x"].to(DEV), t["w"].to(DEV)
    r = t["r"].to(DEV) if res else None
    qraw, q, qn = _guarded((M, H), torch.uint8)
    sraw, s, sn = _guarded(scale_shape(fmt, M, H, layout), torch.uint8 if fmt == "mxfp8" else torch.float32)
    nraw, n, nn = _guarded((M, H), torch.bfloat16)
    rraw, ro, rn = _guarded((M, H), torch.bfloat16)
    kw = dict(fmt=fmt, gemma=gemma, quant_from_fp32=from32, scale_layout=layout)
    rmsnorm_add_quant(x, w, residual_in=r, residual_out=ro if res else None, q_out=q, scale_out=s,
                      normed_out=n if normed else None, **kw)
    torch.cuda.synchronize()
    for raw, nb, what in ((qraw, qn, "q"), (sraw, sn, "scale"), (nraw, nn, "normed"), (rraw, rn, "residual")):
        assert _intact(raw, nb), f"bytes written past {what}"
    if res:
        r2 = r.clone()
        q2, s2, n2, _ = rmsnorm_add_quant(x, w, residual_in=r2, normed=normed, **kw)   # in place
        torch.cuda.synchronize()
        assert torch.equal(q, q2) and torch.equal(s, s2) and torch.equal(ro, r2)
        if normed:
            assert torch.equal(n, n2)
    ref = oracle.rmsnorm_add_quant(fmt, _bits(t["x"]), _bits(t["r"]) if res else None, _bits(t["w"]), eps=1e-6,
                                   gemma=gemma, from_fp32=from32, normed=normed)
    check_norm(fmt, ref, q.cpu().numpy(), _unlayout(fmt, s, M, H, layout), _bits(n) if normed else None,
               _bits(ro) if res else None, from_fp32=from32)


def test_wide_norm_fp16_and_graph_replay():
    M, H = 6, 32768                              # 2 CTAs a row, fp16 rows, launched from a CUDA graph
    g = torch.Generator().manual_seed(32768)
    x = (torch.randn(M, H, generator=g) * 3.0).to(torch.float16).to(DEV)
    r = torch.randn(M, H, generator=g).to(torch.float16).to(DEV)
    w = (0.1 * torch.randn(H, generator=g)).to(torch.float16).to(DEV)
    ro = torch.empty_like(r)
    q = torch.empty(M, H, dtype=torch.uint8, device=DEV)
    s = torch.empty(M, H // 32, dtype=torch.uint8, device=DEV)
    n = torch.empty_like(x)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for _ in range(3):
            rmsnorm_add_quant(x, w, residual_in=r, residual_out=ro, q_out=q, scale_out=s, normed_out=n)
    gr.replay()
    torch.cuda.synchronize()
    ref = oracle.rmsnorm_add_quant("mxfp8", _bits(x), _bits(r), _bits(w), eps=1e-6, gemma=True, from_fp32=False,
                                   normed=True, fp16=True)
    check_norm("mxfp8", ref, q.cpu().numpy(), s.cpu().numpy(), _bits(n), _bits(ro), from_fp32=False)


# (fmt, act, M, I, from_fp32, round_act_bf16, layout)
SWIGLU_CASES = [
    ("mxfp8", "swiglu_oai", 3, 18432, True, False, "row"),        # 2 segments
    ("mxfp8", "swiglu_oai", 37, 24576, True, False, "swizzled"),
    ("block128", "silu_mul", 5, 24576, False, True, "col_major"),
    ("block128", "silu_mul", 2, 16512, False, True, "row"),       # ragged: 2 segments of 1040 and 1024 chunks
    ("per_token", "swiglu_oai", 3, 18432, True, False, "row"),    # a cluster of 2 CTAs a row
    ("per_token", "silu_mul", 37, 24576, False, True, "row"),
    ("per_token", "swiglu_oai", 2, 131072, False, False, "row"),  # 8 CTAs a row
    ("mxfp8", "silu_mul", 2, 131072, True, False, "row"),         # 8 segments
]


@pytest.mark.parametrize("c", SWIGLU_CASES, ids=lambda c: "-".join(map(str, c)))
def test_wide_swiglu(c):
    fmt, act, M, I, from32, rnd, layout = c
    gu = inputs.swiglu_inputs(M, I, seed=I + M, std=3.0)
    qraw, q, qn = _guarded((M, I), torch.uint8)
    sraw, s, sn = _guarded(scale_shape(fmt, M, I, layout), torch.uint8 if fmt == "mxfp8" else torch.float32)
    swiglu_quant(gu.to(DEV), fmt=fmt, act=act, quant_from_fp32=from32, round_act_bf16=rnd, q_out=q, scale_out=s,
                 scale_layout=layout)
    torch.cuda.synchronize()
    assert _intact(qraw, qn) and _intact(sraw, sn), "bytes written past an output"
    ref = oracle.swiglu_quant(fmt, act, _bits(gu), from_fp32=from32, round_act_bf16=rnd)
    check_swiglu(fmt, ref, q.cpu().numpy(), _unlayout(fmt, s, M, I, layout), from_fp32=from32)


def test_wide_swiglu_bf16_out():
    M, I = 3, 20480                               # the unfused activation step, 2 segments
    gu = inputs.swiglu_inputs(M, I, seed=5, std=3.0)
    raw, out, n = _guarded((M, I), torch.bfloat16)
    swiglu(gu.to(DEV), act="silu_mul", round_act_bf16=True, out=out)
    torch.cuda.synchronize()
    assert _intact(raw, n)
    ref = oracle.swiglu_quant("mxfp8", "silu_mul", _bits(gu), from_fp32=True, round_act_bf16=True)
    want = _bits(inputs.to_bf16(ref["a"]))
    got = _bits(out)
    key = lambda b: np.where(b & 0x8000, -(b.astype(np.int64) & 0x7FFF), b.astype(np.int64) & 0x7FFF)
    assert np.abs(key(want) - key(got)).max() <= 1


@pytest.mark.parametrize("fmt,W,dtype", [("mxfp8", 24576, torch.bfloat16), ("block128", 32768, torch.float16),
                                         ("per_token", 24576, torch.bfloat16), ("per_token", 65536, torch.float16),
                                         ("mxfp8", 16416, torch.bfloat16)])
def test_wide_quantize(fmt, W, dtype):
    M = 5
    g = torch.Generator().manual_seed(W)
    src = (torch.randn(M, W, generator=g) * 2.0).to(dtype)
    qraw, q, qn = _guarded((M, W), torch.uint8)
    sraw, s, sn = _guarded(scale_shape(fmt, M, W), torch.uint8 if fmt == "mxfp8" else torch.float32)
    quantize_fp8(src.to(DEV), fmt=fmt, q_out=q, scale_out=s)
    torch.cuda.synchronize()
    assert _intact(qraw, qn) and _intact(sraw, sn), "bytes written past an output"
    ref = oracle.quantize(fmt, _bits(src), fp16=dtype == torch.float16)
    check_quant(fmt, ref, q.cpu().numpy(), s.cpu().numpy(), from_fp32=False)
