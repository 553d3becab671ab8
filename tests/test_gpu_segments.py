"""GPU parity of the launches that split rows into column segments.

SwiGLU: at small M the library runs each row of a wide SwiGLU as up to 16
CTAs, each taking a whole number of scale groups (MXFP8 and 1x128 only; the
per-token format needs the row's amax). The cases below are chosen so that
the launch is segmented on the device under test (checked against the host's
rule), including segments that do not fill their CTA's threads, layouts that
pad rows, SiLU's bf16 roundings and the bf16 output of the unfused chain.
Each result must match the oracle under the usual tolerances, equal bit for
bit the same rows computed inside a batch large enough to run unsegmented,
and leave the bytes around its outputs untouched.

Norms: a row may also run as up to 8 CTAs that each form the whole row's sum
of squares and write one column segment, in every format, but never for an
in-place residual update. The split results must match the oracle, leave the
bytes around every output untouched, and equal bit for bit the in-place
launch of the same inputs (same plan, unsplit).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.parity import check_bf16, check_norm, check_swiglu
from swiglu_fp8_activation_gb300 import inputs, rmsnorm_add_quant, scale_shape, swiglu, swiglu_quant

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GUARD = 4096
BIG_M = 512                      # enough rows that no launch splits them (above two waves)


def _sms():
    return torch.cuda.get_device_properties(DEV).multi_processor_count


def _segments(fmt, rows, I, sms):
    """The host's choice of column segments a row (the C library's rule)."""
    if fmt == "per_token":
        return 1
    nch, gch = I // 8, (16 if fmt == "block128" else 4)
    s = 1
    while s < 16 and rows * 2 * s <= sms and nch % (2 * s * gch) == 0 and nch // (2 * s) >= 64:
        s *= 2
    if s == 1 and sms // 2 < rows <= 2 * sms:          # balance between half a wave and two waves
        best_ctas, best_s = -(-rows // sms), 1
        c = 2
        while c <= 16 and nch % (c * gch) == 0 and nch // c >= 64:
            per = -(-rows * c // sms)
            if per * best_s * 16 < best_ctas * c * 15:
                best_ctas, best_s = per, c
            c *= 2
        s = best_s
    return s


def _rows_of(fmt, M, layout):
    if layout == "swizzled":
        return -(-M // 128) * 128
    if layout == "col_major":
        return -(-M // 4) * 4
    return M


def _guarded(shape, dtype):
    """A tensor of `shape` inside a 0xFF-filled byte buffer, and its byte count."""
    esz = torch.empty((), dtype=dtype).element_size()
    n = int(np.prod(shape)) * esz
    raw = torch.full((n + GUARD,), 0xFF, dtype=torch.uint8, device=DEV)
    return raw, raw[:n].view(dtype).view(shape), n


def _gate_up(M, I, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(M, 2 * I, generator=g) * 3.0).to(torch.bfloat16)


def _bits(t):
    return inputs.bf16_bits(t.detach().cpu())


# (fmt, act, M, I, scale layout, from_fp32, round_act_bf16)
CASES = [
    ("block128", "silu_mul", 1, 12288, "row", False, True),        # 16 segments of 96 chunks
    ("block128", "silu_mul", 32, 12288, "row", False, True),       # 4 segments
    ("block128", "silu_mul", 1, 12288, "col_major", True, False),  # padding rows of the layout
    ("block128", "swiglu_oai", 19, 5120, "col_major", True, False),
    ("mxfp8", "swiglu_oai", 1, 2304, "row", True, False),          # 72-chunk segments in 96 threads
    ("mxfp8", "swiglu_oai", 7, 12288, "row", True, False),
    ("mxfp8", "silu_mul", 3, 4224, "row", False, False),           # 132-chunk segments in 160 threads
    ("mxfp8", "swiglu_oai", 5, 6144, "row", False, False),
]


def _name(c):
    return "-".join(str(v) for v in c)


@pytest.mark.parametrize("c", CASES, ids=_name)
def test_segmented_swiglu_quant(c):
    fmt, act, M, I, layout, from32, rnd = c
    rows = _rows_of(fmt, M, layout)
    assert _segments(fmt, rows, I, _sms()) > 1, "case does not exercise a segmented launch on this device"
    gu = _gate_up(M, I, seed=M * 7919 + I)
    kw = dict(fmt=fmt, act=act, quant_from_fp32=from32, round_act_bf16=rnd)
    qraw, q, qn = _guarded((M, I), torch.uint8)
    sdt = torch.uint8 if fmt == "mxfp8" else torch.float32
    sraw, s, sn = _guarded(scale_shape(fmt, M, I, layout), sdt)
    swiglu_quant(gu.to(DEV), q_out=q, scale_out=s, scale_layout=layout, **kw)
    # the same rows at the top of a batch that runs unsegmented, row-major scales
    big = torch.cat([gu, _gate_up(BIG_M - M, I, seed=I)], dim=0)
    assert _segments(fmt, BIG_M, I, _sms()) == 1
    qb, sb = swiglu_quant(big.to(DEV), **kw)
    torch.cuda.synchronize()
    assert (qraw[qn:] == 0xFF).all(), "bytes written past q_out"
    assert (sraw[sn:] == 0xFF).all(), "bytes written past scale_out"
    assert torch.equal(q, qb[:M])
    s_row = sb[:M].cpu().numpy()
    if layout == "row":
        np.testing.assert_array_equal(s.cpu().numpy(), s_row)
    else:
        np.testing.assert_array_equal(s.cpu().numpy(), oracle.scale_layout(fmt, s_row, layout))
    ref = oracle.swiglu_quant(fmt, act, _bits(gu), from_fp32=from32, round_act_bf16=rnd)
    check_swiglu(fmt, ref, qb[:M].cpu().numpy(), s_row, from_fp32=from32)


@pytest.mark.parametrize("act,M,I,rnd", [("silu_mul", 1, 12288, True), ("swiglu_oai", 5, 2304, False),
                                         ("silu_mul", 3, 4224, False)])
def test_segmented_swiglu_bf16(act, M, I, rnd):
    # the unfused chain's activation step (bf16 out, no quantisation) splits by MXFP8's groups
    assert _segments("mxfp8", M, I, _sms()) > 1
    gu = _gate_up(M, I, seed=M + I)
    raw, out, n = _guarded((M, I), torch.bfloat16)
    swiglu(gu.to(DEV), act=act, round_act_bf16=rnd, out=out)
    big = torch.cat([gu, _gate_up(BIG_M - M, I, seed=I + 1)], dim=0)
    ob = swiglu(big.to(DEV), act=act, round_act_bf16=rnd)
    torch.cuda.synchronize()
    assert (raw[n:] == 0xFF).all(), "bytes written past out"
    assert torch.equal(out, ob[:M])
    ref = oracle.swiglu_quant("mxfp8", act, _bits(gu), from_fp32=True, round_act_bf16=rnd)
    check_bf16("activation", inputs.bf16_bits(inputs.to_bf16(ref["a"])), _bits(out))


def _norm_segments(rows, H, sms):
    """The host's choice of column segments a row for a norm launch."""
    nch = H // 8
    s = 1
    while s < 8 and rows * 2 * s <= sms and nch % (64 * s) == 0 and nch // (2 * s) >= 64:
        s *= 2
    return s


# (fmt, M, H, gemma, residual, normed, from_fp32, scale layout)
NORM_CASES = [
    ("mxfp8", 8, 6144, True, True, True, False, "row"),          # 8 segments of 96 chunks
    ("mxfp8", 16, 6144, True, True, True, False, "row"),
    ("mxfp8", 64, 6144, True, True, False, False, "row"),        # 2 segments
    ("mxfp8", 2, 8704, False, True, True, True, "row"),          # 3 chunks a thread, past the row end
    ("mxfp8", 3, 2560, True, False, True, False, "row"),
    ("block128", 1, 4096, False, False, False, True, "row"),     # 8 segments of 64 chunks
    ("block128", 5, 4096, False, True, True, False, "col_major"),
    ("per_token", 1, 7168, False, False, False, False, "row"),   # 4 segments; the row scale from segment 0
    ("per_token", 3, 1536, False, True, True, True, "row"),
]


def _norm_name(c):
    return "-".join(str(v) for v in c)


@pytest.mark.parametrize("c", NORM_CASES, ids=_norm_name)
def test_segmented_norm(c):
    fmt, M, H, gemma, res, normed, from32, layout = c
    assert _norm_segments(_rows_of(fmt, M, layout), H, _sms()) > 1, "case does not split on this device"
    t = inputs.norm_inputs(M, H, seed=M * 131 + H, x_std=3.0, r_std=1.0 if res else None,
                           w_mean=0.0 if gemma else 1.0, w_std=0.1)
    x, w = t["x"].to(DEV), t["w"].to(DEV)
    r = t["r"].to(DEV) if res else None
    qraw, q, qn = _guarded((M, H), torch.uint8)
    sdt = torch.float32 if fmt != "mxfp8" else torch.uint8
    sraw, s, sn = _guarded(scale_shape(fmt, M, H, layout), sdt)
    nraw, n, nn = _guarded((M, H), torch.bfloat16)
    rraw, ro, rn = _guarded((M, H), torch.bfloat16)
    kw = dict(fmt=fmt, gemma=gemma, quant_from_fp32=from32, scale_layout=layout)
    rmsnorm_add_quant(x, w, residual_in=r, residual_out=ro if res else None, q_out=q, scale_out=s,
                      normed_out=n if normed else None, **kw)
    torch.cuda.synchronize()
    for raw, nbytes, what in ((qraw, qn, "q_out"), (sraw, sn, "scale_out"), (nraw, nn, "normed_out"),
                              (rraw, rn, "residual_out")):
        assert (raw[nbytes:] == 0xFF).all(), f"bytes written past {what}"
    if res:
        # the in-place update of the same residual runs unsplit with the same plan: bit for bit equal
        r2 = r.clone()
        q2, s2, n2, _ = rmsnorm_add_quant(x, w, residual_in=r2, normed=normed, **kw)
        torch.cuda.synchronize()
        assert torch.equal(q, q2) and torch.equal(s, s2) and torch.equal(ro, r2)
        if normed:
            assert torch.equal(n, n2)
    s_row = s.cpu().numpy()
    if layout != "row":
        q3, s3, _, _ = rmsnorm_add_quant(x, w, residual_in=r.clone() if res else None,
                                         **{**kw, "scale_layout": "row"})
        torch.cuda.synchronize()
        assert torch.equal(q, q3)
        np.testing.assert_array_equal(s_row, oracle.scale_layout(fmt, s3.cpu().numpy(), layout))
        s_row = s3.cpu().numpy()
    ref = oracle.rmsnorm_add_quant(fmt, _bits(t["x"]), _bits(t["r"]) if res else None, _bits(t["w"]), eps=1e-6,
                                   gemma=gemma, from_fp32=from32, normed=normed)
    check_norm(fmt, ref, q.cpu().numpy(), s_row, _bits(n) if normed else None, _bits(ro) if res else None,
               from_fp32=from32)


def test_segmented_norm_fp16():
    # fp16 rows with a separate residual, split in 8 (M = 4, H = 4096)
    M, H = 4, 4096
    assert _norm_segments(M, H, _sms()) > 1
    g = torch.Generator().manual_seed(4096)
    x = (torch.randn(M, H, generator=g) * 3.0).to(torch.float16)
    r = torch.randn(M, H, generator=g).to(torch.float16)
    w = (0.1 * torch.randn(H, generator=g)).to(torch.float16)
    xd, rd, wd = x.to(DEV), r.to(DEV), w.to(DEV)
    ro = torch.empty_like(rd)
    q, s, n, _ = rmsnorm_add_quant(xd, wd, residual_in=rd, residual_out=ro, normed=True)
    r2 = rd.clone()
    q2, s2, n2, _ = rmsnorm_add_quant(xd, wd, residual_in=r2, normed=True)   # in place: unsplit
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(s, s2) and torch.equal(n, n2) and torch.equal(ro, r2)
    f16 = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    ref = oracle.rmsnorm_add_quant("mxfp8", f16(x), f16(r), f16(w), eps=1e-6, gemma=True, from_fp32=False,
                                   normed=True, fp16=True)
    check_norm("mxfp8", ref, q.cpu().numpy(), s.cpu().numpy(), f16(n), f16(ro), from_fp32=False)


def test_split_launches_chained():
    # Four layers: norm (8 segments) -> SwiGLU on its bf16 copy (4 segments), the residual carried
    # from layer to layer. Launched back to back (each launch may begin before the previous one
    # ends), and replayed from a CUDA graph, the chain must equal the same chain with a device
    # synchronisation after every launch, and the in-place residual chain (whole rows).
    M, H, L = 8, 6144, 4
    assert _norm_segments(M, H, _sms()) == 8 and _segments("mxfp8", M, H // 2, _sms()) == 4
    g = torch.Generator().manual_seed(77)
    xs = [(torch.randn(M, H, generator=g) * 3.0).to(torch.bfloat16).to(DEV) for _ in range(L)]
    ws = [(0.1 * torch.randn(H, generator=g)).to(torch.bfloat16).to(DEV) for _ in range(L)]
    r0 = torch.randn(M, H, generator=g).to(torch.bfloat16).to(DEV)

    def buffers():
        return dict(r=[torch.empty(M, H, dtype=torch.bfloat16, device=DEV) for _ in range(L)],
                    q=[torch.empty(M, H, dtype=torch.uint8, device=DEV) for _ in range(L)],
                    s=[torch.empty(M, H // 32, dtype=torch.uint8, device=DEV) for _ in range(L)],
                    n=[torch.empty(M, H, dtype=torch.bfloat16, device=DEV) for _ in range(L)],
                    aq=[torch.empty(M, H // 2, dtype=torch.uint8, device=DEV) for _ in range(L)],
                    asc=[torch.empty(M, H // 64, dtype=torch.uint8, device=DEV) for _ in range(L)])

    def chain(b, sync):
        r_in = r0
        for k in range(L):
            rmsnorm_add_quant(xs[k], ws[k], residual_in=r_in, residual_out=b["r"][k], q_out=b["q"][k],
                              scale_out=b["s"][k], normed_out=b["n"][k])
            if sync:
                torch.cuda.synchronize()
            swiglu_quant(b["n"][k], q_out=b["aq"][k], scale_out=b["asc"][k])
            if sync:
                torch.cuda.synchronize()
            r_in = b["r"][k]

    ref, eager, graphed = buffers(), buffers(), buffers()
    chain(ref, sync=True)
    chain(eager, sync=False)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        chain(graphed, sync=False)
    gr.replay()
    torch.cuda.synchronize()
    for key in ref:
        for k in range(L):
            assert torch.equal(ref[key][k], eager[key][k]), (key, k, "back to back")
            assert torch.equal(ref[key][k], graphed[key][k]), (key, k, "graph replay")
    # the in-place residual chain runs whole rows: the same values
    r = r0.clone()
    for k in range(L):
        q, s, n, _ = rmsnorm_add_quant(xs[k], ws[k], residual_in=r, normed=True)
        torch.cuda.synchronize()
        assert torch.equal(r, ref["r"][k]) and torch.equal(q, ref["q"][k]) and torch.equal(s, ref["s"][k])
        assert torch.equal(n, ref["n"][k])


def test_forced_segments_with_swizzled_scales():
    # The swizzled E8M0 layout pads the rows to 128, which never splits on a
    # 152-SM device. Planning for 4096 multiprocessors (sgq_set_sm_budget)
    # splits them: the norm in 8 segments (its segments need W/32 % 16 == 0),
    # and SwiGLU at I = 2240 (70 groups, 70 % 4 == 2) in 2, whose second
    # segment holds the last group, which completes its tile row with zero
    # codes. Each must equal bit for bit what the unsplit launches give.
    from swiglu_fp8_activation_gb300 import set_sm_budget
    budget, M, H, I = 4096, 50, 4096, 2240
    assert _norm_segments(128, H, budget) == 8 and _norm_segments(128, H, _sms()) == 1
    assert _segments("mxfp8", 128, I, budget) == 2 and (I // 32) % 4 == 2
    t = inputs.norm_inputs(M, H, seed=50, x_std=3.0, r_std=1.0, w_mean=0.0, w_std=0.1)
    x, r, w = (t[k].to(DEV) for k in ("x", "r", "w"))
    gu = _gate_up(M, I, seed=2240)
    sraw, s, sn = _guarded(scale_shape("mxfp8", M, H, "swizzled"), torch.uint8)
    ro = torch.empty_like(r)
    araw, a_s, an = _guarded(scale_shape("mxfp8", M, I, "swizzled"), torch.uint8)
    try:
        set_sm_budget(budget)
        q, _, n, _ = rmsnorm_add_quant(x, w, residual_in=r, residual_out=ro, scale_out=s, normed=True,
                                       scale_layout="swizzled")
        r2 = r.clone()   # in place: never split, same plan otherwise
        q2, s2, n2, _ = rmsnorm_add_quant(x, w, residual_in=r2, normed=True, scale_layout="swizzled")
        aq, _ = swiglu_quant(gu.to(DEV), scale_out=a_s, scale_layout="swizzled")
        torch.cuda.synchronize()
    finally:
        set_sm_budget(0)
    aq_row, as_row = swiglu_quant(gu.to(DEV))            # the device's own plan: unsplit, row-major
    torch.cuda.synchronize()
    assert (sraw[sn:] == 0xFF).all() and (araw[an:] == 0xFF).all(), "bytes written past a scale buffer"
    assert torch.equal(q, q2) and torch.equal(s, s2) and torch.equal(n, n2) and torch.equal(ro, r2)
    assert torch.equal(aq, aq_row)
    np.testing.assert_array_equal(a_s.cpu().numpy(), oracle.scale_layout("mxfp8", as_row.cpu().numpy(), "swizzled"))
    ref = oracle.rmsnorm_add_quant("mxfp8", _bits(t["x"]), _bits(t["r"]), _bits(t["w"]), eps=1e-6, gemma=True,
                                   from_fp32=False, normed=True)
    s_sw = s.cpu().numpy()
    s_row = _unswizzle(s_sw, M, H // 32)
    np.testing.assert_array_equal(s_sw, oracle.scale_layout("mxfp8", s_row, "swizzled"))   # padding is code 0
    check_norm("mxfp8", ref, q.cpu().numpy(), s_row, _bits(n), _bits(ro), from_fp32=False)
    ref2 = oracle.swiglu_quant("mxfp8", "swiglu_oai", _bits(gu), from_fp32=True)
    check_swiglu("mxfp8", ref2, aq.cpu().numpy(), as_row.cpu().numpy(), from_fp32=True)


def _unswizzle(flat, M, G):
    """Row-major [M, G] codes read back out of the swizzled [Mp, Gp] buffer."""
    flat = np.asarray(flat).reshape(-1)
    Gp = -(-G // 4) * 4
    out = np.zeros((M, G), dtype=flat.dtype)
    for r in range(M):
        for g in range(G):
            tile = (r // 128) * (Gp // 4) + g // 4
            rr = r % 128
            out[r, g] = flat[tile * 512 + (rr % 32) * 16 + (rr // 32) * 4 + g % 4]
    return out
