"""Seeded random configurations across every entry point, each checked
against the oracle under the same tolerances as the fixed parity tests:
random formats, flags, activation types, scale layouts and shapes (M from 1
to a few hundred, widths any multiple of the format's group up to the
maximum), then the all-reduce norm over 1 to 8 ranks and rows wider than one
CTA covers. Cases are drawn once from fixed seeds, so a failure names a
reproducible configuration."""
import numpy as np
import pytest
import torch

import oracle
from oracle.parity import check_bf16, check_norm, check_quant, check_swiglu
from swiglu_fp8_activation_gb300 import (inputs, quantize_fp8, rmsnorm_add_quant, rmsnorm_dual_quant, swiglu,
                                          swiglu_quant)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GROUP = {"mxfp8": 32, "block128": 128, "per_token": 8}
MAX_ELEMS = 1 << 20


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _width(rng, fmt, lo=1):
    g = GROUP[fmt]
    return int(g * rng.integers(lo, 16384 // g + 1))


def _rows(rng, W, max_rows=300, max_elems=MAX_ELEMS):
    return int(rng.integers(1, max(2, min(max_rows, max_elems // W)) + 1))


def _layout(rng, fmt):
    if fmt == "mxfp8" and rng.random() < 0.3:
        return "swizzled"
    if fmt == "block128" and rng.random() < 0.3:
        return "col_major"
    return "row"


def _cases(n=48, seed=2024, max_rows=300, max_elems=MAX_ELEMS):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        op = ["norm", "swiglu", "quant", "dual"][i % 4]
        fmt = ["mxfp8", "block128", "per_token"][int(rng.integers(3))]
        c = {"op": op, "fmt": fmt, "seed": int(rng.integers(1 << 30)), "from32": bool(rng.random() < 0.5)}
        if op == "norm":
            c.update(W=_width(rng, fmt), gemma=bool(rng.random() < 0.5),
                     residual=["none", "separate", "inplace"][int(rng.integers(3))], normed=bool(rng.random() < 0.5),
                     fp16=bool(rng.random() < 0.3), layout=_layout(rng, fmt))
        elif op == "swiglu":
            c.update(W=_width(rng, fmt), act=["swiglu_oai", "silu_mul"][int(rng.integers(2))], layout=_layout(rng, fmt))
            c["round"] = c["act"] == "silu_mul" and bool(rng.random() < 0.5)
        elif op == "quant":
            c.update(W=_width(rng, fmt), fp16=bool(rng.random() < 0.3), layout=_layout(rng, fmt), from32=False)
        else:
            c.update(W=_width(rng, fmt), Wb=_width(rng, fmt), fp16=bool(rng.random() < 0.3), gemma=bool(rng.random() < 0.5),
                     qb=bool(rng.random() < 0.5))
        c["M"] = _rows(rng, max(c["W"], c.get("Wb", 0)), max_rows, max_elems)
        out.append(c)
    return out


# a second draw of twice as many cases (it found the -0 code, the layout-dependent plan and the
# tie counts of fp32-source FP8 norms that the first draw had missed)
CASES = _cases() + _cases(n=96, seed=7919)


# and cases of up to 9000 rows and 4M elements a launch (the exact-fit and many-rows-a-CTA plans)
CASES += _cases(n=40, seed=4242, max_rows=9000, max_elems=1 << 22)


def _name(c):
    return "-".join(f"{k}{v}" for k, v in c.items() if k != "seed")


def _act_tensor(g, M, W, fp16, scale=3.0):
    x = torch.randn(M, W, generator=g) * scale * torch.exp2(torch.randint(-3, 4, (M, 1), generator=g).float())
    return x.to(torch.float16 if fp16 else torch.bfloat16)


def _check_layout(fmt, layout, s_layout, s_row):
    if layout != "row":
        np.testing.assert_array_equal(s_layout.cpu().numpy(), oracle.scale_layout(fmt, s_row.cpu().numpy(), layout))


@pytest.mark.parametrize("c", CASES, ids=_name)
def test_random_configuration(c):
    g = torch.Generator().manual_seed(c["seed"])
    M, W, fmt = c["M"], c["W"], c["fmt"]
    if c["op"] == "norm":
        x = _act_tensor(g, M, W, c["fp16"])
        w = (torch.randn(W, generator=g) * 0.1 + (0.0 if c["gemma"] else 1.0)).to(x.dtype)
        r = _act_tensor(g, M, W, c["fp16"], 1.0) if c["residual"] != "none" else None
        rd = r.to(DEV) if r is not None else None
        ro = None if rd is None else (rd if c["residual"] == "inplace" else torch.empty_like(rd))
        kw = dict(fmt=fmt, residual_in=rd, residual_out=ro, gemma=c["gemma"], quant_from_fp32=c["from32"],
                  normed=c["normed"])
        q, s, n, rout = rmsnorm_add_quant(x.to(DEV), w.to(DEV), **kw)
        torch.cuda.synchronize()
        ref = oracle.rmsnorm_add_quant(fmt, _bits(x), _bits(r) if r is not None else None, _bits(w), eps=1e-6,
                                       gemma=c["gemma"], from_fp32=c["from32"], normed=c["normed"], fp16=c["fp16"])
        check_norm(fmt, ref, q.cpu().numpy(), s.cpu().numpy(), _bits(n) if c["normed"] else None,
                   _bits(rout) if r is not None else None, from_fp32=c["from32"])
        if c["layout"] != "row":
            rd2 = r.to(DEV) if r is not None else None
            ro2 = None if rd2 is None else (rd2 if c["residual"] == "inplace" else torch.empty_like(rd2))
            q2, s2, _, _ = rmsnorm_add_quant(x.to(DEV), w.to(DEV), **{**kw, "residual_in": rd2, "residual_out": ro2,
                                                                       "scale_layout": c["layout"]})
            torch.cuda.synchronize()
            assert torch.equal(q, q2)
            _check_layout(fmt, c["layout"], s2, s)
    elif c["op"] == "swiglu":
        gu = (torch.randn(M, 2 * W, generator=g) * 3.0).to(torch.bfloat16)
        kw = dict(fmt=fmt, act=c["act"], quant_from_fp32=c["from32"], round_act_bf16=c["round"])
        q, s = swiglu_quant(gu.to(DEV), **kw)
        a = swiglu(gu.to(DEV), act=c["act"], round_act_bf16=c["round"])
        torch.cuda.synchronize()
        ref = oracle.swiglu_quant(fmt, c["act"], _bits(gu), from_fp32=c["from32"], round_act_bf16=c["round"])
        check_swiglu(fmt, ref, q.cpu().numpy(), s.cpu().numpy(), from_fp32=c["from32"])
        check_bf16("activation", inputs.bf16_bits(inputs.to_bf16(ref["a"])), _bits(a))
        if c["layout"] != "row":
            q2, s2 = swiglu_quant(gu.to(DEV), **kw, scale_layout=c["layout"])
            torch.cuda.synchronize()
            assert torch.equal(q, q2)
            _check_layout(fmt, c["layout"], s2, s)
    elif c["op"] == "quant":
        src = _act_tensor(g, M, W, c["fp16"])
        q, s = quantize_fp8(src.to(DEV), fmt=fmt, scale_layout=c["layout"])
        q_r, s_r = quantize_fp8(src.to(DEV), fmt=fmt)
        torch.cuda.synchronize()
        ref = oracle.quantize(fmt, _bits(src), fp16=c["fp16"])
        np.testing.assert_array_equal(q_r.cpu().numpy(), ref["q"])
        np.testing.assert_array_equal(s_r.cpu().numpy(), ref["scale"])
        assert torch.equal(q, q_r)
        _check_layout(fmt, c["layout"], s, s_r)
    else:
        Wa, Wb = W, c["Wb"]
        buf = _act_tensor(g, M, Wa + Wb + 16, c["fp16"])
        wa = (1 + 0.1 * torch.randn(Wa, generator=g)).to(buf.dtype)
        wb = (1 + 0.1 * torch.randn(Wb, generator=g)).to(buf.dtype)
        d = buf.to(DEV)
        (qa, sa, na), (qb, sb, nb) = rmsnorm_dual_quant(d[:, :Wa], wa.to(DEV), d[:, Wa:Wa + Wb], wb.to(DEV), fmt=fmt,
                                                       gemma=c["gemma"], quant_from_fp32=c["from32"], quant_a=True,
                                                       normed_a=True, quant_b=c["qb"], normed_b=True)
        torch.cuda.synchronize()
        ra, rb = oracle.rmsnorm_dual_quant(fmt, _bits(buf[:, :Wa]), _bits(wa), _bits(buf[:, Wa:Wa + Wb]), _bits(wb),
                                           eps=1e-6, gemma=c["gemma"], from_fp32=c["from32"], fp16=c["fp16"])
        check_norm(fmt, ra, qa.cpu().numpy(), sa.cpu().numpy(), _bits(na), None, from_fp32=c["from32"])
        check_bf16("normed_b", rb["normed"], _bits(nb))
        if c["qb"]:
            check_quant(fmt, rb, qb.cpu().numpy(), sb.cpu().numpy(), c["from32"])


# --------------------------------------- the all-reduce norm and wide rows

def _wide_width(rng, fmt):
    g = GROUP[fmt]
    return int(g * rng.integers(16384 // g + 1, 65536 // g + 1))


def _more_cases(n=24, seed=2025):
    """Seeded configurations of the all-reduce norm (1-8 ranks, every format,
    residual mode and layout) and of rows wider than one CTA covers (thread
    block clusters and column segments, every op). Quantisation from fp32
    only for MXFP8 here, whose power-of-two scales leave no quotient ties:
    the fixed parity tests cover the ties of fp32-source 1x128 and
    per-token FP8."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        op = ["allreduce", "wide_norm", "wide_swiglu", "wide_quant"][i % 4]
        fmt = ["mxfp8", "block128", "per_token"][int(rng.integers(3))]
        c = {"op": op, "fmt": fmt, "seed": int(rng.integers(1 << 30)),
             "from32": fmt == "mxfp8" and bool(rng.random() < 0.5), "layout": _layout(rng, fmt)}
        if op == "allreduce":
            c.update(W=_width(rng, fmt), n=int(rng.integers(1, 9)), gemma=bool(rng.random() < 0.5),
                     residual=["none", "separate", "inplace"][int(rng.integers(3))], normed=bool(rng.random() < 0.5))
            c["M"] = int(rng.integers(1, 65))
        elif op == "wide_norm":
            c.update(W=_wide_width(rng, fmt), gemma=bool(rng.random() < 0.5), fp16=bool(rng.random() < 0.3),
                     residual=["none", "separate", "inplace"][int(rng.integers(3))], normed=bool(rng.random() < 0.5))
            c["M"] = int(rng.integers(1, 9))
        elif op == "wide_swiglu":
            c.update(W=_wide_width(rng, fmt), act=["swiglu_oai", "silu_mul"][int(rng.integers(2))])
            c["round"] = c["act"] == "silu_mul" and bool(rng.random() < 0.5)
            c["M"] = int(rng.integers(1, 9))
        else:
            c.update(W=_wide_width(rng, fmt), fp16=bool(rng.random() < 0.3), from32=False)
            c["M"] = int(rng.integers(1, 9))
        out.append(c)
    return out


MORE_CASES = _more_cases() + _more_cases(n=48, seed=104729)


def _row_scales(fmt, layout, s, M, W):
    """Row-major scales from a launch's layout (checked against the oracle's rearrangement)."""
    if layout == "row":
        return s.cpu().numpy()
    G = W // (32 if fmt == "mxfp8" else 128)
    sl = s.cpu().numpy()
    if layout == "col_major":
        row = np.ascontiguousarray(sl[:, :M].T)
    else:
        flat, Gp = sl.reshape(-1), -(-G // 4) * 4
        row = np.zeros((M, G), dtype=sl.dtype)
        for r in range(M):
            for gi in range(G):
                rr = r % 128
                row[r, gi] = flat[((r // 128) * (Gp // 4) + gi // 4) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + gi % 4]
    np.testing.assert_array_equal(sl, oracle.scale_layout(fmt, row, layout))
    return row


@pytest.mark.parametrize("c", MORE_CASES, ids=_name)
def test_random_allreduce_and_wide_configuration(c):
    from swiglu_fp8_activation_gb300 import SgqError, allreduce_rmsnorm_add_quant
    g = torch.Generator().manual_seed(c["seed"])
    M, W, fmt, layout = c["M"], c["W"], c["fmt"], c["layout"]
    if c["op"] in ("allreduce", "wide_norm"):
        fp16 = c.get("fp16", False)
        if c["op"] == "allreduce":
            parts = [_act_tensor(g, M, W, False, 1.0) for _ in range(c["n"])]
        else:
            parts = [_act_tensor(g, M, W, fp16)]
        w = (torch.randn(W, generator=g) * 0.1 + (0.0 if c["gemma"] else 1.0)).to(parts[0].dtype)
        r = _act_tensor(g, M, W, fp16, 1.0) if c["residual"] != "none" else None
        rd = r.to(DEV) if r is not None else None
        ro = None if rd is None else (rd if c["residual"] == "inplace" else torch.empty_like(rd))
        kw = dict(fmt=fmt, residual_in=rd, residual_out=ro, gemma=c["gemma"], quant_from_fp32=c["from32"],
                  normed=c["normed"], scale_layout=layout)
        if c["op"] == "allreduce":
            pd = [p.to(DEV) for p in parts]
            try:
                q, s, n, rout = allreduce_rmsnorm_add_quant(pd, w.to(DEV), **kw)
            except SgqError as e:
                # the staging limit: a CTA stages 16 bytes a chunk of every partial and the
                # residual, at most 2048 chunks; only rows wider than 8192 columns with eight
                # staged inputs (ranks + residual) reach 227 KB
                assert e.status == 2 and W > 8192 and c["n"] + (r is not None) >= 8, (e.status, W, c["n"])
                return
            summed = pd[0].float()
            for p in pd[1:]:
                summed = summed + p.float()     # the kernel's all-reduce: fp32 sum in rank order, then bf16
            r2 = r.to(DEV) if r is not None else None
            ro2 = None if r2 is None else (r2 if c["residual"] == "inplace" else torch.empty_like(r2))
            q2, s2, n2, rout2 = rmsnorm_add_quant(summed.to(torch.bfloat16), w.to(DEV),
                                                  **{**kw, "residual_in": r2, "residual_out": ro2})
            torch.cuda.synchronize()
            assert torch.equal(q, q2) and torch.equal(s, s2)
            assert (n is None or torch.equal(n, n2)) and (rout is None or torch.equal(rout, rout2))
            ref = oracle.allreduce_rmsnorm_add_quant(fmt, [_bits(p) for p in parts], _bits(r) if r is not None else None,
                                                     _bits(w), eps=1e-6, gemma=c["gemma"], from_fp32=c["from32"],
                                                     normed=c["normed"])
        else:
            q, s, n, rout = rmsnorm_add_quant(parts[0].to(DEV), w.to(DEV), **kw)
            torch.cuda.synchronize()
            ref = oracle.rmsnorm_add_quant(fmt, _bits(parts[0]), _bits(r) if r is not None else None, _bits(w),
                                           eps=1e-6, gemma=c["gemma"], from_fp32=c["from32"], normed=c["normed"],
                                           fp16=fp16)
        check_norm(fmt, ref, q.cpu().numpy(), _row_scales(fmt, layout, s, M, W), _bits(n) if c["normed"] else None,
                   _bits(rout) if r is not None else None, from_fp32=c["from32"])
    elif c["op"] == "wide_swiglu":
        gu = (torch.randn(M, 2 * W, generator=g) * 3.0).to(torch.bfloat16)
        q, s = swiglu_quant(gu.to(DEV), fmt=fmt, act=c["act"], quant_from_fp32=c["from32"], round_act_bf16=c["round"],
                            scale_layout=layout)
        torch.cuda.synchronize()
        ref = oracle.swiglu_quant(fmt, c["act"], _bits(gu), from_fp32=c["from32"], round_act_bf16=c["round"])
        check_swiglu(fmt, ref, q.cpu().numpy(), _row_scales(fmt, layout, s, M, W), from_fp32=c["from32"])
    else:
        src = _act_tensor(g, M, W, c["fp16"])
        q, s = quantize_fp8(src.to(DEV), fmt=fmt, scale_layout=layout)
        torch.cuda.synchronize()
        ref = oracle.quantize(fmt, _bits(src), fp16=c["fp16"])
        check_quant(fmt, ref, q.cpu().numpy(), _row_scales(fmt, layout, s, M, W), from_fp32=False)
