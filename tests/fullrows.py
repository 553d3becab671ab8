"""Parity over every row of a launch: the oracle and the checker run on row
blocks, one block per task, on all host threads (the C oracle and numpy's
loops run outside the interpreter lock). The code-mismatch budgets (1e-4
away from exact ties, 1e-3 at them) are applied to the totals over all
blocks; every other tolerance applies in each block. Used by the GPU parity tests for launches too large for one oracle
call."""
from __future__ import annotations

import concurrent.futures as cf
import os

import oracle
from oracle.parity import budget_result, check_norm, check_swiglu

BLOCK = 256


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _merge(parts: list) -> dict:
    out = {}
    for st in parts:
        for k, v in st.items():
            if k.endswith("_frac") or k.startswith("scale_max"):
                out[k] = max(out.get(k, v), v) if k.startswith("scale_max") else out.get(k, 0.0) + v * st.get("n_plain", 0)
            else:
                out[k] = out.get(k, 0) + v
    n = out.get("n_plain", 0)
    for k in list(out):
        if k.endswith("_frac"):
            out[k] = out[k] / max(n, 1)
    out["code_mismatch_frac"] = out.get("code_mismatch", 0) / max(n, 1)
    return out


def _finish(parts: list) -> dict:
    st = _merge(parts)
    ok, msg = budget_result(st.get("code_mismatch", 0), st.get("tie_mismatch", 0), st.get("n_plain", 0))
    assert ok, msg
    return st


def norm_all_rows(fmt, x, r, w, q, s, normed, residual, *, eps, gemma, from_fp32, fp16=False) -> dict:
    """x, r (or None), w: 16-bit patterns; q, s, normed (or None), residual
    (or None): the library's outputs as numpy arrays, all rows."""
    M = x.shape[0]

    def block(a):
        b = min(a + BLOCK, M)
        ref = oracle.rmsnorm_add_quant(fmt, x[a:b], None if r is None else r[a:b], w, eps=eps, gemma=gemma,
                                       from_fp32=from_fp32, normed=normed is not None, fp16=fp16)
        return check_norm(fmt, ref, q[a:b], s[a:b], None if normed is None else normed[a:b],
                          None if residual is None else residual[a:b], from_fp32=from_fp32, budget=False)

    with cf.ThreadPoolExecutor(_threads()) as ex:
        return _finish(list(ex.map(block, range(0, M, BLOCK))))


def swiglu_all_rows(fmt, act, gu, q, s, *, from_fp32, round_act_bf16=False, alpha=1.702, beta=1.0,
                    limit=7.0) -> dict:
    """gu: bf16 patterns [M, 2I]; q, s: the library's outputs, all rows."""
    M = gu.shape[0]

    def block(a):
        b = min(a + BLOCK, M)
        ref = oracle.swiglu_quant(fmt, act, gu[a:b], from_fp32=from_fp32, round_act_bf16=round_act_bf16,
                                  alpha=alpha, beta=beta, limit=limit)
        return check_swiglu(fmt, ref, q[a:b], s[a:b], from_fp32=from_fp32, budget=False)

    with cf.ThreadPoolExecutor(_threads()) as ex:
        return _finish(list(ex.map(block, range(0, M, BLOCK))))
