"""CPU oracle of the fused norm / SwiGLU + FP8 quantisation ops.

TEST INFRASTRUCTURE ONLY: the tests, `__graft_entry__.smoke()` and the
benchmark's CPU-baseline leg use it; the library's product path never imports
it. It wraps `sgq_oracle.c` (plain fp64 C, scalar loops) through ctypes and
takes and returns numpy arrays. Inputs are raw bf16 bit patterns (uint16).

Every function computes the definitions stated in `sgq_oracle.c`, except
`scale_layout`, a plain Python rearrangement of finished scales. Parity pins
(closed forms, brute force and the pages' printed statistics) are in
tests/test_oracle_*.py.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from .build import build_oracle

FORMATS = {"mxfp8": 0, "block128": 1, "per_token": 2}
ACTS = {"swiglu_oai": 0, "silu_mul": 1}
F_GEMMA, F_FROM_FP32, F_ACT_ROUND_BF16, F_FP16 = 1, 2, 4, 32
AMB_SRC, AMB_CODE, AMB_TIE = 1, 2, 4
REL_WINDOW = 2.0 ** -20

_lib = None


def lib() -> C.CDLL:
    """The oracle library: built beside its source, or the prebuilt library
    named by SGQ_ORACLE_LIBRARY (the mutation tests' planted-mistake builds)."""
    global _lib
    if _lib is None:
        L = C.CDLL(os.environ.get("SGQ_ORACLE_LIBRARY") or build_oracle())
        L.ora_bf16_decode.restype = C.c_double
        L.ora_bf16_decode.argtypes = [C.c_uint16]
        L.ora_bf16_round.restype = C.c_uint16
        L.ora_bf16_round.argtypes = [C.c_double]
        L.ora_f16_decode.restype = C.c_double
        L.ora_f16_decode.argtypes = [C.c_uint16]
        L.ora_f16_round.restype = C.c_uint16
        L.ora_f16_round.argtypes = [C.c_double]
        L.ora_e4m3_decode.restype = C.c_double
        L.ora_e4m3_decode.argtypes = [C.c_uint8]
        L.ora_e4m3_encode.restype = C.c_uint8
        L.ora_e4m3_encode.argtypes = [C.c_double]
        L.ora_mx_scale_exp.restype = C.c_int
        L.ora_mx_scale_exp.argtypes = [C.c_double]
        p = C.c_void_p
        L.ora_rmsnorm_add_quant.restype = C.c_int
        L.ora_rmsnorm_add_quant.argtypes = [C.c_int, C.c_uint, C.c_long, C.c_long, C.c_float,
                                            p, p, p, p, p, p, p, p, p, p, p, C.c_double]
        L.ora_swiglu_quant.restype = C.c_int
        L.ora_swiglu_quant.argtypes = [C.c_int, C.c_int, C.c_uint, C.c_long, C.c_long, C.c_float,
                                       C.c_float, C.c_float, p, p, p, p, p, p, p, C.c_double]
        L.ora_allreduce_sum.restype = C.c_int
        L.ora_allreduce_sum.argtypes = [C.c_int, C.POINTER(C.c_void_p), C.c_long, C.c_uint, p, p, C.c_double]
        L.ora_quantize.restype = C.c_int
        L.ora_quantize.argtypes = [C.c_int, C.c_uint, C.c_long, C.c_long, p, p, p, p, p, p, C.c_double]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def bf16_decode(b: int) -> float:
    return lib().ora_bf16_decode(int(b) & 0xFFFF)


def bf16_round(v: float) -> int:
    return int(lib().ora_bf16_round(float(v)))


def e4m3_decode(c: int) -> float:
    return lib().ora_e4m3_decode(int(c) & 0xFF)


def e4m3_encode(v: float) -> int:
    return int(lib().ora_e4m3_encode(float(v)))


def mx_scale_exp(amax: float) -> int:
    return int(lib().ora_mx_scale_exp(float(amax)))


def _group(fmt: str, width: int) -> int:
    return {"mxfp8": 32, "block128": 128, "per_token": width}[fmt]


def _scale_array(fmt: str, M: int, width: int) -> np.ndarray:
    ng = width // _group(fmt, width)
    return np.zeros((M, ng), dtype=np.uint8 if fmt == "mxfp8" else np.float32)


def _u16(a, shape):
    a = np.ascontiguousarray(a, dtype=np.uint16)
    assert a.shape == shape, (a.shape, shape)
    return a


def rmsnorm_add_quant(fmt: str, x: np.ndarray, r: np.ndarray | None, w: np.ndarray, *,
                      eps: float, gemma: bool, from_fp32: bool, normed: bool = True,
                      diagnostics: bool = True, rel: float = REL_WINDOW, fp16: bool = False) -> dict:
    """Residual add + RMSNorm + FP8 quantisation of rows x [M,H] (bf16 bits,
    or fp16 bits with fp16=True, which also makes the written rows fp16).

    Returns q (uint8 [M,H]), scale ([M,G] uint8 E8M0 codes or float32),
    residual (uint16 bits or None), normed (uint16 bits or None) and, with
    diagnostics, y (fp64 normed values), t (fp64 E4M3 arguments), amb and gamb.
    """
    M, H = x.shape
    x = _u16(x, (M, H))
    r = None if r is None else _u16(r, (M, H))
    w = _u16(w, (H,))
    q = np.zeros((M, H), np.uint8)
    s = _scale_array(fmt, M, H)
    r_out = np.zeros((M, H), np.uint16) if r is not None else None
    n_out = np.zeros((M, H), np.uint16) if normed else None
    y = t = amb = gamb = None
    if diagnostics:
        y, t = np.zeros((M, H)), np.zeros((M, H))
        amb, gamb = np.zeros((M, H), np.uint8), np.zeros(s.shape, np.uint8)
    flags = (F_GEMMA if gemma else 0) | (F_FROM_FP32 if from_fp32 else 0) | (F_FP16 if fp16 else 0)
    rc = lib().ora_rmsnorm_add_quant(FORMATS[fmt], flags, M, H, float(eps), _ptr(x), _ptr(r), _ptr(w),
                                     _ptr(r_out), _ptr(n_out), _ptr(q), _ptr(s), _ptr(y), _ptr(t),
                                     _ptr(amb), _ptr(gamb), rel)
    if rc != 0:
        raise ValueError(f"oracle rejected arguments (fmt={fmt}, M={M}, H={H})")
    return {"q": q, "scale": s, "residual": r_out, "normed": n_out, "y": y, "t": t,
            "amb": amb, "gamb": gamb}


def swiglu_quant(fmt: str, act: str, gate_up: np.ndarray, *, from_fp32: bool,
                 round_act_bf16: bool = False, alpha: float = 1.702, beta: float = 1.0,
                 limit: float = 7.0, diagnostics: bool = True, rel: float = REL_WINDOW) -> dict:
    """SwiGLU (OAI clamped or SiLU-and-mul) + FP8 quantisation of gate_up [M, 2I] (bf16 bits).

    Returns q (uint8 [M,I]), scale, and with diagnostics a (fp64 activation),
    t, amb and gamb.
    """
    M, I2 = gate_up.shape
    I = I2 // 2
    gu = _u16(gate_up, (M, I2))
    q = np.zeros((M, I), np.uint8)
    s = _scale_array(fmt, M, I)
    a = t = amb = gamb = None
    if diagnostics:
        a, t = np.zeros((M, I)), np.zeros((M, I))
        amb, gamb = np.zeros((M, I), np.uint8), np.zeros(s.shape, np.uint8)
    flags = (F_FROM_FP32 if from_fp32 else 0) | (F_ACT_ROUND_BF16 if round_act_bf16 else 0)
    rc = lib().ora_swiglu_quant(FORMATS[fmt], ACTS[act], flags, M, I, float(alpha), float(beta),
                                float(limit), _ptr(gu), _ptr(q), _ptr(s), _ptr(a), _ptr(t),
                                _ptr(amb), _ptr(gamb), rel)
    if rc != 0:
        raise ValueError(f"oracle rejected arguments (fmt={fmt}, act={act}, M={M}, I={I})")
    return {"q": q, "scale": s, "a": a, "t": t, "amb": amb, "gamb": gamb}


def quantize(fmt: str, src: np.ndarray, *, diagnostics: bool = True, rel: float = REL_WINDOW,
             fp16: bool = False) -> dict:
    """Standalone FP8 quantisation of bf16 rows src [M, W] (bf16 bits, or fp16
    bits with fp16=True): the quant of the unfused chains. Returns q, scale
    and, with diagnostics, t, amb and gamb."""
    M, W = src.shape
    src = _u16(src, (M, W))
    q = np.zeros((M, W), np.uint8)
    s = _scale_array(fmt, M, W)
    t = amb = gamb = None
    if diagnostics:
        t, amb, gamb = np.zeros((M, W)), np.zeros((M, W), np.uint8), np.zeros(s.shape, np.uint8)
    rc = lib().ora_quantize(FORMATS[fmt], F_FP16 if fp16 else 0, M, W, _ptr(src), _ptr(q), _ptr(s), _ptr(t), _ptr(amb), _ptr(gamb), rel)
    if rc != 0:
        raise ValueError(f"oracle rejected arguments (fmt={fmt}, M={M}, W={W})")
    return {"q": q, "scale": s, "t": t, "amb": amb, "gamb": gamb}


def scale_layout(fmt: str, scale: np.ndarray, layout: str) -> np.ndarray:
    """Rearrange row-major scales [M, G] into another consumer layout.

    "row":       unchanged.
    "swizzled":  (MXFP8) the tiled scale-factor layout of block-scaled MMA
                 operands: rows padded to a multiple of 128 and columns to a
                 multiple of 4 with zeros; the padded [Mp, Gp] array is cut
                 into tiles of 128 rows x 4 columns, which are laid out one
                 after another, tile columns fastest; inside a tile, row r
                 and column g go to position (r % 32) * 16 + (r // 32) * 4 + g.
                 Returned as [Mp, Gp] (the flat buffer, reshaped).
    "col_major": (1x128) the transpose [G, Mp], rows padded to a multiple of 4
                 with zeros.

    Scale layouts are a convention of the consumer GEMM: the review section
    "Scale layout / scheme contract" of "[ROCm][MiniMax-M3.1] Fuse MXFP8 quant
    into the add+RMSNorm and SwiGLU epilogues" separates consumers of
    row-major [M, N/32] E8M0 scales from consumers of swizzled ones. Written
    as plain loops over the entries.
    """
    scale = np.asarray(scale)
    M, G = scale.shape
    if layout == "row":
        return scale.copy()
    if layout == "swizzled":
        assert fmt == "mxfp8"
        Mp, Gp = -(-M // 128) * 128, -(-G // 4) * 4
        flat = np.zeros(Mp * Gp, dtype=scale.dtype)
        tiles_per_band = Gp // 4
        for r in range(M):
            for g in range(G):
                tile = (r // 128) * tiles_per_band + g // 4
                rr, gg = r % 128, g % 4
                flat[tile * 512 + (rr % 32) * 16 + (rr // 32) * 4 + gg] = scale[r, g]
        return flat.reshape(Mp, Gp)
    if layout == "col_major":
        assert fmt == "block128"
        Mp = -(-M // 4) * 4
        out = np.zeros((G, Mp), dtype=scale.dtype)
        for r in range(M):
            for g in range(G):
                out[g, r] = scale[r, g]
        return out
    raise ValueError(f"unknown scale layout {layout!r}")


def f16_decode(b: int) -> float:
    return lib().ora_f16_decode(int(b))


def f16_round(v: float) -> int:
    return lib().ora_f16_round(float(v))


def rmsnorm_dual_quant(fmt: str, xa: np.ndarray, wa: np.ndarray, xb: np.ndarray, wb: np.ndarray, *, eps: float,
                       gemma: bool, from_fp32: bool, fp16: bool = False, **kw) -> tuple:
    """Two independent RMSNorms (no residual) + quantisation over the same
    rows: the q and kv latent norms of multi-head latent attention, which
    "[ROCm] Fuse per-token activation quant into RMSNorm for per-channel
    quantized attention" (sglang PR 34502), "Change", runs as one fused q/kv
    RMSNorm. Each half is exactly rmsnorm_add_quant of its own rows and
    weight; returns the two result dicts."""
    a = rmsnorm_add_quant(fmt, xa, None, wa, eps=eps, gemma=gemma, from_fp32=from_fp32, fp16=fp16, **kw)
    b = rmsnorm_add_quant(fmt, xb, None, wb, eps=eps, gemma=gemma, from_fp32=from_fp32, fp16=fp16, **kw)
    return a, b


def allreduce_sum(parts: list, *, fp16: bool = False, rel: float = REL_WINDOW) -> tuple:
    """The all-reduce over tensor-parallel ranks that precedes the norm: the
    element-wise sum of the ranks' partial tensors (16-bit patterns, all of
    one shape) in fp64, rounded once to the activation type. Returns (the
    sum's 16-bit patterns, a uint8 mask of the elements whose fp64 sum lies
    within `rel` of a rounding boundary of that type)."""
    parts = [np.ascontiguousarray(a, dtype=np.uint16) for a in parts]
    shape = parts[0].shape
    assert all(a.shape == shape for a in parts)
    out = np.zeros(shape, np.uint16)
    near = np.zeros(shape, np.uint8)
    ptrs = (C.c_void_p * len(parts))(*[a.ctypes.data for a in parts])
    rc = lib().ora_allreduce_sum(len(parts), ptrs, out.size, F_FP16 if fp16 else 0, _ptr(out), _ptr(near), rel)
    if rc != 0:
        raise ValueError("oracle rejected arguments (allreduce_sum)")
    return out, near


def allreduce_rmsnorm_add_quant(fmt: str, parts: list, r: np.ndarray | None, w: np.ndarray, **kw) -> dict:
    """All-reduce + residual add + RMSNorm + FP8 quantisation, in the order of
    its steps: x = allreduce_sum(parts) (the all-reduce's output), then
    rmsnorm_add_quant(x, r, w). The result carries x and its boundary mask
    (`x`, `x_near`) beside rmsnorm_add_quant's outputs."""
    x, near = allreduce_sum(parts, fp16=kw.get("fp16", False))
    ref = rmsnorm_add_quant(fmt, x, r, w, **kw)
    ref["x"], ref["x_near"] = x, near
    return ref
