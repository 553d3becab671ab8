"""ctypes binding of libsgq.so (include/sgq.h), with the same entry-point names.

Argument marshalling only: shape, dtype and device checks, output allocation
with torch.empty, and the call. Every arithmetic step runs in the CUDA kernels.
If the library is missing, the first call raises SgqError: there is no
fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libsgq.so"

FORMATS = {"mxfp8": 0, "block128": 1, "per_token": 2}
ACTS = {"swiglu_oai": 0, "silu_mul": 1}
F_GEMMA_WEIGHT, F_QUANT_FROM_FP32, F_ACT_ROUND_BF16 = 1, 2, 4
F_SCALE_SWIZZLED, F_SCALE_COL_MAJOR = 8, 16
F_FP16 = 32
ACT_DTYPES = (torch.bfloat16, torch.float16)   # the 16-bit activation types of the norms and the quant
GROUP = {"mxfp8": 32, "block128": 128}
# scale layouts: name -> (flag, the one format it applies to, or None for all)
SCALE_LAYOUTS = {"row": (0, None), "swizzled": (F_SCALE_SWIZZLED, "mxfp8"), "col_major": (F_SCALE_COL_MAJOR, "block128")}

_lib = None


class NormSeg(C.Structure):
    """sgq_norm_seg_t: one row set of rmsnorm_dual_quant."""
    _fields_ = [("H", C.c_int64), ("ld", C.c_int64), ("x", C.c_void_p), ("weight", C.c_void_p),
                ("q_out", C.c_void_p), ("scale_out", C.c_void_p), ("normed_out", C.c_void_p)]


class SgqError(RuntimeError):
    """A non-zero status from the library, or a missing library."""

    def __init__(self, msg: str, status: int | None = None):
        super().__init__(msg)
        self.status = status


def library_path() -> str:
    return os.environ.get("SGQ_LIBRARY", os.path.join(HERE, LIB_NAME))


def library() -> C.CDLL:
    """Load libsgq.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise SgqError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(path)
        vp, i64 = C.c_void_p, C.c_int64
        L.rmsnorm_add_quant.restype = C.c_int
        L.rmsnorm_add_quant.argtypes = [C.c_int, C.c_uint32, i64, i64, C.c_float,
                                        vp, vp, vp, vp, vp, vp, vp, vp]
        L.swiglu_quant.restype = C.c_int
        L.swiglu_quant.argtypes = [C.c_int, C.c_int, C.c_uint32, i64, i64, C.c_float, C.c_float,
                                   C.c_float, vp, vp, vp, vp]
        L.rmsnorm_add.restype = C.c_int
        L.rmsnorm_add.argtypes = [C.c_uint32, i64, i64, C.c_float, vp, vp, vp, vp, vp, vp]
        L.swiglu.restype = C.c_int
        L.swiglu.argtypes = [C.c_int, C.c_uint32, i64, i64, C.c_float, C.c_float, C.c_float, vp, vp, vp]
        L.quantize_fp8.restype = C.c_int
        L.quantize_fp8.argtypes = [C.c_int, C.c_uint32, i64, i64, vp, vp, vp, vp]
        L.rmsnorm_dual_quant.restype = C.c_int
        L.rmsnorm_dual_quant.argtypes = [C.c_int, C.c_uint32, i64, C.c_float, C.POINTER(NormSeg),
                                         C.POINTER(NormSeg), vp]
        L.sgq_status_string.restype = C.c_char_p
        L.sgq_status_string.argtypes = [C.c_int]
        L.sgq_abi_version.restype = C.c_int
        L.sgq_abi_version.argtypes = []
        L.sgq_launch_error.restype = C.c_char_p
        L.sgq_launch_error.argtypes = []
        L.allreduce_rmsnorm_add_quant.restype = C.c_int
        L.allreduce_rmsnorm_add_quant.argtypes = [C.c_int, C.c_uint32, C.c_int, i64, i64, C.c_float,
                                                  C.POINTER(C.c_void_p), vp, vp, vp, vp, vp, vp, vp]
        L.sgq_set_sm_budget.restype = C.c_int
        L.sgq_set_sm_budget.argtypes = [C.c_int]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return library().sgq_status_string(int(status)).decode()


def set_sm_budget(sms: int) -> None:
    """Plan launches as if the device had `sms` multiprocessors (0: the
    device's own count). Process-wide; see sgq_set_sm_budget in sgq.h."""
    _check(library().sgq_set_sm_budget(int(sms)), "sgq_set_sm_budget")


def _check(status: int, what: str):
    if status != 0:
        detail = f": {library().sgq_launch_error().decode()}" if status == 4 else ""
        raise SgqError(f"{what}: {status_string(status)} (status {status}){detail}", status)


def _ptr(t: torch.Tensor | None):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _round_up(v: int, m: int) -> int:
    return (v + m - 1) // m * m


def scale_shape(fmt: str, M: int, W: int, layout: str = "row") -> tuple:
    """Shape of the scale tensor: row-major [M, groups] ([M, 1] per-token);
    swizzled MXFP8 [M rounded up to 128, groups rounded up to 4] holding the
    512-byte tiles in order; column-major 1x128 [groups, M rounded up to 4]."""
    if layout == "swizzled":
        return (_round_up(M, 128), _round_up(W // 32, 4))
    if layout == "col_major":
        return (W // 128, _round_up(M, 4))
    return (M, 1) if fmt == "per_token" else (M, W // GROUP[fmt])


def _layout_flag(fmt: str, layout: str) -> int:
    if layout not in SCALE_LAYOUTS:
        raise SgqError(f"unknown scale layout {layout!r}")
    flag, only = SCALE_LAYOUTS[layout]
    if only is not None and fmt != only:
        raise SgqError(f"scale layout {layout!r} applies to {only} only, not {fmt}")
    return flag


def scale_dtype(fmt: str) -> torch.dtype:
    return torch.uint8 if fmt == "mxfp8" else torch.float32


def _act_dtype(t: torch.Tensor, name: str) -> torch.dtype:
    if t.dtype not in ACT_DTYPES:
        raise SgqError(f"{name}: expected bfloat16 or float16, got {t.dtype}")
    return t.dtype


def _want(t: torch.Tensor, shape, dtype, name):
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise SgqError(f"{name}: expected {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")
    if t.numel() and not t.is_contiguous():
        raise SgqError(f"{name}: must be contiguous")


def rmsnorm_add_quant(x: torch.Tensor, weight: torch.Tensor, *, fmt: str = "mxfp8",
                      residual_in: torch.Tensor | None = None,
                      residual_out: torch.Tensor | None = None, eps: float = 1e-6,
                      gemma: bool = True, quant_from_fp32: bool = False, normed: bool = False,
                      q_out: torch.Tensor | None = None, scale_out: torch.Tensor | None = None,
                      normed_out: torch.Tensor | None = None, scale_layout: str = "row", stream=None):
    """Residual add + RMSNorm + FP8 quantisation (one kernel launch).

    x [M,H] bf16; weight [H] bf16; residual_in [M,H] bf16 or None;
    residual_out defaults to residual_in (in-place update) when residual_in is
    given. x, weight and the residual are all bfloat16 or all float16 (the
    written rows then have the same type). Returns (q [M,H] uint8 E4M3,
    scale, normed [M,H] or None, residual_out or None).
    """
    M, H = x.shape
    dt = _act_dtype(x, "x")
    _want(x, (M, H), dt, "x")
    _want(weight, (H,), dt, "weight")
    if residual_in is not None:
        _want(residual_in, (M, H), dt, "residual_in")
        if residual_out is None:
            residual_out = residual_in
    if residual_out is not None:
        _want(residual_out, (M, H), dt, "residual_out")
    dev = x.device
    if q_out is None:
        q_out = torch.empty((M, H), dtype=torch.uint8, device=dev)
    if fmt not in FORMATS:
        raise SgqError(f"unknown format {fmt!r}")
    lflag = _layout_flag(fmt, scale_layout)
    if scale_out is None:
        scale_out = torch.empty(scale_shape(fmt, M, H, scale_layout), dtype=scale_dtype(fmt), device=dev)
    if normed and normed_out is None:
        normed_out = torch.empty((M, H), dtype=dt, device=dev)
    _want(q_out, (M, H), torch.uint8, "q_out")
    _want(scale_out, scale_shape(fmt, M, H, scale_layout), scale_dtype(fmt), "scale_out")
    if normed_out is not None:
        _want(normed_out, (M, H), dt, "normed_out")
    flags = (F_GEMMA_WEIGHT if gemma else 0) | (F_QUANT_FROM_FP32 if quant_from_fp32 else 0) | lflag
    flags |= F_FP16 if dt == torch.float16 else 0
    st = library().rmsnorm_add_quant(FORMATS[fmt], flags, M, H, float(eps), _ptr(x),
                                     _ptr(residual_in), _ptr(residual_out), _ptr(weight),
                                     _ptr(q_out), _ptr(scale_out), _ptr(normed_out), _stream(stream))
    _check(st, "rmsnorm_add_quant")
    return q_out, scale_out, normed_out, residual_out


def swiglu_quant(gate_up: torch.Tensor, *, fmt: str = "mxfp8", act: str = "swiglu_oai",
                 quant_from_fp32: bool = True, round_act_bf16: bool = False, alpha: float = 1.702,
                 beta: float = 1.0, limit: float = 7.0, q_out: torch.Tensor | None = None,
                 scale_out: torch.Tensor | None = None, scale_layout: str = "row", stream=None):
    """SwiGLU + FP8 quantisation (one kernel launch).

    gate_up [M, 2I] bf16 (gate = first half, up = second half). Returns
    (q [M,I] uint8 E4M3, scale).
    """
    M, I2 = gate_up.shape
    I = I2 // 2
    _want(gate_up, (M, 2 * I), torch.bfloat16, "gate_up")
    if I2 % 2:
        raise SgqError("gate_up: width must be even")
    if fmt not in FORMATS or act not in ACTS:
        raise SgqError(f"unknown format/activation {fmt!r}/{act!r}")
    dev = gate_up.device
    lflag = _layout_flag(fmt, scale_layout)
    if q_out is None:
        q_out = torch.empty((M, I), dtype=torch.uint8, device=dev)
    if scale_out is None:
        scale_out = torch.empty(scale_shape(fmt, M, I, scale_layout), dtype=scale_dtype(fmt), device=dev)
    _want(q_out, (M, I), torch.uint8, "q_out")
    _want(scale_out, scale_shape(fmt, M, I, scale_layout), scale_dtype(fmt), "scale_out")
    flags = (F_QUANT_FROM_FP32 if quant_from_fp32 else 0) | (F_ACT_ROUND_BF16 if round_act_bf16 else 0) | lflag
    st = library().swiglu_quant(FORMATS[fmt], ACTS[act], flags, M, I, float(alpha), float(beta),
                                float(limit), _ptr(gate_up), _ptr(q_out), _ptr(scale_out), _stream(stream))
    _check(st, "swiglu_quant")
    return q_out, scale_out


def rmsnorm_add(x: torch.Tensor, weight: torch.Tensor, *, residual_in: torch.Tensor | None = None,
                residual_out: torch.Tensor | None = None, eps: float = 1e-6, gemma: bool = True,
                normed_out: torch.Tensor | None = None, stream=None):
    """Residual add + RMSNorm to bf16 (the norm step of the unfused chain).

    Returns (normed [M,H] in x's type, residual_out or None); residual_out
    defaults to residual_in (in-place update) when residual_in is given.
    """
    M, H = x.shape
    dt = _act_dtype(x, "x")
    _want(x, (M, H), dt, "x")
    _want(weight, (H,), dt, "weight")
    if residual_in is not None:
        _want(residual_in, (M, H), dt, "residual_in")
        if residual_out is None:
            residual_out = residual_in
    if residual_out is not None:
        _want(residual_out, (M, H), dt, "residual_out")
    if normed_out is None:
        normed_out = torch.empty((M, H), dtype=dt, device=x.device)
    _want(normed_out, (M, H), dt, "normed_out")
    flags = (F_GEMMA_WEIGHT if gemma else 0) | (F_FP16 if dt == torch.float16 else 0)
    st = library().rmsnorm_add(flags, M, H, float(eps), _ptr(x), _ptr(residual_in),
                               _ptr(residual_out), _ptr(weight), _ptr(normed_out), _stream(stream))
    _check(st, "rmsnorm_add")
    return normed_out, residual_out


def swiglu(gate_up: torch.Tensor, *, act: str = "swiglu_oai", round_act_bf16: bool = False,
           alpha: float = 1.702, beta: float = 1.0, limit: float = 7.0, out: torch.Tensor | None = None,
           stream=None):
    """SwiGLU to bf16 (the activation step of the unfused chain).

    gate_up [M, 2I] bf16. Returns out [M, I] bf16.
    """
    M, I2 = gate_up.shape
    I = I2 // 2
    _want(gate_up, (M, 2 * I), torch.bfloat16, "gate_up")
    if I2 % 2:
        raise SgqError("gate_up: width must be even")
    if act not in ACTS:
        raise SgqError(f"unknown activation {act!r}")
    if out is None:
        out = torch.empty((M, I), dtype=torch.bfloat16, device=gate_up.device)
    _want(out, (M, I), torch.bfloat16, "out")
    st = library().swiglu(ACTS[act], F_ACT_ROUND_BF16 if round_act_bf16 else 0, M, I, float(alpha), float(beta),
                          float(limit), _ptr(gate_up), _ptr(out), _stream(stream))
    _check(st, "swiglu")
    return out


def quantize_fp8(src: torch.Tensor, *, fmt: str = "mxfp8", q_out: torch.Tensor | None = None,
                 scale_out: torch.Tensor | None = None, scale_layout: str = "row", stream=None):
    """FP8 quantisation of bf16 rows (the separate quant of the unfused chain).

    src [M, W] bfloat16 or float16. Returns (q [M,W] uint8 E4M3, scale).
    """
    M, W = src.shape
    dt = _act_dtype(src, "src")
    _want(src, (M, W), dt, "src")
    if fmt not in FORMATS:
        raise SgqError(f"unknown format {fmt!r}")
    lflag = _layout_flag(fmt, scale_layout)
    if q_out is None:
        q_out = torch.empty((M, W), dtype=torch.uint8, device=src.device)
    if scale_out is None:
        scale_out = torch.empty(scale_shape(fmt, M, W, scale_layout), dtype=scale_dtype(fmt), device=src.device)
    _want(q_out, (M, W), torch.uint8, "q_out")
    _want(scale_out, scale_shape(fmt, M, W, scale_layout), scale_dtype(fmt), "scale_out")
    lflag |= F_FP16 if dt == torch.float16 else 0
    st = library().quantize_fp8(FORMATS[fmt], lflag, M, W, _ptr(src), _ptr(q_out), _ptr(scale_out),
                                _stream(stream))
    _check(st, "quantize_fp8")
    return q_out, scale_out


def _seg_input(x: torch.Tensor, name: str):
    """A 2-D activation whose rows may be strided (a column range of a wider
    tensor): unit column stride, row stride ld >= width."""
    if x.dim() != 2 or (x.shape[0] > 1 and x.stride(1) != 1) or (x.shape[1] > 1 and x.stride(1) != 1):
        raise SgqError(f"{name}: expected a 2-D tensor with unit column stride")
    ld = x.stride(0) if x.shape[0] > 1 else x.shape[1]
    if ld < x.shape[1]:
        raise SgqError(f"{name}: row stride {ld} below the width {x.shape[1]}")
    return ld


def rmsnorm_dual_quant(xa: torch.Tensor, wa: torch.Tensor, xb: torch.Tensor, wb: torch.Tensor, *,
                       fmt: str = "per_token", eps: float = 1e-6, gemma: bool = False,
                       quant_from_fp32: bool = False, quant_a: bool = True, quant_b: bool = False,
                       normed_a: bool = False, normed_b: bool = True, stream=None):
    """Two RMSNorms over the same rows in one launch (the q and kv latent
    norms): segment a (xa [M,Ha], wa [Ha]) and b (xb [M,Hb], wb [Hb]). xa and
    xb may be column ranges of one tensor (strided rows). Each segment is
    quantised (quant_*) and/or written in its activation type (normed_*).
    Returns ((qa, sa, na), (qb, sb, nb)) with None for what was not asked.
    """
    M = xa.shape[0]
    if xb.shape[0] != M:
        raise SgqError("xa and xb must have the same number of rows")
    if fmt not in FORMATS:
        raise SgqError(f"unknown format {fmt!r}")
    dt = _act_dtype(xa, "xa")
    segs, outs = [], []
    for name, x, w, quant, normed in (("a", xa, wa, quant_a, normed_a), ("b", xb, wb, quant_b, normed_b)):
        if x.dtype != dt:
            raise SgqError(f"x{name}: expected {dt}, got {x.dtype}")
        H = x.shape[1]
        ld = _seg_input(x, f"x{name}")
        _want(w, (H,), dt, f"w{name}")
        if not (quant or normed):
            raise SgqError(f"segment {name}: nothing to write")
        q = torch.empty((M, H), dtype=torch.uint8, device=x.device) if quant else None
        s = torch.empty(scale_shape(fmt, M, H), dtype=scale_dtype(fmt), device=x.device) if quant else None
        n = torch.empty((M, H), dtype=dt, device=x.device) if normed else None
        segs.append(NormSeg(H, ld, x.data_ptr(), w.data_ptr(), q.data_ptr() if quant else None,
                            s.data_ptr() if quant else None, n.data_ptr() if normed else None))
        outs.append((q, s, n))
    flags = (F_GEMMA_WEIGHT if gemma else 0) | (F_QUANT_FROM_FP32 if quant_from_fp32 else 0)
    flags |= F_FP16 if dt == torch.float16 else 0
    st = library().rmsnorm_dual_quant(FORMATS[fmt], flags, M, float(eps), C.byref(segs[0]), C.byref(segs[1]),
                                      _stream(stream))
    _check(st, "rmsnorm_dual_quant")
    return outs[0], outs[1]


MAX_RANKS = 8


def allreduce_rmsnorm_add_quant(partials: list, weight: torch.Tensor, *, fmt: str = "mxfp8",
                                residual_in: torch.Tensor | None = None,
                                residual_out: torch.Tensor | None = None, eps: float = 1e-6,
                                gemma: bool = True, quant_from_fp32: bool = False, normed: bool = False,
                                q_out: torch.Tensor | None = None, scale_out: torch.Tensor | None = None,
                                normed_out: torch.Tensor | None = None, scale_layout: str = "row", stream=None):
    """Tensor-parallel all-reduce + residual add + RMSNorm + FP8 quantisation
    (one kernel launch): x = bf16 of the partials' fp32 sum in rank order,
    then rmsnorm_add_quant(x, ...). partials: the ranks' [M, H] bf16 tensors
    (this device's memory, or peers' mapped into it); every partial must be
    complete before the launch. Returns (q, scale, normed or None,
    residual_out or None); residual_out defaults to residual_in.
    """
    if not 1 <= len(partials) <= MAX_RANKS:
        raise SgqError(f"partials: 1 to {MAX_RANKS} tensors, got {len(partials)}")
    M, H = partials[0].shape
    for k, p in enumerate(partials):
        _want(p, (M, H), torch.bfloat16, f"partials[{k}]")
    _want(weight, (H,), torch.bfloat16, "weight")
    if residual_in is not None:
        _want(residual_in, (M, H), torch.bfloat16, "residual_in")
        if residual_out is None:
            residual_out = residual_in
    if residual_out is not None:
        _want(residual_out, (M, H), torch.bfloat16, "residual_out")
    if fmt not in FORMATS:
        raise SgqError(f"unknown format {fmt!r}")
    dev = partials[0].device
    lflag = _layout_flag(fmt, scale_layout)
    if q_out is None:
        q_out = torch.empty((M, H), dtype=torch.uint8, device=dev)
    if scale_out is None:
        scale_out = torch.empty(scale_shape(fmt, M, H, scale_layout), dtype=scale_dtype(fmt), device=dev)
    if normed and normed_out is None:
        normed_out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    _want(q_out, (M, H), torch.uint8, "q_out")
    _want(scale_out, scale_shape(fmt, M, H, scale_layout), scale_dtype(fmt), "scale_out")
    if normed_out is not None:
        _want(normed_out, (M, H), torch.bfloat16, "normed_out")
    flags = (F_GEMMA_WEIGHT if gemma else 0) | (F_QUANT_FROM_FP32 if quant_from_fp32 else 0) | lflag
    ptrs = (C.c_void_p * len(partials))(*[p.data_ptr() for p in partials])
    st = library().allreduce_rmsnorm_add_quant(FORMATS[fmt], flags, len(partials), M, H, float(eps), ptrs,
                                               _ptr(residual_in), _ptr(residual_out), _ptr(weight), _ptr(q_out),
                                               _ptr(scale_out), _ptr(normed_out), _stream(stream))
    _check(st, "allreduce_rmsnorm_add_quant")
    return q_out, scale_out, normed_out, residual_out
