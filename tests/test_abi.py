"""The C ABI of libsgq.so (include/sgq.h), checked without a GPU: the library
loads, exports every declared function, agrees with the Python binding and
the oracle on enum and flag values, and rejects bad arguments on the host
with the documented status before anything is launched (fake, never
dereferenced pointers)."""
import ctypes as C
import os
import re

import pytest

import oracle
from swiglu_fp8_activation_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "sgq.h")
OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3
BASE = 1 << 40          # fake device addresses: aligned, far apart, never touched
MB = 1 << 20


def _header():
    with open(HEADER) as f:
        return f.read()


def _declared_functions():
    return re.findall(r"^(?:int|const char\*)\s+(\w+)\(", _header(), flags=re.M)


def _header_value(name):
    m = re.search(rf"\b{name}\s*=\s*(\d+)", _header()) or re.search(rf"#define\s+{name}\s+\(1u << (\d+)\)", _header())
    assert m, name
    v = int(m.group(1))
    return (1 << v) if "<<" in m.group(0) else v


def test_library_exports_every_declared_function(sgq_lib):
    names = _declared_functions()
    assert set(names) == {"rmsnorm_add_quant", "swiglu_quant", "rmsnorm_add", "swiglu", "quantize_fp8",
                          "rmsnorm_dual_quant", "sgq_status_string", "sgq_abi_version", "sgq_launch_error",
                          "sgq_set_sm_budget", "allreduce_rmsnorm_add_quant"}
    for n in names:
        assert hasattr(sgq_lib, n), n
    m = re.search(r"#define SGQ_ABI_VERSION (\d+)", _header())
    assert sgq_lib.sgq_abi_version() == int(m.group(1))


def test_enum_and_flag_values_agree():
    for name, key in (("SGQ_FMT_MXFP8", "mxfp8"), ("SGQ_FMT_FP8_BLOCK128", "block128"),
                      ("SGQ_FMT_FP8_PER_TOKEN", "per_token")):
        assert _header_value(name) == binding.FORMATS[key] == oracle.FORMATS[key]
    for name, key in (("SGQ_ACT_SWIGLU_OAI", "swiglu_oai"), ("SGQ_ACT_SILU_MUL", "silu_mul")):
        assert _header_value(name) == binding.ACTS[key] == oracle.ACTS[key]
    assert _header_value("SGQ_F_GEMMA_WEIGHT") == binding.F_GEMMA_WEIGHT == oracle.F_GEMMA
    assert _header_value("SGQ_F_QUANT_FROM_FP32") == binding.F_QUANT_FROM_FP32 == oracle.F_FROM_FP32
    assert _header_value("SGQ_F_ACT_ROUND_BF16") == binding.F_ACT_ROUND_BF16 == oracle.F_ACT_ROUND_BF16
    assert _header_value("SGQ_F_FP16") == binding.F_FP16 == oracle.F_FP16
    assert _header_value("SGQ_F_SCALE_SWIZZLED") == binding.F_SCALE_SWIZZLED
    assert _header_value("SGQ_F_SCALE_COL_MAJOR") == binding.F_SCALE_COL_MAJOR


def test_launch_error_text_without_a_failure(sgq_lib):
    sgq_lib.sgq_launch_error.restype = C.c_char_p
    assert sgq_lib.sgq_launch_error() == b"no launch error"


def test_sm_budget_rejects_a_negative_count(sgq_lib):
    assert sgq_lib.sgq_set_sm_budget(-1) == 1
    assert sgq_lib.sgq_set_sm_budget(0) == 0


def test_status_strings(sgq_lib):
    for s, word in ((0, "ok"), (1, "invalid"), (2, "unsupported"), (3, "misaligned"), (4, "launch"), (99, "unknown")):
        assert word in sgq_lib.sgq_status_string(s).decode()


def _p(i):
    return C.c_void_p(BASE + i * 64 * MB)


def _host_checked(status):
    """Every call here passes fake pointers, so it must be refused (or be
    empty) before anything launches: a launch status means a case got past
    the host checks and would touch fake addresses on a GPU."""
    assert status != 4, "a fake-pointer call passed the host checks"
    return status


def norm(lib, fmt=0, flags=1, M=8, H=256, eps=1e-6, x=_p(0), r=_p(1), ro=_p(2), w=_p(3), q=_p(4), s=_p(5),
         n=_p(6)):
    return _host_checked(lib.rmsnorm_add_quant(fmt, flags, M, H, eps, x, r, ro, w, q, s, n, None))


def swiglu(lib, fmt=0, act=0, flags=2, M=8, I=256, alpha=1.702, beta=1.0, limit=7.0, gu=_p(0), q=_p(1), s=_p(2)):
    return _host_checked(lib.swiglu_quant(fmt, act, flags, M, I, alpha, beta, limit, gu, q, s, None))


def test_norm_argument_errors(sgq_lib):
    L = sgq_lib
    assert norm(L, M=0) == OK                         # empty: no launch
    assert norm(L, M=0, x=None, q=None) == OK
    assert norm(L, fmt=3) == INVALID
    assert norm(L, fmt=-1) == INVALID
    assert norm(L, flags=1 | 4) == INVALID            # ACT_ROUND_BF16 is not a norm flag
    assert norm(L, flags=1 << 7) == INVALID
    assert norm(L, M=-1) == INVALID
    assert norm(L, H=0) == INVALID
    assert norm(L, eps=-1e-6) == INVALID
    assert norm(L, eps=float("nan")) == INVALID
    assert norm(L, eps=float("inf")) == INVALID
    assert norm(L, H=48) == UNSUPPORTED               # MX needs H % 32 == 0
    assert norm(L, fmt=1, H=96) == UNSUPPORTED        # 1x128 needs H % 128 == 0
    assert norm(L, fmt=2, H=20) == UNSUPPORTED        # per-token needs H % 8 == 0
    assert norm(L, H=131072 + 32) == UNSUPPORTED      # above SGQ_MAX_WIDTH
    for kw in ("x", "w", "q", "s"):
        assert norm(L, **{kw: None}) == INVALID, kw
    assert norm(L, r=None) == INVALID                 # residual_out without residual_in
    assert norm(L, x=C.c_void_p(BASE + 8)) == MISALIGNED
    assert norm(L, q=C.c_void_p(BASE + 4 * 64 * MB + 8)) == MISALIGNED
    assert norm(L, fmt=1, s=C.c_void_p(BASE + 5 * 64 * MB + 2)) == MISALIGNED
    assert norm(L, n=C.c_void_p(BASE + 6 * 64 * MB + 1)) == MISALIGNED
    assert norm(L, q=_p(0)) == INVALID                # q_out overlaps x
    assert norm(L, n=_p(1)) == INVALID                # normed_out overlaps residual_in
    assert norm(L, ro=C.c_void_p(BASE + 64 * MB + 256)) == INVALID   # partial residual overlap
    assert norm(L, s=_p(4)) == INVALID                # scale overlaps q
    assert norm(L, M=1 << 45, H=16384) == INVALID     # 2^59 elements: sizes would overflow
    assert swiglu(L, M=1 << 45, I=16384) == INVALID


def test_swiglu_argument_errors(sgq_lib):
    L = sgq_lib
    assert swiglu(L, M=0) == OK
    assert swiglu(L, fmt=7) == INVALID
    assert swiglu(L, act=2) == INVALID
    assert swiglu(L, flags=4) == INVALID              # ACT_ROUND_BF16 needs SiLU-and-mul
    assert swiglu(L, flags=1) == INVALID              # GEMMA_WEIGHT is not a SwiGLU flag
    assert swiglu(L, limit=0.0) == INVALID
    assert swiglu(L, limit=float("nan")) == INVALID
    assert swiglu(L, alpha=float("inf")) == INVALID
    assert swiglu(L, I=-32) == INVALID
    assert swiglu(L, I=48) == UNSUPPORTED
    assert swiglu(L, fmt=1, I=64) == UNSUPPORTED
    assert swiglu(L, gu=None) == INVALID
    assert swiglu(L, gu=C.c_void_p(BASE + 4)) == MISALIGNED
    assert swiglu(L, q=_p(0)) == INVALID              # q_out overlaps gate_up


def norm_only(lib, flags=1, M=8, H=256, eps=1e-6, x=_p(0), r=_p(1), ro=_p(2), w=_p(3), n=_p(6)):
    return _host_checked(lib.rmsnorm_add(flags, M, H, eps, x, r, ro, w, n, None))


def act_only(lib, act=0, flags=0, M=8, I=256, alpha=1.702, beta=1.0, limit=7.0, gu=_p(0), out=_p(1)):
    return _host_checked(lib.swiglu(act, flags, M, I, alpha, beta, limit, gu, out, None))


def quant(lib, fmt=0, flags=0, M=8, W=256, src=_p(0), q=_p(1), s=_p(2)):
    return _host_checked(lib.quantize_fp8(fmt, flags, M, W, src, q, s, None))


def test_unfused_norm_argument_errors(sgq_lib):
    L = sgq_lib
    assert norm_only(L, M=0, x=None, n=None) == OK
    assert norm_only(L, flags=2) == INVALID           # no quantisation, so no QUANT_FROM_FP32
    assert norm_only(L, M=-1) == INVALID
    assert norm_only(L, H=0) == INVALID
    assert norm_only(L, eps=float("nan")) == INVALID
    assert norm_only(L, H=20) == UNSUPPORTED          # H % 8 == 0 is the only width rule
    assert norm_only(L, H=131072 + 8) == UNSUPPORTED
    for kw in ("x", "w", "n"):
        assert norm_only(L, **{kw: None}) == INVALID, kw
    assert norm_only(L, r=None) == INVALID            # residual_out without residual_in
    assert norm_only(L, n=C.c_void_p(BASE + 6 * 64 * MB + 8)) == MISALIGNED
    assert norm_only(L, n=_p(0)) == INVALID           # normed_out overlaps x
    assert norm_only(L, ro=_p(6)) == INVALID          # residual_out overlaps normed_out


def test_unfused_swiglu_argument_errors(sgq_lib):
    L = sgq_lib
    assert act_only(L, M=0, gu=None, out=None) == OK
    assert act_only(L, act=2) == INVALID
    assert act_only(L, flags=2) == INVALID            # no quantisation, so no QUANT_FROM_FP32
    assert act_only(L, flags=4) == INVALID            # ACT_ROUND_BF16 needs SiLU-and-mul
    assert act_only(L, limit=-1.0) == INVALID
    assert act_only(L, I=36) == UNSUPPORTED           # I % 8 == 0 is the only width rule
    assert act_only(L, gu=None) == INVALID
    assert act_only(L, out=None) == INVALID
    assert act_only(L, out=C.c_void_p(BASE + 64 * MB + 2)) == MISALIGNED
    assert act_only(L, out=C.c_void_p(BASE + 4096)) == INVALID     # out inside gate_up


def test_quantize_argument_errors(sgq_lib):
    L = sgq_lib
    assert quant(L, M=0, src=None) == OK
    assert quant(L, fmt=3) == INVALID
    assert quant(L, M=-2) == INVALID
    assert quant(L, W=0) == INVALID
    assert quant(L, W=48) == UNSUPPORTED
    assert quant(L, fmt=1, W=192) == UNSUPPORTED
    assert quant(L, fmt=2, W=12) == UNSUPPORTED
    assert quant(L, W=131072 + 32) == UNSUPPORTED
    for kw in ("src", "q", "s"):
        assert quant(L, **{kw: None}) == INVALID, kw
    assert quant(L, src=C.c_void_p(BASE + 8)) == MISALIGNED
    assert quant(L, fmt=2, s=C.c_void_p(BASE + 2 * 64 * MB + 2)) == MISALIGNED
    assert quant(L, q=_p(0)) == INVALID               # q_out overlaps src
    assert quant(L, M=1 << 45, W=16384) == INVALID
    assert quant(L, flags=1) == INVALID               # GEMMA_WEIGHT is not a quant flag
    assert quant(L, flags=2) == INVALID               # nor QUANT_FROM_FP32 (the source is bf16)


SWZ, COL = 1 << 3, 1 << 4


def test_scale_layout_flags(sgq_lib):
    L = sgq_lib
    # each layout flag belongs to one format
    assert quant(L, fmt=1, flags=SWZ) == INVALID
    assert quant(L, fmt=2, flags=SWZ) == INVALID
    assert quant(L, fmt=0, flags=COL) == INVALID
    assert quant(L, fmt=2, flags=COL) == INVALID
    assert quant(L, fmt=0, flags=SWZ | COL) == INVALID
    assert norm(L, fmt=1, flags=1 | SWZ) == INVALID
    assert norm(L, fmt=0, flags=1 | COL) == INVALID
    assert swiglu(L, fmt=2, flags=2 | COL) == INVALID
    assert norm_only(L, flags=1 | SWZ) == INVALID     # no quantisation, so no scale layout
    assert act_only(L, flags=COL) == INVALID
    # the overlap checks use the padded sizes: 8 rows swizzled take 128 * 8 scale bytes at W = 256
    base = BASE + 2 * 64 * MB
    assert quant(L, M=0, flags=SWZ) == OK
    assert quant(L, flags=SWZ, s=C.c_void_p(base), q=C.c_void_p(base + 128 * 8 - 16)) == INVALID
    # column-major 1x128 at M = 5, W = 512: 4 groups x 8 padded rows x 4 bytes
    assert quant(L, fmt=1, flags=COL, M=5, W=512, s=C.c_void_p(base), q=C.c_void_p(base + 4 * 8 * 4 - 16)) == INVALID


def test_binding_rejects_wrong_tensors():
    import torch
    x = torch.zeros(4, 64, dtype=torch.float32)
    w = torch.zeros(64, dtype=torch.bfloat16)
    with pytest.raises(binding.SgqError):
        binding.rmsnorm_add_quant(x, w)
    with pytest.raises(binding.SgqError):
        binding.swiglu_quant(torch.zeros(4, 64, dtype=torch.bfloat16), fmt="nope")
    with pytest.raises(binding.SgqError):
        binding.rmsnorm_add(x, w)
    with pytest.raises(binding.SgqError):
        binding.swiglu(torch.zeros(4, 63, dtype=torch.bfloat16))
    with pytest.raises(binding.SgqError):
        binding.quantize_fp8(torch.zeros(4, 64, dtype=torch.bfloat16), fmt="fp4")


FP16 = 1 << 5


def test_fp16_flag_is_taken_by_the_norms_and_the_quant_only(sgq_lib):
    L = sgq_lib
    assert swiglu(L, flags=2 | FP16) == INVALID       # SwiGLU is bf16 only
    assert act_only(L, flags=FP16) == INVALID
    assert norm(L, M=0, flags=1 | FP16) == OK
    assert norm_only(L, M=0, flags=1 | FP16) == OK
    assert quant(L, M=0, flags=FP16) == OK


def _seg(H=512, ld=None, x=0, w=1, q=2, s=3, n=4):
    f = lambda i: None if i is None else BASE + i * 64 * MB
    return binding.NormSeg(H, H if ld is None else ld, f(x), f(w), f(q), f(s), f(n))


def dual(lib, a=None, b=None, fmt=2, flags=0, M=8, eps=1e-6):
    a = a or _seg()
    b = b or _seg(x=5, w=6, q=None, s=None, n=7)
    return _host_checked(lib.rmsnorm_dual_quant(fmt, flags, M, eps, C.byref(a), C.byref(b), None))


def test_dual_norm_argument_errors(sgq_lib):
    L = sgq_lib
    assert dual(L, M=0) == OK
    assert dual(L, fmt=3) == INVALID
    assert dual(L, flags=4) == INVALID                # ACT_ROUND_BF16 is not a norm flag
    assert dual(L, flags=1 << 3) == INVALID           # no scale layouts
    assert dual(L, M=-1) == INVALID
    assert dual(L, eps=float("nan")) == INVALID
    assert _host_checked(L.rmsnorm_dual_quant(2, 0, 8, 1e-6, None, C.byref(_seg()), None)) == INVALID
    assert dual(L, a=_seg(H=0)) == INVALID
    assert dual(L, a=_seg(ld=256)) == INVALID         # row stride below the width
    assert dual(L, fmt=0, a=_seg(H=520)) == UNSUPPORTED              # quantised: MX group of 32
    # an unquantised segment needs H % 8 only: H = 520 passes the width rule and fails later on the overlap
    assert dual(L, fmt=0, b=_seg(H=520, x=5, w=6, q=None, s=None, n=0)) == INVALID
    assert dual(L, b=_seg(H=20, x=5, w=6, q=None, s=None, n=7)) == UNSUPPORTED
    assert dual(L, a=_seg(H=16384 + 8)) == UNSUPPORTED
    assert dual(L, a=_seg(x=None)) == INVALID
    assert dual(L, a=_seg(w=None)) == INVALID
    assert dual(L, a=_seg(s=None)) == INVALID         # q_out without scale_out
    assert dual(L, a=_seg(q=None)) == INVALID         # scale_out without q_out
    assert dual(L, b=_seg(x=5, w=6, q=None, s=None, n=None)) == INVALID   # nothing to write
    assert dual(L, a=_seg(ld=516)) == MISALIGNED      # rows must start 16-byte aligned
    assert dual(L, a=_seg(n=7)) == INVALID            # two outputs in one place
    assert dual(L, a=_seg(q=5)) == INVALID            # an output over an input
    assert dual(L, M=1 << 45, a=_seg(H=16384)) == INVALID


def allreduce(lib, fmt=0, flags=1, n=2, M=8, H=256, eps=1e-6, parts=None, r=_p(2), ro=_p(3), w=_p(4), q=_p(5),
              s=_p(6), nrm=_p(7)):
    if parts is None:
        parts = [_p(0), _p(1)][:n] + [_p(8 + k) for k in range(max(0, n - 2))]
    arr = (C.c_void_p * max(1, len(parts)))(*parts)
    return _host_checked(lib.allreduce_rmsnorm_add_quant(fmt, flags, n, M, H, eps, arr, r, ro, w, q, s, nrm, None))


def test_allreduce_norm_argument_errors(sgq_lib):
    L = sgq_lib
    L.allreduce_rmsnorm_add_quant.restype = C.c_int
    L.allreduce_rmsnorm_add_quant.argtypes = [C.c_int, C.c_uint32, C.c_int, C.c_int64, C.c_int64, C.c_float,
                                              C.POINTER(C.c_void_p)] + [C.c_void_p] * 7
    assert allreduce(L, M=0) == OK                           # empty: no launch
    assert allreduce(L, n=0, parts=[]) == INVALID
    assert allreduce(L, n=9) == INVALID                      # above SGQ_MAX_RANKS
    assert allreduce(L, flags=1 << 5) == INVALID             # bf16 only
    assert allreduce(L, fmt=3) == INVALID
    assert allreduce(L, parts=[_p(0), None]) == INVALID      # a null partial
    assert allreduce(L, parts=[_p(0), C.c_void_p(BASE + 64 * MB + 2)]) == MISALIGNED
    assert allreduce(L, H=48) == UNSUPPORTED                 # MX group
    assert allreduce(L, H=16384 + 32) == UNSUPPORTED         # whole rows only
    assert allreduce(L, q=_p(1)) == INVALID                  # an output over a partial
    assert allreduce(L, nrm=_p(0)) == INVALID
    assert allreduce(L, r=None) == INVALID                   # residual_out without residual_in
    assert allreduce(L, w=None) == INVALID
    assert allreduce(L, n=8, H=16384, M=1024) == UNSUPPORTED     # eight staged partials of a 16384 row do not fit
