"""Seeded synthetic inputs for the fused norm / SwiGLU + FP8 quantisation ops.

This module is shared by the tests, the benchmark and the CPU oracle's callers.
It holds no arithmetic of the method: it only draws random numbers and rounds
them to bfloat16 (through PyTorch's own conversion) to make input tensors.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) gives 64-bit words. Uniforms take the top 53
bits. Normals use the Box-Muller transform on two uniforms (cosine branch).
Every tensor draws from its own stream, keyed by (seed, tag), so a tensor does
not change when another tensor's shape changes.

The workload table below follows the input recipes of the pages:
  * "[ROCm][MiniMax-M3.1] ... MXFP8 quant ..." (vllm PR 65478), section
    "Microbenchmark script": hidden 6144, x ~ 3*randn, r ~ randn, w ~ 0.1*randn,
    eps 1e-6; shared-expert intermediate 768 with gate_up of width 1536;
    alpha 1.702, beta 1.0, limit 7.0; M from 8 to 192.
  * "[Perf] [AMD] qwen3: Fuse the 1x128 FP8 input quant ..." (sglang PR 48043),
    section "Modifications": Qwen3-like widths.
  * "[ROCm] Fuse per-token activation quant into RMSNorm ..." (sglang PR 34502),
    section "Change": MLA-like per-token widths.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TWO_NEG53 = 2.0 ** -53


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function applied to an array of uint64 states."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, tag: int) -> np.uint64:
    """Starting state of the stream keyed by (seed, tag)."""
    key = np.array([(int(seed) & 0xFFFFFFFF) << 16 | (int(tag) & 0xFFFF)], dtype=np.uint64)
    return _mix(key * _GAMMA + _GAMMA)[0]


_CHUNK = 1 << 18          # draws per piece: keeps every temporary in cache


def _pieces(n: int, fill) -> np.ndarray:
    """An array of n draws filled piece by piece by fill(out_slice, start, stop)
    on a few host threads (numpy releases the interpreter lock inside its
    loops). Every draw depends on its index alone, so the result does not
    depend on the piece size or the thread count."""
    out = np.empty(n, dtype=np.float64)
    starts = range(0, n, _CHUNK)
    if n <= 4 * _CHUNK:
        for a in starts:
            fill(out, a, min(a + _CHUNK, n))
        return out
    import concurrent.futures as cf
    import os
    with cf.ThreadPoolExecutor(min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(lambda a: fill(out, a, min(a + _CHUNK, n)), starts))
    return out


def _words_at(base: np.uint64, first: int, count: int) -> np.ndarray:
    """SplitMix64 outputs number first .. first + count - 1 of a stream."""
    idx = np.arange(first, first + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + idx * _GAMMA)


def words(n: int, seed: int, tag: int) -> np.ndarray:
    """n consecutive SplitMix64 outputs of stream (seed, tag)."""
    return _words_at(_stream_base(seed, tag), 1, n)


def uniform(n: int, seed: int, tag: int) -> np.ndarray:
    """n uniforms in [0, 1) from the top 53 bits of each word."""
    base = _stream_base(seed, tag)

    def fill(out, a, b):
        out[a:b] = (_words_at(base, a + 1, b - a) >> np.uint64(11)).astype(np.float64) * _TWO_NEG53
    return _pieces(n, fill)


def normal(n: int, seed: int, tag: int) -> np.ndarray:
    """n standard normals by Box-Muller (cosine branch), two words per draw."""
    base = _stream_base(seed, tag)

    def fill(out, a, b):
        w = _words_at(base, 2 * a + 1, 2 * (b - a))
        u1 = ((w[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * _TWO_NEG53  # (0, 1]
        u2 = (w[1::2] >> np.uint64(11)).astype(np.float64) * _TWO_NEG53  # [0, 1)
        out[a:b] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return _pieces(n, fill)


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """Round an array to a CPU bfloat16 tensor with PyTorch's conversion."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw 16-bit patterns of a CPU bfloat16 tensor, as uint16."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _outliers_and_zero_blocks(a: np.ndarray, seed: int, tag: int, outlier_frac: float,
                              outlier_gain: float, zero_blocks: np.ndarray | None) -> np.ndarray:
    if outlier_frac > 0.0:
        pick = uniform(a.size, seed, tag).reshape(a.shape) < outlier_frac
        a = np.where(pick, a * outlier_gain, a)
    if zero_blocks is not None:
        rows, cols = a.shape
        a = a.reshape(rows, cols // 32, 32).copy()
        a[zero_blocks] = 0.0
        a = a.reshape(rows, cols)
    return a


def _zero_block_mask(rows: int, cols: int, frac: float, seed: int, tag: int) -> np.ndarray | None:
    if frac <= 0.0:
        return None
    return (uniform(rows * (cols // 32), seed, tag) < frac).reshape(rows, cols // 32)


@dataclass(frozen=True)
class Stress:
    """Prefill-stress structure: a fraction of elements scaled by a gain and a
    fraction of 32-aligned blocks set to zero (in every input of the op)."""

    outlier_frac: float = 0.0
    outlier_gain: float = 100.0
    zero_block_frac: float = 0.0


NO_STRESS = Stress()


def norm_inputs(M: int, H: int, *, seed: int, x_std: float, r_std: float | None,
                w_mean: float, w_std: float, stress: Stress = NO_STRESS) -> dict:
    """x [M,H], optional r [M,H] and w [H], all CPU bfloat16.

    x ~ N(0, x_std^2), r ~ N(0, r_std^2) (None: no residual), w ~ w_mean + N(0, w_std^2).
    Under `stress`, the same zero blocks are applied to x and r, so the sum h
    is zero there too.
    """
    zb = _zero_block_mask(M, H, stress.zero_block_frac, seed, 10)
    x = normal(M * H, seed, 1).reshape(M, H) * x_std
    x = _outliers_and_zero_blocks(x, seed, 11, stress.outlier_frac, stress.outlier_gain, zb)
    out = {"x": to_bf16(x)}
    if r_std is not None:
        r = normal(M * H, seed, 2).reshape(M, H) * r_std
        r = _outliers_and_zero_blocks(r, seed, 12, stress.outlier_frac, stress.outlier_gain, zb)
        out["r"] = to_bf16(r)
    else:
        out["r"] = None
    out["w"] = to_bf16(w_mean + normal(H, seed, 3) * w_std)
    return out


def swiglu_inputs(M: int, I: int, *, seed: int, std: float, stress: Stress = NO_STRESS) -> torch.Tensor:
    """gate_up [M, 2I] CPU bfloat16, ~ N(0, std^2); gate = columns [0, I), up = [I, 2I).

    Under `stress`, the same 32-blocks are zeroed in the gate half and the up half.
    """
    zb = _zero_block_mask(M, I, stress.zero_block_frac, seed, 20)
    g = normal(M * I, seed, 4).reshape(M, I) * std
    u = normal(M * I, seed, 5).reshape(M, I) * std
    g = _outliers_and_zero_blocks(g, seed, 21, stress.outlier_frac, stress.outlier_gain, zb)
    u = _outliers_and_zero_blocks(u, seed, 22, stress.outlier_frac, stress.outlier_gain, zb)
    return to_bf16(np.concatenate([g, u], axis=1))


# ---------------------------------------------------------------------------
# Workload table. Formats, flags and activations are named by strings here so
# that this module depends on neither side of the parity check.
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class NormCase:
    name: str
    fmt: str              # "mxfp8" | "block128" | "per_token"
    M: int
    H: int
    seed: int
    x_std: float
    r_std: float | None   # None: no residual input
    w_mean: float
    w_std: float
    gemma: bool           # y = h*inv*(1+w) (True) or h*inv*w (False)
    from_fp32: bool       # quantise the fp32 normed value (True) or its bf16 rounding
    normed_copy: bool     # also write the bf16 normed rows
    eps: float = 1e-6
    stress: Stress = NO_STRESS


@dataclass(frozen=True)
class SwigluCase:
    name: str
    fmt: str
    act: str              # "swiglu_oai" | "silu_mul"
    M: int
    I: int
    seed: int
    std: float
    from_fp32: bool
    round_act_bf16: bool  # SiLU-and-mul: round silu(g) to bf16 before the product
    alpha: float = 1.702
    beta: float = 1.0
    limit: float = 7.0
    stress: Stress = NO_STRESS


PREFILL_STRESS = Stress(outlier_frac=0.001, outlier_gain=100.0, zero_block_frac=0.01)


def norm_case_gemma_mx(M: int, H: int = 6144, seed: int = 0, stress: Stress = NO_STRESS,
                       name: str = "gemma_add_rmsnorm_mxfp8") -> NormCase:
    """Add + Gemma RMSNorm + MXFP8 + bf16 copy (MiniMax-M3.1 post-attention norm)."""
    if stress is NO_STRESS:
        x_std, r_std = 3.0, 1.0
    else:
        x_std, r_std = 1.0, 1.0
    return NormCase(name, "mxfp8", M, H, seed, x_std, r_std, 0.0, 0.1, True, False, True, stress=stress)


def swiglu_case_oai_mx(M: int, I: int = 768, seed: int = 1, std: float = 2.0,
                       stress: Stress = NO_STRESS, name: str = "swiglu_oai_mxfp8") -> SwigluCase:
    """fp32 OAI SwiGLU + MXFP8 directly from fp32 (MiniMax-M3.1 shared expert)."""
    return SwigluCase(name, "mxfp8", "swiglu_oai", M, I, seed, std, True, False, stress=stress)


def norm_case_block128(M: int, H: int = 4096, seed: int = 2) -> NormCase:
    """Qwen3-like RMSNorm + 1x128 FP8, quantised from the fp32 normed value."""
    return NormCase("rmsnorm_block128", "block128", M, H, seed, 1.0, None, 1.0, 0.1, False, True, False)


def swiglu_case_silu_block128(M: int, I: int = 12288, seed: int = 2) -> SwigluCase:
    """Qwen3-like SiLU-and-mul + 1x128 FP8, rounded like the unfused SiLU-and-mul."""
    return SwigluCase("silu_mul_block128", "block128", "silu_mul", M, I, seed, 1.0, False, True)


def norm_case_per_token(M: int, W: int, seed: int = 3) -> NormCase:
    """MLA-like RMSNorm + per-token FP8 ([M,1] scale) of the bf16 normed rows."""
    return NormCase("rmsnorm_per_token", "per_token", M, W, seed, 1.0, None, 1.0, 0.1, False, False, False)


def workloads() -> dict:
    """The five workload families: decode sweeps, Qwen3-like, MLA-like, prefill stress."""
    return {
        "cfg1_norm_mx": [norm_case_gemma_mx(8)],
        "cfg1_norm_mx_sweep": [norm_case_gemma_mx(m) for m in (8, 16, 32, 64, 128, 192)],
        "cfg2_swiglu_mx": [swiglu_case_oai_mx(m) for m in (8, 16, 32, 64, 128, 192)],
        "cfg3_block128": [norm_case_block128(m) for m in (1, 32, 256)]
        + [swiglu_case_silu_block128(m) for m in (1, 32, 256)],
        "cfg4_per_token": [norm_case_per_token(m, w) for w in (7168, 1536, 512) for m in (1, 4096)],
        "cfg5_prefill": [
            norm_case_gemma_mx(8192, 6144, seed=4, stress=PREFILL_STRESS, name="prefill_gemma_add_rmsnorm_mxfp8"),
            swiglu_case_oai_mx(8192, 3072, seed=4, std=1.0, stress=PREFILL_STRESS, name="prefill_swiglu_oai_mxfp8"),
        ],
    }


def make_norm(case: NormCase) -> dict:
    """CPU bf16 tensors x, r (or None), w for a NormCase."""
    return norm_inputs(case.M, case.H, seed=case.seed, x_std=case.x_std, r_std=case.r_std,
                       w_mean=case.w_mean, w_std=case.w_std, stress=case.stress)


def make_swiglu(case: SwigluCase) -> torch.Tensor:
    """CPU bf16 gate_up [M, 2I] for a SwigluCase."""
    return swiglu_inputs(case.M, case.I, seed=case.seed, std=case.std, stress=case.stress)
