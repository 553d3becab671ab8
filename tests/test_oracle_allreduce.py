"""Pins of the oracle's all-reduce step (the sum over tensor-parallel ranks
in front of the fused norm): exact sums of small integer grids against
PyTorch's rounding of the same (exactly representable) fp32 sums, ties to
even at a bf16 midpoint, one rank as the identity, invariance under a
permutation of the ranks (the fp64 sum of these values is exact), and the
fused result equal to the plain norm of the summed rows."""
import numpy as np
import torch

import oracle
from swiglu_fp8_activation_gb300 import inputs


def _bf16(a):
    return inputs.bf16_bits(torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


def test_sum_of_integer_grids_matches_a_rounding_of_the_exact_sum():
    rng = np.random.default_rng(0)
    for n in (1, 2, 3, 4, 8):
        parts_f = [rng.integers(-2000, 2000, size=(7, 96)).astype(np.float64) * 2.0 ** -6 for _ in range(n)]
        parts = [_bf16(p) for p in parts_f]
        vals = [torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
                for b in parts]
        exact = np.sum(vals, axis=0)                     # integers / 64 below 2^24 / 64: exact in fp32 too
        want = _bf16(exact.astype(np.float32))
        got, _ = oracle.allreduce_sum(parts)
        np.testing.assert_array_equal(got, want)


def test_ties_round_to_even_and_one_rank_is_the_identity():
    one, tiny = _bf16([1.0])[0], _bf16([2.0 ** -8])[0]
    got, near = oracle.allreduce_sum([np.array([one]), np.array([tiny])])
    assert got[0] == one and near[0] == 1                # 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7
    three = _bf16([3 * 2.0 ** -8])[0]
    got, _ = oracle.allreduce_sum([np.array([one]), np.array([three])])
    assert got[0] == _bf16([1.0 + 2.0 ** -6])[0]         # 1 + 3 * 2^-8: the midpoint above 1 + 2^-7 -> 1 + 2^-6
    x = inputs.bf16_bits(inputs.norm_inputs(3, 256, seed=1, x_std=3.0, r_std=None, w_mean=0, w_std=0.1)["x"])
    got, _ = oracle.allreduce_sum([x])
    np.testing.assert_array_equal(got, x)


def test_rank_order_does_not_change_the_sum():
    rng = np.random.default_rng(3)
    parts = [_bf16(rng.standard_normal((4, 128)) * 2.0) for _ in range(4)]
    a, _ = oracle.allreduce_sum(parts)
    b, _ = oracle.allreduce_sum(parts[::-1])
    c, _ = oracle.allreduce_sum([parts[2], parts[0], parts[3], parts[1]])
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, c)


def test_fused_result_is_the_norm_of_the_summed_rows():
    rng = np.random.default_rng(4)
    M, H = 5, 512
    parts = [_bf16(rng.standard_normal((M, H))) for _ in range(4)]
    t = inputs.norm_inputs(M, H, seed=4, x_std=1.0, r_std=1.0, w_mean=0.0, w_std=0.1)
    r, w = inputs.bf16_bits(t["r"]), inputs.bf16_bits(t["w"])
    fused = oracle.allreduce_rmsnorm_add_quant("mxfp8", parts, r, w, eps=1e-6, gemma=True, from_fp32=False)
    x, _ = oracle.allreduce_sum(parts)
    plain = oracle.rmsnorm_add_quant("mxfp8", x, r, w, eps=1e-6, gemma=True, from_fp32=False)
    for k in ("q", "scale", "residual", "normed"):
        np.testing.assert_array_equal(fused[k], plain[k])
    np.testing.assert_array_equal(fused["x"], x)
