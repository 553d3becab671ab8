"""The parity checker accepts the oracle's own result and rejects planted
mistakes (a code two steps off, a scale off by one, too many one-step code
mismatches, a bf16 output two ulps off). Runs on the CPU."""
import numpy as np
import pytest

import oracle
from oracle.parity import check_norm, check_swiglu
from swiglu_fp8_activation_gb300 import inputs


def _norm(fmt, from_fp32=False):
    case = inputs.norm_case_gemma_mx(16, 1024)
    t = inputs.make_norm(case)
    return oracle.rmsnorm_add_quant(fmt, inputs.bf16_bits(t["x"]), inputs.bf16_bits(t["r"]),
                                    inputs.bf16_bits(t["w"]), eps=case.eps, gemma=True, from_fp32=from_fp32)


@pytest.mark.parametrize("fmt", ["mxfp8", "block128", "per_token"])
@pytest.mark.parametrize("from_fp32", [False, True])
def test_checker_accepts_the_oracle(fmt, from_fp32):
    ref = _norm(fmt, from_fp32)
    st = check_norm(fmt, ref, ref["q"].copy(), ref["scale"].copy(), ref["normed"], ref["residual"],
                    from_fp32=from_fp32)
    assert st["code_mismatch"] == 0


@pytest.mark.parametrize("fmt", ["mxfp8", "block128", "per_token"])
def test_checker_rejects_planted_mistakes(fmt):
    ref = _norm(fmt)
    # a code two steps away
    q = ref["q"].copy()
    j = np.argmax((q & 0x7F) > 8)
    q.flat[j] = q.flat[j] - 2
    with pytest.raises(AssertionError):
        check_norm(fmt, ref, q, ref["scale"], from_fp32=False)
    # a scale off by one code / one fp32 ulp in a non-excused group
    s = ref["scale"].copy()
    k = int(np.argmin(ref["gamb"].reshape(-1)))
    assert ref["gamb"].reshape(-1)[k] == 0
    if fmt == "mxfp8":
        s.reshape(-1)[k] += 1
    else:
        s.reshape(-1)[k] = np.nextafter(s.reshape(-1)[k], np.float32(1e30))
    with pytest.raises(AssertionError):
        check_norm(fmt, ref, ref["q"], s, from_fp32=False)
    # one-step code mismatches on more than 1e-4 of the elements
    q = ref["q"].copy()
    idx = np.flatnonzero(((q & 0x7F) > 8) & ((q & 0x7F) < 0x7E))[:20]
    q.flat[idx] += 1
    with pytest.raises(AssertionError):
        check_norm(fmt, ref, q, ref["scale"], from_fp32=False)
    # bf16 copy two ulps off
    n = ref["normed"].copy()
    n.flat[5] += 2
    with pytest.raises(AssertionError):
        check_norm(fmt, ref, ref["q"], ref["scale"], n, None, from_fp32=False)


def test_checker_accepts_one_ulp_and_one_rare_step():
    ref = _norm("mxfp8")
    n = ref["normed"].copy()
    n.flat[3] += 1
    r = ref["residual"].copy()
    r.flat[7] -= 1
    check_norm("mxfp8", ref, ref["q"], ref["scale"], n, r, from_fp32=False)
    big = oracle.swiglu_quant("mxfp8", "swiglu_oai", inputs.bf16_bits(inputs.swiglu_inputs(64, 768, seed=3, std=2.0)),
                              from_fp32=True)
    q = big["q"].copy()
    j = int(np.flatnonzero(((q & 0x7F) > 8) & ((q & 0x7F) < 0x7E) & (big["gamb"].repeat(32, axis=1).reshape(q.shape) == 0))[0])
    q.flat[j] += 1   # 1 of 49152 elements: below 1e-4
    st = check_swiglu("mxfp8", big, q, big["scale"], from_fp32=True)
    assert st["code_mismatch"] == 1


def test_ties_have_their_own_bound_and_must_be_within_one_step():
    # fp32-source 1x128 norm with plain weights: exact ties are common
    case = inputs.norm_case_block128(64, 4096)
    t = inputs.make_norm(case)
    ref = oracle.rmsnorm_add_quant("block128", inputs.bf16_bits(t["x"]), None, inputs.bf16_bits(t["w"]),
                                   eps=case.eps, gemma=False, from_fp32=True)
    tie = (ref["amb"] & oracle.AMB_TIE) != 0
    assert tie.sum() > 30          # about 4e-4 of the elements
    q0 = ref["q"].copy()
    inner = ((q0 & 0x7F) > 8) & ((q0 & 0x7F) < 0x7E)
    idx = np.flatnonzero(tie & inner)
    q = q0.copy()
    q.flat[idx] += 1               # every tie on the other neighbour: under the 1e-3 tie bound, accepted
    st = check_norm("block128", ref, q, ref["scale"], from_fp32=True)
    assert st["tie_mismatch"] == idx.size and st["code_mismatch"] == idx.size
    budget = int(1e-4 * q0.size)   # 26 of 262144
    plain = np.flatnonzero(~tie & inner)
    q = q0.copy()
    q.flat[plain[:budget]] += 1    # non-tie mismatches within 1e-4: accepted
    check_norm("block128", ref, q, ref["scale"], from_fp32=True)
    q.flat[plain[budget:budget + 2]] += 1       # beyond 1e-4 away from ties: rejected
    with pytest.raises(AssertionError):
        check_norm("block128", ref, q, ref["scale"], from_fp32=True)
    # more than 1e-3 of the elements at (marked) ties: rejected
    many = dict(ref, amb=ref["amb"].copy())
    fake = plain[: int(2e-3 * q0.size)]
    many["amb"].flat[fake] |= oracle.AMB_TIE
    q = q0.copy()
    q.flat[fake] += 1
    with pytest.raises(AssertionError):
        check_norm("block128", many, q, ref["scale"], from_fp32=True)
    q = q0.copy()
    q.flat[idx[0]] += 2            # two steps at a tie: rejected
    with pytest.raises(AssertionError):
        check_norm("block128", ref, q, ref["scale"], from_fp32=True, budget=False)


def test_full_row_blocks_apply_the_budget_to_the_totals():
    import fullrows
    gu = inputs.bf16_bits(inputs.swiglu_inputs(600, 256, seed=4, std=2.0))
    ref = oracle.swiglu_quant("mxfp8", "swiglu_oai", gu, from_fp32=True, diagnostics=False)
    q0 = ref["q"]
    st = fullrows.swiglu_all_rows("mxfp8", "swiglu_oai", gu, q0, ref["scale"], from_fp32=True)
    assert st["code_mismatch"] == 0 and st["n_plain"] <= q0.size
    ok = np.flatnonzero(((q0 & 0x7F) > 8) & ((q0 & 0x7F) < 0x7E))
    allowed = int(1e-4 * st["n_plain"])                 # 15 of 153600
    # one step off in two row blocks: within the budget over all rows, though
    # one block alone holds more than 1e-4 of its own elements
    first = ok[ok < 256 * 256][:allowed - 2]
    last = ok[ok >= 512 * 256][:2]
    q = q0.copy()
    q.flat[np.r_[first, last]] += 1
    st = fullrows.swiglu_all_rows("mxfp8", "swiglu_oai", gu, q, ref["scale"], from_fp32=True)
    assert st["code_mismatch"] == allowed
    q.flat[ok[ok >= 256 * 256][:20]] += 1               # over the budget in total: rejected
    with pytest.raises(AssertionError):
        fullrows.swiglu_all_rows("mxfp8", "swiglu_oai", gu, q, ref["scale"], from_fp32=True)


def test_single_row_ties_and_non_ties():
    # one fp32-source 1x128 row of 8192 elements: the 1e-4 budget is under one
    # element, the tie bound eight
    t = inputs.norm_inputs(1, 8192, seed=0, x_std=1.0, r_std=None, w_mean=1.0, w_std=0.1)
    ref = oracle.rmsnorm_add_quant("block128", inputs.bf16_bits(t["x"]), None, inputs.bf16_bits(t["w"]),
                                   eps=1e-6, gemma=False, from_fp32=True)
    q0 = ref["q"]
    tie = (ref["amb"] & oracle.AMB_TIE) != 0
    inner = ((q0 & 0x7F) > 8) & ((q0 & 0x7F) < 0x7E)
    it, nt = np.flatnonzero(tie & inner), np.flatnonzero(~tie & inner)
    assert it.size >= 2
    q = q0.copy()
    q.flat[it[:2]] += 1            # two ties on the other neighbour: accepted
    st = check_norm("block128", ref, q, ref["scale"], from_fp32=True)
    assert st["tie_mismatch"] == 2
    q = q0.copy()
    q.flat[nt[0]] += 1             # one element away from ties: rejected
    with pytest.raises(AssertionError):
        check_norm("block128", ref, q, ref["scale"], from_fp32=True)
