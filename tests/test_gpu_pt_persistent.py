"""GPU parity of the persistent per-token norm: narrow rows at large M with
no residual (several rows a CTA, at least two waves of row blocks) run as
one wave of CTAs that loop over the row blocks, prefetching the next block's
rows. Its outputs must equal, bit for bit, the unfused chain (the norm to
16 bits, then the standalone quant, which keep the row-block kernel's plan),
and the same launch planned for a two-multiprocessor device (so that every
CTA loops over hundreds of row blocks); and match the oracle on every row.
The plan mirror below is the C library's (plan_rows)."""
import numpy as np
import pytest
import torch

import oracle
from oracle.parity import check_norm
from swiglu_fp8_activation_gb300 import inputs, quantize_fp8, rmsnorm_add, rmsnorm_add_quant, set_sm_budget

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _sms():
    return torch.cuda.get_device_properties(DEV).multi_processor_count


def _plan(M, W, sms):
    """(chunks a thread, threads a row, rows a CTA) as the library plans a row-block launch."""
    nch = W // 8
    small = M * nch <= sms * 1024
    order = [1, 2, 3, 4] if small else [4, 3, 2, 1]
    for nv in order:
        if nch % (32 * nv) == 0 and nch // nv <= 512:
            tpr = nch // nv
            break
    else:
        raise AssertionError("no exact fit")
    rpc = max(256 // tpr, 1)
    per_sm = -(-M // sms)
    if per_sm < rpc:
        rpc = max(per_sm, 1)
    return nv, tpr, rpc


def _persistent(M, W, sms):
    nv, tpr, rpc = _plan(M, W, sms)
    return M % rpc == 0 and rpc >= 2 and M // rpc >= 2 * sms


# (W, M, fp16, from_fp32, gemma, normed)
CASES = [
    (512, 4096, False, False, False, False),     # the latent-attention widths of the per-token workload
    (1536, 4096, False, False, False, True),
    (2048, 2048, True, False, True, True),
    (1024, 4096, False, True, False, False),
    (512, 8192, True, True, True, True),
]


@pytest.mark.parametrize("c", CASES, ids=lambda c: "W{}-M{}-f16{}-f32{}-gemma{}-normed{}".format(*c))
def test_persistent_per_token_norm(c):
    W, M, f16, f32, gemma, normed = c
    assert _persistent(M, W, _sms()), "shape expected to take the persistent kernel"
    dt = torch.float16 if f16 else torch.bfloat16
    t = inputs.norm_inputs(M, W, seed=W + M, x_std=1.0, r_std=None, w_mean=0.0 if gemma else 1.0, w_std=0.1)
    x, w = t["x"].to(dt), t["w"].to(dt)
    xd, wd = x.to(DEV), w.to(DEV)
    kw = dict(fmt="per_token", gemma=gemma, quant_from_fp32=f32, normed=normed)
    q, s, n, _ = rmsnorm_add_quant(xd, wd, **kw)
    try:
        set_sm_budget(2)                         # the same plan, 2 x (CTAs an SM) CTAs looping over the blocks
        assert _plan(M, W, 2) == _plan(M, W, _sms())
        q2, s2, n2, _ = rmsnorm_add_quant(xd, wd, **kw)
        torch.cuda.synchronize()
    finally:
        set_sm_budget(0)
    assert torch.equal(q, q2) and torch.equal(s, s2)
    if normed:
        assert torch.equal(n, n2)
    if not f32:                                  # the unfused chain, row-block kernels with the same plan
        nb, _ = rmsnorm_add(xd, wd, gemma=gemma)
        q3, s3 = quantize_fp8(nb, fmt="per_token")
        torch.cuda.synchronize()
        assert torch.equal(q, q3) and torch.equal(s, s3)
        if normed:
            assert torch.equal(n, nb)
    ref = oracle.rmsnorm_add_quant("per_token", _bits(x), None, _bits(w), eps=1e-6, gemma=gemma, from_fp32=f32,
                                   normed=normed, fp16=f16)
    check_norm("per_token", ref, q.cpu().numpy(), s.cpu().numpy(), _bits(n) if normed else None, None,
               from_fp32=f32)


def test_first_persistent_launch_inside_graph_capture():
    # fp16 rows of 768 (3 chunks a thread, 32 threads a row): a kernel and
    # shape no other test launches, so its first launch (which asks the
    # occupancy calculator) happens while the stream is being captured
    M, W = 4096, 768
    assert _persistent(M, W, _sms())
    t = inputs.norm_inputs(M, W, seed=768, x_std=1.0, r_std=None, w_mean=1.0, w_std=0.1)
    x, w = t["x"].to(torch.float16).to(DEV), t["w"].to(torch.float16).to(DEV)
    q = torch.empty(M, W, dtype=torch.uint8, device=DEV)
    s = torch.empty(M, 1, dtype=torch.float32, device=DEV)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        rmsnorm_add_quant(x, w, fmt="per_token", gemma=False, q_out=q, scale_out=s)
    g.replay()
    q2, s2, _, _ = rmsnorm_add_quant(x, w, fmt="per_token", gemma=False)
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(s, s2)
    ref = oracle.quantize("per_token", _bits(rmsnorm_add(x, w, gemma=False)[0]), fp16=True)
    np.testing.assert_array_equal(q.cpu().numpy(), ref["q"])


_rng = np.random.default_rng(99)
# seeded narrow per-token shapes at large M: width a multiple of 8 up to 2048, 2400-12000 rows,
# fp16 or bf16, either quant source, either weight form
RANDOM = [(int(8 * _rng.integers(1, 257)), int(_rng.integers(2400, 12000)), bool(_rng.random() < 0.3),
           bool(_rng.random() < 0.5), bool(_rng.random() < 0.5)) for _ in range(24)]


@pytest.mark.parametrize("c", RANDOM, ids=lambda c: "W{}-M{}-f16{}-f32{}-gemma{}".format(*c))
def test_random_large_m_per_token_shapes(c):
    W, M, f16, f32, gemma = c
    dt = torch.float16 if f16 else torch.bfloat16
    t = inputs.norm_inputs(M, W, seed=W + M, x_std=1.0, r_std=None, w_mean=0.0 if gemma else 1.0, w_std=0.1)
    x, w = t["x"].to(dt), t["w"].to(dt)
    q, s, n, _ = rmsnorm_add_quant(x.to(DEV), w.to(DEV), fmt="per_token", gemma=gemma, quant_from_fp32=f32,
                                   normed=True)
    nb, _ = rmsnorm_add(x.to(DEV), w.to(DEV), gemma=gemma)
    torch.cuda.synchronize()
    assert torch.equal(n, nb)
    if not f32:
        q2, s2 = quantize_fp8(nb, fmt="per_token")
        torch.cuda.synchronize()
        assert torch.equal(q, q2) and torch.equal(s, s2)
    rows = np.unique(np.r_[0, np.random.default_rng(W + M).integers(0, M, 64), M - 1])
    ref = oracle.rmsnorm_add_quant("per_token", _bits(x)[rows], None, _bits(w), eps=1e-6, gemma=gemma, from_fp32=f32,
                                   normed=True, fp16=f16)
    check_norm("per_token", ref, q.cpu().numpy()[rows], s.cpu().numpy()[rows], _bits(n)[rows], None, from_fp32=f32,
               budget=False)
