"""GPU parity of the tensor-parallel all-reduce folded into the fused norm
(allreduce_rmsnorm_add_quant). The ranks' partial rows live on this one GPU
here (on a multi-GPU node they would be peer memory, read the same way).
The result must match the oracle (the partials' exact sum rounded once to
bf16, then the norm), equal bit for bit the plain fused norm of the rows a
rank-order fp32 sum gives, and, in the two-shot form, each rank's slice must
equal the same rows computed alone."""
import numpy as np
import pytest
import torch

import oracle
from oracle.parity import check_norm
from swiglu_fp8_activation_gb300 import allreduce_rmsnorm_add_quant, inputs, rmsnorm_add_quant, scale_shape, tp

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GUARD = 4096


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _parts(n, M, H, seed):
    return [inputs.norm_inputs(M, H, seed=seed + 31 * k, x_std=1.5, r_std=None, w_mean=0.0, w_std=0.1)["x"].to(DEV)
            for k in range(n)]


def _summed(parts):
    """The all-reduce's output as the kernel defines it: fp32 sum in rank order, rounded to bf16."""
    s = parts[0].float()
    for p in parts[1:]:
        s = s + p.float()
    return s.to(torch.bfloat16)


CASES = [  # (fmt, n, M, H, residual, from_fp32, gemma, layout)
    ("mxfp8", 4, 8, 6144, True, False, True, "row"),          # the MiniMax-M3.1 TP4 decode shape
    ("mxfp8", 2, 300, 6144, True, False, True, "swizzled"),
    ("per_token", 8, 1, 7168, False, False, False, "row"),    # the latent-attention entry projection, TP8
    ("per_token", 8, 9, 7168, True, True, False, "row"),
    ("block128", 1, 37, 4096, False, True, False, "col_major"),
    ("block128", 3, 64, 2176, True, False, False, "row"),
    ("mxfp8", 8, 4096, 1536, True, False, True, "row"),       # many rows a CTA
]


@pytest.mark.parametrize("c", CASES, ids=lambda c: "-".join(map(str, c)))
def test_allreduce_norm_matches_oracle_and_the_plain_norm(c):
    fmt, n, M, H, res, from32, gemma, layout = c
    parts = _parts(n, M, H, seed=M * 7 + H + n)
    t = inputs.norm_inputs(M, H, seed=H + n, x_std=1.0, r_std=1.0 if res else None,
                           w_mean=0.0 if gemma else 1.0, w_std=0.1)
    w = t["w"].to(DEV)
    r = t["r"].to(DEV) if res else None
    ro = torch.empty_like(r) if res else None
    kw = dict(fmt=fmt, gemma=gemma, quant_from_fp32=from32, scale_layout=layout, normed=True)
    q, s, nrm, _ = allreduce_rmsnorm_add_quant(parts, w, residual_in=r, residual_out=ro, **kw)
    q2, s2, n2, ro2 = rmsnorm_add_quant(_summed(parts), w, residual_in=r.clone() if res else None, **kw)
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(s, s2) and torch.equal(nrm, n2)
    if res:
        assert torch.equal(ro, ro2)
    s_row = s.cpu().numpy()
    if layout != "row":
        _, s3, _, _ = rmsnorm_add_quant(_summed(parts), w, residual_in=r.clone() if res else None,
                                        **{**kw, "scale_layout": "row"})
        s_row = s3.cpu().numpy()
        np.testing.assert_array_equal(s.cpu().numpy(), oracle.scale_layout(fmt, s_row, layout))
    ref = oracle.allreduce_rmsnorm_add_quant(fmt, [_bits(p) for p in parts], _bits(t["r"]) if res else None,
                                             _bits(t["w"]), eps=1e-6, gemma=gemma, from_fp32=from32)
    check_norm(fmt, ref, q.cpu().numpy(), s_row, _bits(nrm), _bits(ro) if res else None, from_fp32=from32)


def test_outputs_stay_inside_their_buffers_and_graph_replay():
    M, H, n = 5, 6144, 4
    parts = _parts(n, M, H, seed=3)
    t = inputs.norm_inputs(M, H, seed=4, x_std=1.0, r_std=1.0, w_mean=0.0, w_std=0.1)
    r, w = t["r"].to(DEV), t["w"].to(DEV)
    bufs = {k: torch.full((nb + GUARD,), 0xA7, dtype=torch.uint8, device=DEV)
            for k, nb in (("q", M * H), ("s", M * H // 32), ("n", 2 * M * H), ("r", 2 * M * H))}
    q = bufs["q"][: M * H].view(M, H)
    s = bufs["s"][: M * H // 32].view(M, H // 32)
    nrm = bufs["n"][: 2 * M * H].view(torch.bfloat16).view(M, H)
    ro = bufs["r"][: 2 * M * H].view(torch.bfloat16).view(M, H)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        allreduce_rmsnorm_add_quant(parts, w, residual_in=r, residual_out=ro, q_out=q, scale_out=s, normed_out=nrm)
    g.replay()
    torch.cuda.synchronize()
    for k, nb in (("q", M * H), ("s", M * H // 32), ("n", 2 * M * H), ("r", 2 * M * H)):
        assert (bufs[k][nb:] == 0xA7).all(), f"bytes written past {k}"
    q2, s2, n2, ro2 = rmsnorm_add_quant(_summed(parts), w, residual_in=r.clone(), normed=True)
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(s, s2) and torch.equal(nrm, n2) and torch.equal(ro, ro2)


@pytest.mark.parametrize("world", [2, 4])
def test_two_shot_slices(world):
    # every rank computes its own rows from views of all partials; the slices
    # put together match the oracle over all rows, and each slice is the
    # plain fused norm of its summed rows
    M, H = 203, 7168
    parts = _parts(world, M, H, seed=world)
    t = inputs.norm_inputs(M, H, seed=9, x_std=1.0, r_std=1.0, w_mean=1.0, w_std=0.1)
    r, w = t["r"].to(DEV), t["w"].to(DEV)
    outs = []
    for k in range(world):
        a, b = tp.rank_rows(M, world, k)
        rs = r[a:b].clone()
        q, s, _, _ = allreduce_rmsnorm_add_quant([p[a:b] for p in parts], w, fmt="per_token", gemma=False,
                                                 residual_in=rs)
        q2, s2, _, _ = rmsnorm_add_quant(_summed([p[a:b] for p in parts]), w, fmt="per_token", gemma=False,
                                         residual_in=r[a:b].clone())
        torch.cuda.synchronize()
        assert torch.equal(q, q2) and torch.equal(s, s2)
        outs.append((q, s, rs))
    q = torch.cat([o[0] for o in outs]).cpu().numpy()
    s = torch.cat([o[1] for o in outs]).cpu().numpy()
    ro = torch.cat([o[2] for o in outs])
    ref = oracle.allreduce_rmsnorm_add_quant("per_token", [_bits(p) for p in parts], _bits(t["r"]), _bits(t["w"]),
                                             eps=1e-6, gemma=False, from_fp32=False)
    check_norm("per_token", ref, q, s, None, _bits(ro), from_fp32=False)
