"""Host side of the tensor-parallel all-reduce folded into the norm, on the
CPU: the two-shot row partition, and the two-shot form run by two and by
three gloo ranks with the oracle as each rank's compute step. Every rank
holds only its own partial and receives the others' through the process
group (in place of mapped peer memory); the gathered outputs of every rank
must equal the oracle's one-shot result over all rows, bit for bit (the
oracle is row-independent, so the partition must not change any byte)."""
import os
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
from swiglu_fp8_activation_gb300 import tp  # noqa: E402


def test_rank_rows_partition():
    for world in range(1, 9):
        for M in range(0, 60):
            rows = [tp.rank_rows(M, world, k) for k in range(world)]
            assert rows[0][0] == 0 and rows[-1][1] == M
            assert all(rows[k][1] == rows[k + 1][0] for k in range(world - 1))
            sizes = [b - a for a, b in rows]
            assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)
    with pytest.raises(ValueError):
        tp.rank_rows(4, 2, 2)
    assert tp.one_shot(9, 7168) and not tp.one_shot(10, 7168)     # 128 KiB of bf16 at hidden 7168: nine rows


M, H, FMT = 37, 256, "mxfp8"


def _inputs(world):
    from swiglu_fp8_activation_gb300 import inputs
    parts = [inputs.norm_inputs(M, H, seed=100 + k, x_std=1.5, r_std=None, w_mean=0.0, w_std=0.1)["x"]
             for k in range(world)]
    t = inputs.norm_inputs(M, H, seed=7, x_std=1.0, r_std=1.0, w_mean=0.0, w_std=0.1)
    return parts, t["r"], t["w"]


def _oracle_compute(w):
    """The oracle standing in for the fused kernel on one rank's rows."""
    import oracle
    from swiglu_fp8_activation_gb300 import inputs

    def compute(part_slices, r_slice):
        ref = oracle.allreduce_rmsnorm_add_quant(FMT, [inputs.bf16_bits(p) for p in part_slices],
                                                 inputs.bf16_bits(r_slice), inputs.bf16_bits(w), eps=1e-6,
                                                 gemma=True, from_fp32=False, diagnostics=False)
        as16 = lambda b: torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16)
        return (torch.from_numpy(ref["q"]), torch.from_numpy(ref["scale"]), as16(ref["normed"]),
                as16(ref["residual"]))
    return compute


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        parts, r, w = _inputs(world)
        mine = parts[rank].view(torch.uint8)
        got = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(got, mine)                     # the other ranks' partials, as mapped peer memory
        partials = [g.view(torch.bfloat16) for g in got]
        outs = tp.two_shot(_oracle_compute(w), partials, r, rank=rank, world=world)
        q.put((rank, [o.view(torch.uint8).numpy().tobytes() for o in outs]))
    except Exception as e:                             # report at once instead of leaving the queue empty
        q.put((rank, f"rank {rank} failed: {e!r}"))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_two_shot_on_gloo_ranks_equals_one_shot(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29600 + world * 17 + os.getpid() % 500
    procs = [ctx.Process(target=_rank, args=(k, world, port, q)) for k in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in procs)
    errors = [v for v in res.values() if isinstance(v, str)]
    assert not errors, errors
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    parts, r, w = _inputs(world)
    want = _oracle_compute(w)(parts, r)
    want = [o.view(torch.uint8).numpy().tobytes() for o in want]
    for k in range(world):
        assert res[k] == want, f"rank {k}'s gathered outputs differ from the one-shot result"
