"""Host-side logic of bench.py, on the CPU: algorithmic byte counts, the
clock-sample parser, the max-over-ranks reduction across two gloo ranks, and
the reference arm's JSON line (the CPU oracle on a bounded sample)."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes():
    # norm at M=8192, H=6144: x, r read; residual, bf16 copy, E4M3, E8M0 written; w once
    assert bench.norm_bytes(8192, 6144) == 8192 * (2 * 6144 * 4 + 6144 + 6144 // 32) + 2 * 6144 == 454_569_984
    # SwiGLU at M=8192, I=3072: gate_up read, E4M3 + E8M0 written
    assert bench.swiglu_bytes(8192, 3072) == 126_615_552
    assert bench.step_bytes() == 454_569_984 + 126_615_552
    # 1x128 and per-token scale bytes
    assert bench.norm_bytes(1, 4096, False, False, "block128") == 2 * 4096 + 4096 + 4 * 32 + 2 * 4096
    assert bench.swiglu_bytes(2, 512, "per_token") == 2 * (4 * 512 + 512 + 4)


def test_clock_summary_parses_samples():
    c = bench.ClockSampler(None)
    c.lines = ["1965, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
               "2070, 2070, 1200.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
               "2025, 2070, 1100.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
               "garbage line"]
    s = c.summary()
    assert s == {"sm_mhz": 2025.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    m = bench.max_over_ranks(float(10 + rank * 5), world)
    bench.barrier(world)
    q.put((rank, m, bench.dist_env()))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [m for _, m, _ in out] == [15.0, 15.0]
    assert [e for _, _, e in out] == [(2, 0, 0), (2, 1, 0)]


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["metric"] == bench.METRIC


def test_warmup_below_three_is_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])
