"""bench.py host logic without a GPU: the whole-job aggregation over ranks
(world size 2 on gloo), the clock-sample parser, and the reference arm."""

import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t, b = bench.aggregate(0.5 + rank, 1000.0 * (rank + 1), world)
    q.put((rank, t, b))
    dist.destroy_process_group()


def test_aggregate_max_time_sum_bytes_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, b in got:
        assert t == 1.5, "time must be the max over ranks"
        assert b == 3000.0, "bytes must be summed over ranks"


def test_aggregate_single_rank_is_identity():
    assert bench.aggregate(0.25, 123.0, 1) == (0.25, 123.0)


def test_clock_summary_parses_samples():
    c = bench.ClockSampler(0)
    c.lines = [
        "0, 300, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1995, 2070, 950.5, 0x4, Not Active, Not Active, Not Active, Active",
    ]
    s = c.summary()
    assert s["sm_max_mhz"] == 2070.0
    assert s["sm_mhz"] == pytest.approx(1987.5)
    assert s["reasons"] == ["sw_power_cap"]


def test_reference_arm_json_line(capsys):
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_oracle_sample_shards_cover_every_unit_once():
    s = bench.OracleSample(bn_f32_channels=3, bn_bf16_channels=2, rms_rows=10, ln_rows=7)
    for n in (1, 4, 16):
        lists = s.shards(n)
        assert len(lists) == n
        # every op's units are split into contiguous ranges; ops with fewer
        # units than shards leave some shards without a call for that op
        expect = sum(min(units, n) for _, units, _, _ in s.items)
        assert sum(len(fns) for fns in lists) == expect
    par = bench.cpu_parallel(s, 0.05)
    assert par["value"] > 0 and par["cores"] == (os.cpu_count() or 1)
    assert bench.cpu_model()


def test_johnson_order_minimises_two_stage_makespan():
    """The end-to-end pipeline order: for random upload / download sizes the
    order must reach the smallest two-stage flow-shop makespan found by
    trying every permutation."""
    import itertools
    import random
    import types
    import torch

    def makespan(seq):
        t_up = t_down = 0
        for up, down in seq:
            t_up += up
            t_down = max(t_down, t_up) + down
        return t_down

    rng = random.Random(7)
    for _ in range(20):
        jobs = [(rng.randint(1, 40), rng.randint(1, 40)) for _ in range(6)]
        ops = [types.SimpleNamespace(name=str(i), h2d=[(torch.empty(u, dtype=torch.uint8), None)],
                                     d2h=[(None, torch.empty(d, dtype=torch.uint8))])
               for i, (u, d) in enumerate(jobs)]
        got = [jobs[int(op.name)] for op in bench.johnson_order(ops)]
        assert sorted(got) == sorted(jobs)
        assert makespan(got) == min(makespan(p) for p in itertools.permutations(jobs))
