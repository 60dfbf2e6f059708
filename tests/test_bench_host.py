"""bench.py's host-side logic without a GPU: argument handling, the FLOP count,
clock summaries, the oracle sampling step, and the multi-rank coordination
(barrier, max/sum over ranks, rank-0-only reference arm) on two gloo ranks."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench
from exact_io_aware_attention_gb300 import inputs as gen


def test_parse_args_defaults_and_limits():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.impl == "cuda" and a.warmup >= 3 and a.steps >= 1
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])
    with pytest.raises(SystemExit):
        bench.parse_args(["--steps", "0"])


def test_flop_count_follows_the_method():
    w = gen.WORKLOADS["gpt2_medium_causal"]
    fwd, bwd = bench.attention_flops(w)
    assert fwd == 4 * 4096 ** 2 * 128 * 4 * 16 / 2
    assert bwd == 2.5 * fwd
    wd = gen.WORKLOADS["gpt2_medium_dense"]
    assert bench.attention_flops(wd)[0] == 2 * fwd
    assert bench.attention_flops(wd, 0.25)[0] == 0.5 * fwd


def test_clock_summary():
    rows = [["0", "2070", "2070", "900.5", "0x0", "Not Active", "Not Active", "Not Active",
             "Not Active"],
            ["0", "1980", "2070", "1200.0", "0x4", "Not Active", "Not Active", "Not Active",
             "Active"],
            ["0", "345", "2070", "120.0", "0x1", "Not Active", "Not Active", "Not Active",
             "Not Active"]]
    s = bench.summarize_clocks(rows, timed_ms=18.3, period_ms=50)
    assert s["sm_max_mhz"] == 2070 and s["samples"] == 3 and s["samples_under_load"] == 2
    assert s["sm_mhz"] == (2070 + 1980) / 2 and s["sm_mhz_basis"] == "samples under load"
    assert s["reasons"] == ["sw_power_cap"]
    assert s["timed_region_ms"] == 18.3 and s["sample_period_ms"] == 50
    empty = bench.summarize_clocks([])
    assert empty["samples"] == 0 and empty["samples_under_load"] == 0


def test_clock_summary_without_load_samples():
    """No sample above the load threshold: nothing is counted as under load."""
    idle = [["0", "2070", "2070", "165.3", "0x0", "Not Active", "Not Active", "Not Active",
             "Not Active"],
            ["0", "1965", "2070", "150.0", "0x0", "Not Active", "Not Active", "Not Active",
             "Not Active"],
            ["0", "2055", "2070", "[N/A]", "0x0", "Not Active", "Not Active", "Not Active",
             "Not Active"]]
    s = bench.summarize_clocks(idle, timed_ms=18.0, period_ms=50)
    assert s["samples"] == 3 and s["samples_under_load"] == 0
    assert s["sm_mhz"] == 2055 and s["sm_mhz_basis"].startswith("all samples")
    assert s["power_w_max"] == 165.3


def test_oracle_sample_step_credits_visible_keys():
    w = gen.Workload(99, "tiny", 1, 2, 256, 64, True)
    inp = gen.make_inputs(1, 2, 256, 64, case=99)
    dt, fl = bench.oracle_sample_step(inp, w, head=1, rows_per_step=16)
    assert dt > 0
    rows = [i * 16 + (37 % 16) for i in range(16)]
    assert fl == 3.5 * 4.0 * 64 * sum(r + 1 for r in rows)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    d = bench.Dist()
    d.barrier()
    mx = d.reduce(10.0 + rank, "max")
    sm = d.reduce(1.0 + rank, "sum")
    ref = bench.run_reference(bench.parse_args(["--impl", "reference"]), d) if rank == 1 else "skip"
    d.close()
    q.put((rank, mx, sm, ref))


def test_two_gloo_ranks_coordinate_timing():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [11.0, 11.0]      # max over ranks, seen by both
    assert [o[2] for o in out] == [3.0, 3.0]        # sum over ranks
    assert out[1][3] is None                         # the reference arm runs on rank 0 only
