"""Host logic of bench.py: replica barrier and max-over-ranks (gloo, world
size 2, CPU), the nvidia-smi clock summary, and the reference arm's rank
handling."""

import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    rep = bench.Replicas(backend="gloo")
    rep.barrier()
    m = rep.max(10.0 + rank)          # each rank's elapsed time; all ranks see the slowest
    rep.barrier()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"rank": rep.rank, "world": rep.world, "max": m}, f)
    rep.close()


def test_replicas_barrier_and_max_over_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    assert [r["rank"] for r in res] == [0, 1]
    assert all(r["world"] == 2 and r["max"] == 11.0 for r in res)


def test_single_process_replicas_are_trivial(monkeypatch):
    for v in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(v, raising=False)
    rep = bench.Replicas()
    assert rep.world == 1 and rep.max(3.5) == 3.5
    rep.barrier()


def test_clock_summary():
    text = "\n".join([
        "0, 345, 2070, 200.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1890, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1905, 2070, 1150.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1920, 2070, 1170.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ])
    c = bench.summarise_clocks(text)
    assert c["sm_max_mhz"] == 2070 and c["sm_mhz"] == 1905 and c["reasons"] == ["sw_power_cap"]
    assert bench.summarise_clocks("") is None


def test_reference_arm_non_zero_rank_does_nothing(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert capsys.readouterr().out == ""


def test_row_flops_counts_real_lengths():
    import numpy as np
    cu = [0, 10, 30]
    rows = np.array([0, 9, 10, 29])
    assert bench.row_flops(cu, rows, 2, 4, True) == 4 * 4 * 2 * (1 + 10 + 1 + 20)
    assert bench.row_flops(cu, rows, 2, 4, False) == 4 * 4 * 2 * (10 + 10 + 20 + 20)


def test_useful_mma_area_of_the_workloads(cpattn):
    """The bench line's useful share of the forward kernel's tile area: about
    0.85 on the micro-batch (short zigzag chunks, tiles packed across chunk
    edges), near 1 on one long sequence."""
    import inputs
    w = inputs.workload("dynamic_cp_microbatch")
    plan = cpattn.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    f = bench.useful_mma_fraction(plan, True)
    assert 0.85 < f < 0.86
    assert 0.85 < bench.useful_mma_fraction(plan, True, backward=True) < 0.86
    one = cpattn.cpattn_plan([0, 4096], 2, "zigzag")
    # 4096 tokens, 4 chunks of 1024: only each tile's diagonal 128 x 128 block is
    # partly masked, about half of it over a mean of ~2,100 keys per tile row
    assert 0.96 < bench.useful_mma_fraction(one, True) < 0.98
    full = cpattn.cpattn_plan([0, 4096], 2, "zigzag")
    assert bench.useful_mma_fraction(full, False) == 1.0


def test_sustained_fraction_only_under_the_power_cap(monkeypatch):
    monkeypatch.setattr(bench, "measured_sustained", lambda: 1700.0)
    capped = {}
    bench.add_sustained(capped, 850.0, {"reasons": ["sw_power_cap"], "sm_mhz": 1777.0})
    assert capped == {"frac_of_sustained": 0.5, "peak_sustained": 1700.0}
    free = {}
    bench.add_sustained(free, 850.0, {"reasons": [], "sm_mhz": 2070.0})
    bench.add_sustained(free, 850.0, None)
    assert free == {}
