"""bench.py's multi-rank host logic on the CPU (gloo, world size 2).

The layer does not shard across GPUs (no expert parallelism), so N GPUs run N
independent replicas; the only cross-rank steps are a barrier around every
timed region and the slowest rank's time, which sets the job's throughput.
Those run here over gloo between two spawned processes, on 127.0.0.1.  The
reference arm does its work on rank 0 only; the other ranks exit at once."""
import argparse
import os
import socket
import tempfile

import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_worker(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ranks = bench._Ranks(world, "cpu")
        ranks.barrier()
        got = ranks.max(10.0 + 0.5 * rank)  # the last rank is the slowest
        ranks.barrier()
        with open(os.path.join(out_dir, f"rank{rank}"), "w") as f:
            f.write(repr(got))
    finally:
        dist.destroy_process_group()


def test_every_rank_gets_the_slowest_ranks_time_over_gloo():
    world = 2
    with tempfile.TemporaryDirectory() as out:
        mp.start_processes(_rank_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        got = [float(open(os.path.join(out, f"rank{r}")).read()) for r in range(world)]
    assert got == [10.5, 10.5]


def test_single_rank_needs_no_process_group():
    ranks = bench._Ranks(1, "cpu")
    ranks.barrier()
    assert ranks.max(3.25) == 3.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(workload="tiny", tokens=0, experts=0, zipf=False, zero_experts=0,
                              ref_tokens=1, warmup=0, steps=1, gpus=2)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_contract_line_on_rank_zero(monkeypatch, capsys):
    import json
    monkeypatch.setenv("RANK", "0")
    args = argparse.Namespace(workload="tiny", tokens=0, experts=0, zipf=False, zero_experts=0,
                              ref_tokens=2, warmup=0, steps=1, gpus=1)
    assert bench.run_reference(args) == 0
    lines = capsys.readouterr().out.strip().splitlines()
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["config"]["tokens_per_step"] == 2
