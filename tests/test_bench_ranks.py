"""Host logic of bench.py's multi-process path, on CPU. With N > 1 every
rank is an independent replica: the job's time is the slowest rank's (max
over ranks, checked here with two gloo processes), rank 0 alone prints, and
the reference arm runs on rank 0 only while the other ranks exit without
work. Rank 0's reference line is checked for the contract's keys on the
smallest layer."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

import bench
from workloads import get_config


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, values, outdir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(values[rank], dist, torch.device("cpu"))
        with open(os.path.join(outdir, f"rank{rank}.json"), "w") as fh:
            json.dump(got, fh)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    values = [1.25, 3.5]
    mp.spawn(_rank_main, args=(2, _free_port(), values, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert json.loads((tmp_path / f"rank{r}.json").read_text()) == 3.5


def _error_rank_main(rank, world, port, bad, outdir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.error_on_any_rank(bad[rank], dist, torch.device("cpu"))
        with open(os.path.join(outdir, f"err{rank}.json"), "w") as fh:
            json.dump(got, fh)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("bad", [(False, True), (False, False)])
def test_device_error_seen_by_every_rank(tmp_path, bad):
    # one rank's error makes every rank raise, so none waits in a later
    # collective for a rank that has left
    mp.spawn(_error_rank_main, args=(2, _free_port(), list(bad), str(tmp_path)), nprocs=2,
             join=True)
    for r in range(2):
        assert json.loads((tmp_path / f"err{r}.json").read_text()) is any(bad)


def test_device_error_one_process():
    assert bench.error_on_any_rank(True, None, None) is True
    assert bench.error_on_any_rank(False, None, None) is False


def test_max_over_ranks_one_process():
    assert bench.max_over_ranks(2.75, None, None) == 2.75


def _args(monkeypatch, *argv):
    monkeypatch.setattr(sys, "argv", ["bench.py", *argv])
    return bench.parse()


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = _args(monkeypatch, "--impl", "reference", "--gpus", "2", "--steps", "1")
    assert bench.run_reference(args, get_config("tiny_T256_d128_E8_k2_f256_fp32")) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank_zero(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "0")
    args = _args(monkeypatch, "--impl", "reference", "--steps", "1", "--warmup", "0")
    assert bench.run_reference(args, get_config("tiny_T256_d128_E8_k2_f256_fp32")) == 0
    lines = capsys.readouterr().out.strip().splitlines()
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "tiny_T256_d128_E8_k2_f256_fp32"
