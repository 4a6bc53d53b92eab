"""The replica path of bench.py under torch.distributed, on CPU with the gloo backend and two
ranks: the slowest rank's step time reaches every rank, the whole-job value counts every
rank's tokens, only rank 0 prints, and the oracle arm runs on rank 0 alone."""
import contextlib
import io
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.0, 3.5][rank]            # rank 1 is the slower replica
    worst = bench.max_over_ranks(ms, world, "cpu")
    dec = bench.whole_job(worst, 1, world, 6, False)
    pre = bench.whole_job(worst, 16384, world, 6, True)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        printed = bench.emit({"value": dec[0], "rank": rank}, rank)
    ref = bench.run_reference(None, rank, world, "cpu") if rank != 0 else "rank 0 runs it"
    dist.barrier()
    dist.destroy_process_group()
    json.dump({"worst": worst, "dec": dec, "pre": pre, "printed": printed,
               "stdout": buf.getvalue(), "ref": ref},
              open(os.path.join(out_dir, f"rank{rank}.json"), "w"))


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(worker, args=(world, free_port(), str(tmp_path)), nprocs=world, join=True)
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(world)]
    for x in r:
        assert x["worst"] == 3.5
        # decode: 3.5 ms over 2 ranks x 1 token x 6 layers
        assert x["dec"][1] == "us/token/layer" and x["dec"][0] == pytest.approx(3500.0 / 12)
        # prefill: both ranks' 16384 tokens over the slowest step
        assert x["pre"][1] == "tokens/s" and x["pre"][0] == pytest.approx(2 * 16384 / 3.5e-3)
    assert r[0]["printed"] and json.loads(r[0]["stdout"])["rank"] == 0
    assert not r[1]["printed"] and r[1]["stdout"] == ""
    assert r[1]["ref"] is None          # the oracle arm: rank 1 exits without work


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(1.25, 1, "cpu") == 1.25
    assert bench.whole_job(2.0, 8, 1, 1, False) == (pytest.approx(250.0), "us/token/layer")
