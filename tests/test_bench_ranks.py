"""The bench's multi-rank logic on CPU: two gloo ranks, max-over-ranks time, whole-job rate.

Rows are independent, so N GPUs run N replicas with no collective on the data path; the only
exchange is the max of the ranks' times.  These tests run it over gloo, with no GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as tdist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(times[rank], tdist, "cpu")
        out.put((rank, t, bench.job_rate(world, 4, 10, t)))
        tdist.barrier()
    finally:
        tdist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [0.75, 1.25]
    mp.start_processes(_rank_main, args=(2, _free_port(), times, q), nprocs=2, join=True, start_method="spawn")
    got = sorted(q.get(timeout=30) for _ in range(2))
    for rank, t, rate in got:
        assert t == 1.25  # every rank sees the slowest rank's time
        assert rate == pytest.approx(2 * 4 * 10 / 1.25)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(0.5, None, "cpu") == 0.5
    assert bench.job_rate(1, 1, 100, 2.0) == 50.0


def test_reference_arm_rank1_exits_quietly():
    # under torchrun only rank 0 runs the oracle arm; the others exit 0 without work or output
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_work_model_counts_groups_and_slots():
    import numpy as np
    import synth
    cfg = synth.CONFIGS["c2_decode_b4_hash"]
    idx = np.array([[0, 1, 2, 3, 4, 5], [0, 1, 2, 3, 4, 6], [-1, 7, 7, 7, 7, 7], [8] * 6], np.int32)[:, :cfg.top_k]
    wm = bench.work_model(cfg, idx)
    valid = idx[(idx >= 0) & (idx < cfg.experts)]
    assert wm["groups"] == len(set(valid.tolist())) + 1
    assert wm["slots"] == valid.size + cfg.rows
    one = 3 * cfg.inter * cfg.hidden * 2
    assert wm["w_gateup"] + wm["w_down"] == wm["groups"] * one
    # the binding roofline of the decode kernel is HBM; a big prefill GEMM's may be the tensor pipe
    rl = bench.roofline_entry("decode", 0.1, wm, cfg, bench.FALLBACK_PEAKS, "fallback")
    assert rl["bound"] == "hbm" and rl["unit"] == "GB/s" and rl["alg"] > wm["w_gateup"] + wm["w_down"]
