"""The bench's multi-rank path on CPU: two gloo ranks run the same reduction
the GPU ranks run (max over ranks of every time, whole-job throughput = the
units all ranks processed over that time), and the reference arm does no
work on ranks other than 0."""
from __future__ import annotations

import os
import socket
import sys
import json
import types

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from quantized_attention_smooth_gb300 import workloads as wl  # noqa: E402

STEPS = 10


def _rank_result(rank: int) -> dict:
    # rank 1 is the slow one for the step time, rank 0 for the e2e time
    return dict(total_ms=100.0 + 50.0 * rank, pro_ms=2.0 + rank, att_ms=7.0 - rank,
                e2e_ms=40.0 - 10.0 * rank, ops=4.0e11, ops_padded=4.0e11,
                ops_effective=2.0e11, ops_padded_effective=2.0e11, launches=20 + rank)


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r = bench.reduce_over_ranks(_rank_result(rank), world, "cpu")
        q.put((rank, r, bench.job_figures(r, world, STEPS)))
    finally:
        dist.destroy_process_group()


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_reduce_to_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(world):
            rank, r, fig = q.get(timeout=120)
            got[rank] = (r, fig)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    assert sorted(got) == [0, 1]
    for rank, (r, fig) in got.items():
        assert r["total_ms"] == 150.0 and r["e2e_ms"] == 40.0
        assert r["pro_ms"] == 3.0 and r["att_ms"] == 7.0
        assert r["launches"] == 20 + rank            # counts stay per rank
        # 2 ranks x 4e11 ops per step, 15 ms per step (the slow rank's)
        assert fig["value"] == pytest.approx(2 * 4.0e11 / 15e-3 / 1e12)
        assert fig["value_causal_effective"] == pytest.approx(fig["value"] / 2)
        assert fig["e2e"] == pytest.approx(2 * 4.0e11 / 40e-3 / 1e12)
    assert got[0][1] == got[1][1]                    # every rank agrees


def test_single_rank_needs_no_process_group():
    r = _rank_result(0)
    assert bench.reduce_over_ranks(r, 1) is r
    fig = bench.job_figures(r, 1, STEPS)
    assert fig["value"] == pytest.approx(4.0e11 / 10e-3 / 1e12)


def test_reference_arm_is_rank_zero_only(capsys):
    args = types.SimpleNamespace(oracle_pairs=4096, warmup=3, steps=1, gpus=2, variant="fp8")
    bench.reference_arm(args, wl.WORKLOADS["small_d64"], rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_oracle_sample_is_bounded_and_covers_small_workloads():
    """Both arms time the oracle on the same bounded sample: the whole small
    workload, one head of the 4096 x 4096 one, and >= 512 rows of the
    longest, so that attention (not the prologue) dominates the sample."""
    plan = bench.oracle_sample_plan
    assert plan(wl.WORKLOADS["small_d64"]) == (2, 2, 256)
    assert plan(wl.WORKLOADS["b2_h24_l4096_d128"]) == (1, 1, 4096)
    heads, kv, rows = plan(wl.WORKLOADS["dit_self_l32768"])
    assert (heads, kv) == (1, 1) and rows == 512
    heads, kv, rows = plan(wl.WORKLOADS["gqa_causal_b4_l8192"])
    assert heads % (32 // 8) == 0 or (heads, kv) == (1, 1)
    assert rows * 8192 <= bench.ORACLE_PAIR_BUDGET


def test_reference_arm_line_on_rank_zero(capsys):
    args = types.SimpleNamespace(oracle_pairs=256 * 64, warmup=3, steps=1, gpus=1,
                                 variant="fp8")
    bench.reference_arm(args, wl.WORKLOADS["small_d64"], rank=0, world=1)
    line = json.loads(capsys.readouterr().out)
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
