"""Host-side logic of bench.py, on the CPU: the visible-pair count it uses,
the profile-summary lookup, argument defaults and the multi-rank timing
reduction (gloo, world size 2)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle


def test_closed_form_pairs_match_oracle_for_bench_workload():
    w = bench.workload()
    raw, comp = bench.visible_pairs_closed_form(w.S, w.W, w.m)
    oraw, ocomp = oracle.visible_pairs(None, 1, w.S, w.W, w.m)
    assert (raw, comp) == (int(oraw[0]), int(ocomp[0]))
    assert (raw + comp) * w.H == 1608028160


def test_default_arguments():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1 and a.impl == "ours"


def test_profiled_traffic_lookup(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    digest = bench.source_digest("hca_bwd_dkv")
    assert digest
    w = bench.workload()
    (tmp_path / "hca_bwd_dkv_x.md").write_text(
        f"workload: {w.name}\ntraffic_bytes_per_launch: 1.5e9\nsource_sha256_16: {digest}\n")
    assert bench.profiled_traffic("hca_bwd_dkv", w.name) == 1.5e9
    # a summary taken on an older kernel source is not used
    (tmp_path / "hca_bwd_dkv_x.md").write_text(
        f"workload: {w.name}\ntraffic_bytes_per_launch: 1.5e9\nsource_sha256_16: 0000000000000000\n")
    assert bench.profiled_traffic("hca_bwd_dkv", w.name) is None
    assert bench.profiled_traffic("hca_fwd_tc", w.name) is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    d = bench.init_dist(world, "gloo")
    bench.barrier(d)
    m = bench.max_over_ranks(10.0 + 5.0 * rank, d)
    out[rank] = m
    d.destroy_process_group()


def test_max_over_ranks_gloo_world_size_2():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 15.0


def test_single_rank_needs_no_process_group():
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(3.5, None) == 3.5
