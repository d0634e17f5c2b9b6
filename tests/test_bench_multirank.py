"""The bench's multi-rank logic on CPU: two gloo ranks, the slowest rank's time sets the job's time,
and the job's value is the work of all ranks over that time (replicas of the whole workload)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 100.0 + 50.0 * rank                 # rank 1 is the slow one
        slowest = bench.reduce_max(local_ms, dist)
        dist.barrier()
        out[rank] = (slowest, bench.whole_job_rate(2.0e12, world, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    slowest, rate = res[0]
    assert slowest == 150.0
    assert rate == pytest.approx(2 * 2.0e12 / 0.150)


def test_single_rank_helpers():
    assert bench.reduce_max(3.5, None) == 3.5
    assert bench.whole_job_rate(1.0e12, 1, 1000.0) == pytest.approx(1.0e12)
    assert bench.measured_traffic("no_such_workload") == (None, None)


def test_source_key_ignores_comments_only():
    """The traffic bookkeeping's key: comment and spacing edits keep it, any code edit changes it."""
    base = bench.source_key("int a = 1;  // one\n/* block\n comment */ float b;\n")
    assert bench.source_key("int a = 1;\nfloat b;   // other words\n") == base
    assert bench.source_key("int a = 2;\nfloat b;\n") != base
    assert bench.source_key("int a = 1;\ndouble b;\n") != base


def test_hop_summary_slack_and_exposure():
    """The ring-step timelines' arithmetic: a forward hop must end before its own step's compute,
    a backward gradient hop before the next step's; the last step's hop is not counted."""
    c_end = [10.0, 20.0, 30.0]
    fwd = bench.hop_summary(c_end, [9.0, 20.5, 31.0], next_step_bound=False)
    assert fwd["steps"] == 3 and fwd["step_ms_min"] == 10.0 and fwd["step_ms_max"] == 10.0
    assert not fwd["hops_hidden"] and fwd["min_slack_ms"] == -0.5 and fwd["exposed_ms_total"] == 0.5
    bwd = bench.hop_summary(c_end, [12.0, 25.0, 40.0], next_step_bound=True)
    assert bwd["hops_hidden"] and bwd["min_slack_ms"] == 5.0 and bwd["exposed_ms_total"] == 0.0
    one = bench.hop_summary([7.0], [8.0], next_step_bound=False)
    assert one["hops_hidden"] and one["min_slack_ms"] is None


@pytest.mark.parametrize("name", sorted(__import__("synth").CONFIGS))
def test_effective_flops_follow_the_visible_pairs(name):
    """The bench's FLOP count against the plan's exact visible pairs (bit-exact against the
    oracle's brute force elsewhere): 4 B h d per pair, with a causal diagonal counted as half, so
    T^2/2 = T(T+1)/2 - T/2 pairs per (b, head)."""
    import synth
    import context_ring_attention_blockwise_gb300 as cp
    w = synth.workload(name)
    plan = cp.Plan(w.T, w.h, w.n_kv, w.d, w.n_cp, w.layouts[0], w.causal)
    exact = int(plan.counts(1)["pairs"].sum())
    assert exact == (w.T * (w.T + 1) // 2 if w.causal else w.T * w.T)
    effective = exact - w.T / 2 if w.causal else exact
    assert bench.flops_eff(w) == 4.0 * w.B * w.h * w.d * effective


def test_config_names_each_path():
    """The JSON line's config says which path and parallelism a run measured."""
    import argparse
    w = bench.synth.workload("llama70b_zigzag_T128k")
    def cfg(path, gpus):
        return bench.config_of(w, argparse.Namespace(path=path, gpus=gpus, layout=1))
    assert cfg("fused", 1)["parallelism"] == "single GPU" and cfg("fused", 8)["parallelism"] == "replicas"
    assert cfg("steps", 1)["path"] == "steps" and "one launch per ring step" in cfg("steps", 1)["parallelism"]
    assert cfg("ring", 2)["parallelism"].startswith("ring over 2 processes")
    assert cfg("ring", 1)["parallelism"] == "single GPU, one process holding all ranks"
