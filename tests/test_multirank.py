"""The N > 1 path on CPU: two `gloo` ranks, no GPU.

bench.py under torchrun runs one independent copy of the workload per rank
(heads and problems are independent; no collective in the data path) and
reports the whole job's throughput over the slowest rank's time.  These tests
run its rank helpers in two spawned processes, check that a reference run on
a nonzero rank does no work, and check the property the sharding rests on:
the plan and the output of every head depend on that head's inputs only, so
heads split across ranks and gathered give the single-process result.
"""

import os
import socket

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys

    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle as O
        from workloads import make_workload

        out = {}
        # slowest rank's time; identity on one rank
        out["max"] = bench.max_over_ranks(1.5 + rank, world, "cpu")
        out["single"] = bench.max_over_ranks(1.5 + rank, 1, "cpu")
        out["value"] = bench.weak_scaling_value(2.0e12, 4.0, world)

        # heads rank::world of the tiny workload, gathered on every rank
        arrays, prm = make_workload("tiny")
        sz = O.derive_sizes(prm["T"], prm["H"], prm["video_tokens"], prm["topk_ratio"],
                            prm["radius"], prm["tail_mode"])
        mine = list(range(rank, prm["H"], world))
        qh = np.ascontiguousarray(arrays["q"][:, mine])
        kh = np.ascontiguousarray(arrays["k"][:, mine])
        vh = np.ascontiguousarray(arrays["v"][:, mine])
        szh = O.derive_sizes(prm["T"], len(mine), prm["video_tokens"], prm["topk_ratio"],
                             prm["radius"], prm["tail_mode"])
        ref = O.plan(qh, kh, szh)
        o = O.forward(qh, kh, vh, arrays["bias"], ref["idx"], ref["cnt"], szh)
        parts = [None] * world
        dist.all_gather_object(parts, (mine, ref["idx"], ref["cnt"], o))
        out["parts"] = parts
        # reblocking of this rank's heads (independent per head as well)
        rb = O.spark_reblock(kh, 4)
        rparts = [None] * world
        dist.all_gather_object(rparts, (mine, rb["perm"], rb["inv"]))
        out["rparts"] = rparts
        out["H"] = prm["H"]
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def _run(world=2):
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return res


@pytest.fixture(scope="module")
def two_ranks():
    pytest.importorskip("torch")
    return _run(2)


def test_time_is_the_slowest_rank(two_ranks):
    for r in (0, 1):
        assert two_ranks[r]["max"] == 2.5
        assert two_ranks[r]["single"] == 1.5 + r


def test_weak_scaling_value_counts_every_rank(two_ranks):
    # two copies of 2 TFLOP in 4 ms
    assert two_ranks[0]["value"] == pytest.approx(2 * 2.0e12 / 4.0e-3 / 1e12)


def test_heads_split_across_ranks_give_the_single_process_result(two_ranks):
    import oracle as O
    from workloads import make_workload

    arrays, prm = make_workload("tiny")
    sz = O.derive_sizes(prm["T"], prm["H"], prm["video_tokens"], prm["topk_ratio"],
                        prm["radius"], prm["tail_mode"])
    ref = O.plan(arrays["q"], arrays["k"], sz)
    o = O.forward(arrays["q"], arrays["k"], arrays["v"], arrays["bias"], ref["idx"], ref["cnt"], sz)
    for r in (0, 1):
        parts = two_ranks[r]["parts"]
        seen = []
        for heads, idx, cnt, oh in parts:
            for j, h in enumerate(heads):
                seen.append(h)
                # lists are [H, nq, maxl] and [H, nq]; outputs [T, H, 128]
                assert np.array_equal(idx[j], ref["idx"][h])
                assert np.array_equal(cnt[j], ref["cnt"][h])
                assert np.array_equal(oh[:, j], o[:, h])
        assert sorted(seen) == list(range(two_ranks[r]["H"]))


def test_reblocking_heads_split_across_ranks(two_ranks):
    import oracle as O
    from workloads import make_workload

    arrays, prm = make_workload("tiny")
    rb = O.spark_reblock(arrays["k"], 4)
    for r in (0, 1):
        seen = []
        for heads, perm, inv in two_ranks[r]["rparts"]:
            for j, h in enumerate(heads):
                seen.append(h)
                assert np.array_equal(perm[j], rb["perm"][h]) and np.array_equal(inv[j], rb["inv"][h])
        assert sorted(seen) == list(range(prm["H"]))


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import bench

    class Args:
        steps, warmup, gpus = 1, 0, 2

    # a nonzero rank returns before loading the workload or starting a pool
    assert bench.run_reference(Args(), 1, 2) is None
    assert capsys.readouterr().out == ""
