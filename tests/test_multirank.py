"""The N > 1 path on CPU: two `gloo` ranks, no GPU.

bench.py under torchrun splits the heads into contiguous slices, one per rank
(heads are independent; no collective in the data path), and reports the
whole job's kept work over the slowest rank's time (strong scaling).  These
tests run its rank helpers (bench.head_range, bench.split_heads) in two
spawned processes, check that a reference run on a nonzero rank does no work,
and check the property the sharding rests on: the plan and the output of
every head depend on that head's inputs only, so the ranks' slices, gathered,
give the single-process result.
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
        out["value"] = bench.strong_scaling_value(2.0e12, 4.0)

        # heads rank::world of the tiny workload, gathered on every rank
        arrays, prm = make_workload("tiny")
        sz = O.derive_sizes(prm["T"], prm["H"], prm["video_tokens"], prm["topk_ratio"],
                            prm["radius"], prm["tail_mode"])
        h0, h1 = bench.head_range(prm["H"], rank, world)
        mine = list(range(h0, h1))
        sl = bench.split_heads(arrays, h0, h1)
        qh, kh, vh = sl["q"], sl["k"], sl["v"]
        assert qh.flags["C_CONTIGUOUS"] and qh.shape[1] == len(mine)
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


def test_strong_scaling_value_is_the_job_work_over_the_slowest_rank(two_ranks):
    # one workload of 2 TFLOP split over the ranks, 4 ms for the slowest
    assert two_ranks[0]["value"] == pytest.approx(2.0e12 / 4.0e-3 / 1e12)


def test_head_ranges_partition_the_heads():
    import bench

    for H in (1, 2, 5, 24, 56):
        for world in (1, 2, 3, 4, 8):
            rs = [bench.head_range(H, r, world) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == H
            assert all(rs[i][1] == rs[i + 1][0] for i in range(world - 1))
            sizes = [b - a for a, b in rs]
            assert max(sizes) - min(sizes) <= 1


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
