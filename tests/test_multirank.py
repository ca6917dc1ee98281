"""Multi-process (world size 2, gloo, CPU) coverage of the N > 1 paths.

The attention forward shards over (batch, head, query block) with no data
exchange, so the benchmark runs one independent batch per rank (weak
scaling) and reduces only its timings. These tests run that host logic on
two gloo ranks: distinct per-rank problems, the max-over-ranks time and the
summed work. They also run the one exchange the method would have across
devices: key chunks of the same (b, h) attended on different ranks and
merged by log-sum-exp ("Lecture 06 — Making Decode Fast", section 5), which
must equal the unsplit result.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    os.environ["RANK"] = str(rank)
    os.environ["WORLD_SIZE"] = str(world)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _bench_logic(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    _init(rank, world, port)
    try:
        import bench
        from exact_tiled_attention_03_gb300.inputs import HEADLINE

        w = bench.rank_workload(HEADLINE, rank)
        seeds = [None] * world
        dist.all_gather_object(seeds, w.seed)
        t_max = bench.reduce_max(1.0 + rank, world)
        work = bench.reduce_sum(float(w.exact_flops()), world)
        out[rank] = (seeds, t_max, work, w.exact_flops())
    finally:
        dist.destroy_process_group()


def _split_exchange(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    _init(rank, world, port)
    try:
        import oracle
        from exact_tiled_attention_03_gb300.inputs import custom, make_qkv

        # verify-shaped problem: query i sees keys [0, Sk - Sq + i]
        w = custom(2, 3, 5, 300, 16, True, seed=77, q_factor=3.0)
        q, k, v = make_qkv(w)
        cut = 150                                  # fully visible to every query
        if rank == 0:
            o, l = oracle.attention(q, k[:, :, :cut], v[:, :, :cut], False, w.scale)
        else:                                      # last chunk keeps its bottom-right offset
            o, l = oracle.attention(q, k[:, :, cut:], v[:, :, cut:], True, w.scale)
        parts_o = [torch.empty(o.size, dtype=torch.float64) for _ in range(world)]
        parts_l = [torch.empty(l.size, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(parts_o, torch.from_numpy(np.ascontiguousarray(o.reshape(-1))))
        dist.all_gather(parts_l, torch.from_numpy(np.ascontiguousarray(l.reshape(-1))))
        d = w.d
        oc, lc = oracle.combine(np.stack([p.numpy().reshape(-1, d) for p in parts_o]),
                                np.stack([p.numpy() for p in parts_l]))
        o_ref, l_ref = oracle.attention(q, k, v, True, w.scale)
        out[rank] = (float(np.max(np.abs(oc - o_ref.reshape(-1, d)))),
                     float(np.max(np.abs(lc - l_ref.reshape(-1)))))
    finally:
        dist.destroy_process_group()


def _run(fn, world=2):
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=fn, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0, f"rank exited with {p.exitcode}"
    return dict(out)


def _dead_rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    os.environ["RANK"] = str(rank)
    os.environ["WORLD_SIZE"] = str(world)
    import bench

    bench.init_dist(world, "gloo", timeout_s=20.0)
    if rank == 1:
        os._exit(3)  # fails between steps, before the timing reduction
    try:
        bench.reduce_max(1.0, world)
        out[rank] = "no error"
    except Exception as e:  # the backend's error type differs across versions
        out[rank] = "error: " + type(e).__name__


def test_a_dead_rank_ends_the_others_reduction_with_an_error():
    """A rank that exits between steps makes the survivor's next collective
    raise (bounded by the process-group timeout) rather than wait for it."""
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_dead_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert procs[1].exitcode == 3
    assert procs[0].exitcode == 0, procs[0].exitcode
    assert out.get(0, "").startswith("error"), dict(out)


def test_bench_rank_logic_two_gloo_ranks():
    out = _run(_bench_logic)
    seeds, t_max, work, per_rank = out[0]
    assert len(set(seeds)) == 2, "each rank must run its own independent problem"
    assert t_max == 2.0, "the job is as slow as its slowest rank"
    assert work == 2 * per_rank, "value counts the work of every rank"
    assert out[1][1] == 2.0 and out[1][2] == work


def test_split_kv_exchange_across_two_gloo_ranks():
    out = _run(_split_exchange)
    for rank in (0, 1):
        err_o, err_l = out[rank]
        assert err_o < 1e-12 and err_l < 1e-12


def test_bench_launches_its_own_ranks_when_started_without_a_launcher(capfd, monkeypatch):
    """`bench.py --gpus 2` with no WORLD_SIZE in the environment starts two
    ranks under torchrun itself (rendezvous on 127.0.0.1). The reference arm
    runs on host cores, so the launch, the rendezvous of both ranks and rank
    0's single JSON line are exercised without a GPU."""
    import json
    import sys
    sys.path.insert(0, ROOT)
    import bench

    for var in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        monkeypatch.delenv(var, raising=False)
    cmd = bench.launch_command(["--gpus", "2"], 2, 12345)
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"]
    assert "--nproc-per-node=2" in cmd and "127.0.0.1" in cmd
    rc = bench.main(["--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
                     "--workload", "tiny_b1h1s256d64_causal", "--ref-budget", "2"])
    assert rc == 0
    lines = [l for l in capfd.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1, lines       # rank 0 alone prints
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["steps"] == 2
    assert rec["value"] > 0 and rec["config"]["workload"] == "tiny_b1h1s256d64_causal"


def test_bench_refuses_a_rank_count_other_than_its_launcher(monkeypatch):
    import sys
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "2", "--impl", "reference"])
