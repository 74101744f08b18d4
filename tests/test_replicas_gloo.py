"""Several ranks as independent replicas (the host side of `bench.py --gpus N`),
run as two gloo processes on the CPU.

The layer needs no exchange between GPUs: every rank runs its own handle,
cache and inputs, and the ranks share only a barrier and the max-over-ranks of
their timed durations. These tests check exactly those pieces. Each rank draws
inputs of its own. A rank's layer result (here from the oracle) depends only on
its own inputs. The job's time is that of its slowest rank, and the whole-job
tokens/s counts every rank's tokens."""
import hashlib
import multiprocessing as mp
import os
import socket

import numpy as np

import synth

SHAPE = synth.Shape("replica", L=2, E=8, k=2, H=64, I=32, fmt=synth.FMT_NVFP4, act=synth.ACT_BF16)
STEPS, T = 3, 4


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_result(rank):
    """The oracle's output for the first layer of a rank's first step."""
    import bench
    import oracle
    hid = bench.rank_hidden_states(SHAPE, rank, STEPS, SHAPE.L, T, 0.0)
    experts = {e: synth.expert_weights(SHAPE, 0, 0, e) for e in range(SHAPE.E)}
    r = oracle.layer(SHAPE, experts, synth.router_weights(SHAPE, 0, 0), hid[0, 0])
    return hid, r["out"]


def _digest(a):
    return hashlib.sha1(np.ascontiguousarray(a).tobytes()).hexdigest()


def _worker(rank, world, port, q):
    try:
        import torch.distributed as dist
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import bench
        hid, out = _rank_result(rank)
        reuse = synth.reuse_flags(rank, 64, 0.7)
        ms = 10.0 + 5.0 * rank
        ms_max = bench.max_over_ranks(dist, ms)
        got = [None] * world
        dist.all_gather_object(got, (_digest(hid), _digest(out), _digest(reuse)))
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, ms_max, got, _digest(out)))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, "error", repr(e), None))


def test_two_gloo_ranks_run_independent_replicas():
    import bench
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, ms_max, got, out_digest = q.get(timeout=180)
        assert ms_max != "error", got
        res[rank] = (ms_max, got, out_digest)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # the job takes as long as its slowest rank
    assert res[0][0] == res[1][0] == 15.0
    # every rank saw the same gathered digests
    assert res[0][1] == res[1][1]
    (h0, o0, f0), (h1, o1, f1) = res[0][1]
    # inputs, results and step-reuse draws differ between ranks
    assert h0 != h1 and o0 != o1 and f0 != f1
    # a rank's result depends on its own inputs only: recomputed here, alone
    for r in range(world):
        _, out = _rank_result(r)
        assert _digest(out) == res[r][2]
    # whole-job tokens/s counts the tokens of every rank over the slowest rank's time
    assert bench.job_value(world, STEPS, T, 15.0) == world * STEPS * T / 15e-3


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(None, 12.5) == 12.5
    assert bench.job_value(1, 300, 1, 600.0) == 500.0
