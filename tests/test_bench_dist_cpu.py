"""Host logic of the multi-process bench path, on CPU with gloo (world size 2).

The operator shards into independent units with no exchange, so N GPUs run N replicas;
the job's time is the slowest rank's and its throughput counts every replica's work.
"""
import io
import os
import socket
import sys
import contextlib

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank                       # rank 1 is the slow replica
        slowest = bench.max_over_ranks(mine)
        value = bench.job_tflops(1e12, world, 4, slowest)
        # the reference arm: ranks other than 0 return at once and print nothing
        out = io.StringIO()
        ran = None
        if rank != 0:
            class A:
                steps, warmup, ref_units, impl = 1, 0, 1, "reference"
            from block_causal_video_attention_b300 import synth
            with contextlib.redirect_stdout(out):
                ran = bench.run_reference(A, None, False)
                # the decode and variable-length reference arms likewise
                assert bench.run_decode(A, synth.WORKLOADS["minecraft_decode"]) is None
                assert bench.run_varlen(A, synth.WORKLOADS["tokenizer_enc"]) is None
        dist.barrier()
        results[rank] = (slowest, value, out.getvalue(), ran)
    finally:
        dist.destroy_process_group()


def test_replicas_max_over_ranks_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(results)
    assert set(res) == {0, 1}
    for r in range(world):
        slowest, value, printed, ran = res[r]
        assert slowest == pytest.approx(15.0)                 # the max, on every rank
        # 2 replicas x 4 steps x 1 TFLOP in 15 ms
        assert value == pytest.approx(2 * 4 * 1.0 / 15e-3)
    assert res[1][2] == "" and res[1][3] is None


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(2e12, 1, 10, 1000.0) == pytest.approx(20.0)
