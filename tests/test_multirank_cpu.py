"""The N > 1 path of the bench on CPU: two processes over a gloo process group.

With N GPUs the bench runs N independent replicas (the path partitions into
independent problems, so there is no collective on the data path).  The host
logic that turns the ranks' timings into one job-wide number is checked here
without a GPU: the timed span is the slowest rank's, the value counts every
rank's tokens, and only rank 0 reports.  The reference arm under a launcher
does its work on rank 0 only; the other ranks return at once.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, spans, tokens, queue):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        out = bench.combine_ranks(spans[rank], tokens, world, rank)
        queue.put((rank, out))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run_ranks(spans, tokens):
    import multiprocessing as mp

    ctx = mp.get_context("spawn")  # a fresh interpreter per rank
    queue = ctx.Queue()
    port = _free_port()
    world = len(spans)
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, spans, tokens, queue))
             for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in range(world):
            rank, out = queue.get(timeout=120)
            results[rank] = out
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return results


def test_two_ranks_take_the_slowest_span_and_count_all_tokens():
    tokens = 4096 * 50
    results = _run_ranks([10.0, 12.5], tokens)
    assert results[1] is None  # only rank 0 reports
    span, value = results[0]
    assert span == 12.5
    assert value == pytest.approx(2 * tokens / 12.5e-3)


def test_two_ranks_order_does_not_matter():
    tokens = 1000
    results = _run_ranks([7.0, 3.0], tokens)
    span, value = results[0]
    assert span == 7.0
    assert value == pytest.approx(2 * tokens / 7.0e-3)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    span, value = bench.combine_ranks(4.0, 500, 1, 0)
    assert span == 4.0 and value == pytest.approx(500 / 4.0e-3)
    assert bench.combine_ranks(4.0, 500, 1, 1) is None


def test_reference_arm_other_ranks_return_without_work():
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        workload = "layer_t4096"
        steps = 1
        warmup = 3

    assert bench.run_reference(Args(), rank=1, world=2) is None
