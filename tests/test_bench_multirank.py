"""The benchmark's multi-rank host logic on CPU: two ranks over a gloo
process group (the GPU runs use NCCL with one rank per GPU; the layer's
calls are independent per rank, so the only exchange is the timing
reduction)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.cpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank step times: rank 1 is the slow one
        mine = [10.0 + 5.0 * rank, 3.0 - rank]
        got = bench.max_over_ranks(mine, world)
        calls = list(bench.rank_calls(rank, 3, 5))
        dist.barrier()
        q.put((rank, got, calls))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_partition():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank holds the element-wise maximum
    for _, got, _ in res:
        assert got == [15.0, 3.0]
    # the ranks' token streams are disjoint and cover W + K calls each
    c0, c1 = res[0][2], res[1][2]
    assert len(c0) == len(c1) == 8 and not set(c0) & set(c1)


def test_whole_job_value_uses_the_slowest_rank():
    import bench
    # 2 ranks x 5 steps x 4 tokens over the slowest rank's 20 ms
    assert bench.whole_job_tokens_per_s(4, 5, 2, 20.0) == pytest.approx(2000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    from mixture_experts_ffn_gate_gb300 import synth
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup = 1, 1
    # rank 1 returns at once, without touching the oracle
    assert bench.reference_arm(A(), synth.WORKLOADS["tiny_t4_h256_i128_e8_k2"], 4) is None
