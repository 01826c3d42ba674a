"""The benchmark's multi-rank path on CPU (gloo, world size 2): each rank
runs an independent replica, the timing is the max over ranks and nothing
else is exchanged. Runs without a GPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    elapsed = [3.5, 7.25][rank]
    got = bench.max_over_ranks(elapsed, world)
    bench.barrier(world)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    results = dict(q.get(timeout=5) for _ in range(2))
    assert all(p.exitcode == 0 for p in procs)
    assert results == {0: 7.25, 1: 7.25}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    bench.barrier(1)


def test_kv_read_bytes_counts_valid_tokens_only():
    import bench
    # 2 sequences of 3 and 5 tokens, 8 KV heads, head size 128, 2-byte dtype
    assert bench.kv_read_bytes([3, 5], 8, 128, 2) == 8 * 2 * 8 * 128 * 2


def test_attention_flops_counts_visible_keys():
    """The prefill roofline's algorithmic flops: new token i of a sequence
    with c cached tokens sees c + i + 1 keys; 4 flops per key and head dim
    (q.k and p.v) per query head. Checked against a direct count."""
    import bench
    for ctx, n, hq, d in (([0], 1, 1, 1), ([0, 5, 17], 3, 8, 128), ([1000, 0], 64, 64, 64)):
        direct = sum(4 * d * hq * (c + i + 1) for c in ctx for i in range(n))
        assert bench.attention_flops(ctx, n, hq, d) == direct
    # one new token: decode, 4 * D * Hq per cached-or-new key
    assert bench.attention_flops([9], 1, 2, 16) == 4 * 16 * 2 * 10
