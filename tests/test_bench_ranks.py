"""The benchmark's multi-GPU host logic on CPU: N replicas (one process per
GPU) report the slowest rank's time, and the whole-job value counts the
layer-rounds of every replica.  Two gloo ranks on 127.0.0.1 stand in for two
GPUs; no GPU is touched."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank 1 is the slow replica for the round time, rank 0 for e2e
        got = bench.max_over_ranks([2.0 + rank * 0.5, 3.0 - rank], dist)
        out[rank] = (got, bench.us_per_layer_round(got[0], 16, world))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replicas_take_the_slowest_rank(world):
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        got, value = res[rank]
        assert got == [2.5, 3.0]  # every rank sees the maxima
        assert value == pytest.approx(2.5e3 / (16 * world))


def test_single_process_is_unchanged():
    assert bench.max_over_ranks([1.25, 7.0]) == [1.25, 7.0]
    assert bench.us_per_layer_round(3.2, 16, 1) == pytest.approx(200.0)


def test_algorithmic_bytes_per_format():
    """Per token and KV head, K + V: 3-bit 2 x (96 B codes + 16 B group
    scales) = 224 B; int4 2 x (128 B codes + one 2 B scale) = 260 B; plus Q
    (and O for the layer-round)."""
    ctx, t, hq, hkv = [1000, 24], 16, 24, 4
    q = len(ctx) * t * hq * 256 * 2
    keys = (1000 + 16 + 24 + 16) * hkv
    assert bench.verify_kernel_bytes(ctx, t, hq, hkv) == keys * 224 + q
    assert bench.verify_kernel_bytes(ctx, t, hq, hkv, "int4") == keys * 260 + q
    assert bench.algorithmic_bytes_per_layer_round(ctx, t, hq, hkv, "int4") == keys * 260 + 2 * q
