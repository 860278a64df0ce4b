"""Expert sharding on the CPU: the shard ranges, and the exchange of partial
outputs between two gloo ranks (the same all-gather the GPU ranks use), with
the partials computed by the oracle over each rank's expert range. The sum of
the gathered partials in rank order equals the whole layer ("多卡 CUDA 张量并行：
DwarfStar 如何在 8 张 L40S 上跑出 120 t/s", section "8 张卡是怎么配对的": routed experts
split 50/50 across a pair, router replicated)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_expert_shard_partitions():
    from quantized_moe_expert_route_gb300.shard import expert_shard
    for E in (1, 7, 8, 512, 1000):
        for world in (1, 2, 3, 4, 8):
            if world > E:
                continue
            r = [expert_shard(E, i, world) for i in range(world)]
            assert r[0][0] == 0 and r[-1][1] == E
            assert all(r[i][1] == r[i + 1][0] for i in range(world - 1))
            sizes = [hi - lo for lo, hi in r]
            assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)
    assert expert_shard(512, 0, 2) == (0, 256) and expert_shard(512, 1, 2) == (256, 512)
    with pytest.raises(ValueError):
        expert_shard(8, 2, 2)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import synth
    from oracle import ffn
    from quantized_moe_expert_route_gb300.shard import expert_shard, gather_partials
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = synth.LayerConfig("sh", 16, 4, 256, 64, 5, "mixed", True, 61)
        L = synth.make_layer(cfg, 0)
        lo, hi = expert_shard(cfg.n_experts, rank, world)
        part = ffn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k, expert_lo=lo, expert_hi=hi)
        got = gather_partials(torch.from_numpy(part))
        q.put((rank, [g.numpy() for g in got], part))
    finally:
        dist.destroy_process_group()


def test_two_rank_exchange_sums_to_the_layer():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, got, own = q.get(timeout=240)
        res[rank] = (got, own)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import synth
    from oracle import ffn
    cfg = synth.LayerConfig("sh", 16, 4, 256, 64, 5, "mixed", True, 61)
    L = synth.make_layer(cfg, 0)
    full = ffn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k)
    for rank in range(world):
        got, own = res[rank]
        # every rank receives every partial, in rank order
        for r in range(world):
            np.testing.assert_array_equal(got[r], res[r][1])
        acc = got[0].copy()
        for r in range(1, world):
            acc += got[r]
        np.testing.assert_allclose(acc, full, rtol=1e-12, atol=1e-12 * np.abs(full).max())
    # the split is not trivial: both ranks contribute
    assert np.abs(res[0][1]).max() > 0 and np.abs(res[1][1]).max() > 0
