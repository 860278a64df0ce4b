"""Expert sharding on the GPU ("多卡 CUDA 张量并行：DwarfStar 如何在 8 张 L40S 上跑出 120
t/s", section "8 张卡是怎么配对的": routed experts split across a pair of GPUs,
router replicated, partial outputs summed): the fixed-order partial sum of
the library bit for bit against an ordered fp32 sum; the shards of a layer,
each evaluated over its expert range with the other experts' table entries
pointing at placeholder weights that must never be read, summed back to the
oracle's layer; and two processes (ranks) on this GPU exchanging their
partials over gloo, which must end with bit-identical outputs."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import synth
from oracle import ffn as offn
from tests.gpu_util import assert_parity, ensure_built, host_layer_to_device, oracle_full_layer

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def M():
    ensure_built()
    import quantized_moe_expert_route_gb300 as M
    M.load()
    return M


@pytest.mark.parametrize("n,count,offset", [(1, 4096, 0), (2, 4096, 0), (3, 4099, 0), (5, 1, 0), (4, 2048, 1)])
def test_sum_partials_ordered(M, n, count, offset):
    rng = np.random.default_rng(n * 1000 + count)
    parts = (rng.standard_normal((n, count)) * 1e3 ** rng.integers(-1, 2, (n, 1))).astype(np.float32)
    dev = torch.from_numpy(parts).cuda()
    out_buf = torch.zeros(count + 1, dtype=torch.float32, device="cuda")
    out = out_buf[offset:offset + count]           # offset 1: not 16-byte aligned (scalar kernel)
    M.sum_partials(dev, out=out)
    ref = parts[0].copy()
    for p in range(1, n):
        ref = (ref + parts[p]).astype(np.float32)   # one fp32 add at a time, ascending order
    np.testing.assert_array_equal(out.cpu().numpy(), ref)


def _shard_table(M, experts, lo, hi, hidden, inter, n_shared=0):
    """The table of a rank holding experts [lo, hi): the other entries point
    at expert lo's tensors (placeholders of the right shape, never read)."""
    ph = experts[lo]
    own = [experts[e] if lo <= e < hi else ph for e in range(len(experts))]
    return M.WeightTable(own, hidden, inter, n_shared=n_shared)


@pytest.mark.parametrize("name,world", [("decode16", 2), ("mtp6", 2), ("decode1", 3), ("decode16_shared", 2)])
def test_shards_sum_to_the_layer(M, name, world):
    """With a shared expert (the last table entry) the last shard computes it."""
    from synth import gpu as sgpu
    cfg = synth.CONFIGS[name]
    DL = sgpu.make_device_layer(cfg, 5)
    parts = []
    for r in range(world):
        lo, hi = M.expert_shard(cfg.n_entries, r, world)
        table = _shard_table(M, DL.experts, lo, hi, cfg.hidden, cfg.inter, cfg.n_shared)
        opt = M.make_options(n_experts=cfg.n_entries, expert_lo=lo, expert_hi=hi)
        parts.append(M.ffn_forward(table, DL.x_bf16, DL.logits, cfg.k, options=opt))
    out = M.sum_partials(torch.stack(parts)).cpu().numpy()
    assert_parity(out, oracle_full_layer(cfg, DL), f"{name} in {world} expert shards")
    del DL
    torch.cuda.empty_cache()


def test_small_mixed_layer_three_shards(M):
    cfg = synth.LayerConfig("shm", 24, 6, 512, 128, 9, "mixed", True, 73)
    L = synth.make_layer(cfg, 0)
    experts, x, logits = host_layer_to_device(L)
    parts = []
    for r in range(3):
        lo, hi = M.expert_shard(cfg.n_experts, r, 3)
        table = _shard_table(M, experts, lo, hi, cfg.hidden, cfg.inter)
        parts.append(M.ffn_forward(table, x, logits, cfg.k,
                                   options=M.make_options(n_experts=cfg.n_experts, expert_lo=lo, expert_hi=hi)))
    out = M.sum_partials(torch.stack(parts)).cpu().numpy()
    assert_parity(out, offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k), "mixed layer in 3 shards")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import quantized_moe_expert_route_gb300 as M
    from synth import gpu as sgpu
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = synth.CONFIGS["decode16"]
        DL = sgpu.make_device_layer(cfg, 6)
        lo, hi = M.expert_shard(cfg.n_experts, rank, world)
        table = _shard_table(M, DL.experts, lo, hi, cfg.hidden, cfg.inter)
        layer = M.ShardedLayer(table, cfg.n_experts, rank, world)
        out = layer.forward(DL.x_bf16, DL.logits, cfg.k)
        torch.cuda.synchronize()
        q.put((rank, out.cpu().numpy()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_over_gloo(M):
    """Two processes on this GPU, each holding half of the experts: their
    kernels never wait on each other (the exchange goes through the host),
    and both end with the same bits, equal to the oracle's layer."""
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    outs = {}
    for _ in range(world):
        rank, out = q.get(timeout=600)
        outs[rank] = out
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    np.testing.assert_array_equal(outs[0], outs[1])
    from synth import gpu as sgpu
    cfg = synth.CONFIGS["decode16"]
    DL = sgpu.make_device_layer(cfg, 6, fill_weights=False)
    assert_parity(outs[0], oracle_full_layer(cfg, DL), "decode16 over two gloo ranks")
