"""The cold-expert tier ("三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80 Token 每秒的高效推理
优化指南", section 优化策略一: the coldest experts by router frequency stay in host
RAM): the tail 20% of the experts by router-bias rank are kept in pinned host
memory (on GB300 the Grace CPU's memory, read by the GPU over NVLink-C2C). The
layer's routed cold experts are staged into the workspace by the GPU after
routing, so the grouped GEMV kernels compute on the same bytes as with every
expert in device memory: the outputs must be bit-identical to that, and match
the oracle."""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import assert_parity, ensure_built, oracle_full_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    ensure_built()
    import quantized_moe_expert_route_gb300 as M
    M.load()
    return M


def _cold_experts(DL, frac=0.2):
    """The experts of the coldest `frac` of ranks, with their matrices copied
    into pinned host memory."""
    E = DL.cfg.n_experts
    perm = synth.permutation(DL.seed, E)
    cold = set(int(e) for e in perm[E - int(E * frac):])
    experts = []
    for e, ex in enumerate(DL.experts):
        if e in cold:
            experts.append({n: (f, r, c, st, v.cpu().pin_memory()) for n, (f, r, c, st, v) in ex.items()})
        else:
            experts.append(ex)
    return experts, cold


@pytest.mark.parametrize("name,tokens", [("decode16", None), ("mtp6", None), ("decode1", None), ("mtp6", 24)])
def test_cold_tier_matches_all_device(M, name, tokens):
    from synth import gpu as sgpu
    cfg = synth.CONFIGS[name]
    DL = sgpu.make_device_layer(cfg, 21, tokens=tokens)
    T = DL.x_host.shape[0]
    experts, cold = _cold_experts(DL)
    hot = M.WeightTable(DL.experts, cfg.hidden, cfg.inter)
    mixed = M.WeightTable(experts, cfg.hidden, cfg.inter)
    assert mixed.c.n_cold == len(cold) and hot.c.n_cold == 0
    # a table with cold experts runs on the grouped GEMV path (fused and tensor paths refuse it)
    assert M.ffn_path(mixed, T, cfg.k) == M.PATH_GEMV
    assert M.ffn_path(mixed, T, cfg.k, M.make_options(n_experts=cfg.n_experts, path=M.PATH_TENSOR)) == -1
    gemv = M.make_options(n_experts=cfg.n_experts, path=M.PATH_GEMV)
    ws = M.Workspace(mixed, T, cfg.k)
    got = M.ffn_forward(mixed, DL.x_bf16, DL.logits, cfg.k, ws=ws).cpu().numpy()
    assert ws.read_status() == 0
    ref_dev = M.ffn_forward(hot, DL.x_bf16, DL.logits, cfg.k, options=gemv).cpu().numpy()
    assert np.array_equal(got, ref_dev)
    # some routed pairs reach cold experts
    R = ws.routing()
    act = R["active"].cpu().numpy()
    assert any(int(e) in cold for e in act[1:1 + act[0]]) or T < 6
    assert_parity(got, oracle_full_layer(cfg, DL), f"{name} T={T} with a cold tier")
    # a second call reuses the workspace (the staging is rewritten every call)
    again = M.ffn_forward(mixed, DL.x_bf16, DL.logits, cfg.k, ws=ws).cpu().numpy()
    assert np.array_equal(again, got)


def test_cold_expert_must_be_whole(M):
    from synth import gpu as sgpu
    cfg = synth.LayerConfig("cw", 8, 2, 256, 64, 3, "q4k", True, 31)
    DL = sgpu.make_device_layer(cfg, 0)
    experts = [dict(e) for e in DL.experts]
    f, r, c, st, v = experts[3]["down"]
    experts[3]["down"] = (f, r, c, st, v.cpu().pin_memory())    # only one matrix on the host
    with pytest.raises(M.MoeError) as ei:
        M.WeightTable(experts, cfg.hidden, cfg.inter)
    assert ei.value.code == 1
