"""GPU parity of shared-expert fusion ("多卡 CUDA 张量并行：DwarfStar 如何在 8 张 L40S 上跑出
120 t/s", memory layout: shared experts beside the routed ones, stored there in
Q8_0) against the fp64 oracle, through the C ABI. The shared expert is table
entry E and slot k of every token (weight 1), so it runs in the same grouped
kernels as the routed experts: small layers on every output, the 512-expert
decode and prefill layers with one Q8_0 shared expert on every token, on the
streaming and tiled GEMV kernels and on the tensor path; the routing views;
the expert-range split (the shared expert goes to the last shard); and the
fused decode kernel, which has no shared slots, refusing the layer."""
import numpy as np
import pytest
import torch

import synth
from oracle import ffn as offn
from tests.gpu_util import assert_parity, ensure_built, host_layer_to_device, oracle_full_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    ensure_built()
    import quantized_moe_expert_route_gb300 as M
    M.load()
    return M


def _small(E=12, k=3, H=512, I=128, T=40, tiers="mixed", seed=101, S=1):
    cfg = synth.LayerConfig("sh", E, k, H, I, T, tiers, True, seed, S)
    return cfg, synth.make_layer(cfg, 0)


@pytest.mark.parametrize("S", [1, 2])
@pytest.mark.parametrize("path", ["TENSOR", "GEMV"])
def test_shared_small(M, path, S):
    cfg, L = _small(S=S, seed=101 + S)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, cfg.hidden, cfg.inter, n_shared=S)
    assert table.n_experts == cfg.n_experts and table.n_entries == cfg.n_entries
    p = getattr(M, "PATH_" + path)
    opt = M.make_options(n_experts=table.n_entries, path=p)
    assert M.ffn_path(table, cfg.tokens, cfg.k, opt) == p
    ws = M.Workspace(table, cfg.tokens, cfg.k, path=p)
    out = M.ffn_forward(table, x, logits, cfg.k, ws=ws, options=opt).cpu().numpy()
    assert ws.read_status() == 0
    ref = offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k, n_shared=S)
    assert_parity(out, ref, f"{path} S={S}")
    # routing views: the shared experts fill slots k.. with weight 1
    r = ws.routing()
    ids, w = r["ids"].cpu().numpy(), r["weights"].cpu().numpy()
    assert ids.shape == (cfg.tokens, cfg.k + S)
    np.testing.assert_array_equal(ids[:, cfg.k:], np.broadcast_to(np.arange(cfg.n_experts, cfg.n_entries),
                                                                  (cfg.tokens, S)))
    assert np.all(w[:, cfg.k:] == 1.0)
    oi, ow = offn.token_slots(L.logits, cfg.k, True, S)
    np.testing.assert_array_equal(ids, oi)


@pytest.mark.parametrize("path", ["TENSOR", "GEMV"])
def test_shared_split_and_routed_only(M, path):
    """[0, E) is bit-identical to the same layer without the shared expert;
    [0, E) plus [E, E + 1) is the whole layer."""
    cfg, L = _small(T=24, seed=131)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, cfg.hidden, cfg.inter, n_shared=1)
    plain = M.WeightTable(experts[:cfg.n_experts], cfg.hidden, cfg.inter)
    p = getattr(M, "PATH_" + path)
    E = cfg.n_experts
    routed = M.ffn_forward(table, x, logits, cfg.k,
                           options=M.make_options(n_experts=E + 1, expert_hi=E, path=p)).cpu().numpy()
    ref_plain = M.ffn_forward(plain, x, logits, cfg.k, options=M.make_options(n_experts=E, path=p)).cpu().numpy()
    np.testing.assert_array_equal(routed, ref_plain)
    shared = M.ffn_forward(table, x, logits, cfg.k,
                           options=M.make_options(n_experts=E + 1, expert_lo=E, path=p)).cpu().numpy()
    ref = offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k, n_shared=1)
    assert_parity(routed.astype(np.float64) + shared, ref, f"{path} split")
    assert_parity(shared, offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k, n_shared=1, expert_lo=E),
                  f"{path} shared only")


def test_shared_refuses_fused_and_bad_counts(M):
    cfg, L = _small(E=64, k=8, H=512, I=256, T=1, tiers="q4k", seed=141)
    # a shared expert in the fused kernel's own formats, so that only its
    # being shared keeps the layer off that kernel
    L.experts[-1] = synth.expert_matrices(cfg, L.seed, cfg.n_experts, (synth.Q4_K, synth.Q8_0))
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, cfg.hidden, cfg.inter, n_shared=1)
    as_routed = M.WeightTable(experts, cfg.hidden, cfg.inter)       # the same 65 experts, all routed
    assert M.ffn_path(as_routed, 1, cfg.k) == M.PATH_FUSED
    assert M.ffn_path(table, 1, cfg.k, M.make_options(n_experts=65, path=M.PATH_FUSED)) == -1
    assert M.ffn_path(table, 1, cfg.k) == M.PATH_GEMV
    out = M.ffn_forward(table, x, logits, cfg.k).cpu().numpy()
    assert_parity(out, offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k, n_shared=1), "decode1 shared AUTO")
    with pytest.raises(ValueError):
        M.WeightTable(experts, cfg.hidden, cfg.inter, n_shared=len(experts))
    with pytest.raises(M.MoeError):
        M.WeightTable(experts, cfg.hidden, cfg.inter, n_shared=5)      # above MOE_MAX_SHARED
    # k + n_shared above the slot limit (k = 32, one shared expert)
    with pytest.raises(M.MoeError) as ei:
        M.ffn_forward(table, x, logits, 32, ws=M.Workspace(table, 1, 8))
    assert ei.value.code == 8


@pytest.mark.parametrize("name,paths", [("decode16_shared", ("AUTO", "GEMV_TILED", "TENSOR")),
                                        ("prefill512_shared", ("TENSOR", "GEMV"))])
def test_shared_full_size(M, name, paths):
    from synth import gpu as sgpu
    cfg = synth.CONFIGS[name]
    DL = sgpu.make_device_layer(cfg, 0)
    table = M.WeightTable(DL.experts, cfg.hidden, cfg.inter, n_shared=cfg.n_shared)
    ref = oracle_full_layer(cfg, DL)
    for path in paths:
        x = DL.x_bf16
        if path == "AUTO":
            opt = None
            ws = M.Workspace(table, cfg.tokens, cfg.k)
            assert M.ffn_path(table, cfg.tokens, cfg.k) == M.PATH_GEMV
            assert M.gemv_kernels(table, cfg.tokens, cfg.k) == M.GEMV_STREAMING
        elif path == "GEMV_TILED":
            # the streaming kernels want a 16-byte aligned activation pointer:
            # one off by 2 bytes runs the tiled kernels
            buf = torch.empty(x.numel() + 8, dtype=torch.bfloat16, device="cuda")
            x = buf[1:1 + x.numel()].view(x.shape)
            x.copy_(DL.x_bf16)
            opt = M.make_options(n_experts=table.n_entries, path=M.PATH_GEMV)
            ws = M.Workspace(table, cfg.tokens, cfg.k, path=M.PATH_GEMV)
        else:
            p = getattr(M, "PATH_" + path)
            opt = M.make_options(n_experts=table.n_entries, path=p)
            ws = M.Workspace(table, cfg.tokens, cfg.k, path=p)
        out = M.ffn_forward(table, x, DL.logits, cfg.k, ws=ws, options=opt).cpu().numpy()
        assert ws.read_status() == 0
        assert_parity(out, ref, f"{name} {path}")
    del table, DL
    torch.cuda.empty_cache()
