"""GPU parity of the ternary T5_G128 format ("RTX 4080 SUPER 原生 Windows 跑 27B",
section 九.2: base-3 codes, five weights per byte, one fp16 scale per 128
weights) against the fp64 oracle, through the C ABI, on the tensor-core path
(its T5 kernel variant) and the tiled grouped GEMV path: small layers with
T5_G128 alone and mixed with the IQ and standard formats, shapes whose K ends
inside a 256-weight raw stage, and the 512-expert ternary decode and prefill
layers on every token."""
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


def _grid():
    return torch.from_numpy(synth.iq3_grid().view(np.int32).copy()).cuda()


def _run(M, L, path, grid=None):
    cfg = L.cfg
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, cfg.hidden, cfg.inter, grid=grid)
    p = getattr(M, "PATH_" + path)
    opt = M.make_options(n_experts=cfg.n_experts, path=p)
    assert M.ffn_path(table, cfg.tokens, cfg.k, opt) == p
    ws = M.Workspace(table, cfg.tokens, cfg.k, path=p)
    out = M.ffn_forward(table, x, logits, cfg.k, ws=ws, options=opt).cpu().numpy()
    assert ws.read_status() == 0
    return out


@pytest.mark.parametrize("H,I,T", [(512, 128, 40), (384, 384, 33), (256, 128, 130), (1024, 256, 5)])
@pytest.mark.parametrize("path", ["TENSOR", "GEMV"])
def test_t5_small(M, path, H, I, T):
    cfg = synth.LayerConfig("t5", 12, 3, H, I, T, "t5", True, 151 + H + I + T)
    L = synth.make_layer(cfg, 0)
    out = _run(M, L, path)
    assert_parity(out, offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k), f"{path} T5 H={H} I={I} T={T}")


@pytest.mark.parametrize("path", ["TENSOR", "GEMV"])
def test_t5_mixed_with_every_format(M, path):
    """One layer holding T5_G128 experts beside every other format (the tensor
    path's T5 variant decodes them all)."""
    cfg = synth.LayerConfig("t5m", 16, 4, 512, 128, 24, "q4k", True, 171)
    L = synth.make_layer(cfg, 0, with_weights=False)
    pairs = [(synth.T5_G128, synth.T5_G128), (synth.Q4_K, synth.T5_G128), (synth.T5_G128, synth.Q8_0),
             (synth.Q6_K, synth.Q8_0), (synth.IQ4_XS, synth.IQ4_NL), (synth.IQ3_XXS, synth.MXFP4),
             (synth.Q8_0, synth.IQ4_NL), (synth.MXFP4, synth.MXFP4)]
    L.fmts = [pairs[e % len(pairs)] for e in range(cfg.n_experts)]
    L.experts = [synth.expert_matrices(cfg, L.seed, e, L.fmts[e]) for e in range(cfg.n_experts)]
    out = _run(M, L, path, grid=_grid())
    assert_parity(out, offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k), f"{path} T5 among all formats")


def test_t5_needs_k_multiple_of_128(M):
    cfg = synth.LayerConfig("t5k", 4, 2, 256, 64, 2, "q4k", True, 181)
    experts, x, logits = host_layer_to_device(synth.make_layer(cfg, 0))
    # a down matrix of 64 columns cannot hold 128-weight blocks
    bad = dict(experts[0])
    bad["down"] = (synth.T5_G128, 256, 64, 16, torch.zeros(256 * 16, dtype=torch.uint8, device="cuda"))
    with pytest.raises(M.MoeError):
        M.WeightTable([bad] + experts[1:], cfg.hidden, cfg.inter)


@pytest.mark.parametrize("name,paths", [("decode16_t5", ("AUTO", "GEMV")), ("prefill512_t5", ("TENSOR", "GEMV"))])
def test_t5_full_size(M, name, paths):
    from synth import gpu as sgpu
    cfg = synth.CONFIGS[name]
    DL = sgpu.make_device_layer(cfg, 0)
    table = M.WeightTable(DL.experts, cfg.hidden, cfg.inter)
    ref = oracle_full_layer(cfg, DL)
    for path in paths:
        if path == "AUTO":
            # the streaming decode kernels take only the standard formats
            assert M.gemv_kernels(table, cfg.tokens, cfg.k) == M.GEMV_TILED
            assert M.ffn_path(table, cfg.tokens, cfg.k) == M.PATH_TENSOR
            opt, ws = None, M.Workspace(table, cfg.tokens, cfg.k)
        else:
            p = getattr(M, "PATH_" + path)
            opt = M.make_options(n_experts=cfg.n_experts, path=p)
            ws = M.Workspace(table, cfg.tokens, cfg.k, path=p)
        out = M.ffn_forward(table, DL.x_bf16, DL.logits, cfg.k, ws=ws, options=opt).cpu().numpy()
        assert ws.read_status() == 0
        assert_parity(out, ref, f"{name} {path}")
    del table, DL
    torch.cuda.empty_cache()
