"""GPU parity of the pages' own tier formats ("三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80
Token 每秒的高效推理优化指南", section 优化策略二: Q6_K gate/up with Q8_0 down for the
hottest experts, IQ4_XS with IQ4_NL down in the middle, IQ3_XXS with MXFP4 down
for the tail) against the fp64 oracle, through the C ABI, on the tensor-core
path and the grouped GEMV paths (streaming and tiled): each IQ format alone and the mixed
tiers, small layers on every output and the full-size 512-expert layers (6
and 2048 tokens) on every token. The IQ3_XXS grid is the table's input; the
layers use the seeded synthetic grid."""
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


def _with_formats(L, gu, dn):
    """The layer's experts re-generated with the given formats."""
    experts = []
    for e in range(L.cfg.n_experts):
        experts.append(synth.expert_matrices(L.cfg, L.seed, e, (gu, dn)))
    L.experts = experts
    return L


@pytest.mark.parametrize("gu,dn", [(synth.IQ4_XS, synth.IQ4_NL), (synth.IQ3_XXS, synth.MXFP4),
                                   (synth.IQ4_NL, synth.IQ4_NL), (synth.Q4_K, synth.IQ4_NL)])
@pytest.mark.parametrize("path", ["TENSOR", "GEMV"])
def test_iq_formats_small(M, gu, dn, path):
    cfg = synth.LayerConfig("iq", 12, 3, 512, 128, 40, "q4k", True, 91 + gu + 10 * dn)
    L = _with_formats(synth.make_layer(cfg, 0, with_weights=False), gu, dn)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, cfg.hidden, cfg.inter, grid=_grid())
    p = getattr(M, "PATH_" + path)
    opt = M.make_options(n_experts=cfg.n_experts, path=p)
    assert M.ffn_path(table, cfg.tokens, cfg.k, opt) == p
    ws = M.Workspace(table, cfg.tokens, cfg.k, path=p)
    out = M.ffn_forward(table, x, logits, cfg.k, ws=ws, options=opt).cpu().numpy()
    assert ws.read_status() == 0
    assert_parity(out, offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k), f"{path} gu {gu} dn {dn}")


def test_iq_mixed_tiers_small_and_auto(M):
    cfg = synth.LayerConfig("iqm", 24, 6, 512, 128, 9, "mixed_iq", True, 93)
    L = synth.make_layer(cfg, 0)
    assert {f for f in L.fmts} == {(synth.Q6_K, synth.Q8_0), (synth.IQ4_XS, synth.IQ4_NL),
                                    (synth.IQ3_XXS, synth.MXFP4)}
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, cfg.hidden, cfg.inter, grid=_grid())
    # decode rows: AUTO takes the streaming GEMV kernels, which decode the IQ formats too
    assert M.ffn_path(table, cfg.tokens, cfg.k) == M.PATH_GEMV
    assert M.gemv_kernels(table, cfg.tokens, cfg.k) == M.GEMV_STREAMING
    ref = offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k)
    assert_parity(M.ffn_forward(table, x, logits, cfg.k).cpu().numpy(), ref, "mixed_iq AUTO")
    opt = M.make_options(n_experts=cfg.n_experts, path=M.PATH_GEMV)
    assert_parity(M.ffn_forward(table, x, logits, cfg.k, options=opt).cpu().numpy(), ref, "mixed_iq GEMV")
    # the tier decomposition on the GPU: the layer is the sum of its format-masked runs
    parts = 0
    for f in (synth.Q6_K, synth.IQ4_XS, synth.IQ3_XXS):
        o = M.make_options(n_experts=cfg.n_experts, format_mask=1 << f)
        parts = parts + M.ffn_forward(table, x, logits, cfg.k, options=o).cpu().numpy().astype(np.float64)
    assert_parity(parts, ref, "sum of the three tiers")


def test_iq3_table_needs_grid(M):
    cfg = synth.LayerConfig("iqg", 4, 2, 256, 64, 2, "q4k", True, 95)
    L = _with_formats(synth.make_layer(cfg, 0, with_weights=False), synth.IQ3_XXS, synth.MXFP4)
    experts, x, logits = host_layer_to_device(L)
    with pytest.raises(M.MoeError) as ei:
        M.WeightTable(experts, cfg.hidden, cfg.inter)
    assert ei.value.code == 1


@pytest.mark.parametrize("gu,dn", [(synth.IQ4_XS, synth.IQ4_NL), (synth.IQ3_XXS, synth.MXFP4),
                                   (synth.IQ4_NL, synth.IQ4_NL), (synth.Q4_K, synth.IQ4_NL)])
@pytest.mark.parametrize("T", [1, 6, 16])
def test_iq_formats_streaming(M, gu, dn, T):
    """Each IQ format on the streaming GEMV kernels (1, 6 and 16 rows; two
    64-column groups per lane with H = 4096 up to 6 rows, whose staged
    activations leave room for the ring), against the oracle and bit for bit
    on a second call."""
    H = 4096 if T <= 6 else 2048
    cfg = synth.LayerConfig("iqs", 12, 3, H, 128, T, "q4k", True, 97 + gu + 10 * dn + T)
    L = _with_formats(synth.make_layer(cfg, 0, with_weights=False), gu, dn)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, cfg.hidden, cfg.inter, grid=_grid())
    opt = M.make_options(n_experts=cfg.n_experts, path=M.PATH_GEMV)
    assert M.gemv_kernels(table, T, cfg.k) == M.GEMV_STREAMING
    ws = M.Workspace(table, T, cfg.k, path=M.PATH_GEMV)
    out = M.ffn_forward(table, x, logits, cfg.k, ws=ws, options=opt).cpu().numpy()
    assert ws.read_status() == 0
    assert_parity(out, offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k), f"stream gu {gu} dn {dn} T={T}")
    again = M.ffn_forward(table, x, logits, cfg.k, ws=ws, options=opt).cpu().numpy()
    assert np.array_equal(again, out)


def test_iq3_streaming_full_byte_grid(M):
    """IQ3_XXS grid magnitudes up to 255 (a caller's grid may hold any byte):
    the streaming kernels take them as unsigned bytes."""
    cfg = synth.LayerConfig("iqb", 8, 2, 512, 64, 4, "q4k", True, 131)
    L = _with_formats(synth.make_layer(cfg, 0, with_weights=False), synth.IQ3_XXS, synth.Q8_0)
    rng = np.random.default_rng(5)
    grid_np = rng.integers(0, 256, size=(256, 4), dtype=np.uint32)
    grid_np = (grid_np[:, 0] | (grid_np[:, 1] << 8) | (grid_np[:, 2] << 16) | (grid_np[:, 3] << 24)).astype(np.uint32)
    for ex in L.experts:
        for mat in ex.values():
            if mat.fmt == synth.IQ3_XXS:
                mat.grid = grid_np
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, cfg.hidden, cfg.inter, grid=torch.from_numpy(grid_np.view(np.int32).copy()).cuda())
    opt = M.make_options(n_experts=cfg.n_experts, path=M.PATH_GEMV)
    assert M.gemv_kernels(table, cfg.tokens, cfg.k) == M.GEMV_STREAMING
    out = M.ffn_forward(table, x, logits, cfg.k, options=opt).cpu().numpy()
    ref = offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k)
    assert_parity(out, ref, "IQ3_XXS grid with bytes up to 255")


@pytest.mark.parametrize("name,paths", [("mtp6_iq", ("TENSOR", "GEMV")), ("prefill2048_iq", ("TENSOR",))])
def test_iq_full_size(M, name, paths):
    from synth import gpu as sgpu
    cfg = synth.CONFIGS[name]
    DL = sgpu.make_device_layer(cfg, 0)
    table = M.WeightTable(DL.experts, cfg.hidden, cfg.inter, grid=DL.grid)
    ref = oracle_full_layer(cfg, DL)
    for path in paths:
        p = getattr(M, "PATH_" + path)
        opt = M.make_options(n_experts=cfg.n_experts, path=p)
        ws = M.Workspace(table, cfg.tokens, cfg.k, path=p)
        out = M.ffn_forward(table, DL.x_bf16, DL.logits, cfg.k, ws=ws, options=opt).cpu().numpy()
        assert ws.read_status() == 0
        assert_parity(out, ref, f"{name} {path}")
    del table, DL
    torch.cuda.empty_cache()
