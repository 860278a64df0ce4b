"""GPU parity of the tensor-core path (MOE_PATH_TENSOR: TMEM-resident
dequantised weights, tcgen05 grouped GEMMs) against the fp64 oracle, through
the C ABI, with the tolerance of the other GPU tests.

Small layers cover every format alone and mixed, experts with more rows than
one 128-row chunk, reduction lengths that end in a partial 256-wide raw
stage, and a tiny layer forced onto the path. The full-size layers (16-row
and 6-row decode, the 2048-token prefill chunk) are checked on every token
against the oracle, which evaluates them expert by expert over a process
pool. Also: routing
bit-exact, run-to-run bitwise reproducibility, tier decomposition, empty
selections and the device status word."""
import numpy as np
import pytest
import torch

import synth
from oracle import bucket as obucket
from oracle import ffn as offn
from oracle import router as orouter
from tests.gpu_util import assert_parity, ensure_built, host_layer_to_device, oracle_full_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    ensure_built()
    import quantized_moe_expert_route_gb300 as M
    M.load()
    return M


def run_tensor(M, L, options=None, table=None, dev=None):
    cfg = L.cfg
    experts, x, logits = dev if dev is not None else host_layer_to_device(L)
    table = table or M.WeightTable(experts, cfg.hidden, cfg.inter)
    opt = options or M.make_options(n_experts=cfg.n_experts, path=M.PATH_TENSOR)
    assert M.ffn_path(table, cfg.tokens, cfg.k, opt) == M.PATH_TENSOR
    ws = M.Workspace(table, cfg.tokens, cfg.k, path=M.PATH_TENSOR)
    out = M.ffn_forward(table, x, logits, cfg.k, ws=ws, options=opt)
    torch.cuda.synchronize()
    return out.cpu().numpy(), table, ws


@pytest.mark.parametrize("tiers,E,k,H,I,T", [
    ("q8_0", 8, 2, 256, 128, 4),       # the tiny layer's shape, forced onto the tensor path
    ("q4k", 16, 4, 256, 64, 100),
    ("mixed", 16, 4, 512, 128, 120),   # Q6_K, Q4_K, MXFP4 gate/up; Q8_0, MXFP4 down
    ("mixed", 4, 2, 512, 192, 300),    # ~150 rows per expert: two chunks each; down K = 192 (< 256)
    ("q8_0", 12, 3, 384, 64, 37),      # H = 3 x 128
    ("mixed", 40, 8, 1024, 320, 97),   # down K = 320: a partial second raw stage
    ("q8_0", 64, 8, 256, 64, 400),     # 3200 pairs: the many-pair (multi-CTA) bucketing
])
def test_tensor_small(M, tiers, E, k, H, I, T):
    cfg = synth.LayerConfig("tc", E, k, H, I, T, tiers, tiers != "q8_0", 1000 + 7 * T + E)
    L = synth.make_layer(cfg, 0)
    out, table, ws = run_tensor(M, L)
    ref = offn.moe_ffn(L.experts, L.x_bf16, L.logits, k)
    assert_parity(out, ref, f"tensor {tiers} E{E} k{k} H{H} I{I} T{T}")
    # routing and bucketing are the oracle's, bit for bit
    rid, rw, _ = orouter.route_topk(L.logits, k)
    R = ws.routing()
    np.testing.assert_array_equal(R["ids"].cpu().numpy(), rid)
    roff, rpairs, rpos, ract, _ = obucket.bucket(rid, E)
    np.testing.assert_array_equal(R["offsets"].cpu().numpy(), roff)
    np.testing.assert_array_equal(R["pos"].cpu().numpy(), rpos)
    assert ws.read_status() == 0


def test_tensor_reproducible_and_tiers(M):
    cfg = synth.LayerConfig("tc2", 24, 6, 512, 128, 150, "mixed", True, 4242)
    L = synth.make_layer(cfg, 0)
    dev = host_layer_to_device(L)
    a, table, _ = run_tensor(M, L, dev=dev)
    b, _, _ = run_tensor(M, L, dev=dev, table=table)
    assert np.array_equal(a, b), "tensor path not bitwise reproducible"
    # the layer equals the sum of its format-masked runs
    parts = 0
    for f in (synth.Q4_K, synth.Q6_K, synth.MXFP4):
        opt = M.make_options(n_experts=cfg.n_experts, path=M.PATH_TENSOR, format_mask=1 << f)
        o, _, _ = run_tensor(M, L, options=opt, table=table, dev=dev)
        parts = parts + o.astype(np.float64)
    ref = offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k)
    assert_parity(parts, ref, "sum of format-masked tensor runs")
    # an empty expert range selects nothing: the output is exactly zero
    opt = M.make_options(n_experts=cfg.n_experts, path=M.PATH_TENSOR, expert_lo=5, expert_hi=5)
    z, _, ws = run_tensor(M, L, options=opt, table=table, dev=dev)
    assert not z.any()
    assert ws.read_status() == 0


def full_tensor(M, name, layer=0):
    from synth import gpu as sgpu
    cfg = synth.CONFIGS[name]
    DL = sgpu.make_device_layer(cfg, layer)
    table = M.WeightTable(DL.experts, cfg.hidden, cfg.inter)
    opt = M.make_options(n_experts=cfg.n_experts, path=M.PATH_TENSOR)
    ws = M.Workspace(table, cfg.tokens, cfg.k, path=M.PATH_TENSOR)
    out = M.ffn_forward(table, DL.x_bf16, DL.logits, cfg.k, ws=ws, options=opt).cpu().numpy()
    assert ws.read_status() == 0
    return cfg, DL, table, out


@pytest.mark.parametrize("name", ["decode16", "mtp6"])
def test_tensor_full_decode_shapes(M, name):
    cfg, DL, table, out = full_tensor(M, name)
    assert_parity(out, oracle_full_layer(cfg, DL), f"tensor {name}")
    del table, DL
    torch.cuda.empty_cache()


def test_tensor_full_prefill(M):
    """The 2048-token mixed-tier chunk, as the benchmark runs it: every token
    (all 512 experts, with the rows of the hot experts past the first 128-row
    chunk) against the oracle, on the tensor path and on the grouped GEMV
    path; per-expert rows reach the second chunk."""
    cfg, DL, table, out = full_tensor(M, "prefill2048")
    assert M.ffn_path(table, cfg.tokens, cfg.k) == M.PATH_TENSOR   # AUTO takes it
    routing = M.Workspace(table, cfg.tokens, cfg.k)
    M.ffn_forward(table, DL.x_bf16, DL.logits, cfg.k, ws=routing)
    counts = np.diff(routing.routing()["offsets"].cpu().numpy())
    assert (counts > 0).all() and counts.max() > 128
    ref = oracle_full_layer(cfg, DL)
    assert_parity(out, ref, "tensor prefill2048 (all tokens)")
    opt = M.make_options(n_experts=cfg.n_experts, path=M.PATH_GEMV)
    gemv = M.ffn_forward(table, DL.x_bf16, DL.logits, cfg.k, options=opt).cpu().numpy()
    assert_parity(gemv, ref, "gemv prefill2048 (all tokens)")
    del table, DL
    torch.cuda.empty_cache()
