"""GPU parity of the whole layer (moe_ffn_forward through the C ABI) against
the fp64 oracle: relative L2 error <= 1e-3 and max abs error <= 1e-2 * RMS.

Every layer is compared on every output element, the full-size layers (512
experts, top-10, 2048/640: 1, 16, 6 and 2048 tokens) included, in the launch
configuration the benchmark times; the oracle evaluates those expert by expert
over a process pool.
Also: tier decomposition and expert-range splits on the GPU, run-to-run
bitwise reproducibility, permutation of the expert table, device status
flags, guard bands around the output and the workspace, and argument errors.
"""
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


def run_layer(M, L, k=None, options=None, T=None):
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, L.cfg.hidden, L.cfg.inter)
    out = M.ffn_forward(table, x, logits, k or L.cfg.k, options=options)
    torch.cuda.synchronize()
    return out.cpu().numpy(), table, x, logits


def small_cfg(tiers="mixed", E=16, k=4, H=256, I=64, T=5, seed=11, bias=True):
    return synth.LayerConfig("small", E, k, H, I, T, tiers, bias, seed)


def test_tiny_config(M):
    L = synth.make_layer(synth.CONFIGS["tiny"], 0)
    out, *_ = run_layer(M, L)
    ref = offn.moe_ffn(L.experts, L.x_bf16, L.logits, L.cfg.k)
    assert_parity(out, ref, "tiny")


@pytest.mark.parametrize("tiers,T", [("q8_0", 1), ("q4k", 3), ("mixed", 7), ("mixed", 33), ("mixed", 96),
                                     ("q4k", 130)])
def test_small_layers(M, tiers, T):
    L = synth.make_layer(small_cfg(tiers=tiers, T=T, seed=T), 0)
    out, *_ = run_layer(M, L)
    ref = offn.moe_ffn(L.experts, L.x_bf16, L.logits, L.cfg.k)
    assert_parity(out, ref, f"{tiers} T={T}")


def test_ragged_shapes(M):
    # I not a multiple of the 16-row gate/up tile nor of the 32-row down tile;
    # H spans several Q4_K super-blocks; k odd.
    cfg = synth.LayerConfig("ragged", 9, 3, 512, 96 + 32, 11, "mixed", True, 5)
    L = synth.make_layer(cfg, 0)
    out, *_ = run_layer(M, L)
    assert_parity(out, offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k), "ragged")
    cfg = synth.LayerConfig("ragged2", 5, 5, 256, 32, 2, "q8_0", False, 6)   # k = E, I = one block
    L = synth.make_layer(cfg, 0)
    out, *_ = run_layer(M, L)
    assert_parity(out, offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k), "k=E")


def test_not_renormalized(M):
    L = synth.make_layer(small_cfg(T=6, seed=21), 0)
    opt = M.make_options(renormalize=False, n_experts=L.cfg.n_experts)
    out, *_ = run_layer(M, L, options=opt)
    assert_parity(out, offn.moe_ffn(L.experts, L.x_bf16, L.logits, L.cfg.k, renormalize=False), "no renorm")


def test_tier_decomposition_and_range_split(M):
    L = synth.make_layer(small_cfg(E=20, k=5, T=9, seed=31), 0)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, L.cfg.hidden, L.cfg.inter)
    E, k = L.cfg.n_experts, L.cfg.k
    full = M.ffn_forward(table, x, logits, k).cpu().numpy().astype(np.float64)
    ref = offn.moe_ffn(L.experts, L.x_bf16, L.logits, k)
    assert_parity(full, ref, "full")
    parts = np.zeros_like(full)
    for f in sorted({fm for fm, _ in L.fmts}):
        opt = M.make_options(format_mask=1 << f, n_experts=E)
        part = M.ffn_forward(table, x, logits, k, options=opt).cpu().numpy()
        assert_parity(part, offn.moe_ffn(L.experts, L.x_bf16, L.logits, k, format_mask=1 << f), f"tier {f}")
        parts += part
    assert_parity(parts, ref, "sum of tiers")
    lo = M.ffn_forward(table, x, logits, k, options=M.make_options(expert_lo=0, expert_hi=8, n_experts=E))
    hi = M.ffn_forward(table, x, logits, k, options=M.make_options(expert_lo=8, expert_hi=E, n_experts=E))
    assert_parity(lo.cpu().numpy() + hi.cpu().numpy(), ref, "range split")


def test_bitwise_reproducible(M):
    L = synth.make_layer(small_cfg(T=40, seed=41), 0)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, L.cfg.hidden, L.cfg.inter)
    ws = M.Workspace(table, 40, L.cfg.k)
    a = M.ffn_forward(table, x, logits, L.cfg.k, ws=ws).clone()
    b = M.ffn_forward(table, x, logits, L.cfg.k, ws=ws).clone()
    assert torch.equal(a, b)


def test_permuted_table(M):
    L = synth.make_layer(small_cfg(E=12, k=3, T=8, seed=51), 0)
    experts, x, logits = host_layer_to_device(L)
    t1 = M.WeightTable(experts, L.cfg.hidden, L.cfg.inter)
    a = M.ffn_forward(t1, x, logits, L.cfg.k)
    perm = np.random.default_rng(52).permutation(12)
    t2 = M.WeightTable([experts[int(p)] for p in perm], L.cfg.hidden, L.cfg.inter)
    b = M.ffn_forward(t2, x, logits[:, torch.from_numpy(perm).cuda()].contiguous(), L.cfg.k)
    # the schedule depends only on each expert's data, so the result is bit-identical
    assert torch.equal(a, b)


def test_status_and_nonfinite(M):
    L = synth.make_layer(small_cfg(T=4, seed=61), 0)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, L.cfg.hidden, L.cfg.inter)
    ws = M.Workspace(table, 4, L.cfg.k)
    M.ffn_forward(table, x, logits, L.cfg.k, ws=ws)
    assert ws.read_status() == 0
    lg = logits.clone()
    lg[1, 3] = float("nan")
    lg[2, :] = float("-inf")
    out = M.ffn_forward(table, x, lg, L.cfg.k, ws=ws).cpu().numpy()
    assert ws.read_status() & M.FLAG_NONFINITE_LOGIT
    assert ws.read_status() == 0          # read clears
    lgh = lg.cpu().numpy()
    ref = offn.moe_ffn(L.experts, L.x_bf16, lgh, L.cfg.k)
    assert np.all(out[2] == 0) and np.all(ref[2] == 0)
    assert_parity(out, ref, "nonfinite")


def test_guard_bands(M):
    """Canary bytes around the output and the workspace survive a forward."""
    L = synth.make_layer(small_cfg(T=13, seed=71), 0)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, L.cfg.hidden, L.cfg.inter)
    T, H, k = 13, L.cfg.hidden, L.cfg.k
    G = 4096
    ws_bytes = M.Workspace(table, T, k).nbytes
    big = torch.full((G + ws_bytes + G,), 0xA5, dtype=torch.uint8, device="cuda")
    ws = M.Workspace.__new__(M.Workspace)
    ws.buf, ws.nbytes = big[G:G + ws_bytes], ws_bytes
    torch.zeros(256, dtype=torch.uint8, device="cuda")
    ws.buf[:256].zero_()
    outbig = torch.full((T * H + 2 * 1024,), 7.0, dtype=torch.float32, device="cuda")
    out = outbig[1024:1024 + T * H].view(T, H)
    M.ffn_forward(table, x, logits, k, out=out, ws=ws)
    torch.cuda.synchronize()
    assert torch.all(big[:G] == 0xA5) and torch.all(big[G + ws_bytes:] == 0xA5)
    assert torch.all(outbig[:1024] == 7.0) and torch.all(outbig[1024 + T * H:] == 7.0)
    assert_parity(out.cpu().numpy(), offn.moe_ffn(L.experts, L.x_bf16, L.logits, k), "guarded")


def test_argument_errors(M):
    L = synth.make_layer(small_cfg(T=2, seed=81), 0)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, L.cfg.hidden, L.cfg.inter)
    ws = M.Workspace(table, 2, L.cfg.k)
    with pytest.raises(M.MoeError) as ei:
        M.ffn_forward(table, x, logits, L.cfg.n_experts + 1, ws=ws)   # k > E
    assert ei.value.code == 1
    with pytest.raises(M.MoeError) as ei:
        M.ffn_forward(table, x, logits, 0, ws=ws)
    assert ei.value.code == 1
    bad_opt = M.make_options(expert_lo=3, expert_hi=2, n_experts=L.cfg.n_experts)
    with pytest.raises(M.MoeError) as ei:
        M.ffn_forward(table, x, logits, L.cfg.k, ws=ws, options=bad_opt)
    assert ei.value.code == 1
    small = M.Workspace(table, 1, L.cfg.k)
    with pytest.raises(M.MoeError) as ei:
        M.ffn_forward(table, x, logits, L.cfg.k, ws=small)
    assert ei.value.code == 5
    bad = [dict(e) for e in experts]
    fmt, rows, cols, stride, data = bad[0]["gate"]
    bad[0]["gate"] = (fmt, rows, cols + 32, stride, data)
    with pytest.raises(M.MoeError) as ei:
        M.WeightTable(bad, L.cfg.hidden, L.cfg.inter)
    assert ei.value.code == 2
    bad[0]["gate"] = (9, rows, cols, stride, data)
    with pytest.raises(M.MoeError) as ei:
        M.WeightTable(bad, L.cfg.hidden, L.cfg.inter)
    assert ei.value.code == 3
    bad[0]["gate"] = (fmt, rows, cols, stride + 8, data)
    with pytest.raises(M.MoeError) as ei:
        M.WeightTable(bad, L.cfg.hidden, L.cfg.inter)
    assert ei.value.code == 2
    # gate and up in different formats
    bad[0]["gate"] = experts[0]["gate"]
    f2 = synth.Q8_0 if fmt != synth.Q8_0 else synth.MXFP4
    m2 = synth.gen_matrix(f2, rows, cols, 5)
    bad[0]["up"] = (f2, rows, cols, m2.stride, torch.from_numpy(m2.data).cuda())
    with pytest.raises(M.MoeError) as ei:
        M.WeightTable(bad, L.cfg.hidden, L.cfg.inter)
    assert ei.value.code == 3


def test_zero_tokens(M):
    L = synth.make_layer(small_cfg(T=0, seed=91), 0)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, L.cfg.hidden, L.cfg.inter)
    out = M.ffn_forward(table, x, logits, L.cfg.k)
    assert out.shape == (0, L.cfg.hidden)


# --------------------------------------------------------------- full size
def full_layer_parity(M, name, tokens_to_check=None, layer=0, paths=(None,)):
    """AUTO (None) and any explicitly requested paths against one oracle result."""
    from synth import gpu as sgpu
    cfg = synth.CONFIGS[name]
    DL = sgpu.make_device_layer(cfg, layer)
    table = M.WeightTable(DL.experts, cfg.hidden, cfg.inter)
    outs = {}
    for path in paths:
        opt = None if path is None else M.make_options(n_experts=cfg.n_experts, path=path)
        ws = M.Workspace(table, cfg.tokens, cfg.k, path=path or 0)
        outs[path] = M.ffn_forward(table, DL.x_bf16, DL.logits, cfg.k, ws=ws, options=opt).cpu().numpy()
    tok = list(range(cfg.tokens)) if tokens_to_check is None else tokens_to_check
    ref = oracle_full_layer(cfg, DL, None if tokens_to_check is None else tok)
    for path, out in outs.items():
        assert_parity(out[tok], ref, f"{name} path {path}")
    del table, DL
    torch.cuda.empty_cache()


def test_full_decode1(M):
    full_layer_parity(M, "decode1")
    full_layer_parity(M, "decode1", layer=7)


def test_full_decode16(M):
    full_layer_parity(M, "decode16", paths=(None, M.PATH_GEMV, M.PATH_TENSOR))


def test_full_mtp6(M):
    full_layer_parity(M, "mtp6", paths=(None, M.PATH_GEMV))


def test_full_prefill(M):
    """All 2048 tokens (every one of the 512 experts, the hot experts' rows
    past the first 128-row chunk included) against the oracle."""
    full_layer_parity(M, "prefill2048")


# --------------------------------------------------------------- fused decode path
def run_path(M, L, path, k=None, options=None):
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, L.cfg.hidden, L.cfg.inter)
    opt = options or M.make_options(n_experts=L.cfg.n_experts, path=path)
    assert M.ffn_path(table, L.cfg.tokens, k or L.cfg.k, opt) == path
    ws = M.Workspace(table, L.cfg.tokens, k or L.cfg.k)
    out = M.ffn_forward(table, x, logits, k or L.cfg.k, ws=ws, options=opt)
    torch.cuda.synchronize()
    return out.cpu().numpy(), table, ws


@pytest.mark.parametrize("T,k,E,H,I", [(1, 10, 64, 2048, 640), (2, 4, 16, 256, 64), (3, 8, 40, 512, 96),
                                       (6, 10, 512, 2048, 640), (1, 1, 4, 256, 32), (5, 12, 20, 1024, 1024)])
def test_fused_decode_small(M, T, k, E, H, I):
    cfg = synth.LayerConfig("fz", E, k, H, I, T, "q4k", True, 7 * T + E)
    L = synth.make_layer(cfg, 0)
    out, table, ws = run_path(M, L, M.PATH_FUSED)
    ref = offn.moe_ffn(L.experts, L.x_bf16, L.logits, k)
    assert_parity(out, ref, f"fused T={T} E={E}")
    # the routing it publishes is the oracle's, bit for bit
    from oracle import router as orouter, bucket as obucket
    rid, rw, _ = orouter.route_topk(L.logits, k)
    R = ws.routing()
    np.testing.assert_array_equal(R["ids"].cpu().numpy(), rid)
    roff, rpairs, rpos, ract, _ = obucket.bucket(rid, E)
    np.testing.assert_array_equal(R["offsets"].cpu().numpy(), roff)
    act = R["active"].cpu().numpy()
    np.testing.assert_array_equal(act[1:1 + act[0]], ract)
    np.testing.assert_array_equal(R["pos"].cpu().numpy(), rpos)
    assert ws.read_status() == 0


def test_fused_decode_filters_and_reproducible(M):
    cfg = synth.LayerConfig("ff", 24, 6, 512, 128, 4, "q4k", True, 99)
    L = synth.make_layer(cfg, 0)
    E, k = cfg.n_experts, cfg.k
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, cfg.hidden, cfg.inter)
    ref = offn.moe_ffn(L.experts, L.x_bf16, L.logits, k)
    ws = M.Workspace(table, cfg.tokens, k)
    full = M.ffn_forward(table, x, logits, k, ws=ws, options=M.make_options(n_experts=E, path=M.PATH_FUSED))
    again = M.ffn_forward(table, x, logits, k, ws=ws, options=M.make_options(n_experts=E, path=M.PATH_FUSED))
    assert torch.equal(full, again)
    assert_parity(full.cpu().numpy(), ref, "fused full")
    lo = M.ffn_forward(table, x, logits, k, ws=ws,
                       options=M.make_options(expert_lo=0, expert_hi=10, n_experts=E, path=M.PATH_FUSED))
    hi = M.ffn_forward(table, x, logits, k, ws=ws,
                       options=M.make_options(expert_lo=10, expert_hi=E, n_experts=E, path=M.PATH_FUSED))
    assert_parity(lo.cpu().numpy() + hi.cpu().numpy(), ref, "fused range split")
    nr = M.ffn_forward(table, x, logits, k, ws=ws,
                       options=M.make_options(renormalize=False, n_experts=E, path=M.PATH_FUSED))
    assert_parity(nr.cpu().numpy(), offn.moe_ffn(L.experts, L.x_bf16, L.logits, k, renormalize=False), "fused nr")
    lg = logits.clone()
    lg[2, 5] = float("nan")
    M.ffn_forward(table, x, lg, k, ws=ws, options=M.make_options(n_experts=E, path=M.PATH_FUSED))
    assert ws.read_status() & M.FLAG_NONFINITE_LOGIT


@pytest.mark.parametrize("mode", ["halves", "equal", "two_values"])
def test_fused_decode_tied_logits(M, mode):
    """Tied router logits: the lower expert index wins, as in the oracle.
    Coarse logits leave few candidates per slice; all-equal logits leave
    every candidate (the counting-rank path of the kernel's top-k)."""
    cfg = synth.LayerConfig("tie", 96, 8, 256, 64, 3, "q4k", True, 31)
    L = synth.make_layer(cfg, 0)
    if mode == "halves":
        L.logits = (np.round(L.logits * 2) / 2).astype(np.float32)
    elif mode == "equal":
        L.logits = np.full_like(L.logits, 0.25)
    else:
        L.logits = np.where(L.logits > 0.5, 1.0, -1.0).astype(np.float32)
    out, table, ws = run_path(M, L, M.PATH_FUSED)
    ref = offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k)
    assert_parity(out, ref, f"fused tied logits ({mode})")
    from oracle import router as orouter
    rid, rw, _ = orouter.route_topk(L.logits, cfg.k)
    R = ws.routing()
    np.testing.assert_array_equal(R["ids"].cpu().numpy(), rid)
    np.testing.assert_allclose(R["weights"].cpu().numpy(), rw, rtol=4e-6, atol=0)
    assert ws.read_status() == 0


def test_fused_path_rejects_ineligible(M):
    L = synth.make_layer(small_cfg(tiers="mixed", T=3, seed=5), 0)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, L.cfg.hidden, L.cfg.inter)
    opt = M.make_options(n_experts=L.cfg.n_experts, path=M.PATH_FUSED)
    assert M.ffn_path(table, 3, L.cfg.k, opt) == -1
    with pytest.raises(M.MoeError) as ei:
        M.ffn_forward(table, x, logits, L.cfg.k, options=opt)
    assert ei.value.code == 8
    # AUTO takes the streaming GEMV kernels for this decode batch
    assert M.ffn_path(table, 3, L.cfg.k) == M.PATH_GEMV
    assert M.gemv_kernels(table, 3, L.cfg.k) == M.GEMV_STREAMING
    assert M.gemv_kernels(table, 17, L.cfg.k) == M.GEMV_TILED


@pytest.mark.parametrize("tiers,T,H,I", [("q8_0", 1, 256, 64), ("q4k", 3, 256, 64), ("mixed", 7, 256, 64),
                                         ("mixed", 33, 512, 96 + 32), ("mixed", 96, 256, 64), ("q4k", 130, 256, 64)])
def test_gemv_path_small(M, tiers, T, H, I):
    """The grouped GEMV path requested explicitly, on shapes AUTO sends elsewhere."""
    cfg = synth.LayerConfig("gv", 16, 4, H, I, T, tiers, True, 900 + T)
    L = synth.make_layer(cfg, 0)
    opt = M.make_options(n_experts=cfg.n_experts, path=M.PATH_GEMV)
    out, *_ = run_layer(M, L, options=opt)
    assert_parity(out, offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k), f"gemv {tiers} T={T}")


@pytest.mark.parametrize("tiers,T,H,I", [("q8_0", 2, 256, 64), ("q4k", 5, 512, 96), ("mixed", 16, 256, 64),
                                         ("mixed", 6, 512, 160), ("q4k", 8, 4096, 64), ("q8_0", 16, 2048, 32),
                                         ("mixed", 1, 1024, 32)])
def test_stream_kernels_small(M, tiers, T, H, I):
    """The streaming decode kernels of the GEMV path (up to 16 rows): chunks of
    1, 2 and 4 row pairs, 1 and 2 column groups per lane, one-block rows,
    every gate/up format and both down formats."""
    cfg = synth.LayerConfig("sg", 16, 4, H, I, T, tiers, True, 700 + T + H + I)
    L = synth.make_layer(cfg, 0)
    opt = M.make_options(n_experts=cfg.n_experts, path=M.PATH_GEMV)
    out, table, x, logits = run_layer(M, L, options=opt)
    assert_parity(out, offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k), f"stream {tiers} T={T} H={H} I={I}")
    again = M.ffn_forward(table, x, logits, cfg.k, options=opt)
    assert np.array_equal(again.cpu().numpy(), out)


@pytest.mark.parametrize("tiers,T,H,I", [("q8_0", 4, 256, 512), ("q4k", 3, 256, 544), ("mixed", 5, 256, 576),
                                         ("q4k", 2, 512, 1056), ("mixed", 6, 512, 1024)])
def test_stream_down_block_groups(M, tiers, T, H, I):
    """The streaming down kernel's blocks in groups of 16 (I = 512 .. 1056:
    one or two whole groups, with 0, 1 or 2 blocks after them), Q8_0 and
    MXFP4 down rows, against the oracle and bit for bit on a second call."""
    cfg = synth.LayerConfig("sgd", 16, 4, H, I, T, tiers, True, 810 + T + I)
    L = synth.make_layer(cfg, 0)
    opt = M.make_options(n_experts=cfg.n_experts, path=M.PATH_GEMV)
    out, table, x, logits = run_layer(M, L, options=opt)
    assert M.gemv_kernels(table, T, cfg.k) == M.GEMV_STREAMING
    assert_parity(out, offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k), f"stream down {tiers} T={T} I={I}")
    again = M.ffn_forward(table, x, logits, cfg.k, options=opt)
    assert np.array_equal(again.cpu().numpy(), out)


@pytest.mark.parametrize("tiers,T,H,I", [("q4k", 17, 512, 128), ("q4k", 24, 256, 64), ("q8_0", 32, 512, 96),
                                         ("q4k", 32, 2048, 64)])
def test_stream_kernels_up_to_32_rows(M, tiers, T, H, I):
    """The streaming kernels take up to 32 rows when every gate/up matrix is
    Q8_0 or Q4_K (17, 24 and 32 rows here), and AUTO takes them there."""
    cfg = synth.LayerConfig("sg32", 24, 6, H, I, T, tiers, True, 770 + T + H)
    L = synth.make_layer(cfg, 0)
    opt = M.make_options(n_experts=cfg.n_experts, path=M.PATH_GEMV)
    out, table, x, logits = run_layer(M, L, options=opt)
    assert M.gemv_kernels(table, T, cfg.k) == M.GEMV_STREAMING
    assert M.ffn_path(table, T, cfg.k) == M.PATH_GEMV
    assert_parity(out, offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k), f"stream {tiers} T={T}")


def test_stream_row_limit_by_format(M):
    """With Q6_K or MXFP4 gate/up the streaming kernels stop at 16 rows: AUTO
    takes the tensor path above (it measured faster there)."""
    L = synth.make_layer(small_cfg(tiers="mixed", E=24, k=6, H=512, I=128, T=20, seed=31), 0)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, L.cfg.hidden, L.cfg.inter)
    assert M.gemv_kernels(table, 16, L.cfg.k) == M.GEMV_STREAMING
    assert M.gemv_kernels(table, 17, L.cfg.k) == M.GEMV_TILED
    assert M.ffn_path(table, 20, L.cfg.k) == M.PATH_TENSOR


def test_full_decode24_streaming(M):
    """The 512-expert Q4_K layer at 24 rows on AUTO (the streaming kernels),
    every token against the oracle."""
    from synth import gpu as sgpu
    cfg = synth.LayerConfig("decode24", 512, 10, 2048, 640, 24, "q4k", True, 12524)
    DL = sgpu.make_device_layer(cfg, 0)
    table = M.WeightTable(DL.experts, cfg.hidden, cfg.inter)
    assert M.ffn_path(table, 24, cfg.k) == M.PATH_GEMV and M.gemv_kernels(table, 24, cfg.k) == M.GEMV_STREAMING
    ws = M.Workspace(table, 24, cfg.k)
    out = M.ffn_forward(table, DL.x_bf16, DL.logits, cfg.k, ws=ws).cpu().numpy()
    assert ws.read_status() == 0
    assert_parity(out, oracle_full_layer(cfg, DL), "decode24 streaming")
    del table, DL
    torch.cuda.empty_cache()


def test_full_decode1_gemv_path(M):
    """The general grouped GEMV path on the full-size single-token layer."""
    from synth import gpu as sgpu
    cfg = synth.CONFIGS["decode1"]
    DL = sgpu.make_device_layer(cfg, 2)
    table = M.WeightTable(DL.experts, cfg.hidden, cfg.inter)
    opt = M.make_options(n_experts=cfg.n_experts, path=M.PATH_GEMV)
    out = M.ffn_forward(table, DL.x_bf16, DL.logits, cfg.k, options=opt).cpu().numpy()
    fused = M.ffn_forward(table, DL.x_bf16, DL.logits, cfg.k).cpu().numpy()
    assert M.ffn_path(table, 1, cfg.k) == M.PATH_FUSED
    lazy = synth.LazyExperts(cfg, DL.seed, DL.fmts)
    ref = offn.moe_ffn(lazy, DL.x_host, DL.logits_host, cfg.k, gate_formats=lazy.gate_formats())
    assert_parity(out, ref, "decode1 gemv")
    assert_parity(fused, ref, "decode1 fused")


def test_uniform_layout_matches_descriptor_table(M):
    """Experts stored as one strided tensor (descriptors computed in the
    kernel) and the same bytes in separate allocations (descriptors read from
    the table) give bit-identical outputs on every path."""
    from synth import gpu as sgpu
    cfg = synth.LayerConfig("uni", 48, 6, 512, 128, 3, "q4k", True, 123)
    DL = sgpu.make_device_layer(cfg, 0)
    t_uni = M.WeightTable(DL.experts, cfg.hidden, cfg.inter)
    assert t_uni.c.uniform_layout == 1
    copies = [{n: (f, r, cc, st, v.clone()) for n, (f, r, cc, st, v) in ex.items()} for ex in DL.experts]
    t_sep = M.WeightTable(copies, cfg.hidden, cfg.inter)
    assert t_sep.c.uniform_layout == 0
    for path in (M.PATH_FUSED, M.PATH_GEMV):
        opt = M.make_options(n_experts=cfg.n_experts, path=path)
        a = M.ffn_forward(t_uni, DL.x_bf16, DL.logits, cfg.k, options=opt)
        b = M.ffn_forward(t_sep, DL.x_bf16, DL.logits, cfg.k, options=opt)
        assert torch.equal(a, b), path
    lazy = synth.LazyExperts(cfg, DL.seed, DL.fmts)
    ref = offn.moe_ffn(lazy, DL.x_host, DL.logits_host, cfg.k, gate_formats=lazy.gate_formats())
    assert_parity(a.cpu().numpy(), ref, "uniform layout")


@pytest.mark.parametrize("tiers,T,path", [("q4k", 1, "FUSED"), ("mixed", 6, "GEMV"), ("mixed", 40, "TENSOR")])
def test_timing_events_leave_results_unchanged(M, tiers, T, path):
    """The profiling events (before gate/up, between gate/up and down, after
    down) are recorded on every path and change nothing in the result."""
    cfg = synth.LayerConfig("ev", 16, 4, 512, 128, T, tiers, True, 880 + T)
    L = synth.make_layer(cfg, 0)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, cfg.hidden, cfg.inter)
    p = getattr(M, "PATH_" + path)
    assert M.ffn_path(table, T, cfg.k, M.make_options(n_experts=cfg.n_experts, path=p)) == p
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    plain = M.ffn_forward(table, x, logits, cfg.k, options=M.make_options(n_experts=cfg.n_experts, path=p))
    timed = M.ffn_forward(table, x, logits, cfg.k,
                          options=M.make_options(n_experts=cfg.n_experts, path=p, timing_events=ev))
    torch.cuda.synchronize()
    assert torch.equal(plain, timed)
    assert ev[0].elapsed_time(ev[1]) >= 0.0 and ev[1].elapsed_time(ev[2]) >= 0.0
    assert_parity(timed.cpu().numpy(), offn.moe_ffn(L.experts, L.x_bf16, L.logits, cfg.k), f"events {path}")
