"""Failure detection on the GPU without a fault: with the device-side wait
bound shortened to 1 ns (moe_set_wait_timeout_ns), the kernels' waits for
weights from memory and for other threads give up. Each path (the fused
decode kernel with its grid barrier and ring, the streaming grouped GEMV
kernels with their ring and producer, the tensor-core GEMMs with their
producer, dequantiser, MMA and epilogue handshakes), on full-size layers (512 experts, top-10,
2048/640) whose weight streams take microseconds, must then set
MOE_FLAG_WAIT_TIMEOUT, drain its own copies, return, and leave the context
usable: with the default bound restored, the same workspace gives the
oracle's result and a clean status. (The tiled grouped GEMV kernels wait once
per tile, after staging the activations, by which time the tile's copy has
landed: no bound makes that wait run out.)"""
import pytest

import synth
from tests.gpu_util import assert_parity, ensure_built, oracle_full_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    ensure_built()
    import quantized_moe_expert_route_gb300 as M
    M.load()
    return M


CASES = [("FUSED", None, "decode1", None), ("GEMV", "STREAMING", "decode16", None), ("TENSOR", None, "mtp6", 128)]


@pytest.mark.parametrize("path,kernels,name,tokens", CASES, ids=["fused", "stream", "tensor"])
def test_short_wait_bound_times_out_then_recovers(M, path, kernels, name, tokens):
    from synth import gpu as sgpu
    cfg = synth.CONFIGS[name]
    DL = sgpu.make_device_layer(cfg, 11, tokens=tokens)
    T = DL.x_host.shape[0]
    table = M.WeightTable(DL.experts, cfg.hidden, cfg.inter)
    p = getattr(M, "PATH_" + path)
    opt = M.make_options(n_experts=cfg.n_experts, path=p)
    assert M.ffn_path(table, T, cfg.k, opt) == p
    if kernels:
        assert M.gemv_kernels(table, T, cfg.k) == getattr(M, "GEMV_" + kernels)
    ws = M.Workspace(table, T, cfg.k, path=p)
    timed_out = False
    try:
        M.set_wait_timeout_ns(1)
        for _ in range(5):
            M.ffn_forward(table, DL.x_bf16, DL.logits, cfg.k, ws=ws, options=opt)
            if ws.read_status() & M.FLAG_WAIT_TIMEOUT:
                timed_out = True
                break
    finally:
        M.set_wait_timeout_ns(0)
    assert timed_out, f"{path}: no wait gave up under a 1 ns bound"
    out = M.ffn_forward(table, DL.x_bf16, DL.logits, cfg.k, ws=ws, options=opt).cpu().numpy()
    assert ws.read_status() == 0
    assert_parity(out, oracle_full_layer(cfg, DL), f"{path} after the timeouts")
