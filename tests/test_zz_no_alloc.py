"""moe_ffn_forward_noalloc: the layer for callers that cannot allocate device
memory (a framework whose memory planner owns all device memory, a
latency-critical loop where cudaMalloc/cudaFree would synchronise the device,
a C client that only receives input and output pointers). Its scratch is the
library's own fixed 4 MiB device array. Checked through the C ABI against
moe_ffn_forward (caller workspace): the same kernels on the same inputs, so
the outputs must be bit-identical, on two calls in a row on every path the
array serves (the fused decode kernel, whose grid-barrier counter lives in
the array across calls, the streaming GEMV kernels and the tensor path), and
for its size limit and its status flags.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import ensure_built, host_layer_to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    ensure_built()
    import quantized_moe_expert_route_gb300 as M
    M.load()
    return M


def _same(M, table, x, logits, k, options=None, calls=2):
    ref = M.ffn_forward(table, x, logits, k, options=options).cpu().numpy()
    for _ in range(calls):
        got = M.ffn_forward_noalloc(table, x, logits, k, options=options).cpu().numpy()
        assert np.array_equal(got, ref)
    return ref


def test_noalloc_matches_workspace_forward_twice(M):
    # two different layers in a row: the second call must not see the first
    # call's leftovers in the shared scratch
    cfgs = [synth.LayerConfig("na1", 16, 4, 256, 64, 9, "mixed", True, 101),
            synth.LayerConfig("na2", 24, 6, 512, 128, 5, "mixed", True, 202)]
    for cfg in cfgs:
        L = synth.make_layer(cfg, 0)
        experts, x, logits = host_layer_to_device(L)
        table = M.WeightTable(experts, cfg.hidden, cfg.inter)
        _same(M, table, x, logits, cfg.k)
    assert M.noalloc_read_status() == 0


def test_noalloc_every_path_full_size(M):
    """The 512-expert top-10 2048/640 layer on each path the array serves: a
    16-row batch (streaming GEMV kernels), then one token twice (the fused
    kernel, after a GEMV-path call), then 20 tokens on the tensor path."""
    from synth import gpu as sgpu
    cfg = synth.CONFIGS["decode16"]
    DL = sgpu.make_device_layer(cfg, 3)
    table = M.WeightTable(DL.experts, cfg.hidden, cfg.inter)
    k = cfg.k
    assert M.ffn_path(table, 16, k) == M.PATH_GEMV and M.gemv_kernels(table, 16, k) == M.GEMV_STREAMING
    _same(M, table, DL.x_bf16, DL.logits, k)
    assert M.ffn_path(table, 1, k) == M.PATH_FUSED
    for t in (0, 9):
        _same(M, table, DL.x_bf16[t:t + 1].contiguous(), DL.logits[t:t + 1].contiguous(), k)
    x20 = torch.cat([DL.x_bf16, DL.x_bf16[:4]]).contiguous()
    lg20 = torch.cat([DL.logits, DL.logits[4:8]]).contiguous()
    opt = M.make_options(n_experts=cfg.n_experts, path=M.PATH_TENSOR)
    assert M.ffn_path(table, 20, k, opt) == M.PATH_TENSOR
    _same(M, table, x20, lg20, k, options=opt)
    # and back to the fused kernel
    _same(M, table, DL.x_bf16[3:4].contiguous(), DL.logits[3:4].contiguous(), k)
    assert M.noalloc_read_status() == 0


def test_noalloc_status_flags(M):
    cfg = synth.LayerConfig("nas", 16, 4, 256, 64, 3, "q4k", True, 404)
    L = synth.make_layer(cfg, 0)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, cfg.hidden, cfg.inter)
    M.noalloc_read_status()
    lg = logits.clone()
    lg[1, 2] = float("nan")
    M.ffn_forward_noalloc(table, x, lg, cfg.k)
    assert M.noalloc_read_status() & M.FLAG_NONFINITE_LOGIT
    assert M.noalloc_read_status() == 0           # read clears
    _same(M, table, x, logits, cfg.k, calls=1)


def test_noalloc_rejects_oversize(M):
    cfg = synth.LayerConfig("big", 16, 8, 2048, 640, 64, "q4k", True, 303)
    L = synth.make_layer(cfg, 0)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, cfg.hidden, cfg.inter)
    ws = M.Workspace(table, 64, cfg.k)
    assert ws.nbytes > M.NOALLOC_SCRATCH_BYTES
    with pytest.raises(M.MoeError) as ei:
        M.ffn_forward_noalloc(table, x, logits, cfg.k)
    assert ei.value.code == 8
    # the size check follows the requested path: the tensor path's workspace
    # is larger than the grouped GEMV path's (here 3.1 MB against 4.6 MB)
    cfg = synth.LayerConfig("big2", 64, 22, 2048, 128, 16, "q4k", True, 304)
    L = synth.make_layer(cfg, 0)
    experts, x, logits = host_layer_to_device(L)
    table = M.WeightTable(experts, cfg.hidden, cfg.inter)
    gemv = M.make_options(n_experts=cfg.n_experts, path=M.PATH_GEMV)
    tensor = M.make_options(n_experts=cfg.n_experts, path=M.PATH_TENSOR)
    assert M.Workspace(table, 16, cfg.k, path=M.PATH_GEMV).nbytes <= M.NOALLOC_SCRATCH_BYTES
    assert M.Workspace(table, 16, cfg.k, path=M.PATH_TENSOR).nbytes > M.NOALLOC_SCRATCH_BYTES
    _same(M, table, x, logits, cfg.k, options=gemv, calls=1)
    with pytest.raises(M.MoeError) as ei:
        M.ffn_forward_noalloc(table, x, logits, cfg.k, options=tensor)
    assert ei.value.code == 8
