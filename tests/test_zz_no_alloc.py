"""moe_ffn_forward_noalloc: the layer for callers that cannot allocate device
memory (a framework whose memory planner owns all device memory, a
latency-critical loop where cudaMalloc/cudaFree would synchronise the device,
a C client that only receives input and output pointers). Its scratch is the
library's own fixed 4 MiB device array. Checked through the C ABI against
moe_ffn_forward (caller workspace) on two calls in a row, with the parity
tolerance of the other GPU tests, and for its size limit.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import assert_parity, ensure_built, host_layer_to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    ensure_built()
    import quantized_moe_expert_route_gb300 as M
    M.load()
    return M


def test_noalloc_matches_workspace_forward_twice(M):
    # two different layers in a row: the second call must not see the first
    # call's leftovers in the shared scratch
    cfgs = [synth.LayerConfig("na1", 16, 4, 256, 64, 9, "mixed", True, 101),
            synth.LayerConfig("na2", 24, 6, 512, 128, 5, "mixed", True, 202)]
    for cfg in cfgs:
        L = synth.make_layer(cfg, 0)
        experts, x, logits = host_layer_to_device(L)
        table = M.WeightTable(experts, cfg.hidden, cfg.inter)
        ref = M.ffn_forward(table, x, logits, cfg.k).cpu().numpy()
        got = M.ffn_forward_noalloc(table, x, logits, cfg.k).cpu().numpy()
        assert_parity(got, ref, f"noalloc {cfg.name}")


def test_noalloc_full_size_decode(M):
    from synth import gpu as sgpu
    cfg = synth.CONFIGS["decode16"]
    DL = sgpu.make_device_layer(cfg, 3)
    table = M.WeightTable(DL.experts, cfg.hidden, cfg.inter)
    ref = M.ffn_forward(table, DL.x_bf16, DL.logits, cfg.k).cpu().numpy()
    for _ in range(2):
        got = M.ffn_forward_noalloc(table, DL.x_bf16, DL.logits, cfg.k).cpu().numpy()
        assert_parity(got, ref, "noalloc decode16")


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
