"""The GPU weight filler writes exactly the bytes of the numpy generator
(same SplitMix64 recipe), for every format, including row padding."""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import ensure_built

pytestmark = pytest.mark.gpu


def test_gpu_filler_matches_numpy():
    ensure_built()
    from synth import gpu as sgpu
    cases = [(synth.Q8_0, 7, 640), (synth.Q8_0, 3, 256), (synth.Q4_K, 5, 2048), (synth.Q6_K, 4, 512),
             (synth.MXFP4, 6, 640), (synth.MXFP4, 2, 2048), (synth.IQ4_NL, 5, 640), (synth.IQ4_NL, 3, 96),
             (synth.IQ4_XS, 4, 2048), (synth.IQ3_XXS, 6, 512), (synth.T5_G128, 5, 640),
             (synth.T5_G128, 3, 2048), (synth.T5_G128, 2, 128)]
    mats, refs = [], []
    for i, (fmt, rows, cols) in enumerate(cases):
        key = synth.stream_key(1234, 40 + i)
        ref = synth.gen_matrix(fmt, rows, cols, key)
        t = torch.full((rows * ref.stride,), 0xEE, dtype=torch.uint8, device="cuda")
        mats.append((t, fmt, rows, cols, ref.stride, key))
        refs.append(ref)
    sgpu.fill(mats)
    for (t, *_), ref in zip(mats, refs):
        np.testing.assert_array_equal(t.cpu().numpy(), ref.data)


@pytest.mark.parametrize("name", ["mtp6", "mtp6_iq", "decode16_shared", "decode16_t5"])
def test_device_layer_matches_lazy_experts(name):
    ensure_built()
    from synth import gpu as sgpu
    cfg = synth.CONFIGS[name]
    DL = sgpu.make_device_layer(cfg, 0)
    lazy = synth.LazyExperts(cfg, DL.seed, DL.fmts)
    perm = synth.permutation(DL.seed, cfg.n_experts)
    assert len(DL.experts) == len(lazy) == cfg.n_entries
    for e in [int(perm[0]), int(perm[200]), int(perm[511]), 0] + list(range(cfg.n_experts, cfg.n_entries)):
        for mat in ("gate", "up", "down"):
            fmt, rows, cols, stride, view = DL.experts[e][mat]
            m = lazy[e][mat]
            assert (fmt, rows, cols, stride) == (m.fmt, m.rows, m.cols, m.stride)
            np.testing.assert_array_equal(view.cpu().numpy(), m.data)
    if name == "mtp6_iq":
        np.testing.assert_array_equal(DL.grid.cpu().numpy().view(np.uint32), synth.iq3_grid())
