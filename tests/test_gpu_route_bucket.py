"""GPU parity of the router and the bucketing against the oracle, through the
C ABI: ids, offsets, pairs, pos and the active list bit-exact; router weights
within 4e-6 relative; device status flags for non-finite logits, bad and
duplicate ids."""
import numpy as np
import pytest
import torch

import synth
from oracle import bucket as obucket
from oracle import router as orouter
from tests.gpu_util import W_REL_TOL, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    ensure_built()
    import quantized_moe_expert_route_gb300 as M
    M.load()
    return M


def run_route(M, logits_np, k, renorm=True):
    lg = torch.from_numpy(np.ascontiguousarray(logits_np, dtype=np.float32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids, w = M.route_topk(lg, k, renorm, status=status)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), int(status.item())


def check_route(M, logits_np, k, renorm=True):
    ids, w, st = run_route(M, logits_np, k, renorm)
    rid, rw, flags = orouter.route_topk(logits_np, k, renorm)
    np.testing.assert_array_equal(ids, rid)
    assert np.all(np.abs(w - rw) <= W_REL_TOL * np.abs(rw) + 1e-12), np.abs(w - rw).max()
    assert bool(st & 1) == bool(flags.any())


@pytest.mark.parametrize("T,E,k", [(4, 8, 2), (1, 512, 10), (16, 512, 10), (6, 512, 10), (2048, 512, 10),
                                   (33, 100, 7), (5, 1024, 32), (3, 8, 8), (7, 1, 1), (9, 40, 32), (2, 32, 32)])
def test_route_random(M, T, E, k):
    rng = np.random.default_rng(T * 1000 + E + k)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    check_route(M, logits, k, True)
    check_route(M, logits, k, False)


def test_route_zipf_configs(M):
    for name in ("decode1", "decode16", "mtp6", "prefill2048"):
        cfg = synth.CONFIGS[name]
        lg = synth.gen_logits(synth.layer_seed(cfg, 0), cfg.tokens, cfg.n_experts, True)
        check_route(M, lg, cfg.k)


def test_route_ties(M):
    rng = np.random.default_rng(3)
    logits = (rng.integers(-2, 3, size=(64, 48)) * 0.5).astype(np.float32)
    check_route(M, logits, 12)
    check_route(M, np.zeros((5, 64), np.float32), 10)


def test_route_nonfinite(M):
    logits = np.array([[0.5, np.nan, -np.inf, 2.0, np.inf, -1.0, 0.0, 1.0]], np.float32)
    logits = np.repeat(logits, 3, axis=0)
    logits[1] = np.nan
    logits[2, :] = np.arange(8, dtype=np.float32)
    ids, w, st = run_route(M, logits, 6, False)
    rid, rw, _ = orouter.route_topk(logits, 6, False)
    np.testing.assert_array_equal(ids, rid)
    assert np.all(np.abs(w - rw) <= W_REL_TOL * np.abs(rw) + 1e-12)
    assert st & 1


def test_route_empty(M):
    ids, w, st = run_route(M, np.zeros((0, 16), np.float32), 4)
    assert ids.shape == (0, 4) and st == 0


def run_bucket(M, ids_np, E, lo=0, hi=None):
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    off, pairs, pos, active = M.bucket(ids, E, lo, hi, status=status)
    torch.cuda.synchronize()
    return off.cpu().numpy(), pairs.cpu().numpy(), pos.cpu().numpy(), active.cpu().numpy(), int(status.item())


def check_bucket(M, ids_np, E, lo=0, hi=None):
    off, pairs, pos, active, st = run_bucket(M, ids_np, E, lo, hi)
    roff, rpairs, rpos, ract, rflags = obucket.bucket(ids_np, E, lo, E if hi is None else hi)
    np.testing.assert_array_equal(off, roff)
    n = int(roff[-1])
    np.testing.assert_array_equal(pairs[:n], rpairs)
    np.testing.assert_array_equal(pos, rpos)
    assert active[0] == len(ract)
    np.testing.assert_array_equal(active[1:1 + len(ract)], ract)
    assert st == rflags, (st, rflags)


def topk_ids(rng, T, E, k):
    if T == 0:
        return np.zeros((0, k), np.int32)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k", [(4, 8, 2), (1, 512, 10), (16, 512, 10), (2048, 512, 10), (103, 1024, 32),
                                   (0, 16, 3), (1, 1, 1), (1500, 64, 7)])
def test_bucket_random(M, T, E, k):
    rng = np.random.default_rng(T + 7 * E + k)
    check_bucket(M, topk_ids(rng, T, E, k), E)


def test_bucket_zipf_routing(M):
    cfg = synth.CONFIGS["prefill2048"]
    lg = synth.gen_logits(synth.layer_seed(cfg, 0), cfg.tokens, cfg.n_experts, True)
    ids, _, _ = orouter.route_topk(lg, cfg.k)
    check_bucket(M, ids, cfg.n_experts)          # hot experts: >32 pairs per warp chunk, many chunks


def test_bucket_skips_bad_and_duplicates(M):
    ids = np.array([[3, -1], [-1, -1], [7, 0], [5, 3], [2, 2], [-5, 1]], np.int32)
    check_bucket(M, ids, 6)
    off, pairs, pos, active, st = run_bucket(M, ids, 6)
    assert st & 2 and st & 4


def test_bucket_range_filter(M):
    rng = np.random.default_rng(9)
    ids = topk_ids(rng, 300, 64, 8)
    for lo, hi in [(0, 64), (10, 20), (0, 1), (63, 64), (5, 5)]:
        check_bucket(M, ids, 64, lo, hi)
