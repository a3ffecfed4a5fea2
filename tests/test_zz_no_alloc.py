"""The allocation-free compaction, sga_compact_noalloc, against the plan-based sga_compact.

Some callers cannot allocate device memory. Examples: an engine whose device memory is all
reserved up front by its own allocator, or a plug-in that its host framework forbids to
allocate. Such a caller cannot create a plan, because sga_plan_create allocates the plan's
index buffers and scratch. It calls sga_compact_noalloc instead. That call derives the kept set
from the layer configuration and keeps its only scratch in a fixed array inside the library.
Its results must equal sga_compact's, call after call, even though every call reuses the same
scratch.

Collected last on purpose: if it fails, a run that stops at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import subsampled_global_attention_sga_b300 as sga
from _guard import check_all, guarded
from subsampled_global_attention_sga_b300.inputs import correlated_qkv

pytestmark = pytest.mark.gpu

SUM_REL_TOL = 1e-5   # the dropped-row sums, as in the plan-based compaction test


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def _guarded_outputs(cfg, S, dev):
    """NaN-filled outputs, each between NaN guard regions that must survive the call."""
    ks_shape = (cfg.B, cfg.H, S, 64)
    return [guarded(ks_shape, cfg.torch_dtype, dev), guarded(ks_shape, cfg.torch_dtype, dev),
            guarded((cfg.B, cfg.H, 64), torch.float32, dev), guarded((cfg.B, cfg.H, 64), torch.float32, dev)]


def _outputs(cfg, S, dev):
    return tuple(g.t for g in _guarded_outputs(cfg, S, dev))


def _check_against_plan(cfg, seed, dev):
    q, k, v = correlated_qkv(cfg.B, cfg.H, cfg.N, cfg.L, 64, seed=seed, dtype=cfg.torch_dtype, device=dev)
    del q
    plan = sga.Plan(cfg, dev)
    want = plan.compact(k, v)
    gs = _guarded_outputs(cfg, plan.S, dev)
    got = sga.compact_noalloc(cfg, k, v, *[g.t for g in gs])
    torch.cuda.synchronize(dev)
    assert sga.device_status(dev) == 0
    check_all(gs, "noalloc")
    assert torch.equal(got[0], want[0]) and torch.equal(got[1], want[1])
    for g, w in zip(got[2:], want[2:]):
        w64 = w.double()
        err = (g.double() - w64).abs().max().item()
        assert err <= SUM_REL_TOL * max(1.0, w64.abs().max().item()), err
    plan.close()


CASES = [
    # one 32-frame VGGT-shaped layer (37x37 patches + 5 special tokens), sigma = 4
    dict(B=1, H=16, N=32, sigma=4),
    # phase-shifted non-square window on a 37x28 grid, frame 0 subsampled too, two batch elements
    dict(B=2, H=3, N=13, grid_h=37, grid_w=28, sigma=6, phase_shift=True, ref_frame_dense=False),
    # fp32, 8x8 patches, 3x3 window with phase shift
    dict(B=1, H=2, N=10, grid_h=8, grid_w=8, sigma=9, phase_shift=True, dtype="f32"),
]


@pytest.mark.parametrize("kw", CASES)
def test_noalloc_matches_plan_compaction_twice(dev, kw):
    cfg = sga.SGAConfig(**kw)
    # two calls in a row on different inputs: the second must not see the first one's scratch
    _check_against_plan(cfg, seed=31, dev=dev)
    _check_against_plan(cfg, seed=32, dev=dev)


def test_noalloc_refuses_buffers_of_the_wrong_kept_count(dev):
    # the C call receives no buffer sizes: the binding sizes K_S/V_S by sga_kept_count and refuses
    # any other row count before anything is launched, so nothing is written
    cfg = sga.SGAConfig(B=1, H=2, N=6, grid_h=9, grid_w=7, sigma=4, phase_shift=True)
    _, k, v = correlated_qkv(cfg.B, cfg.H, cfg.N, cfg.L, 64, seed=33, dtype=cfg.torch_dtype, device=dev)
    S = sga.kept_count(cfg)
    for wrong in (S - 1, S + 1):
        outs = _outputs(cfg, wrong, dev)
        with pytest.raises(ValueError):
            sga.compact_noalloc(cfg, k, v, *outs)
        torch.cuda.synchronize(dev)
        assert all(torch.isnan(t).all() for t in outs)
    assert sga.device_status(dev) == 0


def test_noalloc_rejects_problems_beyond_its_scratch(dev):
    # 32 heads x ceil(1,099,200 / 2048) = 17,184 blocks of partial sums > 16,384: refused on the host
    cfg = sga.SGAConfig(B=1, H=32, N=800)
    c = cfg.to_c()
    buf = torch.zeros(64, dtype=torch.float32, device=dev)
    p = ctypes.c_void_p(buf.data_ptr())
    st = sga.lib().sga_compact_noalloc(ctypes.byref(c), p, p, p, p, p, p, None)
    assert st == 7  # SGA_ERR_SCRATCH_LIMIT
    assert np.all(buf.cpu().numpy() == 0)
    assert sga.device_status(dev) == 0
