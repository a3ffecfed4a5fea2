"""HostStream: layers streamed from pinned host memory with copies overlapping compute give the
same bytes as ``Plan.layer`` on the device, for every batch, whatever the buffering depth; and
the first batch matches the fp64 oracle within the bf16 tolerance."""
import numpy as np
import pytest
import torch

import oracle
import subsampled_global_attention_sga_b300 as sga
from subsampled_global_attention_sga_b300.inputs import correlated_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def _batches(cfg, n):
    out = []
    for i in range(n):
        q, k, v = correlated_qkv(cfg.B, cfg.H, cfg.N, cfg.L, 64, seed=100 + 3 * i, dtype=torch.bfloat16)
        out.append(tuple(x.pin_memory() for x in (q, k, v)))
    return out


@pytest.mark.parametrize("depth", [1, 2, 3])
def test_stream_equals_layer(dev, depth):
    cfg = sga.SGAConfig(B=1, H=4, N=6, grid_h=12, grid_w=12, sigma=4)
    plan = sga.Plan(cfg, dev)
    batches = _batches(cfg, 5)
    outs = [torch.empty((cfg.B, cfg.H, cfg.T, 64), dtype=torch.bfloat16, pin_memory=True) for _ in batches]
    hs = sga.HostStream(plan, depth=depth)
    for (q, k, v), o in zip(batches, outs):
        hs.submit(q, k, v, o)
    hs.synchronize()
    assert sga.device_status(dev) == 0
    for (q, k, v), o in zip(batches, outs):
        ref = plan.layer(q.to(dev), k.to(dev), v.to(dev)).cpu()
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))


def test_stream_with_rotation_equals_layer(dev):
    cfg = sga.SGAConfig(B=1, H=2, N=5, grid_h=9, grid_w=9, sigma=4, rope=True)
    plan = sga.Plan(cfg, dev)
    batches = _batches(cfg, 3)
    outs = [torch.empty((cfg.B, cfg.H, cfg.T, 64), dtype=torch.bfloat16, pin_memory=True) for _ in batches]
    hs = sga.HostStream(plan)
    for (q, k, v), o in zip(batches, outs):
        hs.submit(q, k, v, o)
    hs.synchronize()
    for (q, k, v), o in zip(batches, outs):
        ref = plan.layer(q.to(dev), k.to(dev), v.to(dev)).cpu()
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))


def test_stream_matches_oracle(dev):
    cfg = sga.SGAConfig(B=1, H=2, N=4, grid_h=8, grid_w=8, sigma=4)
    plan = sga.Plan(cfg, dev)
    (q, k, v), = _batches(cfg, 1)
    o = torch.empty((cfg.B, cfg.H, cfg.T, 64), dtype=torch.bfloat16, pin_memory=True)
    hs = sga.HostStream(plan)
    hs.submit(q, k, v, o)
    hs.synchronize()
    s_h, s_w = cfg.s_hw
    op = oracle.plan(cfg.N, cfg.grid_h, cfg.grid_w, cfg.n_special, s_h, s_w, False, True)
    rows = np.arange(cfg.T)
    for h in range(cfg.H):
        Q, K, V = (x[0, h].float().numpy() for x in (q, k, v))
        ref, _ = oracle.sga_rows(op, Q, K, V, rows)
        got = o[0, h].double().numpy()
        err = got - ref
        assert np.abs(err).max() <= 2e-2
        assert np.linalg.norm(err) / np.linalg.norm(ref) <= 5e-3
