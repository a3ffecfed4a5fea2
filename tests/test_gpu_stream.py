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


@pytest.mark.parametrize("kind,depth", [("dense", 1), ("frame", 2), ("bias", 3)])
def test_plain_stream_equals_device_call(dev, kind, depth):
    """The plain executor (sga_stream_create_plain / sga_stream_submit_plain) streams dense,
    frame-local and size-aware layers from pinned host memory; every output equals the device
    call on the same inputs bit for bit."""
    B, H, N, L = 1, 2, 3, 333
    Tq = N * L
    Tk = 500 if kind == "bias" else Tq
    batches = []
    for i in range(4):
        q, _, _ = correlated_qkv(B, H, 1, Tq, 64, seed=300 + 5 * i, dtype=torch.bfloat16)
        _, k, v = correlated_qkv(B, H, 1, Tk, 64, seed=301 + 5 * i, dtype=torch.bfloat16)
        bias = torch.log(torch.randint(1, 5, (B, H, Tk), generator=torch.Generator().manual_seed(i)).float())
        batches.append(tuple(x.pin_memory() for x in (q, k, v, bias)))
    outs = [torch.empty((B, H, Tq, 64), dtype=torch.bfloat16, pin_memory=True) for _ in batches]
    ps = sga.PlainHostStream(kind, B, H, Tq, Tk=Tk, N=N, L=L, depth=depth)
    for (q, k, v, bias), o in zip(batches, outs):
        ps.submit(q, k, v, o, bias_host=bias if kind == "bias" else None)
    ps.synchronize()
    assert sga.device_status(dev) == 0
    for (q, k, v, bias), o in zip(batches, outs):
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        if kind == "dense":
            ref = sga.dense_forward(qd, kd, vd)
        elif kind == "frame":
            ref = sga.frame_forward(qd, kd, vd, N, L)
        else:
            ref = sga.bias_forward(qd, kd, vd, bias.to(dev))
        assert torch.equal(o.view(torch.int16), ref.cpu().view(torch.int16))
    ps.close()


def test_plain_stream_refuses_mismatched_calls(dev):
    cfg = sga.SGAConfig(B=1, H=1, N=2, grid_h=4, grid_w=4)
    plan = sga.Plan(cfg, dev)
    hs = sga.HostStream(plan)
    ps = sga.PlainHostStream("dense", 1, 1, cfg.T)
    lib = sga.lib()
    import ctypes
    x = torch.zeros((1, 1, cfg.T, 64), dtype=torch.bfloat16).pin_memory()
    p = ctypes.c_void_p(x.data_ptr())
    # an SGA stream takes only sga_stream_submit, a plain one only sga_stream_submit_plain
    assert lib.sga_stream_submit_plain(hs._h, p, p, p, None, p, ctypes.c_float(0.125)) == 1
    assert lib.sga_stream_submit(ps._h, p, p, p, p, ctypes.c_float(0.125)) == 1
    with pytest.raises(ValueError):
        ps.submit(x, x, x, x, bias_host=torch.zeros((1, 1, cfg.T)))
    hs.close()
    ps.close()
