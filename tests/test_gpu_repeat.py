"""Bitwise repeatability of the attention launches at the benchmarked shapes.

Every kernel of the path is deterministic: a work unit's key tiles are visited in a fixed order
and the compaction's partial sums are added in a fixed order.  So a launch repeated on the same
inputs must give the same bits.  A race between the TMA ring, the tensor pipe and the softmax
warps (a tile read before its copy has landed, or after its stage has been refilled) shows up as
a run-to-run difference.  A tolerance check against the oracle can miss such a race when the
stale data happens to be close to the right data.  The output is overwritten with NaN between
repeats, so a launch that skips rows cannot pass either.

Shapes are chosen to cover both kinds of work unit: two query tiles of one segment, and the
mixed unit that pairs the left-over last tiles of two segments (a segment with an odd tile
count)."""
import pytest
import torch

import subsampled_global_attention_sga_b300 as sga
from subsampled_global_attention_sga_b300.inputs import correlated_qkv

pytestmark = pytest.mark.gpu

REPEATS = 4


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def _repeat(fn, out):
    first = None
    for _ in range(REPEATS):
        out.fill_(float("nan"))
        fn()
        torch.cuda.synchronize(out.device)
        assert sga.device_status(out.device) == 0
        got = out.clone()
        assert not torch.isnan(got).any(), "rows left unwritten"
        if first is None:
            first = got
        else:
            assert torch.equal(got.view(torch.int16), first.view(torch.int16)), "launches differ"


def test_frame_local_repeats(dev):
    # 100 frames x 1374 tokens: 11 query tiles per frame, so every unit after the 5 full pairs
    # of each frame is a mixed unit of two frames' last tiles
    N, L, H = 100, 1374, 16
    q, k, v = correlated_qkv(1, H, N, L, 64, seed=11, dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    _repeat(lambda: sga.frame_forward(q, k, v, N, L, out=out), out)


def test_frame_local_odd_segment_count_repeats(dev):
    # 3 frames x 1 head: the last mixed unit repeats its first frame as its second tile
    N, L, H = 3, 300, 1
    q, k, v = correlated_qkv(1, H, N, L, 64, seed=12, dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    _repeat(lambda: sga.frame_forward(q, k, v, N, L, out=out), out)


def test_dense_repeats(dev):
    N, L, H = 32, 1374, 16
    q, k, v = correlated_qkv(1, H, N, L, 64, seed=13, dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    _repeat(lambda: sga.dense_forward(q, k, v, out=out), out)


@pytest.mark.parametrize("N,sigma,rope", [(200, 9, False), (33, 4, True)])
def test_sga_layer_repeats(dev, N, sigma, rope):
    # 200 x 1374 and 33 x 1374 tokens both give an odd query tile count per head: the heads'
    # last tiles pair up in mixed units
    cfg = sga.SGAConfig(B=1, H=16, N=N, sigma=sigma, rope=rope)
    q, k, v = correlated_qkv(1, cfg.H, cfg.N, cfg.L, 64, seed=14, dtype=torch.bfloat16, device=dev)
    plan = sga.Plan(cfg, dev)
    K_S, V_S, ks, vs = plan.compact(k, v)
    out = torch.empty_like(q)
    _repeat(lambda: plan.forward(q, k, v, K_S, V_S, ks, vs, out=out), out)


def test_size_aware_repeats(dev):
    # the bias variant keeps a segment's left-over tile in a unit of its own
    T, Tk, H = 3 * 1374, 1374, 4
    q, _, _ = correlated_qkv(1, H, 3, 1374, 64, seed=15, dtype=torch.bfloat16, device=dev)
    _, k, v = correlated_qkv(1, H, 1, Tk, 64, seed=16, dtype=torch.bfloat16, device=dev)
    bias = torch.log(torch.randint(1, 5, (1, H, Tk), device=dev).float()).contiguous()
    out = torch.empty_like(q)
    assert q.shape[2] == T
    _repeat(lambda: sga.bias_forward(q, k, v, bias, out=out), out)
