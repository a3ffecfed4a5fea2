"""Failure detection on the GPU without a fault: a wait that nothing completes must expire,
report SGA_ERR_TIMEOUT through the device status word, and leave the context usable.  Host-side
argument errors are covered by the other tests (bad shapes, alignment, plan mismatches)."""
import ctypes

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


def test_expired_wait_reports_timeout_and_context_survives(dev):
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    with torch.cuda.device(dev):
        st = sga.lib().sga_selftest_timeout(stream)
    assert st == 5, sga.lib().sga_status_string(st)          # SGA_ERR_TIMEOUT
    assert sga.device_status(dev) == 0                         # read and cleared
    # the same context still computes correctly
    cfg = sga.SGAConfig(B=1, H=2, N=4, grid_h=8, grid_w=8, sigma=4)
    q, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=0, dtype=torch.bfloat16, device=dev)
    out = sga.Plan(cfg, dev).layer(q, k, v)
    torch.cuda.synchronize(dev)
    assert sga.device_status(dev) == 0
    op = oracle.plan(cfg.N, cfg.grid_h, cfg.grid_w, cfg.n_special, 2, 2, False, True)
    for h in range(2):
        ref, _ = oracle.sga_full(op, q[0, h].float().cpu().numpy(), k[0, h].float().cpu().numpy(),
                                 v[0, h].float().cpu().numpy())
        assert np.abs(out[0, h].float().cpu().numpy() - ref).max() <= 2e-2
