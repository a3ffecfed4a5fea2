"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle, element by element on
seeded inputs: full outputs at sizes the oracle finishes in seconds (several tiles and a ragged
tail), sampled rows at the workloads' full sizes in the launch configuration the benchmark
times, and the edge cases of the method."""
import numpy as np
import pytest
import torch

import oracle
import subsampled_global_attention_sga_b300 as sga
from subsampled_global_attention_sga_b300.inputs import correlated_qkv, sample_rows

pytestmark = pytest.mark.gpu

BF16_MAX_ABS, BF16_REL_L2 = 2e-2, 5e-3
F32_MAX_ABS = 1e-5


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def _oracle_plan(cfg):
    s_h, s_w = cfg.s_hw
    return oracle.plan(cfg.N, cfg.grid_h, cfg.grid_w, cfg.n_special, s_h, s_w, cfg.phase_shift,
                       cfg.ref_frame_dense)


def _host(x):
    return x.float().cpu().numpy()


def _compare(got, ref, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref).max()
    if dtype == "f32":
        assert err <= F32_MAX_ABS, f"{what}: max-abs {err:.3e}"
    else:
        rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
        assert err <= BF16_MAX_ABS and rel <= BF16_REL_L2, f"{what}: max-abs {err:.3e} rel-L2 {rel:.3e}"


def _run(cfg, q, k, v, dev, lse=False):
    plan = sga.Plan(cfg, dev)
    L = torch.empty(q.shape[:3], dtype=torch.float32, device=dev) if lse else None
    K_S, V_S, ks, vs = plan.compact(k, v)
    out = plan.forward(q, k, v, K_S, V_S, ks, vs, lse=L)
    torch.cuda.synchronize(dev)
    assert sga.device_status(dev) == 0
    return plan, out, L, (K_S, V_S, ks, vs)


def _check_full(cfg, q, k, v, out, lse=None, **okw):
    op = _oracle_plan(cfg)
    qf, kf, vf, of = _host(q), _host(k), _host(v), _host(out)
    mm = 0 if cfg.mean_mode == "loo" else 1
    for b in range(cfg.B):
        for h in range(cfg.H):
            ref, rl = oracle.sga_full(op, qf[b, h], kf[b, h], vf[b, h], diag=cfg.diag, mean=cfg.mean,
                                      mean_mode=mm, **okw)
            _compare(of[b, h], ref, cfg.dtype, f"b{b} h{h}")
            if lse is not None:
                assert np.abs(lse[b, h].cpu().numpy() - rl).max() < (1e-5 if cfg.dtype == "f32" else 2e-3)


# ------------------------------------------------------------------------------ small, full outputs
def test_tiny_f32_config(dev):
    # B=1, N=4 frames of 8x8 patches + 5 special tokens (276 tokens), H=2, fp32, sigma=4
    cfg = sga.SGAConfig(B=1, H=2, N=4, grid_h=8, grid_w=8, sigma=4, dtype="f32")
    q, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=0, dtype=torch.float32, device=dev)
    plan, out, lse, _ = _run(cfg, q, k, v, dev, lse=True)
    assert (plan.T, plan.S, plan.dropped) == (276, 132, 144)
    _check_full(cfg, q, k, v, out, lse)


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_tiny_bf16(dev, kernel):
    cfg = sga.SGAConfig(B=1, H=2, N=4, grid_h=8, grid_w=8, sigma=4, dtype="bf16", kernel=kernel)
    q, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=0, dtype=torch.bfloat16, device=dev)
    _, out, lse, _ = _run(cfg, q, k, v, dev, lse=True)
    _check_full(cfg, q, k, v, out, lse)


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_multi_tile_vggt_frames(dev, kernel):
    # 8 frames of 37x37 + 5 (10,992 tokens): 86 query tiles, ragged key tail
    cfg = sga.SGAConfig(B=1, H=2, N=8, sigma=4, dtype="bf16", kernel=kernel)
    q, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=1, dtype=torch.bfloat16, device=dev)
    _, out, lse, _ = _run(cfg, q, k, v, dev, lse=True)
    _check_full(cfg, q, k, v, out, lse)


FLAG_CASES = [
    # sigma, phase, ref_dense, diag, mean, mean_mode
    (1, False, True, True, True, "loo"),
    (2, False, True, True, True, "loo"),
    (4, True, True, True, True, "loo"),
    (6, True, False, True, True, "loo"),
    (9, True, True, True, True, "loo"),
    (9, False, False, True, True, "global"),
    (4, False, True, False, True, "loo"),
    (4, False, True, True, False, "loo"),
    (4, True, True, False, False, "loo"),
]


@pytest.mark.parametrize("case", FLAG_CASES)
@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_flag_matrix(dev, case, kernel):
    sigma, ph, ref, diag, mean, mm = case
    cfg = sga.SGAConfig(B=1, H=2, N=6, grid_h=13, grid_w=11, sigma=sigma, phase_shift=ph,
                        ref_frame_dense=ref, diag=diag, mean=mean, mean_mode=mm, dtype="bf16", kernel=kernel)
    q, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=2, dtype=torch.bfloat16, device=dev)
    _, out, _, _ = _run(cfg, q, k, v, dev)
    _check_full(cfg, q, k, v, out)


def test_flag_matrix_f32(dev):
    for sigma, ph, ref, diag, mean, mm in FLAG_CASES:
        cfg = sga.SGAConfig(B=1, H=1, N=5, grid_h=9, grid_w=7, sigma=sigma, phase_shift=ph,
                            ref_frame_dense=ref, diag=diag, mean=mean, mean_mode=mm, dtype="f32")
        q, k, v = correlated_qkv(1, 1, cfg.N, cfg.L, 64, seed=3, dtype=torch.float32, device=dev)
        _, out, _, _ = _run(cfg, q, k, v, dev)
        _check_full(cfg, q, k, v, out)


def test_compaction_exact(dev):
    for dtype, tdt in (("bf16", torch.bfloat16), ("f32", torch.float32)):
        cfg = sga.SGAConfig(B=2, H=3, N=7, sigma=4, phase_shift=True, dtype=dtype)
        q, k, v = correlated_qkv(2, 3, cfg.N, cfg.L, 64, seed=4, dtype=tdt, device=dev)
        plan, _, _, (K_S, V_S, ks, vs) = _run(cfg, q, k, v, dev)
        op = _oracle_plan(cfg)
        kv, off = plan.indices()
        assert np.array_equal(kv, op.kv_index) and np.array_equal(off, op.frame_off)
        idx = torch.as_tensor(op.kv_index.astype(np.int64), device=dev)
        assert torch.equal(K_S, k[:, :, idx]) and torch.equal(V_S, v[:, :, idx])
        kf, vf = _host(k), _host(v)
        for b in range(2):
            for h in range(3):
                rk, rv, c = oracle.dropped_sums(op, kf[b, h], vf[b, h])
                assert c == plan.dropped
                for got, ref in ((ks[b, h], rk), (vs[b, h], rv)):
                    g = got.cpu().numpy().astype(np.float64)
                    assert np.abs(g - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_dense_and_frame_variants(dev, kernel):
    N, L, H = 3, 300, 2
    q, k, v = correlated_qkv(1, H, N, L, 64, seed=5, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((1, H, N * L), dtype=torch.float32, device=dev)
    od = sga.dense_forward(q, k, v, kernel=kernel, lse=lse)
    of = sga.frame_forward(q, k, v, N, L, kernel=kernel)
    torch.cuda.synchronize(dev)
    qf, kf, vf = _host(q), _host(k), _host(v)
    rows = np.arange(N * L)
    for h in range(H):
        ref, rl = oracle.attention_rows(qf[0, h], kf[0, h], vf[0, h], rows)
        _compare(_host(od)[0, h], ref, "bf16", "dense")
        assert np.abs(lse[0, h].cpu().numpy() - rl).max() < 2e-3
        ref, _ = oracle.attention_rows(qf[0, h], kf[0, h], vf[0, h], rows, frame_len=L)
        _compare(_host(of)[0, h], ref, "bf16", "frame")


def test_dense_frame_f32(dev):
    N, L, H = 2, 70, 2
    q, k, v = correlated_qkv(1, H, N, L, 64, seed=6, dtype=torch.float32, device=dev)
    od = sga.dense_forward(q, k, v, dtype="f32")
    of = sga.frame_forward(q, k, v, N, L, dtype="f32")
    torch.cuda.synchronize(dev)
    rows = np.arange(N * L)
    for h in range(H):
        ref, _ = oracle.attention_rows(_host(q)[0, h], _host(k)[0, h], _host(v)[0, h], rows)
        _compare(_host(od)[0, h], ref, "f32", "dense")
        ref, _ = oracle.attention_rows(_host(q)[0, h], _host(k)[0, h], _host(v)[0, h], rows, frame_len=L)
        _compare(_host(of)[0, h], ref, "f32", "frame")


# ------------------------------------------------------------------------------ edge cases
@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_equal_dropped_rows_match_dense(dev, kernel):
    # identity: all dropped keys/values equal -> SGA equals dense attention (oracle dense)
    cfg = sga.SGAConfig(B=1, H=2, N=5, grid_h=16, grid_w=16, sigma=4, phase_shift=True, kernel=kernel)
    q, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=7, dtype=torch.bfloat16, device=dev)
    op = _oracle_plan(cfg)
    drop = torch.as_tensor(op.kept == 0, device=dev)
    g = torch.Generator(device=dev).manual_seed(9)
    kb = torch.randn(64, generator=g, device=dev).to(torch.bfloat16)
    vb = torch.randn(64, generator=g, device=dev).to(torch.bfloat16)
    k[:, :, drop] = kb
    v[:, :, drop] = vb
    _, out, _, _ = _run(cfg, q, k, v, dev)
    rows = np.arange(cfg.T)
    for h in range(2):
        ref, _ = oracle.attention_rows(_host(q)[0, h], _host(k)[0, h], _host(v)[0, h], rows)
        _compare(_host(out)[0, h], ref, "bf16", f"identity h{h}")


def test_zero_query_gives_mean_of_values(dev):
    cfg = sga.SGAConfig(B=1, H=2, N=6, grid_h=12, grid_w=12, sigma=9)
    _, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=8, dtype=torch.bfloat16, device=dev)
    q = torch.zeros_like(k)
    _, out, lse, _ = _run(cfg, q, k, v, dev, lse=True)
    want = v.float().mean(dim=2, keepdim=True).expand_as(out)
    assert (out.float() - want).abs().max().item() <= 2e-3
    assert (lse - np.log(cfg.T)).abs().max().item() <= 1e-3


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_peaky_softmax(dev, kernel):
    cfg = sga.SGAConfig(B=1, H=2, N=4, grid_h=20, grid_w=20, sigma=4, kernel=kernel)
    q, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=10, dtype=torch.bfloat16, device=dev, q_scale=8.0)
    _, out, _, _ = _run(cfg, q, k, v, dev)
    _check_full(cfg, q, k, v, out)


def test_batch2_and_single_frame(dev):
    cfg = sga.SGAConfig(B=2, H=2, N=3, grid_h=10, grid_w=9, sigma=6, phase_shift=True)
    q, k, v = correlated_qkv(2, 2, cfg.N, cfg.L, 64, seed=11, dtype=torch.bfloat16, device=dev)
    _, out, _, _ = _run(cfg, q, k, v, dev)
    _check_full(cfg, q, k, v, out)
    # a single dense reference frame keeps every key: no dropped tokens, plain attention
    cfg1 = sga.SGAConfig(B=1, H=1, N=1, grid_h=10, grid_w=9, sigma=4)
    q, k, v = correlated_qkv(1, 1, 1, cfg1.L, 64, seed=12, dtype=torch.bfloat16, device=dev)
    plan, out, _, _ = _run(cfg1, q, k, v, dev)
    assert plan.dropped == 0
    _check_full(cfg1, q, k, v, out)


def test_bad_arguments_raise(dev):
    cfg = sga.SGAConfig(B=1, H=1, N=2, grid_h=4, grid_w=4)
    plan = sga.Plan(cfg, dev)
    q = torch.zeros((1, 1, cfg.T, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError):
        plan.compact(q[:, :, :-1], q[:, :, :-1])
    with pytest.raises(TypeError):
        plan.compact(q.float(), q.float())
    lib = sga.lib()
    import ctypes
    # misaligned device pointer -> alignment error, nothing launched
    p = ctypes.c_void_p(q.data_ptr() + 2)
    assert lib.sga_compact(plan._h, p, p, p, p, p, p, None) == 3
    assert sga.device_status(dev) == 0


# ------------------------------------------------------------------------------ full sizes, sampled rows
def _sampled(cfg, dev, n_rows=4096, seed=0):
    q, k, v = correlated_qkv(cfg.B, cfg.H, cfg.N, cfg.L, 64, seed=seed, dtype=torch.bfloat16, device=dev)
    plan = sga.Plan(cfg, dev)
    out = plan.layer(q, k, v)
    torch.cuda.synchronize(dev)
    assert sga.device_status(dev) == 0
    op = _oracle_plan(cfg)
    assert op.S == plan.S
    per_head = max(1, n_rows // (cfg.B * cfg.H))
    mm = 0 if cfg.mean_mode == "loo" else 1
    gots, refs = [], []
    for b in range(cfg.B):
        for h in range(cfg.H):
            rows = sample_rows(cfg.T, cfg.L, per_head, seed=1234 + 97 * (b * cfg.H + h), kept=op.kept).numpy()
            ridx = torch.as_tensor(rows, device=dev)
            kf, vf = _host(k[b, h]), _host(v[b, h])
            ref, _ = oracle.sga_rows(op, _host(q[b, h][ridx]), kf, vf, rows, diag=cfg.diag, mean=cfg.mean,
                                     mean_mode=mm)
            gots.append(_host(out[b, h][ridx]))
            refs.append(ref)
    _compare(np.concatenate(gots), np.concatenate(refs), "bf16", "sampled")


def test_vggt_shaped_sampled(dev):
    _sampled(sga.SGAConfig(B=1, H=16, N=32, sigma=4), dev)


def test_long_sequence_sampled(dev):
    _sampled(sga.SGAConfig(B=1, H=16, N=200, sigma=9), dev)


def test_headline_sampled(dev):
    _sampled(sga.SGAConfig(B=1, H=16, N=800, sigma=4), dev)


SWEEP = [(s, ph, terms) for s in (1, 2, 4, 6, 9) for ph in (False, True) for terms in (True, False)
         if not (s == 1 and ph)]


@pytest.mark.parametrize("sigma,phase,terms", SWEEP)
def test_sweep_sampled(dev, sigma, phase, terms):
    cfg = sga.SGAConfig(B=1, H=16, N=100, sigma=sigma, phase_shift=phase, diag=terms, mean=terms)
    _sampled(cfg, dev, n_rows=1024, seed=sigma)


def test_sweep_frame_local_sampled(dev):
    N, L, H = 100, 1374, 16
    q, k, v = correlated_qkv(1, H, N, L, 64, seed=20, dtype=torch.bfloat16, device=dev)
    out = sga.frame_forward(q, k, v, N, L)
    torch.cuda.synchronize(dev)
    gots, refs = [], []
    for h in range(H):
        rows = sample_rows(N * L, L, 64, seed=h).numpy()
        ridx = torch.as_tensor(rows, device=dev)
        ref, _ = oracle.attention_rows(_host(q[0, h][ridx]), _host(k[0, h]), _host(v[0, h]), rows, frame_len=L)
        gots.append(_host(out[0, h][ridx]))
        refs.append(ref)
    _compare(np.concatenate(gots), np.concatenate(refs), "bf16", "frame sweep")
