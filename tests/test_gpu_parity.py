"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle, element by element on
seeded inputs: full outputs at sizes the oracle finishes in seconds (several tiles and a ragged
tail), sampled rows at the workloads' full sizes in the launch configuration the benchmark
times, and the edge cases of the method."""
import numpy as np
import pytest
import torch

import oracle
import subsampled_global_attention_sga_b300 as sga
from _guard import check_all, guarded
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


def _layer_guarded(plan, cfg, q, k, v, dev, lse=False):
    """Compaction and attention with every output between NaN guards, checked after the call."""
    ks_shape = (cfg.B, cfg.H, plan.S, 64)
    gs = [guarded(ks_shape, cfg.torch_dtype, dev), guarded(ks_shape, cfg.torch_dtype, dev),
          guarded((cfg.B, cfg.H, 64), torch.float32, dev), guarded((cfg.B, cfg.H, 64), torch.float32, dev),
          guarded(q.shape, q.dtype, dev)]
    if lse:
        gs.append(guarded(q.shape[:3], torch.float32, dev))
    K_S, V_S, ks, vs = plan.compact(k, v, *[g.t for g in gs[:4]])
    out = plan.forward(q, k, v, K_S, V_S, ks, vs, out=gs[4].t, lse=gs[5].t if lse else None)
    torch.cuda.synchronize(dev)
    assert sga.device_status(dev) == 0
    check_all(gs, "layer")
    return out, (gs[5].t if lse else None), (K_S, V_S, ks, vs)


def _run(cfg, q, k, v, dev, lse=False):
    plan = sga.Plan(cfg, dev)
    out, L, bufs = _layer_guarded(plan, cfg, q, k, v, dev, lse)
    return plan, out, L, bufs


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
    gs = [guarded((1, H, N * L), torch.float32, dev), guarded(q.shape, q.dtype, dev), guarded(q.shape, q.dtype, dev)]
    lse = gs[0].t
    od = sga.dense_forward(q, k, v, kernel=kernel, lse=lse, out=gs[1].t)
    of = sga.frame_forward(q, k, v, N, L, kernel=kernel, out=gs[2].t)
    torch.cuda.synchronize(dev)
    check_all(gs, "dense/frame")
    qf, kf, vf = _host(q), _host(k), _host(v)
    rows = np.arange(N * L)
    for h in range(H):
        ref, rl = oracle.attention_rows(qf[0, h], kf[0, h], vf[0, h], rows)
        _compare(_host(od)[0, h], ref, "bf16", "dense")
        assert np.abs(lse[0, h].cpu().numpy() - rl).max() < 2e-3
        ref, _ = oracle.attention_rows(qf[0, h], kf[0, h], vf[0, h], rows, frame_len=L)
        _compare(_host(of)[0, h], ref, "bf16", "frame")


@pytest.mark.parametrize("T", [32 * 128, 32 * 128 + 77])
def test_dense_at_the_epilogue_form_boundary(dev, T):
    """Units of up to 32 key tiles run each unit's epilogue after the next unit's first P, longer
    ones straight after the unit (two template instances of the kernel, chosen by the host):
    4096 keys are the last size of the first form, 4173 (33 tiles, the last one ragged) the
    first of the second; both against the oracle on every row, several units per CTA."""
    H = 2
    q, k, v = correlated_qkv(1, H, 1, T, 64, seed=21, dtype=torch.bfloat16, device=dev)
    g = guarded(q.shape, q.dtype, dev)
    od = sga.dense_forward(q, k, v, out=g.t)
    torch.cuda.synchronize(dev)
    g.check("dense")
    qf, kf, vf = _host(q), _host(k), _host(v)
    rows = np.arange(T)
    for h in range(H):
        ref, _ = oracle.attention_rows(qf[0, h], kf[0, h], vf[0, h], rows)
        _compare(_host(od)[0, h], ref, "bf16", f"dense T={T} h{h}")


def test_output_only_16_byte_aligned(dev):
    """The epilogue writes each row as four 32-byte sectors when O is 32-byte aligned; the entry
    points only require 16, and an output at an odd multiple of 16 bytes takes the 16-byte
    stores.  Both must give the oracle's rows and leave the neighbours untouched."""
    N, L, H = 2, 300, 2
    q, k, v = correlated_qkv(1, H, N, L, 64, seed=22, dtype=torch.bfloat16, device=dev)
    n = q.numel()
    buf = torch.full((n + 2 * 4096 + 8,), float("nan"), dtype=torch.bfloat16, device=dev)
    out = buf[4096 + 8:4096 + 8 + n].view(q.shape)          # 8 bf16 = 16 bytes past a 32-byte boundary
    assert out.data_ptr() % 32 == 16
    sga.dense_forward(q, k, v, out=out)
    torch.cuda.synchronize(dev)
    assert torch.isnan(buf[:4096 + 8]).all() and torch.isnan(buf[4096 + 8 + n:]).all()
    qf, kf, vf = _host(q), _host(k), _host(v)
    rows = np.arange(N * L)
    for h in range(H):
        ref, _ = oracle.attention_rows(qf[0, h], kf[0, h], vf[0, h], rows)
        _compare(_host(out)[0, h], ref, "bf16", "dense, 16-byte aligned output")


def test_dense_frame_f32(dev):
    N, L, H = 2, 70, 2
    q, k, v = correlated_qkv(1, H, N, L, 64, seed=6, dtype=torch.float32, device=dev)
    gs = [guarded(q.shape, q.dtype, dev), guarded(q.shape, q.dtype, dev)]
    od = sga.dense_forward(q, k, v, dtype="f32", out=gs[0].t)
    of = sga.frame_forward(q, k, v, N, L, dtype="f32", out=gs[1].t)
    torch.cuda.synchronize(dev)
    check_all(gs, "dense/frame f32")
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
    out, _, _ = _layer_guarded(plan, cfg, q, k, v, dev)
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
    g = guarded(q.shape, q.dtype, dev)
    out = sga.frame_forward(q, k, v, N, L, out=g.t)
    torch.cuda.synchronize(dev)
    g.check("frame sweep")
    gots, refs = [], []
    for h in range(H):
        rows = sample_rows(N * L, L, 64, seed=h).numpy()
        ridx = torch.as_tensor(rows, device=dev)
        ref, _ = oracle.attention_rows(_host(q[0, h][ridx]), _host(k[0, h]), _host(v[0, h]), rows, frame_len=L)
        gots.append(_host(out[0, h][ridx]))
        refs.append(ref)
    _compare(np.concatenate(gots), np.concatenate(refs), "bf16", "frame sweep")


# ------------------------------------------------------------------------------ size-aware bias
# "RegimeVGGT ..." Key design 2: softmax(QK^T/sqrt(d) + log g) V.
def _bias_case(dev, Tq, Tk, H, seed, dtype=torch.bfloat16, g_max=8, real=False):
    q, _, _ = correlated_qkv(1, H, 1, Tq, 64, seed=seed, dtype=dtype, device=dev)
    _, k, v = correlated_qkv(1, H, 1, Tk, 64, seed=seed + 1, dtype=dtype, device=dev)
    gen = torch.Generator(device=dev).manual_seed(seed + 2)
    if real:
        bias = torch.randn((1, H, Tk), generator=gen, device=dev) * 3.0
        bias[..., ::7] = -1e4    # effectively removed keys
    else:
        g = torch.randint(1, g_max + 1, (1, H, Tk), generator=gen, device=dev)
        bias = torch.log(g.float())
    return q, k, v, bias.contiguous()


def _check_bias(q, k, v, bias, out, dtype, lse=None, rows=None):
    H = q.shape[1]
    for h in range(H):
        rr = np.arange(q.shape[2]) if rows is None else rows
        ref, rl = oracle.biased_attention_rows(_host(q[0, h])[rr], _host(k[0, h]), _host(v[0, h]),
                                               bias[0, h].double().cpu().numpy())
        _compare(_host(out[0, h])[rr], ref, dtype, f"bias h{h}")
        if lse is not None:
            assert np.abs(lse[0, h].cpu().numpy()[rr] - rl).max() < (1e-5 if dtype == "f32" else 2e-3)


@pytest.mark.parametrize("kernel", ["tc", "simt"])
@pytest.mark.parametrize("Tq,Tk,real", [(700, 450, False), (256, 1000, True), (130, 129, False), (1, 5, True)])
def test_bias_forward(dev, kernel, Tq, Tk, real):
    q, k, v, bias = _bias_case(dev, Tq, Tk, 2, seed=40 + Tq, real=real)
    gs = [guarded((1, 2, Tq), torch.float32, dev), guarded(q.shape, q.dtype, dev)]
    lse = gs[0].t
    out = sga.bias_forward(q, k, v, bias, kernel=kernel, lse=lse, out=gs[1].t)
    torch.cuda.synchronize(dev)
    assert sga.device_status(dev) == 0
    check_all(gs, "bias")
    _check_bias(q, k, v, bias, out, "bf16", lse)


def test_bias_forward_f32(dev):
    q, k, v, bias = _bias_case(dev, 300, 333, 2, seed=50, dtype=torch.float32, real=True)
    g = guarded(q.shape, q.dtype, dev)
    out = sga.bias_forward(q, k, v, bias, dtype="f32", out=g.t)
    torch.cuda.synchronize(dev)
    g.check("bias f32")
    _check_bias(q, k, v, bias, out, "f32")


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_bias_integer_groups_match_expanded_dense(dev, kernel):
    # the same identity the oracle is pinned with, on the GPU: bias ln g == g copies of the key
    q, k, v, bias = _bias_case(dev, 384, 200, 2, seed=60, g_max=4)
    g = torch.round(torch.exp(bias)).long()
    out = sga.bias_forward(q, k, v, bias, kernel=kernel)
    for h in range(2):
        ke = torch.repeat_interleave(k[:, h:h + 1], g[0, h], dim=2).contiguous()
        ve = torch.repeat_interleave(v[:, h:h + 1], g[0, h], dim=2).contiguous()
        qe = q[:, h:h + 1].contiguous()
        oe = torch.empty_like(qe)
        # dense attention over the expanded keys: queries and keys differ in count, so use the
        # biased entry point with a zero bias (a separate check that zero bias == dense follows)
        sga.bias_forward(qe, ke, ve, torch.zeros(ke.shape[:3], device=dev), kernel=kernel, out=oe)
        torch.cuda.synchronize(dev)
        ref, _ = oracle.biased_attention_rows(_host(qe[0, 0]), _host(ke[0, 0]), _host(ve[0, 0]),
                                              np.zeros(ke.shape[2]))
        _compare(_host(oe[0, 0]), ref, "bf16", "expanded dense")
        _compare(_host(out[0, h]), ref, "bf16", "biased vs expanded")


def test_bias_zero_equals_dense_entry_point(dev):
    q, k, v = correlated_qkv(1, 2, 3, 300, 64, seed=61, dtype=torch.bfloat16, device=dev)
    od = sga.dense_forward(q, k, v)
    ob = sga.bias_forward(q, k, v, torch.zeros(q.shape[:3], device=dev))
    torch.cuda.synchronize(dev)
    # same tensor-core kernel, the bias step only adds exact zeros
    assert torch.equal(od, ob)


def test_bias_bad_arguments(dev):
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device=dev)
    lib = sga.lib()
    import ctypes
    p = ctypes.c_void_p(q.data_ptr())
    assert lib.sga_bias_forward(1, 1, 128, 128, 64, 0, 0, p, p, p, None, p, None, ctypes.c_float(0.125), None) == 1
    with pytest.raises(ValueError):
        sga.bias_forward(q, q, q, torch.zeros((1, 1, 127), device=dev))


def test_bias_merged_keys_sampled(dev):
    # a merged-key layer of 32 VGGT frames: 43,968 queries against 12,000 merged keys that
    # stand for 1-8 tokens each, 16 heads; 2048 sampled query rows against the oracle
    H, Tq, Tk = 16, 43968, 12000
    q, k, v, bias = _bias_case(dev, Tq, Tk, H, seed=70)
    g = guarded(q.shape, q.dtype, dev)
    out = sga.bias_forward(q, k, v, bias, out=g.t)
    torch.cuda.synchronize(dev)
    g.check("merged keys")
    gots, refs = [], []
    for h in range(H):
        rows = sample_rows(Tq, 1374, 128, seed=300 + h).numpy()
        ref, _ = oracle.biased_attention_rows(_host(q[0, h])[rows], _host(k[0, h]), _host(v[0, h]),
                                              bias[0, h].double().cpu().numpy())
        gots.append(_host(out[0, h])[rows])
        refs.append(ref)
    _compare(np.concatenate(gots), np.concatenate(refs), "bf16", "merged keys")


# ------------------------------------------------------------------------------ generalised kept set
# "RegimeVGGT ..." Key design 3: fractional per-axis windows, phase shift, protected tokens; and
# any kept set given as an index list, through the same compaction and attention.
def _general_case(dev, cfg, sh, sw, phase, n_prot, seed, dtype=torch.bfloat16):
    rng = np.random.default_rng(seed)
    prot = rng.integers(0, cfg.T, size=n_prot)
    kv, _, _ = sga.plan_host_general(cfg.N, cfg.grid_h, cfg.grid_w, cfg.n_special, sigma_h=sh, sigma_w=sw,
                                     phase_shift=phase, ref_frame_dense=cfg.ref_frame_dense, protected=prot)
    op = oracle.plan_general(cfg.N, cfg.grid_h, cfg.grid_w, cfg.n_special, sh, sw, phase, cfg.ref_frame_dense,
                             protected=prot)
    q, k, v = correlated_qkv(cfg.B, cfg.H, cfg.N, cfg.L, 64, seed=seed, dtype=dtype, device=dev)
    plan = sga.Plan(cfg, dev, kv_index=kv)
    assert plan.S == op.S
    out, _, _ = _layer_guarded(plan, cfg, q, k, v, dev)
    return op, q, k, v, out


@pytest.mark.parametrize("kernel", ["tc", "simt"])
@pytest.mark.parametrize("sh,sw,phase", [((3, 2), (3, 2), True), ((13, 10), (17, 10), False), ((17, 10), (17, 10), True)])
def test_general_plan_full(dev, kernel, sh, sw, phase):
    cfg = sga.SGAConfig(B=1, H=2, N=6, grid_h=13, grid_w=11, kernel=kernel)
    op, q, k, v, out = _general_case(dev, cfg, sh, sw, phase, n_prot=9, seed=80)
    for h in range(2):
        ref, _ = oracle.sga_full(op, _host(q[0, h]), _host(k[0, h]), _host(v[0, h]))
        _compare(_host(out[0, h]), ref, "bf16", f"general h{h}")


def test_arbitrary_kept_set_f32(dev):
    cfg = sga.SGAConfig(B=1, H=2, N=4, grid_h=9, grid_w=8, dtype="f32")
    rng = np.random.default_rng(81)
    kv = np.sort(rng.choice(cfg.T, size=cfg.T // 3, replace=False)).astype(np.int32)
    q, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=81, dtype=torch.float32, device=dev)
    plan = sga.Plan(cfg, dev, kv_index=kv)
    out, _, _ = _layer_guarded(plan, cfg, q, k, v, dev)
    kept = np.zeros(cfg.T, dtype=np.uint8)
    kept[kv] = 1
    off = np.searchsorted(kv, np.arange(cfg.N + 1) * cfg.L).astype(np.int32)
    op = oracle.Plan(T=cfg.T, L=cfg.L, kept=kept, kv_index=kv, frame_off=off)
    got_kv, got_off = plan.indices()
    assert np.array_equal(got_kv, kv) and np.array_equal(got_off, off)
    for h in range(2):
        ref, _ = oracle.sga_full(op, _host(q[0, h]), _host(k[0, h]), _host(v[0, h]))
        _compare(_host(out[0, h]), ref, "f32", f"arbitrary h{h}")


def test_arbitrary_kept_set_rejected(dev):
    cfg = sga.SGAConfig(B=1, H=1, N=2, grid_h=4, grid_w=4)
    for bad in ([3, 3, 5], [5, 2], [-1, 4], [0, cfg.T]):
        with pytest.raises(sga.SgaError):
            sga.Plan(cfg, dev, kv_index=np.array(bad, dtype=np.int32))


def test_general_plan_vggt_sampled(dev):
    # 32 VGGT frames, RegimeVGGT middle band: sigma_b = 1.3 per axis, phase shift, 10 % of the
    # patches protected as salient; 4096 sampled rows against the oracle
    cfg = sga.SGAConfig(B=1, H=16, N=32)
    op, q, k, v, out = _general_case(dev, cfg, (13, 10), (13, 10), True, n_prot=cfg.T // 10, seed=82)
    gots, refs = [], []
    for h in range(cfg.H):
        rows = sample_rows(cfg.T, cfg.L, 256, seed=400 + h, kept=op.kept).numpy()
        ref, _ = oracle.sga_rows(op, _host(q[0, h])[rows], _host(k[0, h]), _host(v[0, h]), rows)
        gots.append(_host(out[0, h])[rows])
        refs.append(ref)
    _compare(np.concatenate(gots), np.concatenate(refs), "bf16", "general sampled")


# ------------------------------------------------------------------------------ fused 2D RoPE
# VGGT re-applies RoPE in every layer ("HTTM ..." section 3); the convention is a parameter.
def _rope_ref(x, cfg):
    """Oracle rotation of one (batch, head) [T, 64] tensor, rounded once to fp32 for the oracle's
    attention routines (relative 6e-8, far below any tolerance here)."""
    return oracle.rope2d(_host(x), cfg.L, cfg.n_special, cfg.grid_w, cfg.rope_base, cfg.rope_pos_offset).astype(np.float32)


@pytest.mark.parametrize("dtype,tdt", [("bf16", torch.bfloat16), ("f32", torch.float32)])
def test_rope_compaction(dev, dtype, tdt):
    cfg = sga.SGAConfig(B=1, H=2, N=5, grid_h=11, grid_w=9, sigma=4, phase_shift=True, dtype=dtype, rope=True,
                        rope_base=100.0, rope_pos_offset=1)
    _, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=90, dtype=tdt, device=dev)
    plan = sga.Plan(cfg, dev)
    gs = [guarded((1, 2, plan.S, 64), tdt, dev), guarded((1, 2, plan.S, 64), tdt, dev),
          guarded((1, 2, 64), torch.float32, dev), guarded((1, 2, 64), torch.float32, dev)]
    K_S, V_S, ks, vs = plan.compact(k, v, *[g.t for g in gs])
    torch.cuda.synchronize(dev)
    check_all(gs, "rope compaction")
    op = _oracle_plan(cfg)
    idx = torch.as_tensor(op.kv_index.astype(np.int64), device=dev)
    assert torch.equal(V_S, v[:, :, idx])                       # values are never rotated
    for h in range(2):
        kr = _rope_ref(k[0, h], cfg)
        got = _host(K_S[0, h])
        tol = 1e-6 if dtype == "f32" else 8e-3                      # one bf16 rounding of |x| < 2
        assert np.abs(got - kr[op.kv_index]).max() <= tol * max(1.0, np.abs(kr).max())
        rk, _, _ = oracle.dropped_sums(op, kr, _host(v[0, h]))
        g = ks[0, h].cpu().numpy().astype(np.float64)
        assert np.abs(g - rk).max() <= 1e-5 * max(1.0, np.abs(rk).max())


@pytest.mark.parametrize("kernel", ["tc", "simt"])
@pytest.mark.parametrize("sigma,phase,base,off", [(4, False, 100.0, 1), (9, True, 10000.0, 0), (1, False, 100.0, 2)])
def test_rope_sga_full(dev, kernel, sigma, phase, base, off):
    cfg = sga.SGAConfig(B=1, H=2, N=6, grid_h=13, grid_w=11, sigma=sigma, phase_shift=phase, kernel=kernel,
                        rope=True, rope_base=base, rope_pos_offset=off)
    q, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=91, dtype=torch.bfloat16, device=dev)
    _, out, lse, _ = _run(cfg, q, k, v, dev, lse=True)
    op = _oracle_plan(cfg)
    for h in range(2):
        ref, rl = oracle.sga_full(op, _rope_ref(q[0, h], cfg), _rope_ref(k[0, h], cfg), _host(v[0, h]))
        _compare(_host(out[0, h]), ref, "bf16", f"rope h{h}")
        assert np.abs(lse[0, h].cpu().numpy() - rl).max() < 2e-3


def test_rope_sga_odd_heads_and_tiles(dev):
    """Three heads of 258 tokens: 3 query tiles per head, so the last tiles of heads 0 and 1 share
    a mixed unit and head 2's sits in one that repeats it (odd segment count); the units are short,
    so each epilogue runs after the next unit's first P.  Every row against the oracle."""
    cfg = sga.SGAConfig(B=1, H=3, N=3, grid_h=9, grid_w=9, sigma=4, kernel="tc", rope=True, rope_base=100.0,
                        rope_pos_offset=1)
    assert cfg.T == 258
    q, k, v = correlated_qkv(1, 3, cfg.N, cfg.L, 64, seed=95, dtype=torch.bfloat16, device=dev)
    _, out, lse, _ = _run(cfg, q, k, v, dev, lse=True)
    op = _oracle_plan(cfg)
    for h in range(3):
        ref, rl = oracle.sga_full(op, _rope_ref(q[0, h], cfg), _rope_ref(k[0, h], cfg), _host(v[0, h]))
        _compare(_host(out[0, h]), ref, "bf16", f"rope odd h{h}")
        assert np.abs(lse[0, h].cpu().numpy() - rl).max() < 2e-3


def test_rope_sga_f32(dev):
    cfg = sga.SGAConfig(B=1, H=2, N=4, grid_h=9, grid_w=7, sigma=6, phase_shift=True, dtype="f32", rope=True)
    q, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=92, dtype=torch.float32, device=dev)
    _, out, _, _ = _run(cfg, q, k, v, dev)
    op = _oracle_plan(cfg)
    for h in range(2):
        ref, _ = oracle.sga_full(op, _rope_ref(q[0, h], cfg), _rope_ref(k[0, h], cfg), _host(v[0, h]))
        _compare(_host(out[0, h]), ref, "f32", f"rope f32 h{h}")


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_rope_standalone_dense_and_frame(dev, kernel):
    cfg = sga.SGAConfig(B=1, H=2, N=3, grid_h=10, grid_w=12, sigma=1, rope=True, rope_base=100.0, rope_pos_offset=1)
    q, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=93, dtype=torch.bfloat16, device=dev)
    qr, kr = q.clone(), k.clone()
    plan = sga.Plan(cfg, dev)
    plan.rope2d(qr)
    plan.rope2d(kr)
    gs = [guarded(q.shape, q.dtype, dev), guarded(q.shape, q.dtype, dev)]
    od = sga.dense_forward(qr, kr, v, kernel=kernel, out=gs[0].t)
    of = sga.frame_forward(qr, kr, v, cfg.N, cfg.L, kernel=kernel, out=gs[1].t)
    torch.cuda.synchronize(dev)
    check_all(gs, "rope dense/frame")
    rows = np.arange(cfg.T)
    for h in range(2):
        qo, ko = _rope_ref(q[0, h], cfg), _rope_ref(k[0, h], cfg)
        assert np.abs(_host(qr[0, h]) - qo).max() <= 8e-3 * max(1.0, np.abs(qo).max())
        ref, _ = oracle.attention_rows(qo, ko, _host(v[0, h]), rows)
        _compare(_host(od[0, h]), ref, "bf16", "rope dense")
        ref, _ = oracle.attention_rows(qo, ko, _host(v[0, h]), rows, frame_len=cfg.L)
        _compare(_host(of[0, h]), ref, "bf16", "rope frame")


def test_rope_rejected_where_unsupported(dev):
    cfg = sga.SGAConfig(B=1, H=1, N=2, grid_h=4, grid_w=4, rope=True)
    k = torch.zeros((1, 1, cfg.T, 64), dtype=torch.bfloat16, device=dev)
    _, S = None, sga.plan_host(cfg)[0].shape[0]
    out = [torch.zeros((1, 1, S, 64), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    sums = [torch.zeros((1, 1, 64), dtype=torch.float32, device=dev) for _ in range(2)]
    with pytest.raises(sga.SgaError):
        sga.compact_noalloc(cfg, k, k, *out, *sums)
    with pytest.raises(sga.SgaError):
        sga.Plan(sga.SGAConfig(B=1, H=1, N=2, grid_h=4, grid_w=4, rope=True, rope_base=1.0), dev)


def test_rope_vggt_sampled(dev):
    cfg = sga.SGAConfig(B=1, H=16, N=32, sigma=4, rope=True, rope_base=100.0, rope_pos_offset=1)
    q, k, v = correlated_qkv(1, cfg.H, cfg.N, cfg.L, 64, seed=94, dtype=torch.bfloat16, device=dev)
    plan = sga.Plan(cfg, dev)
    out, _, _ = _layer_guarded(plan, cfg, q, k, v, dev)
    op = _oracle_plan(cfg)
    gots, refs = [], []
    for h in range(cfg.H):
        rows = sample_rows(cfg.T, cfg.L, 256, seed=500 + h, kept=op.kept).numpy()
        qr, kr = _rope_ref(q[0, h], cfg), _rope_ref(k[0, h], cfg)
        ref, _ = oracle.sga_rows(op, qr[rows], kr, _host(v[0, h]), rows)
        gots.append(_host(out[0, h])[rows])
        refs.append(ref)
    _compare(np.concatenate(gots), np.concatenate(refs), "bf16", "rope sampled")


# ------------------------------------------------------------------------------ token merging
# "HTTM ..." section 2 (head-wise temporal merging, first-frame anchors, unmerge); merged keys
# carry ln g ("RegimeVGGT ..." Key design 2).
def _merge_check(mc, X, Y, Xm, Ym, lg, mp, b, h):
    """The GPU's grouping equals the oracle's bit for bit; merged rows are the group means."""
    m_or = oracle.merge_match(_host(X[b, h]), mc.N, mc.grid_h, mc.grid_w, mc.n_special, mc.n_t,
                              min(mc.n_s, mc.grid_h * mc.grid_w), mc.r_permille)
    kept, gid, sizes = oracle.merge_groups(m_or)
    g = mp[b, h].cpu().numpy().astype(np.int64)
    pairs = set(zip(gid.tolist(), g.tolist()))
    assert len(pairs) == len(kept) == len(set(g.tolist())) == Xm.shape[2], "partitions differ"
    perm = np.zeros(len(kept), dtype=np.int64)            # oracle group -> GPU merged row
    perm[gid] = g
    ref = oracle.merge_apply(_host(X[b, h]), gid, len(kept))
    _compare(_host(Xm[b, h])[perm], ref, mc.dtype, "merged X")
    if Y is not None:
        _compare(_host(Ym[b, h])[perm], oracle.merge_apply(_host(Y[b, h]), gid, len(kept)), mc.dtype, "merged Y")
    np.testing.assert_allclose(lg[b, h].cpu().numpy()[perm], np.log(sizes), atol=1e-6)
    return kept, gid, sizes, perm


def _merge_guarded(mc, X, Y=None):
    """sga.merge with every output between guards, checked after the call."""
    M = sga.merge_size(mc)
    dev, tdt = X.device, X.dtype
    gs = [guarded((mc.B, mc.H, M, 64), tdt, dev), guarded((mc.B, mc.H, M, 64), tdt, dev) if Y is not None else None,
          guarded((mc.B, mc.H, M), torch.float32, dev), guarded((mc.B, mc.H, mc.T), torch.int32, dev)]
    out = sga.merge(mc, X, Y, out=tuple(g.t if g is not None else None for g in gs))
    torch.cuda.synchronize(dev)
    check_all([g for g in gs if g is not None], "merge")
    return out


def _unmerge_guarded(mc, mp, Ym):
    g = guarded((mc.B, mc.H, mc.T, 64), Ym.dtype, Ym.device)
    out = sga.unmerge(mc, mp, Ym, out=g.t)
    torch.cuda.synchronize(Ym.device)
    g.check("unmerge")
    return out


@pytest.mark.parametrize("dtype,tdt", [("bf16", torch.bfloat16), ("f32", torch.float32)])
@pytest.mark.parametrize("n_t,n_s,r", [(4, 8, 500), (3, 13, 1000), (2, 64, 250)])
def test_merge_matches_oracle(dev, dtype, tdt, n_t, n_s, r):
    mc = sga.MergeConfig(B=2, H=2, N=9, grid_h=6, grid_w=7, n_t=n_t, n_s=n_s, r_permille=r, dtype=dtype)
    _, k, v = correlated_qkv(2, 2, mc.N, mc.n_special + mc.grid_h * mc.grid_w, 64, seed=100 + n_s, dtype=tdt,
                             device=dev)
    Km, Vm, lg, mp = _merge_guarded(mc, k, v)
    torch.cuda.synchronize(dev)
    assert sga.device_status(dev) == 0
    for b in range(2):
        for h in range(2):
            _merge_check(mc, k, v, Km, Vm, lg, mp, b, h)


def test_merge_ties_zero_rows_and_near_ties(dev):
    """Inputs built to stress the tensor-core shortlist (approximate cosines, exact decision):
    two identical destinations with a source equal to both (an exact tie: the lower index wins),
    an all-zero source (every cosine is 0: the first destination wins), and a destination one
    bf16 step away from another with a source equal to the first.  The partition must equal the
    oracle's bit for bit."""
    mc = sga.MergeConfig(B=1, H=1, N=4, grid_h=6, grid_w=7, n_t=4, n_s=7, r_permille=500)
    L = mc.n_special + mc.grid_h * mc.grid_w
    _, k, v = correlated_qkv(1, 1, mc.N, L, 64, seed=131, dtype=torch.bfloat16, device=dev)
    tok = lambda f, p: f * L + mc.n_special + p              # frame f, patch p
    x = k[0, 0]
    x[tok(0, 1)] = x[tok(0, 0)]                             # window 0: duplicate destinations
    x[tok(1, 3)] = x[tok(0, 0)]                             #   and a source equal to both
    x[tok(2, 9)] = 0                                        # window 1: an all-zero source
    x[tok(0, 15)] = x[tok(0, 14)]                           # window 2: destinations one step apart
    e = x[tok(0, 15), 5:6].clone()
    x[tok(0, 15), 5:6] = (e.view(torch.int16) + 1).view(torch.bfloat16)   # one bf16 step
    x[tok(3, 16)] = x[tok(0, 14)]                           #   and a source equal to the first
    Km, Vm, lg, mp = _merge_guarded(mc, k, v)
    torch.cuda.synchronize(dev)
    assert sga.device_status(dev) == 0
    _merge_check(mc, k, v, Km, Vm, lg, mp, 0, 0)


@pytest.mark.parametrize("dtype,tdt", [("bf16", torch.bfloat16), ("f32", torch.float32)])
def test_merge_largest_block(dev, dtype, tdt):
    # 8 frames x 64 patches = 512 entries per block, the largest supported; in fp32 the values
    # no longer fit in shared memory beside the keys and are read from global memory
    mc = sga.MergeConfig(B=1, H=2, N=9, grid_h=8, grid_w=8, n_t=8, n_s=64, r_permille=500, dtype=dtype)
    _, k, v = correlated_qkv(1, 2, mc.N, mc.n_special + 64, 64, seed=130, dtype=tdt, device=dev)
    Km, Vm, lg, mp = _merge_guarded(mc, k, v)
    torch.cuda.synchronize(dev)
    assert sga.device_status(dev) == 0
    for h in range(2):
        _merge_check(mc, k, v, Km, Vm, lg, mp, 0, h)


@pytest.mark.parametrize("dtype,tdt", [("bf16", torch.bfloat16), ("f32", torch.float32)])
def test_merge_nothing_is_identity(dev, dtype, tdt):
    # r = 0: every token is its own group, so unmerging the merged rows restores X exactly and
    # every group's ln g is 0
    mc = sga.MergeConfig(B=1, H=2, N=7, grid_h=6, grid_w=7, n_t=3, n_s=10, r_permille=0, dtype=dtype)
    _, k, v = correlated_qkv(1, 2, mc.N, mc.n_special + 42, 64, seed=140, dtype=tdt, device=dev)
    Km, Vm, lg, mp = _merge_guarded(mc, k, v)
    assert Km.shape[2] == mc.T
    assert torch.equal(_unmerge_guarded(mc, mp, Km), k) and torch.equal(_unmerge_guarded(mc, mp, Vm), v)
    assert torch.count_nonzero(lg) == 0
    for h in range(2):                                      # the map is a permutation per head
        assert torch.equal(torch.sort(mp[0, h]).values, torch.arange(mc.T, device=dev, dtype=mp.dtype))


def test_unmerge_gives_each_token_its_group_mean(dev):
    mc = sga.MergeConfig(B=1, H=2, N=8, grid_h=6, grid_w=7, n_t=4, n_s=7, r_permille=700, dtype="f32")
    _, k, _ = correlated_qkv(1, 2, mc.N, mc.n_special + 42, 64, seed=150, dtype=torch.float32, device=dev)
    Km, _, lg, mp = _merge_guarded(mc, k)
    back = _unmerge_guarded(mc, mp, Km)
    torch.cuda.synchronize(dev)
    for h in range(2):
        kept, gid, sizes, _ = _merge_check(mc, k, None, Km, None, lg, mp, 0, h)
        ref = oracle.merge_apply(_host(k[0, h]), gid, len(kept))[gid]      # every token's group mean
        _compare(_host(back[0, h]), ref, "f32", "unmerged means")


@pytest.mark.parametrize("merge_queries", [False, True])
def test_merged_attention(dev, merge_queries):
    mc = sga.MergeConfig(B=1, H=2, N=8, grid_h=9, grid_w=10, n_t=4, n_s=10, r_permille=600)
    L = mc.n_special + mc.grid_h * mc.grid_w
    q, k, v = correlated_qkv(1, 2, mc.N, L, 64, seed=110, dtype=torch.bfloat16, device=dev)
    out = sga.merged_attention(mc, q, k, v, merge_queries=merge_queries)
    Km, Vm, lg, mp = _merge_guarded(mc, k, v)
    torch.cuda.synchronize(dev)
    for h in range(2):
        kept, gid, sizes, _ = _merge_check(mc, k, v, Km, Vm, lg, mp, 0, h)
        km = oracle.merge_apply(_host(k[0, h]), gid, len(kept))
        vm = oracle.merge_apply(_host(v[0, h]), gid, len(kept))
        if merge_queries:
            mq = oracle.merge_match(_host(q[0, h]), mc.N, mc.grid_h, mc.grid_w, mc.n_special, mc.n_t, mc.n_s,
                                    mc.r_permille)
            qk, qgid, _ = oracle.merge_groups(mq)
            qm = oracle.merge_apply(_host(q[0, h]), qgid, len(qk))
            om, _ = oracle.biased_attention_rows(qm, km, vm, np.log(sizes))
            ref = om[qgid]                                  # unmerge: every query gets its group's row
        else:
            ref, _ = oracle.biased_attention_rows(_host(q[0, h]), km, vm, np.log(sizes))
        _compare(_host(out[0, h]), ref, "bf16", f"merged attention h{h}")


def test_merge_vggt_sampled(dev):
    # 32 VGGT frames, chunks of 4 frames, one patch row per run, half of the sources merged
    mc = sga.MergeConfig(B=1, H=16, N=32, n_t=4, n_s=37, r_permille=500)
    L = 1374
    q, k, v = correlated_qkv(1, mc.H, mc.N, L, 64, seed=120, dtype=torch.bfloat16, device=dev)
    Km, Vm, lg, mp = _merge_guarded(mc, k, v)
    out = sga.bias_forward(q, Km, Vm, lg)
    torch.cuda.synchronize(dev)
    assert sga.device_status(dev) == 0
    gots, refs = [], []
    for h in range(mc.H):
        kept, gid, sizes, _ = _merge_check(mc, k, v, Km, Vm, lg, mp, 0, h)
        km = oracle.merge_apply(_host(k[0, h]), gid, len(kept))
        vm = oracle.merge_apply(_host(v[0, h]), gid, len(kept))
        rows = sample_rows(mc.T, L, 128, seed=600 + h).numpy()
        ref, _ = oracle.biased_attention_rows(_host(q[0, h])[rows], km, vm, np.log(sizes))
        gots.append(_host(out[0, h])[rows])
        refs.append(ref)
    _compare(np.concatenate(gots), np.concatenate(refs), "bf16", "merged sampled")


# ------------------------------------------------------------------------------ the benchmarked shapes
# Every workload the benchmark times, at its own shape and in its launch configuration, against
# the oracle on sampled rows (outputs between guards).
def test_dense_benched_shape_sampled(dev):
    # dense global attention over 32 VGGT frames: 43,968 tokens, 16 heads
    N, L, H = 32, 1374, 16
    q, k, v = correlated_qkv(1, H, N, L, 64, seed=160, dtype=torch.bfloat16, device=dev)
    g = guarded(q.shape, q.dtype, dev)
    out = sga.dense_forward(q, k, v, out=g.t)
    torch.cuda.synchronize(dev)
    g.check("dense")
    gots, refs = [], []
    for h in range(H):
        rows = sample_rows(N * L, L, 128, seed=700 + h).numpy()
        ref, _ = oracle.attention_rows(_host(q[0, h])[rows], _host(k[0, h]), _host(v[0, h]), rows)
        gots.append(_host(out[0, h])[rows])
        refs.append(ref)
    _compare(np.concatenate(gots), np.concatenate(refs), "bf16", "dense benched shape")


def test_size_aware_benched_shape_sampled(dev):
    # 274,800 queries (200 frames) against 137,400 merged keys standing for 1-3 tokens (ln g)
    H, Tq, Tk = 16, 274800, 137400
    q, _, _ = correlated_qkv(1, H, 1, Tq, 64, seed=170, dtype=torch.bfloat16, device=dev)
    _, k, v = correlated_qkv(1, H, 1, Tk, 64, seed=171, dtype=torch.bfloat16, device=dev)
    gen = torch.Generator(device=dev).manual_seed(172)
    bias = torch.log(torch.randint(1, 4, (1, H, Tk), generator=gen, device=dev).float()).contiguous()
    g = guarded(q.shape, q.dtype, dev)
    out = sga.bias_forward(q, k, v, bias, out=g.t)
    torch.cuda.synchronize(dev)
    g.check("size-aware")
    gots, refs = [], []
    for h in range(H):
        rows = sample_rows(Tq, 1374, 48, seed=800 + h).numpy()
        ref, _ = oracle.biased_attention_rows(_host(q[0, h])[rows], _host(k[0, h]), _host(v[0, h]),
                                              bias[0, h].double().cpu().numpy())
        gots.append(_host(out[0, h])[rows])
        refs.append(ref)
    _compare(np.concatenate(gots), np.concatenate(refs), "bf16", "size-aware benched shape")


@pytest.mark.parametrize("N,sigma", [(800, 4), (200, 9)])
def test_rope_benched_shapes_sampled(dev, N, sigma):
    # the SGA layer with the fused rotation (base 100, position offset 1)
    cfg = sga.SGAConfig(B=1, H=16, N=N, sigma=sigma, rope=True, rope_base=100.0, rope_pos_offset=1)
    q, k, v = correlated_qkv(1, cfg.H, cfg.N, cfg.L, 64, seed=180 + N, dtype=torch.bfloat16, device=dev)
    plan = sga.Plan(cfg, dev)
    out, _, _ = _layer_guarded(plan, cfg, q, k, v, dev)
    op = _oracle_plan(cfg)
    gots, refs = [], []
    for h in range(cfg.H):
        rows = sample_rows(cfg.T, cfg.L, 96, seed=900 + h, kept=op.kept).numpy()
        qr, kr = _rope_ref(q[0, h], cfg), _rope_ref(k[0, h], cfg)
        ref, _ = oracle.sga_rows(op, qr[rows], kr, _host(v[0, h]), rows)
        gots.append(_host(out[0, h])[rows])
        refs.append(ref)
    _compare(np.concatenate(gots), np.concatenate(refs), "bf16", f"rope N={N}")


def test_general_plan_benched_shape_sampled(dev):
    # 200 frames, per-axis sigma_b = 1.3 with phase shift, 10 % of the tokens protected
    cfg = sga.SGAConfig(B=1, H=16, N=200)
    op, q, k, v, out = _general_case(dev, cfg, (13, 10), (13, 10), True, n_prot=cfg.T // 10, seed=190)
    gots, refs = [], []
    for h in range(cfg.H):
        rows = sample_rows(cfg.T, cfg.L, 96, seed=1000 + h, kept=op.kept).numpy()
        ref, _ = oracle.sga_rows(op, _host(q[0, h])[rows], _host(k[0, h]), _host(v[0, h]), rows)
        gots.append(_host(out[0, h])[rows])
        refs.append(ref)
    _compare(np.concatenate(gots), np.concatenate(refs), "bf16", "general benched shape")


def test_merge_benched_shape(dev):
    # head-wise temporal merging at 200 frames (chunks of 4 frames, 37-patch runs, half of the
    # sources merged), then size-aware attention of all queries over the merged keys: the
    # partition bit for bit on three heads, and sampled attention rows there
    mc = sga.MergeConfig(B=1, H=16, N=200, n_t=4, n_s=37, r_permille=500)
    L = 1374
    q, k, v = correlated_qkv(1, mc.H, mc.N, L, 64, seed=200, dtype=torch.bfloat16, device=dev)
    Km, Vm, lg, mp = _merge_guarded(mc, k, v)
    g = guarded(q.shape, q.dtype, dev)
    out = sga.bias_forward(q, Km, Vm, lg, out=g.t)
    torch.cuda.synchronize(dev)
    assert sga.device_status(dev) == 0
    g.check("merged attention")
    gots, refs = [], []
    for h in (0, 7, 15):
        kept, gid, sizes, _ = _merge_check(mc, k, v, Km, Vm, lg, mp, 0, h)
        km = oracle.merge_apply(_host(k[0, h]), gid, len(kept))
        vm = oracle.merge_apply(_host(v[0, h]), gid, len(kept))
        rows = sample_rows(mc.T, L, 96, seed=1100 + h).numpy()
        ref, _ = oracle.biased_attention_rows(_host(q[0, h])[rows], km, vm, np.log(sizes))
        gots.append(_host(out[0, h])[rows])
        refs.append(ref)
    _compare(np.concatenate(gots), np.concatenate(refs), "bf16", "merge benched shape")


def test_last_device_status_reads_the_plan_device(dev):
    cfg = sga.SGAConfig(B=1, H=2, N=4, grid_h=8, grid_w=8, sigma=4)
    q, k, v = correlated_qkv(1, 2, cfg.N, cfg.L, 64, seed=210, dtype=torch.bfloat16, device=dev)
    plan = sga.Plan(cfg, dev)
    plan.layer(q, k, v)
    assert sga.last_device_status(plan) == 0
    plan.close()
    with pytest.raises(sga.SgaError):
        sga.last_device_status(plan)        # the handle is gone: refused on the host
