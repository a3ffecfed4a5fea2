"""CPU-side checks of the library: the C ABI loads and exports every declared symbol, the host
plan builder matches the oracle's kept set bit for bit, and argument validation rejects bad
configurations before any device work."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import subsampled_global_attention_sga_b300 as sga
from subsampled_global_attention_sga_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "sga.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sga_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    L = sga.lib()
    declared = _declared_functions()
    assert declared, "no declarations parsed"
    assert set(declared) == set(_lib.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name
    assert b"sm_103a" in L.sga_build_info()


def test_library_carries_its_source_fingerprint(monkeypatch):
    """The library names the sources it was compiled from, and the binding refuses a library
    whose fingerprint differs from the tree's (a stale build)."""
    from subsampled_global_attention_sga_b300 import _build
    info = _lib.lib().sga_build_info().decode()
    assert info.endswith("src=" + _build.source_hash())
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "_tree_source_hash", lambda: "0000000000000000")
    with pytest.raises(RuntimeError, match="other sources"):
        _lib.lib()


def test_debug_report_only_in_debug_builds():
    # the normal build has no index checks to report; its debug twin carries the same sources
    import ctypes as C
    w = [C.c_int64(0) for _ in range(4)]
    assert sga.lib().sga_debug_report(*[C.byref(x) for x in w]) == 2
    assert b"debug" not in sga.lib().sga_build_info()
    from subsampled_global_attention_sga_b300 import _build
    if os.path.exists(_build.LIB_DEBUG):
        L = C.CDLL(_build.LIB_DEBUG)
        L.sga_build_info.restype = C.c_char_p
        info = L.sga_build_info().decode()
        assert "debug" in info and info.endswith("src=" + _build.source_hash())


def test_status_strings():
    L = sga.lib()
    for s in range(7):
        assert L.sga_status_string(s)


def test_sigma_windows_match_golden():
    rows = [list(map(int, l.split())) for l in open(os.path.join(GOLDEN, "sigma_map.txt"))
            if l.strip() and not l.startswith("#")]
    assert {s: (a, b) for s, a, b in rows} == sga.SIGMA_WINDOWS
    with pytest.raises(ValueError):
        sga.sigma_window(3)


PLAN_CASES = [
    (4, 8, 8, 5, 4, None, False, True),
    (32, 37, 37, 5, 4, None, False, True),
    (32, 37, 37, 5, 4, None, True, True),
    (200, 37, 37, 5, 9, None, False, True),
    (200, 37, 37, 5, 9, None, True, True),
    (17, 37, 28, 5, 6, None, True, True),
    (9, 7, 5, 5, 2, None, True, False),
    (9, 7, 5, 0, 9, None, True, False),
    (3, 1, 1, 5, 4, None, True, True),
    (5, 6, 6, 2, 1, None, True, False),
    (6, 9, 10, 5, 0, (3, 2), True, True),
]


@pytest.mark.parametrize("case", PLAN_CASES)
def test_host_plan_bit_exact_vs_oracle(case):
    N, gh, gw, nsp, sigma, window, phase, ref = case
    cfg = sga.SGAConfig(B=1, H=1, N=N, grid_h=gh, grid_w=gw, n_special=nsp,
                        sigma=sigma if sigma else 4, window=window, phase_shift=phase, ref_frame_dense=ref)
    s_h, s_w = cfg.s_hw
    kv, off, slot = sga.plan_host(cfg)
    op = oracle.plan(N, gh, gw, nsp, s_h, s_w, phase, ref)
    assert np.array_equal(kv, op.kv_index)
    assert np.array_equal(off, op.frame_off)
    want_slot = np.full(op.T, -1, dtype=np.int32)
    want_slot[op.kv_index] = np.arange(op.S, dtype=np.int32)
    assert np.array_equal(slot, want_slot)


def test_headline_plan_counts():
    for ph, S in ((False, 293808), (True, 278808)):
        cfg = sga.SGAConfig(B=1, H=16, N=800, sigma=4, phase_shift=ph)
        kv, off, _ = sga.plan_host(cfg)
        assert len(kv) == S and off[-1] == S and cfg.T == 1099200


@pytest.mark.parametrize("bad", [dict(head_dim=32), dict(N=0), dict(grid_h=0), dict(window=(0, 2)),
                                 dict(mean_mode="loo", dtype="f32", kernel="tc")])
def test_invalid_configs_rejected(bad):
    kw = dict(B=1, H=1, N=2, grid_h=4, grid_w=4)
    kw.update(bad)
    cfg = sga.SGAConfig(**kw)
    with pytest.raises(sga.SgaError):
        sga.plan_host(cfg)


def test_null_arguments_rejected_without_device():
    L = sga.lib()
    assert L.sga_plan_host(None, None, None, None, None) == 1
    assert L.sga_plan_info(None, None, None, None) == 6
    assert L.sga_compact(None, None, None, None, None, None, None, None) == 6
    L.sga_plan_destroy(None)
    # dense/frame validate shapes and pointers before touching the device
    assert L.sga_dense_forward(1, 1, 128, 32, 0, 0, None, None, None, None, None, ctypes.c_float(0.125), None) == 2
    assert L.sga_dense_forward(1, 1, 128, 64, 0, 0, None, None, None, None, None, ctypes.c_float(0.125), None) == 1
    assert L.sga_frame_forward(1, 1, 0, 10, 64, 0, 0, None, None, None, None, None, ctypes.c_float(0.125), None) == 1
    buf = (ctypes.c_char * 64)()
    p = ctypes.addressof(buf) + 1  # misaligned
    assert L.sga_dense_forward(1, 1, 4, 64, 0, 0, p, p, p, p, None, ctypes.c_float(0.125), None) == 3
    # the host-streaming executor rejects a missing plan or object before any CUDA call
    h = ctypes.c_void_p()
    assert L.sga_stream_create(None, 2, ctypes.byref(h)) == 1 and not h.value
    assert L.sga_stream_submit(None, p, p, p, p, ctypes.c_float(0.125)) == 1
    assert L.sga_stream_synchronize(None) == 1
    assert L.sga_stream_handles(None, None, None, None) == 1
    L.sga_stream_destroy(None)
    # the plain executor validates its description before any CUDA call
    spec = sga._lib.SgaPlainSpec()
    spec.kind, spec.B, spec.H, spec.Tq, spec.head_dim = 7, 1, 1, 128, 64
    assert L.sga_stream_create_plain(ctypes.byref(spec), 2, ctypes.byref(h)) == 1 and not h.value
    spec.kind, spec.N, spec.L = 2, 3, 40                      # frame-local with N*L != Tq
    assert L.sga_stream_create_plain(ctypes.byref(spec), 2, ctypes.byref(h)) == 1
    spec.kind, spec.head_dim = 1, 32
    assert L.sga_stream_create_plain(ctypes.byref(spec), 2, ctypes.byref(h)) == 2
    assert L.sga_stream_create_plain(None, 2, ctypes.byref(h)) == 1
    assert L.sga_stream_submit_plain(None, p, p, p, None, p, ctypes.c_float(0.125)) == 1


KEPT_COUNT_CASES = [
    # N, grid_h, grid_w, n_special, window, phase, ref_dense
    (4, 8, 8, 5, (2, 2), False, True),
    (13, 37, 28, 5, (2, 3), True, False),
    (9, 37, 37, 5, (3, 3), True, True),
    (6, 13, 11, 0, (1, 2), True, True),
    (1, 5, 7, 3, (3, 3), False, False),
    (5, 2, 2, 5, (3, 3), True, False),       # grid smaller than the window
    (3, 9, 7, 5, (1, 1), False, True),       # sigma = 1 keeps every token
    (800, 37, 37, 5, (2, 2), False, True),
    (800, 37, 37, 5, (2, 2), True, True),
]


@pytest.mark.parametrize("case", KEPT_COUNT_CASES)
def test_kept_count_matches_oracle(case):
    """sga_kept_count (the closed form that sizes sga_compact_noalloc's outputs) equals |S| of
    the oracle's plan, which enumerates the kept set token by token."""
    N, gh, gw, nsp, win, ph, ref = case
    cfg = sga.SGAConfig(B=1, H=2, N=N, grid_h=gh, grid_w=gw, n_special=nsp, window=win, phase_shift=ph,
                        ref_frame_dense=ref)
    op = oracle.plan(N, gh, gw, nsp, win[0], win[1], ph, ref)
    assert sga.kept_count(cfg) == op.S


def test_kept_count_rejects_bad_arguments():
    with pytest.raises(sga.SgaError):
        sga.kept_count(sga.SGAConfig(B=1, H=1, N=0, grid_h=4, grid_w=4))
    c = sga.SGAConfig(B=1, H=1, N=2, grid_h=4, grid_w=4).to_c()
    assert sga.lib().sga_kept_count(ctypes.byref(c), None) == 1
    assert sga.lib().sga_kept_count(None, None) == 1
    # the plan-based status read refuses a missing plan before any CUDA call
    assert sga.lib().sga_last_device_status(None, None) == 6


GENERAL_CASES = [
    # N, gh, gw, nsp, sigma_h, sigma_w, phase, ref, n_protected
    (7, 11, 13, 5, (3, 2), (3, 2), False, True, 0),
    (7, 11, 13, 5, (13, 10), (17, 10), True, True, 12),
    (5, 37, 28, 5, (17, 10), (3, 2), True, False, 40),
    (9, 37, 37, 5, (2, 1), (2, 1), True, True, 0),
    (3, 4, 6, 0, (7, 3), (1, 1), True, False, 5),
    (800, 37, 37, 5, (3, 2), (3, 2), True, True, 1000),
]


@pytest.mark.parametrize("case", GENERAL_CASES)
def test_general_plan_bit_exact_vs_oracle(case):
    N, gh, gw, nsp, sh, sw, phase, ref, n_prot = case
    T = N * (nsp + gh * gw)
    prot = np.random.default_rng(N * 7 + gh).integers(0, T, size=n_prot)
    kv, off, slot = sga.plan_host_general(N, gh, gw, nsp, sigma_h=sh, sigma_w=sw, phase_shift=phase,
                                          ref_frame_dense=ref, protected=prot)
    op = oracle.plan_general(N, gh, gw, nsp, sh, sw, phase, ref, protected=prot)
    assert np.array_equal(kv, op.kv_index)
    assert np.array_equal(off, op.frame_off)
    want_slot = np.full(op.T, -1, dtype=np.int32)
    want_slot[op.kv_index] = np.arange(op.S, dtype=np.int32)
    assert np.array_equal(slot, want_slot)


def test_general_plan_rejects_bad_specs():
    with pytest.raises(sga.SgaError):
        sga.plan_host_general(2, 4, 4, 5, sigma_h=(1, 2))          # sigma < 1
    with pytest.raises(sga.SgaError):
        sga.plan_host_general(2, 4, 4, 5, protected=[2 * 21])      # outside [0, N*L)


@pytest.mark.parametrize("N,gh,gw,nsp,n_t,n_s,r", [(9, 6, 7, 5, 4, 8, 500), (800, 37, 37, 5, 4, 37, 500),
                                                   (7, 5, 5, 0, 3, 25, 1000), (5, 4, 9, 5, 5, 13, 0),
                                                   (11, 37, 28, 5, 2, 100, 333)])
def test_merge_size_matches_oracle_merge_count(N, gh, gw, nsp, n_t, n_s, r):
    mc = sga.MergeConfig(B=1, H=1, N=N, grid_h=gh, grid_w=gw, n_special=nsp, n_t=n_t, n_s=n_s, r_permille=r)
    if N > 100:   # count per block in closed form (the oracle merges exactly floor(#src * r / 1000))
        P, ns = gh * gw, min(n_s, gh * gw)
        merged = sum(((min(n_t, N - f0) - 1) * min(ns, P - w0) * r) // 1000
                     for f0 in range(0, N, n_t) for w0 in range(0, P, ns))
    else:
        X = np.random.default_rng(N).standard_normal((mc.T, 64)).astype(np.float32)
        merged = int((oracle.merge_match(X, N, gh, gw, nsp, n_t, min(n_s, gh * gw), r) >= 0).sum())
    assert sga.merge_size(mc) == mc.T - merged


def test_merge_rejects_bad_configs():
    for bad in (dict(n_t=0), dict(r_permille=1001), dict(n_t=9, n_s=100)):   # 9 x 64 > 512
        kw = dict(B=1, H=1, N=4, grid_h=8, grid_w=8, n_s=16)
        kw.update(bad)
        with pytest.raises(sga.SgaError):
            sga.merge_size(sga.MergeConfig(**kw))
