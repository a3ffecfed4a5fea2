"""Pins for the fp64 CPU oracle: each test checks the oracle against something other than
itself -- the pages' printed rules (golden fixtures), closed forms, textbook/library attention,
exact identities and a brute-force re-derivation on tiny inputs.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from subsampled_global_attention_sga_b300.inputs import correlated_qkv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SCALE = 0.125  # 1/sqrt(64)


def _rows(path):
    out = []
    for line in open(os.path.join(GOLDEN, path)):
        line = line.strip()
        if line and not line.startswith("#"):
            out.append([int(x) for x in line.split()])
    return out


def _sdpa(q, k, v, scale=SCALE):
    q = torch.as_tensor(q, dtype=torch.float64)[None, None]
    k = torch.as_tensor(k, dtype=torch.float64)[None, None]
    v = torch.as_tensor(v, dtype=torch.float64)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)[0, 0].numpy()


def _textbook(q, k, v, scale=SCALE):
    s = (q.astype(np.float64) @ k.astype(np.float64).T) * scale
    s -= s.max(axis=1, keepdims=True)
    w = np.exp(s)
    w /= w.sum(axis=1, keepdims=True)
    return w @ v.astype(np.float64)


def _qkv(N, L, H=1, seed=0, q_scale=1.0):
    q, k, v = correlated_qkv(1, H, N, L, 64, seed=seed, dtype=torch.float32, q_scale=q_scale)
    return q[0].numpy(), k[0].numpy(), v[0].numpy()


# ------------------------------------------------------------------------------ plan pins
def test_plan_counts_closed_form_golden():
    for N, gh, gw, nsp, sh, sw, ph, rd, T, S, c in _rows("plan_counts.txt"):
        p = oracle.plan(N, gh, gw, nsp, sh, sw, bool(ph), bool(rd))
        assert (p.T, p.S, p.dropped) == (T, S, c)


@pytest.mark.parametrize("gh,gw", [(8, 8), (7, 5), (37, 28), (1, 1), (2, 9)])
@pytest.mark.parametrize("sigma", [1, 2, 4, 6, 9])
@pytest.mark.parametrize("phase", [False, True])
@pytest.mark.parametrize("ref", [False, True])
def test_plan_per_frame_counts(gh, gw, sigma, phase, ref):
    smap = {s: (a, b) for s, a, b in _rows("sigma_map.txt")}
    sh, sw = smap[sigma]
    N, nsp = 11, 5
    p = oracle.plan(N, gh, gw, nsp, sh, sw, phase, ref)
    L = nsp + gh * gw
    for f in range(N):
        got = p.frame_off[f + 1] - p.frame_off[f]
        if f == 0 and ref:
            want = L
        else:
            pr, pc = ((f // sw) % sh, f % sw) if phase else (0, 0)
            want = nsp + math.ceil(max(0, gh - pr) / sh) * math.ceil(max(0, gw - pc) / sw)
        assert got == want, (f, got, want)
    assert np.all(np.diff(p.kv_index) > 0)
    assert p.kept.sum() == p.S
    assert np.array_equal(np.nonzero(p.kept)[0], p.kv_index)


def test_sigma_map_golden_windows():
    # the first patch of every s_h x s_w window is kept and nothing else (fixed grid)
    for sigma, sh, sw in _rows("sigma_map.txt"):
        assert sh * sw == sigma
        gh, gw, nsp = 7, 8, 5
        p = oracle.plan(2, gh, gw, nsp, sh, sw, False, True)
        L = nsp + gh * gw
        frame1 = p.kept[L:2 * L]
        assert frame1[:nsp].all()
        kept_rc = {divmod(int(x) - nsp, gw) for x in np.nonzero(frame1[nsp:])[0] + nsp}
        windows = {(wr * sh, wc * sw) for wr in range(math.ceil(gh / sh)) for wc in range(math.ceil(gw / sw))}
        assert kept_rc == windows
        assert p.kept[:L].all()  # frame 0 dense


def test_phase_offsets_golden():
    for t, f, ro, co in _rows("phase_offsets.txt"):
        gh = gw = 6
        nsp = 5
        N = f + 1
        p = oracle.plan(N, gh, gw, nsp, t, t, True, False)
        L = nsp + gh * gw
        fr = p.kept[f * L:(f + 1) * L]
        kept_rc = sorted(divmod(int(x), gw) for x in np.nonzero(fr[nsp:])[0])
        assert kept_rc[0] == (ro, co)  # the first kept patch sits at the frame's offset
        assert all(r % t == ro and c % t == co for r, c in kept_rc)


@pytest.mark.parametrize("sh,sw", [(1, 2), (2, 2), (2, 3), (3, 3)])
def test_phase_coverage(sh, sw):
    # with the phase shift, any sigma consecutive frames together cover every grid position once
    gh, gw, nsp = 9, 10, 5
    sigma = sh * sw
    N = 2 * sigma + 3
    p = oracle.plan(N, gh, gw, nsp, sh, sw, True, False)
    L = nsp + gh * gw
    for f0 in range(N - sigma + 1):
        cover = np.zeros(gh * gw, dtype=int)
        for f in range(f0, f0 + sigma):
            cover += p.kept[f * L + nsp:(f + 1) * L]
        assert np.all(cover == 1), f0


def test_sigma1_keeps_everything():
    p = oracle.plan(3, 5, 4, 5, 1, 1, True, False)
    assert p.S == p.T and p.dropped == 0


# ------------------------------------------------------------------------------ attention pins
def test_dense_equals_textbook_and_sdpa():
    q, k, v = _qkv(4, 69)
    rows = np.arange(q.shape[1])
    out, lse = oracle.attention_rows(q[0], k[0], v[0], rows)
    np.testing.assert_allclose(out, _sdpa(q[0], k[0], v[0]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out, _textbook(q[0], k[0], v[0]), rtol=0, atol=1e-12)
    s = (q[0].astype(np.float64) @ k[0].astype(np.float64).T) * SCALE
    m = s.max(axis=1)
    np.testing.assert_allclose(lse, m + np.log(np.exp(s - m[:, None]).sum(axis=1)), atol=1e-12)


def test_frame_equals_per_frame_sdpa():
    N, L = 5, 23
    q, k, v = _qkv(N, L)
    out, _ = oracle.attention_rows(q[0], k[0], v[0], np.arange(N * L), frame_len=L)
    for f in range(N):
        sl = slice(f * L, (f + 1) * L)
        np.testing.assert_allclose(out[sl], _sdpa(q[0][sl], k[0][sl], v[0][sl]), atol=1e-12)


def test_sigma1_sga_equals_dense():
    N, gh, gw, nsp = 4, 8, 8, 5
    p = oracle.plan(N, gh, gw, nsp, 1, 1, False, True)
    q, k, v = _qkv(N, p.L, H=2)
    for h in range(2):
        out, lse = oracle.sga_full(p, q[h], k[h], v[h])
        np.testing.assert_allclose(out, _sdpa(q[h], k[h], v[h]), atol=1e-12)


def _equal_dropped(p, k, v, rng):
    k = k.copy()
    v = v.copy()
    kb = rng.standard_normal(64).astype(np.float32)
    vb = rng.standard_normal(64).astype(np.float32)
    d = p.kept == 0
    k[d] = kb
    v[d] = vb
    return k, v


@pytest.mark.parametrize("sh,sw,phase,ref", [(2, 2, False, True), (2, 3, True, True),
                                             (3, 3, True, False), (1, 2, False, False)])
def test_identity_equal_dropped_rows_equals_dense(sh, sw, phase, ref):
    # every dropped key/value equal: the diagonal plus the log(count)-biased mean reproduce the
    # dropped keys exactly, so SGA equals dense attention for kept and dropped queries alike
    N, gh, gw, nsp = 4, 8, 7, 5
    p = oracle.plan(N, gh, gw, nsp, sh, sw, phase, ref)
    q, k, v = _qkv(N, p.L, seed=3)
    rng = np.random.default_rng(7)
    k2, v2 = _equal_dropped(p, k[0], v[0], rng)
    out, _ = oracle.sga_full(p, q[0], k2, v2)
    np.testing.assert_allclose(out, _sdpa(q[0], k2, v2), atol=1e-12)


def test_identity_is_sensitive_to_each_term():
    # planted mistakes (each switches off or alters one part of the oracle): the identity must fail
    N, gh, gw, nsp = 4, 8, 8, 5
    p = oracle.plan(N, gh, gw, nsp, 2, 2, False, True)
    q, k, v = _qkv(N, p.L, seed=5)
    k2, v2 = _equal_dropped(p, k[0], v[0], np.random.default_rng(1))
    ref = _sdpa(q[0], k2, v2)
    drop = p.kept == 0
    for kw in (dict(diag=False), dict(mean=False), dict(mean_mode=1)):
        out, _ = oracle.sga_full(p, q[0], k2, v2, **kw)
        assert np.abs(out[drop] - ref[drop]).max() > 1e-4, kw
    # a wrong bias (log2 instead of ln, or no bias) is caught as well: emulate it by feeding
    # sums scaled so that the mean key is unchanged but the count differs
    ks, vs, c = oracle.dropped_sums(p, k2, v2)
    out, _ = oracle.sga_full(p, q[0], k2, v2, sums=(ks * 2, vs * 2, c))
    assert np.abs(out - ref).max() > 1e-4


def test_zero_query_gives_mean_of_all_values():
    N, gh, gw, nsp = 4, 8, 8, 5
    for (sh, sw, ph) in [(2, 2, False), (3, 3, True), (1, 1, False)]:
        p = oracle.plan(N, gh, gw, nsp, sh, sw, ph, True)
        _, k, v = _qkv(N, p.L, seed=11)
        q0 = np.zeros((p.T, 64), np.float32)
        out, lse = oracle.sga_full(p, q0, k[0], v[0])
        want = v[0].astype(np.float64).mean(axis=0)
        np.testing.assert_allclose(out, np.broadcast_to(want, out.shape), atol=1e-12)
        np.testing.assert_allclose(lse, np.log(p.T), atol=1e-12)
        outd, _ = oracle.attention_rows(q0, k[0], v[0], np.arange(p.T))
        np.testing.assert_allclose(outd, np.broadcast_to(want, out.shape), atol=1e-12)


# ------------------------------------------------------------------------------ brute force
def _bf_kept(N, gh, gw, nsp, sh, sw, phase, ref):
    """Kept tokens by enumerating windows (a formulation independent of the oracle's)."""
    L = nsp + gh * gw
    kept = set()
    for f in range(N):
        if f == 0 and ref:
            kept.update(range(0, L))
            continue
        kept.update(f * L + p for p in range(nsp))
        r0, c0 = ((f // sw) % sh, f % sw) if phase else (0, 0)
        for wr in range(r0, gh, sh):
            for wc in range(c0, gw, sw):
                kept.add(f * L + nsp + wr * gw + wc)  # top-left token of the window
    return kept


def _bf_row(i, q, k, v, kept, T, diag, mean, mean_mode, scale=SCALE):
    entries = []  # (token ids it stands for, key, value, bias)
    for t in sorted(kept):
        entries.append(([t], k[t].astype(np.float64), v[t].astype(np.float64), 0.0))
    dropped = [t for t in range(T) if t not in kept]
    if diag and i not in kept:
        entries.append(([i], k[i].astype(np.float64), v[i].astype(np.float64), 0.0))
    if mean:
        src = [t for t in dropped if (t != i or mean_mode == 1)]
        if src:
            kb = np.mean([k[t].astype(np.float64) for t in src], axis=0)
            vb = np.mean([v[t].astype(np.float64) for t in src], axis=0)
            entries.append((src, kb, vb, math.log(len(src))))
    logits = [scale * float(np.dot(q.astype(np.float64), e[1])) + e[3] for e in entries]
    m = max(logits)
    ws = [math.exp(x - m) for x in logits]
    z = math.fsum(ws)
    o = sum(w * e[2] for w, e in zip(ws, entries)) / z
    srcs = [t for e in entries for t in e[0]]
    return o, m + math.log(z), [w / z for w in ws], srcs


CASES = [
    # N, gh, gw, nsp, sh, sw, phase, ref, diag, mean, mode
    (4, 8, 8, 5, 2, 2, False, True, True, True, 0),
    (4, 8, 8, 5, 2, 2, True, True, True, True, 0),
    (3, 7, 5, 5, 2, 3, True, False, True, True, 0),
    (3, 6, 6, 5, 3, 3, False, True, True, False, 0),
    (3, 6, 6, 5, 3, 3, False, True, False, True, 0),
    (3, 6, 6, 5, 3, 3, True, True, True, True, 1),
    (2, 4, 5, 0, 1, 2, False, False, True, True, 0),
    (2, 3, 3, 2, 3, 3, False, False, True, True, 0),  # one kept patch per frame
]


@pytest.mark.parametrize("case", CASES)
def test_bruteforce_agrees(case):
    N, gh, gw, nsp, sh, sw, ph, ref, diag, mean, mode = case
    p = oracle.plan(N, gh, gw, nsp, sh, sw, ph, ref)
    kept = _bf_kept(N, gh, gw, nsp, sh, sw, ph, ref)
    assert kept == set(p.kv_index.tolist())
    q, k, v = _qkv(N, p.L, seed=2, q_scale=3.0)
    rows = np.arange(p.T)
    out, lse = oracle.sga_rows(p, q[0], k[0], v[0], rows, diag=diag, mean=mean, mean_mode=mode)
    for i in rows:
        o, l, w, srcs = _bf_row(int(i), q[0][i], k[0], v[0], kept, p.T, diag, mean, mode)
        np.testing.assert_allclose(out[i], o, atol=1e-12)
        assert abs(lse[i] - l) < 1e-12
        assert abs(math.fsum(w) - 1.0) < 1e-12
        if diag and mean and mode == 0:
            # the three components partition the keys: S, {i} if dropped, D \ {i}
            assert sorted(srcs) == list(range(p.T))


def test_mean_count_zero_drops_the_term():
    # one dropped token only: for that query c_i = 0 (no mean term), the others see count 1
    N, gh, gw, nsp = 2, 1, 2, 0
    p = oracle.plan(N, gh, gw, nsp, 1, 2, False, True)
    assert p.dropped == 1
    q, k, v = _qkv(N, p.L, seed=9)
    out, _ = oracle.sga_full(p, q[0], k[0], v[0])
    np.testing.assert_allclose(out, _sdpa(q[0], k[0], v[0]), atol=1e-12)


def test_appended_column_identity():
    # RegimeVGGT's size-aware bias absorbed into an extra column: [q, 1] . [k, sqrt(d) ln g]
    # scaled by 1/sqrt(d) equals q.k/sqrt(d) + ln g.  Rebuild each row's SGA softmax that way
    # and run it through torch SDPA (d + 1 = 65 columns, scale kept at 1/sqrt(64)).
    N, gh, gw, nsp = 4, 8, 8, 5
    p = oracle.plan(N, gh, gw, nsp, 2, 2, True, True)
    q, k, v = _qkv(N, p.L, seed=4)
    out, _ = oracle.sga_full(p, q[0], k[0], v[0])
    ks, vs, c = oracle.dropped_sums(p, k[0], v[0])
    for i in [0, 7, 80, 100, 200, p.T - 1]:
        keys = [np.append(k[0][t].astype(np.float64), 0.0) for t in p.kv_index]
        vals = [v[0][t].astype(np.float64) for t in p.kv_index]
        if not p.kept[i]:
            keys.append(np.append(k[0][i].astype(np.float64), 0.0))
            vals.append(v[0][i].astype(np.float64))
            ci = c - 1
            kb = (ks - k[0][i]) / ci
            vb = (vs - v[0][i]) / ci
        else:
            ci = c
            kb, vb = ks / ci, vs / ci
        keys.append(np.append(kb, math.sqrt(64) * math.log(ci)))
        vals.append(vb)
        qq = np.append(q[0][i].astype(np.float64), 1.0)[None]
        got = _sdpa(qq, np.array(keys), np.array(vals), scale=SCALE)[0]
        np.testing.assert_allclose(out[i], got, atol=1e-12)


# ------------------------------------------------------------------------------ size-aware bias
# "RegimeVGGT ..." Key design 2: softmax(QK^T/sqrt(d) + log g) V, a key standing for g tokens.
def test_biased_integer_groups_equal_expanded_keys():
    # a key with bias ln g is exactly g copies of that key: compare with fp64 SDPA over the
    # key set in which every key is repeated g times
    rng = np.random.default_rng(21)
    q, k, v = _qkv(3, 40, seed=13)
    q, k, v = q[0][:50], k[0][:37], v[0][:37]
    g = rng.integers(1, 6, size=37)
    out, lse = oracle.biased_attention_rows(q, k, v, np.log(g))
    ke, ve = np.repeat(k, g, axis=0), np.repeat(v, g, axis=0)
    np.testing.assert_allclose(out, _sdpa(q, ke, ve), atol=1e-12)
    s = (q.astype(np.float64) @ ke.astype(np.float64).T) * SCALE
    m = s.max(axis=1)
    np.testing.assert_allclose(lse, m + np.log(np.exp(s - m[:, None]).sum(axis=1)), atol=1e-12)
    # planted mistake: a base-2 logarithm instead of ln no longer reproduces the copies
    bad, _ = oracle.biased_attention_rows(q, k, v, np.log2(g))
    assert np.abs(bad - out).max() > 1e-3


def test_biased_constant_and_removed_keys():
    q, k, v = _qkv(2, 30, seed=14)
    q, k, v = q[0], k[0], v[0]
    out, lse = oracle.biased_attention_rows(q, k, v, np.full(len(k), 2.5))
    dense, dlse = oracle.attention_rows(q, k, v, np.arange(len(q)))
    np.testing.assert_allclose(out, _sdpa(q, k, v), atol=1e-12)        # shift invariance
    np.testing.assert_allclose(lse, dlse + 2.5, atol=1e-12)
    keep = np.arange(len(k)) % 3 != 1
    bias = np.where(keep, 0.0, -np.inf)
    out, _ = oracle.biased_attention_rows(q, k, v, bias)
    np.testing.assert_allclose(out, _sdpa(q, k[keep], v[keep]), atol=1e-12)


def test_sga_mean_term_is_a_size_aware_key():
    # the SGA mean term is one merged key: for every query, SGA equals size-aware attention
    # over S, the query's own key when it was dropped, and the (leave-one-out) mean key with
    # bias ln(count)
    N, gh, gw, nsp = 4, 8, 8, 5
    p = oracle.plan(N, gh, gw, nsp, 2, 2, True, True)
    q, k, v = _qkv(N, p.L, seed=15)
    q, k, v = q[0], k[0], v[0]
    out, _ = oracle.sga_full(p, q, k, v)
    ks, vs, c = oracle.dropped_sums(p, k, v)
    for i in range(p.T):
        keys = [k[t].astype(np.float64) for t in p.kv_index]
        vals = [v[t].astype(np.float64) for t in p.kv_index]
        bias = [0.0] * p.S
        ci = c
        kb, vb = ks.copy(), vs.copy()
        if not p.kept[i]:
            keys.append(k[i].astype(np.float64)); vals.append(v[i].astype(np.float64)); bias.append(0.0)
            ci = c - 1
            kb -= k[i]; vb -= v[i]
        keys.append(kb / ci); vals.append(vb / ci); bias.append(math.log(ci))
        got, _ = oracle.biased_attention_rows(q[i:i + 1], np.array(keys), np.array(vals), np.array(bias))
        np.testing.assert_allclose(got[0], out[i], atol=1e-6)   # keys pass through fp32 here


# ------------------------------------------------------------------------------ generalised plan
# "RegimeVGGT ..." Key design 3: fractional per-axis sampling factors, phase shift, frame-0 and
# camera/register protection, protected salient tokens.
from fractions import Fraction


def _bf_general_kept(N, gh, gw, nsp, sh, sw, phase, ref, protected=()):
    """Kept set by enumerating the windows with exact fractions (independent of the oracle)."""
    L = nsp + gh * gw
    sh, sw = Fraction(*sh), Fraction(*sw)
    th, tw = math.ceil(sh), math.ceil(sw)
    kept = set(int(x) for x in protected)
    for f in range(N):
        if f == 0 and ref:
            kept.update(range(L))
            continue
        kept.update(f * L + p for p in range(nsp))
        pr, pc = ((f // tw) % th, f % tw) if phase else (0, 0)
        rows, i = [], 0
        while pr + math.ceil(i * sh) < gh:
            rows.append(pr + math.ceil(i * sh)); i += 1
        cols, i = [], 0
        while pc + math.ceil(i * sw) < gw:
            cols.append(pc + math.ceil(i * sw)); i += 1
        kept.update(f * L + nsp + r * gw + c for r in rows for c in cols)
    return kept


@pytest.mark.parametrize("sh,sw", [((3, 2), (3, 2)), ((13, 10), (13, 10)), ((17, 10), (17, 10)),
                                   ((3, 2), (17, 10)), ((2, 1), (3, 1)), ((7, 3), (1, 1))])
@pytest.mark.parametrize("phase", [False, True])
@pytest.mark.parametrize("ref", [False, True])
def test_general_plan_matches_window_enumeration(sh, sw, phase, ref):
    N, gh, gw, nsp = 7, 11, 13, 5
    rng = np.random.default_rng(hash((sh, sw, phase, ref)) % 2**32)
    prot = rng.integers(0, N * (nsp + gh * gw), size=9)
    p = oracle.plan_general(N, gh, gw, nsp, sh, sw, phase, ref, protected=prot)
    want = _bf_general_kept(N, gh, gw, nsp, sh, sw, phase, ref, prot)
    assert set(p.kv_index.tolist()) == want
    assert np.all(np.diff(p.kv_index) > 0)
    assert np.array_equal(np.nonzero(p.kept)[0], p.kv_index)
    L = nsp + gh * gw
    for f in range(N):
        assert p.frame_off[f + 1] - p.frame_off[f] == sum(1 for t in want if f * L <= t < (f + 1) * L)


@pytest.mark.parametrize("phase", [False, True])
def test_general_plan_integer_windows_equal_grid_plan(phase):
    for sigma, sh, sw in _rows("sigma_map.txt"):
        a = oracle.plan_general(9, 37, 28, 5, (sh, 1), (sw, 1), phase, True)
        b = oracle.plan(9, 37, 28, 5, sh, sw, phase, True)
        assert np.array_equal(a.kv_index, b.kv_index) and np.array_equal(a.frame_off, b.frame_off)


def test_general_plan_per_axis_closed_form_and_page_retention():
    gh = gw = 37
    for num, den, pct in _rows("fractional_retention.txt"):
        s = Fraction(num, den)
        p = oracle.plan_general(2, gh, gw, 0, (num, den), (num, den), False, True)
        per_axis = (gh - 1) * den // num + 1          # #{i : ceil(i * sigma) <= G - 1}
        assert p.S - gh * gw == per_axis * per_axis
        # the share of kept patches is close to the page's stated retention
        assert abs(100.0 * per_axis ** 2 / (gh * gw) - pct) < 3.0, (num, den)


# ------------------------------------------------------------------------------ 2D RoPE
def _rope_complex(X, L, nsp, gw, base, off):
    """The same rotation written with complex numbers: z_j = x_j + i x_{j+q}, z_j * e^{i pos theta_j}."""
    T, d = X.shape
    h, q = d // 2, d // 4
    Y = np.array(X, dtype=np.float64)
    p = np.arange(T) % L
    patch = p >= nsp
    pos = np.zeros((T, 2))
    pos[patch, 0] = (p[patch] - nsp) // gw + off
    pos[patch, 1] = (p[patch] - nsp) % gw + off
    theta = base ** (-2.0 * np.arange(q) / h)
    for a in range(2):
        z = X[:, a * h:a * h + q].astype(np.float64) + 1j * X[:, a * h + q:(a + 1) * h].astype(np.float64)
        z = z * np.exp(1j * pos[:, a:a + 1] * theta[None, :])
        Y[:, a * h:a * h + q], Y[:, a * h + q:(a + 1) * h] = z.real, z.imag
    return Y


@pytest.mark.parametrize("base,off", [(100.0, 1), (10000.0, 0), (100.0, 3)])
def test_rope2d_matches_complex_rotation(base, off):
    N, gh, gw, nsp = 3, 6, 7, 5
    L = nsp + gh * gw
    _, k, _ = _qkv(N, L, seed=30)
    got = oracle.rope2d(k[0], L, nsp, gw, base, off)
    np.testing.assert_allclose(got, _rope_complex(k[0], L, nsp, gw, base, off), atol=1e-12)
    # special tokens (position 0) are not rotated; norms are preserved
    sp = (np.arange(N * L) % L) < nsp
    np.testing.assert_allclose(got[sp], k[0][sp].astype(np.float64), atol=0)
    np.testing.assert_allclose(np.linalg.norm(got, axis=1), np.linalg.norm(k[0].astype(np.float64), axis=1),
                               rtol=1e-12)


def test_rope2d_scores_depend_on_relative_position_only():
    # RoPE's defining property: q(p1) . k(p2) depends only on p1 - p2; shifting every position by
    # the same amount (a different pos_offset) leaves all patch-patch scores unchanged
    N, gh, gw, nsp = 2, 5, 6, 5
    L = nsp + gh * gw
    q, k, _ = _qkv(N, L, seed=31)
    patch = (np.arange(N * L) % L) >= nsp
    s = {}
    for off in (0, 4):
        qr = oracle.rope2d(q[0], L, nsp, gw, 100.0, off)[patch]
        kr = oracle.rope2d(k[0], L, nsp, gw, 100.0, off)[patch]
        s[off] = qr @ kr.T
    np.testing.assert_allclose(s[0], s[4], atol=1e-10)
    # and a sign error in the rotation (a planted mistake) breaks the match with the complex form
    bad = _rope_complex(k[0], L, nsp, gw, 100.0, 1)
    bad[:, 16:32] *= -1
    assert np.abs(oracle.rope2d(k[0], L, nsp, gw, 100.0, 1) - bad).max() > 1e-3


# ------------------------------------------------------------------------------ token merging
# "HTTM: Head-wise Temporal Token Merging for Faster VGGT" section 2 (head-wise matching, temporal
# blocks, first-frame anchors); merged keys carry log g ("RegimeVGGT ..." Key design 2).
def _blocks(N, gh, gw, nsp, n_t, n_s):
    L, P = nsp + gh * gw, gh * gw
    for f0 in range(0, N, n_t):
        nf = min(n_t, N - f0)
        for w0 in range(0, P, n_s):
            ws = min(n_s, P - w0)
            dst = [f0 * L + nsp + w0 + k for k in range(ws)]
            src = [f * L + nsp + w0 + k for f in range(f0 + 1, f0 + nf) for k in range(ws)]
            yield dst, src


def _match_fp64(X, N, gh, gw, nsp, n_t, n_s, r_permille):
    """An independent fp64 statement of the matching rule (valid where the fp32 decisions are
    not near-ties)."""
    Xn = X.astype(np.float64)
    nrm = np.linalg.norm(Xn, axis=1)
    match = np.full(len(X), -1)
    for dst, src in _blocks(N, gh, gw, nsp, n_t, n_s):
        if not src:
            continue
        c = (Xn[src] @ Xn[dst].T) / np.outer(nrm[src], nrm[dst])
        best = np.array(dst)[np.argmax(c, axis=1)]
        sim = c.max(axis=1)
        order = sorted(range(len(src)), key=lambda a: (-sim[a], src[a]))
        r = len(src) * r_permille // 1000
        for a in order[:r]:
            match[src[a]] = best[a]
    return match


def _separated_tokens(N, L, d, rng, nsp, gh, gw, n_t, n_s):
    """Sources = a destination of their block plus noise of a distinct size each, so every
    similarity decision is far from a tie."""
    X = rng.standard_normal((N * L, d)).astype(np.float32)
    for dst, src in _blocks(N, gh, gw, nsp, n_t, n_s):
        for i, s in enumerate(src):
            X[s] = X[dst[rng.integers(len(dst))]] + (0.02 + 0.01 * i) * rng.standard_normal(d).astype(np.float32)
    return X


@pytest.mark.parametrize("n_t,n_s,r", [(4, 8, 500), (3, 13, 250), (2, 5, 1000), (5, 64, 600)])
def test_merge_match_rule(n_t, n_s, r):
    N, gh, gw, nsp = 9, 6, 7, 5
    L = nsp + gh * gw
    rng = np.random.default_rng(n_t * 100 + n_s)
    X = _separated_tokens(N, L, 64, rng, nsp, gh, gw, n_t, n_s)
    m = oracle.merge_match(X, N, gh, gw, nsp, n_t, n_s, r)
    np.testing.assert_array_equal(m, _match_fp64(X, N, gh, gw, nsp, n_t, n_s, r))
    p = np.arange(N * L) % L
    assert np.all(m[p < nsp] == -1)                          # special tokens are never merged
    f = np.arange(N * L) // L
    assert np.all(m[f % n_t == 0] == -1)                     # a chunk's first frame anchors
    assert np.all(m[m >= 0] // L % n_t == 0)                 # ... and receives the sources
    m0 = oracle.merge_match(X, N, gh, gw, nsp, n_t, n_s, 0)
    assert np.all(m0 == -1)


def test_merge_exact_copies_keep_attention_exact():
    # every source an exact copy (key and value) of a destination of its block: whichever sources
    # are merged, mean key/value = the copy and bias ln g, so size-aware attention over the
    # merged keys equals dense attention over all tokens
    N, gh, gw, nsp, n_t, n_s = 6, 5, 6, 5, 3, 7
    L = nsp + gh * gw
    rng = np.random.default_rng(3)
    q, k, v = _qkv(N, L, seed=33)
    k, v = k[0].copy(), v[0].copy()
    for dst, src in _blocks(N, gh, gw, nsp, n_t, n_s):
        for s in src:
            j = dst[rng.integers(len(dst))]
            k[s], v[s] = k[j], v[j]
    m = oracle.merge_match(k, N, gh, gw, nsp, n_t, n_s, 700)
    assert (m >= 0).sum() > 0
    kept, gid, sizes = oracle.merge_groups(m)
    km, vm = oracle.merge_apply(k, gid, len(kept)), oracle.merge_apply(v, gid, len(kept))
    out, _ = oracle.biased_attention_rows(q[0], km, vm, np.log(sizes))
    np.testing.assert_allclose(out, _sdpa(q[0], k, v), atol=1e-12)
    # without the ln g bias the merged attention is wrong (the bias is what keeps it exact)
    bad, _ = oracle.biased_attention_rows(q[0], km, vm, np.zeros(len(kept)))
    assert np.abs(bad - out).max() > 1e-4


def test_merge_groups_and_unmerge():
    N, gh, gw, nsp, n_t, n_s = 5, 4, 5, 5, 2, 6
    L = nsp + gh * gw
    X = _separated_tokens(N, L, 64, np.random.default_rng(5), nsp, gh, gw, n_t, n_s)
    m = oracle.merge_match(X, N, gh, gw, nsp, n_t, n_s, 800)
    kept, gid, sizes = oracle.merge_groups(m)
    assert sizes.sum() == N * L and np.all(sizes >= 1)
    # unmerging a per-group quantity copies it to every member: group means of group means
    means = oracle.merge_apply(X, gid, len(kept))
    np.testing.assert_allclose(oracle.merge_apply(means[gid], gid, len(kept)), means, atol=1e-12)
    for t in range(N * L):
        members = np.nonzero(gid == gid[t])[0]
        np.testing.assert_allclose(means[gid[t]], X[members].astype(np.float64).mean(axis=0), atol=1e-12)
