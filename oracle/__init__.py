"""fp64 CPU oracle for Subsampling Global Attention (SGA).

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg are the only callers.  The product package never imports this module and
shares no code with it.  The arithmetic lives in ``sga_oracle.c`` (plain C, fp64, OpenMP over
query rows); this file compiles it with gcc and marshals numpy arrays through ctypes.

Pages followed (by title and section): "AVGGT: Rethinking Global Attention for Accelerating
VGGT" Key designs 1-3; "RegimeVGGT: Layer-Wise Spatially Preserving Redundancy Removal for
Visual Geometry Grounded Transformer" Core mechanism and Key designs 2-3.  The readings taken
where the pages are silent are listed at the top of ``sga_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sga_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``sga_oracle.c`` into ``liboracle.so`` (gcc, -O2, OpenMP, no fast-math, no FMA
    contraction: the fp32 decisions of the token merging use explicit fmaf only)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-o", _LIB_PATH,
               _SRC, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        p = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_plan.restype = i64
        lib.oracle_plan.argtypes = [i32] * 8 + [p, p, p]
        lib.oracle_dropped_sums.restype = i64
        lib.oracle_dropped_sums.argtypes = [i64, i32, p, p, p, p, p]
        lib.oracle_sga_rows.restype = None
        lib.oracle_sga_rows.argtypes = [i64, i32, p, p, i64, p, p, i64, p, p, p, p, i64,
                                        i32, i32, i32, f64, p, p]
        lib.oracle_attention_rows.restype = None
        lib.oracle_attention_rows.argtypes = [i64, i32, i64, p, p, p, p, i64, f64, p, p]
        lib.oracle_plan_general.restype = i64
        lib.oracle_plan_general.argtypes = [i32] * 10 + [p, i64, p, p, p]
        lib.oracle_biased_attention_rows.restype = None
        lib.oracle_biased_attention_rows.argtypes = [i64, i32, p, p, p, p, i64, f64, p, p]
        lib.oracle_rope2d.restype = None
        lib.oracle_rope2d.argtypes = [i64, i32, i64, i32, i32, f64, i32, p, p]
        lib.oracle_merge_match.restype = i64
        lib.oracle_merge_match.argtypes = [i32] * 8 + [p, p]
        lib.oracle_num_threads.restype = i32
        lib.oracle_num_threads.argtypes = []
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


@dataclass
class Plan:
    """The kept key/value set S of one layer (same for every batch element and head)."""
    T: int
    L: int
    kept: np.ndarray        # uint8 [T]
    kv_index: np.ndarray    # int32 [|S|], ascending token indices
    frame_off: np.ndarray   # int32 [N+1]

    @property
    def S(self) -> int:
        return int(self.kv_index.shape[0])

    @property
    def dropped(self) -> int:
        return self.T - self.S


def plan(N: int, grid_h: int, grid_w: int, n_special: int, s_h: int, s_w: int,
         phase_shift: bool, ref_frame_dense: bool) -> Plan:
    L = n_special + grid_h * grid_w
    T = N * L
    kept = np.zeros(T, dtype=np.uint8)
    kv = np.zeros(T, dtype=np.int32)
    off = np.zeros(N + 1, dtype=np.int32)
    n = _load().oracle_plan(N, grid_h, grid_w, n_special, s_h, s_w, int(phase_shift),
                            int(ref_frame_dense), _ptr(kept), _ptr(kv), _ptr(off))
    if n < 0:
        raise ValueError("oracle_plan: bad argument")
    return Plan(T=T, L=L, kept=kept, kv_index=kv[:n].copy(), frame_off=off)


def plan_general(N: int, grid_h: int, grid_w: int, n_special: int, sigma_h, sigma_w,
                 phase_shift: bool, ref_frame_dense: bool, protected=()) -> Plan:
    """Generalised kept set: per-axis rational window sizes ``sigma_h``, ``sigma_w`` given as
    (num, den) pairs, and a list of protected token indices kept in full."""
    L = n_special + grid_h * grid_w
    T = N * L
    kept = np.zeros(T, dtype=np.uint8)
    kv = np.zeros(T, dtype=np.int32)
    off = np.zeros(N + 1, dtype=np.int32)
    prot = np.ascontiguousarray(np.asarray(list(protected), dtype=np.int32).reshape(-1))
    n = _load().oracle_plan_general(N, grid_h, grid_w, n_special, int(sigma_h[0]), int(sigma_h[1]),
                                    int(sigma_w[0]), int(sigma_w[1]), int(phase_shift), int(ref_frame_dense),
                                    _ptr(prot) if len(prot) else None, len(prot), _ptr(kept), _ptr(kv), _ptr(off))
    if n < 0:
        raise ValueError("oracle_plan_general: bad argument")
    return Plan(T=T, L=L, kept=kept, kv_index=kv[:n].copy(), frame_off=off)


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def dropped_sums(p: Plan, K: np.ndarray, V: np.ndarray):
    """fp64 sums of K and V over the dropped set of one (batch, head); returns (k_sum, v_sum, c)."""
    K, V = _f32(K), _f32(V)
    d = K.shape[1]
    ks = np.zeros(d, dtype=np.float64)
    vs = np.zeros(d, dtype=np.float64)
    c = _load().oracle_dropped_sums(p.T, d, _ptr(p.kept), _ptr(K), _ptr(V), _ptr(ks), _ptr(vs))
    return ks, vs, int(c)


def sga_rows(p: Plan, Qrows, K, V, rows, *, diag=True, mean=True, mean_mode=0,
             scale=0.125, sums=None):
    """SGA outputs (fp64) of the query rows ``rows`` of one (batch, head).

    ``Qrows`` holds those rows' query vectors; ``K`` and ``V`` hold all T rows of the head.
    Returns (out [n, d], lse [n]).
    """
    Qrows, K, V = _f32(Qrows), _f32(K), _f32(V)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n, d = Qrows.shape
    if sums is None:
        sums = dropped_sums(p, K, V)
    ks, vs, c = sums
    ks = np.ascontiguousarray(ks, dtype=np.float64)
    vs = np.ascontiguousarray(vs, dtype=np.float64)
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    kv = np.ascontiguousarray(p.kv_index, dtype=np.int32)
    _load().oracle_sga_rows(p.T, d, _ptr(p.kept), _ptr(kv), p.S, _ptr(ks), _ptr(vs), c,
                            _ptr(Qrows), _ptr(K), _ptr(V), _ptr(rows), n,
                            int(diag), int(mean), int(mean_mode), float(scale),
                            _ptr(out), _ptr(lse))
    return out, lse


def attention_rows(Qrows, K, V, rows, *, frame_len=0, scale=0.125):
    """Dense (frame_len == 0) or frame-local attention outputs (fp64) of the rows ``rows``."""
    Qrows, K, V = _f32(Qrows), _f32(K), _f32(V)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n, d = Qrows.shape
    T = K.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    _load().oracle_attention_rows(T, d, int(frame_len), _ptr(Qrows), _ptr(K), _ptr(V),
                                  _ptr(rows), n, float(scale), _ptr(out), _ptr(lse))
    return out, lse


def biased_attention_rows(Qrows, K, V, bias, *, scale=0.125):
    """Size-aware attention softmax(scale * q K^T + bias) V (fp64) of the query vectors
    ``Qrows`` against all Tk keys; ``bias`` is the per-key natural-log bias [Tk]."""
    Qrows, K, V = _f32(Qrows), _f32(K), _f32(V)
    bias = np.ascontiguousarray(np.asarray(bias, dtype=np.float64))
    n, d = Qrows.shape
    Tk = K.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    _load().oracle_biased_attention_rows(Tk, d, _ptr(Qrows), _ptr(K), _ptr(V), _ptr(bias), n,
                                         float(scale), _ptr(out), _ptr(lse))
    return out, lse


def rope2d(X, L: int, n_special: int, grid_w: int, base: float, pos_offset: int) -> np.ndarray:
    """2D rotary position embedding of one (batch, head)'s tokens X [T, d] (fp64 result)."""
    X = _f32(X)
    T, d = X.shape
    Y = np.zeros((T, d), dtype=np.float64)
    _load().oracle_rope2d(T, d, L, n_special, grid_w, float(base), int(pos_offset), _ptr(X), _ptr(Y))
    return Y


def merge_match(X, N, grid_h, grid_w, n_special, n_t, n_s, r_permille):
    """Head-wise temporal token merging of one (batch, head)'s tokens X [T, d]: match[t] = the
    destination token a merged source t joins, else -1 (see the C source for the rules)."""
    X = _f32(X)
    T, d = X.shape
    match = np.zeros(T, dtype=np.int32)
    n = _load().oracle_merge_match(N, grid_h, grid_w, n_special, n_t, n_s, r_permille, d, _ptr(X), _ptr(match))
    if n < 0:
        raise ValueError("oracle_merge_match: bad argument")
    return match


def merge_groups(match):
    """The merged sequence of a match vector: kept tokens (every token that is not a merged
    source) in token order; returns (kept tokens, group id of every token, group sizes)."""
    T = len(match)
    kept = np.nonzero(match < 0)[0]
    gid = np.full(T, -1, dtype=np.int64)
    gid[kept] = np.arange(len(kept))
    srcs = np.nonzero(match >= 0)[0]
    gid[srcs] = gid[match[srcs]]
    sizes = np.bincount(gid, minlength=len(kept))
    return kept, gid, sizes


def merge_apply(X, gid, n_groups):
    """Group means (fp64) of the tokens X [T, d] by group id."""
    X = np.asarray(X, dtype=np.float64)
    out = np.zeros((n_groups, X.shape[1]))
    np.add.at(out, gid, X)
    return out / np.bincount(gid, minlength=n_groups)[:, None]


def sga_full(p: Plan, Q, K, V, **kw):
    """SGA over every row of one (batch, head): Q, K, V are [T, d]."""
    rows = np.arange(p.T, dtype=np.int64)
    return sga_rows(p, Q, K, V, rows, **kw)
