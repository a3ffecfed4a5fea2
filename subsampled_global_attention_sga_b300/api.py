"""Python front end of libsga: argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; this module turns torch tensors
into device pointers plus the current CUDA stream and raises on a non-OK status.  Output
tensors that the caller does not pass are allocated here with torch (device memory is
PyTorch's job); the C entry points themselves never allocate.
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass, field

import numpy as np
import torch

from . import _lib
from ._lib import SgaConfig, SgaGridSpec, SgaMergeConfig, check, lib

# sigma -> (s_h, s_w): "AVGGT: Rethinking Global Attention for Accelerating VGGT", Key design 2
# (sigma = s_h * s_w; 2 -> (1,2), 4 -> (2,2), 6 -> (2,3), 9 -> (3,3)); sigma = 1 keeps every key.
SIGMA_WINDOWS = {1: (1, 1), 2: (1, 2), 4: (2, 2), 6: (2, 3), 9: (3, 3)}

_DTYPES = {"bf16": (_lib.SGA_BF16, torch.bfloat16), "f32": (_lib.SGA_F32, torch.float32)}
_KERNELS = {"auto": _lib.SGA_KERNEL_AUTO, "tc": _lib.SGA_KERNEL_TC, "simt": _lib.SGA_KERNEL_SIMT}
_MEAN_MODES = {"loo": _lib.SGA_MEAN_LOO, "global": _lib.SGA_MEAN_GLOBAL}


def sigma_window(sigma: int):
    """The (s_h, s_w) window of a subsampling factor sigma."""
    if sigma not in SIGMA_WINDOWS:
        raise ValueError(f"sigma must be one of {sorted(SIGMA_WINDOWS)}, got {sigma}")
    return SIGMA_WINDOWS[sigma]


@dataclass
class SGAConfig:
    """One SGA layer: B x H heads over N frames of n_special + grid_h*grid_w tokens, d = 64."""
    B: int
    H: int
    N: int
    grid_h: int = 37
    grid_w: int = 37
    n_special: int = 5
    sigma: int = 4
    window: tuple | None = None        # explicit (s_h, s_w); overrides sigma
    phase_shift: bool = False
    ref_frame_dense: bool = True
    diag: bool = True
    mean: bool = True
    mean_mode: str = "loo"
    dtype: str = "bf16"
    kernel: str = "auto"
    head_dim: int = 64
    rope: bool = False                  # fused 2D rotary embedding of Q and K
    rope_base: float = 100.0
    rope_pos_offset: int = 1

    @property
    def L(self) -> int:
        return self.n_special + self.grid_h * self.grid_w

    @property
    def T(self) -> int:
        return self.N * self.L

    @property
    def s_hw(self):
        return tuple(self.window) if self.window is not None else sigma_window(self.sigma)

    @property
    def torch_dtype(self):
        return _DTYPES[self.dtype][1]

    def to_c(self) -> SgaConfig:
        s_h, s_w = self.s_hw
        c = SgaConfig()
        c.B, c.H, c.N = self.B, self.H, self.N
        c.grid_h, c.grid_w, c.n_special, c.head_dim = self.grid_h, self.grid_w, self.n_special, self.head_dim
        c.s_h, c.s_w = s_h, s_w
        c.phase_shift, c.ref_frame_dense = int(self.phase_shift), int(self.ref_frame_dense)
        c.diag, c.mean = int(self.diag), int(self.mean)
        c.mean_mode = _MEAN_MODES[self.mean_mode]
        c.dtype = _DTYPES[self.dtype][0]
        c.kernel = _KERNELS[self.kernel]
        c.rope, c.rope_base, c.rope_pos_offset = int(self.rope), float(self.rope_base), int(self.rope_pos_offset)
        return c


def plan_host(cfg: SGAConfig):
    """Kept set S computed by the library's host builder: (kv_index, frame_off, slot)."""
    c = cfg.to_c()
    kv = np.zeros(cfg.T, dtype=np.int32)
    off = np.zeros(cfg.N + 1, dtype=np.int32)
    slot = np.zeros(cfg.T, dtype=np.int32)
    n = ctypes.c_int64(0)
    check("sga_plan_host", lib().sga_plan_host(ctypes.byref(c), kv.ctypes.data, off.ctypes.data,
                                              slot.ctypes.data, ctypes.byref(n)))
    return kv[: n.value].copy(), off, slot


def plan_host_general(N: int, grid_h: int = 37, grid_w: int = 37, n_special: int = 5, *,
                      sigma_h=(2, 1), sigma_w=(2, 1), phase_shift: bool = False,
                      ref_frame_dense: bool = True, protected=()):
    """Generalised kept set ("RegimeVGGT ..." Key design 3) computed by the library's host
    builder: per-axis rational window sizes (num, den), e.g. (3, 2) for 1.5, plus protected
    tokens kept in full.  Returns (kv_index, frame_off, slot)."""
    g = SgaGridSpec()
    g.N, g.grid_h, g.grid_w, g.n_special = N, grid_h, grid_w, n_special
    g.sh_num, g.sh_den = int(sigma_h[0]), int(sigma_h[1])
    g.sw_num, g.sw_den = int(sigma_w[0]), int(sigma_w[1])
    g.phase_shift, g.ref_frame_dense = int(phase_shift), int(ref_frame_dense)
    T = N * (n_special + grid_h * grid_w)
    prot = np.ascontiguousarray(np.asarray(list(protected), dtype=np.int32).reshape(-1))
    kv = np.zeros(T, dtype=np.int32)
    off = np.zeros(N + 1, dtype=np.int32)
    slot = np.zeros(T, dtype=np.int32)
    n = ctypes.c_int64(0)
    check("sga_plan_host_general",
          lib().sga_plan_host_general(ctypes.byref(g), prot.ctypes.data if len(prot) else None, len(prot),
                                      kv.ctypes.data, off.ctypes.data, slot.ctypes.data, ctypes.byref(n)))
    return kv[: n.value].copy(), off, slot


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check_tensor(name, t, shape, dtype, device):
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


class Plan:
    """Device-resident kept set of one layer configuration (owns the library's plan)."""

    def __init__(self, cfg: SGAConfig, device=None, kv_index=None):
        """The grid kept set of ``cfg``, or -- with ``kv_index`` (strictly ascending token
        indices) -- an arbitrary kept set over cfg's frames (``sga_plan_create_from_index``)."""
        if device is None:
            device = torch.device("cuda", torch.cuda.current_device())
        self.device = torch.device(device)
        self.cfg = cfg
        self._h = ctypes.c_void_p()
        c = cfg.to_c()
        with torch.cuda.device(self.device):
            if kv_index is None:
                check("sga_plan_create", lib().sga_plan_create(ctypes.byref(c), self.device.index,
                                                               ctypes.byref(self._h)))
            else:
                kv = np.ascontiguousarray(np.asarray(kv_index, dtype=np.int32).reshape(-1))
                check("sga_plan_create_from_index",
                      lib().sga_plan_create_from_index(ctypes.byref(c), kv.ctypes.data if len(kv) else None,
                                                       len(kv), self.device.index, ctypes.byref(self._h)))
        T, S, D = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        check("sga_plan_info", lib().sga_plan_info(self._h, ctypes.byref(T), ctypes.byref(S), ctypes.byref(D)))
        self.T, self.S, self.dropped = T.value, S.value, D.value

    def indices(self):
        kv = np.zeros(max(self.S, 1), dtype=np.int32)
        off = np.zeros(self.cfg.N + 1, dtype=np.int32)
        check("sga_plan_copy_indices", lib().sga_plan_copy_indices(self._h, kv.ctypes.data, off.ctypes.data))
        return kv[: self.S], off

    def close(self):
        if self._h:
            lib().sga_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ steps of the layer
    def compact(self, K, V, K_S=None, V_S=None, k_sum=None, v_sum=None):
        """K_S, V_S (kept rows) and k_sum, v_sum (sums of the dropped rows, fp32)."""
        cfg, dev = self.cfg, self.device
        shp = (cfg.B, cfg.H, self.T, 64)
        _check_tensor("K", K, shp, cfg.torch_dtype, dev)
        _check_tensor("V", V, shp, cfg.torch_dtype, dev)
        ks_shape = (cfg.B, cfg.H, self.S, 64)
        K_S = torch.empty(ks_shape, dtype=cfg.torch_dtype, device=dev) if K_S is None else K_S
        V_S = torch.empty(ks_shape, dtype=cfg.torch_dtype, device=dev) if V_S is None else V_S
        k_sum = torch.empty((cfg.B, cfg.H, 64), dtype=torch.float32, device=dev) if k_sum is None else k_sum
        v_sum = torch.empty((cfg.B, cfg.H, 64), dtype=torch.float32, device=dev) if v_sum is None else v_sum
        _check_tensor("K_S", K_S, ks_shape, cfg.torch_dtype, dev)
        _check_tensor("V_S", V_S, ks_shape, cfg.torch_dtype, dev)
        _check_tensor("k_sum", k_sum, (cfg.B, cfg.H, 64), torch.float32, dev)
        _check_tensor("v_sum", v_sum, (cfg.B, cfg.H, 64), torch.float32, dev)
        with torch.cuda.device(dev):
            check("sga_compact", lib().sga_compact(self._h, _ptr(K), _ptr(V), _ptr(K_S), _ptr(V_S),
                                                   _ptr(k_sum), _ptr(v_sum), _stream(dev)))
        return K_S, V_S, k_sum, v_sum

    def forward(self, Q, K, V, K_S, V_S, k_sum, v_sum, out=None, lse=None, scale=None):
        """SGA attention output [B, H, T, 64]; ``lse`` (fp32 [B, H, T]) is filled when given."""
        cfg, dev = self.cfg, self.device
        shp = (cfg.B, cfg.H, self.T, 64)
        for n, t in (("Q", Q), ("K", K), ("V", V)):
            _check_tensor(n, t, shp, cfg.torch_dtype, dev)
        out = torch.empty(shp, dtype=cfg.torch_dtype, device=dev) if out is None else out
        _check_tensor("out", out, shp, cfg.torch_dtype, dev)
        if lse is not None:
            _check_tensor("lse", lse, shp[:3], torch.float32, dev)
        scale = 1.0 / math.sqrt(64) if scale is None else float(scale)
        with torch.cuda.device(dev):
            check("sga_forward", lib().sga_forward(self._h, _ptr(Q), _ptr(K), _ptr(V), _ptr(K_S), _ptr(V_S),
                                                   _ptr(k_sum), _ptr(v_sum), _ptr(out), _ptr(lse),
                                                   ctypes.c_float(scale), _stream(dev)))
        return out

    def rope2d(self, X):
        """Rotate X [B, H, T, 64] in place with this plan's 2D rotary embedding."""
        cfg, dev = self.cfg, self.device
        _check_tensor("X", X, (cfg.B, cfg.H, self.T, 64), cfg.torch_dtype, dev)
        with torch.cuda.device(dev):
            check("sga_rope2d", lib().sga_rope2d(self._h, _ptr(X), _stream(dev)))
        return X

    def layer(self, Q, K, V, out=None, lse=None, scale=None):
        """The whole SGA layer: compaction, then attention."""
        K_S, V_S, k_sum, v_sum = self.compact(K, V)
        return self.forward(Q, K, V, K_S, V_S, k_sum, v_sum, out=out, lse=lse, scale=scale)


def kept_count(cfg: SGAConfig) -> int:
    """|S| of a layer configuration, from the library's closed form (host only)."""
    c = cfg.to_c()
    n = ctypes.c_int64(0)
    check("sga_kept_count", lib().sga_kept_count(ctypes.byref(c), ctypes.byref(n)))
    return n.value


def compact_noalloc(cfg: SGAConfig, K, V, K_S, V_S, k_sum, v_sum):
    """Compaction through ``sga_compact_noalloc``: no plan and no device allocation inside the
    library (its scratch is a fixed array in the library).  Every output is passed in by the
    caller on the inputs' CUDA device; K_S/V_S must be [B, H, |S|, 64] with |S| =
    ``kept_count(cfg)``: the C call receives no buffer sizes, so a wrong shape is refused here,
    before anything is launched."""
    dev = K.device
    if dev.type != "cuda":
        raise ValueError(f"K: on {dev}, expected a CUDA device")
    shp = (cfg.B, cfg.H, cfg.T, 64)
    _check_tensor("K", K, shp, cfg.torch_dtype, dev)
    _check_tensor("V", V, shp, cfg.torch_dtype, dev)
    S = kept_count(cfg)
    for n, t in (("K_S", K_S), ("V_S", V_S)):
        _check_tensor(n, t, (cfg.B, cfg.H, S, 64), cfg.torch_dtype, dev)
    for n, t in (("k_sum", k_sum), ("v_sum", v_sum)):
        _check_tensor(n, t, (cfg.B, cfg.H, 64), torch.float32, dev)
    c = cfg.to_c()
    with torch.cuda.device(dev):
        check("sga_compact_noalloc", lib().sga_compact_noalloc(ctypes.byref(c), _ptr(K), _ptr(V), _ptr(K_S),
                                                               _ptr(V_S), _ptr(k_sum), _ptr(v_sum), _stream(dev)))
    return K_S, V_S, k_sum, v_sum


def _plain(kind, Q, K, V, N, L, dtype, kernel, out, lse, scale):
    B, H, T, d = Q.shape
    tdt = _DTYPES[dtype][1]
    dev = Q.device
    for n, t in (("Q", Q), ("K", K), ("V", V)):
        _check_tensor(n, t, (B, H, T, d), tdt, dev)
    out = torch.empty_like(Q) if out is None else out
    _check_tensor("out", out, (B, H, T, d), tdt, dev)
    if lse is not None:
        _check_tensor("lse", lse, (B, H, T), torch.float32, dev)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with torch.cuda.device(dev):
        if kind == "dense":
            st = lib().sga_dense_forward(B, H, T, d, _DTYPES[dtype][0], _KERNELS[kernel], _ptr(Q), _ptr(K),
                                         _ptr(V), _ptr(out), _ptr(lse), ctypes.c_float(scale), _stream(dev))
        else:
            if N * L != T:
                raise ValueError(f"N*L = {N * L} does not match T = {T}")
            st = lib().sga_frame_forward(B, H, N, L, d, _DTYPES[dtype][0], _KERNELS[kernel], _ptr(Q), _ptr(K),
                                         _ptr(V), _ptr(out), _ptr(lse), ctypes.c_float(scale), _stream(dev))
    check(f"sga_{kind}_forward", st)
    return out


def dense_forward(Q, K, V, *, dtype="bf16", kernel="auto", out=None, lse=None, scale=None):
    """Dense global attention over all N*L tokens ("AVGGT ...", the standard attention, sigma = 1)."""
    return _plain("dense", Q, K, V, 0, 0, dtype, kernel, out, lse, scale)


def frame_forward(Q, K, V, N, L, *, dtype="bf16", kernel="auto", out=None, lse=None, scale=None):
    """Frame-local attention ("AVGGT ..." Key design 1, Global-to-Frame)."""
    return _plain("frame", Q, K, V, N, L, dtype, kernel, out, lse, scale)


def bias_forward(Q, K, V, bias, *, dtype="bf16", kernel="auto", out=None, lse=None, scale=None):
    """Size-aware attention softmax(scale * Q K^T + bias) V ("RegimeVGGT ..." Key design 2):
    Q [B, H, Tq, 64], K/V [B, H, Tk, 64], bias fp32 [B, H, Tk] (ln g for a key standing for g
    tokens)."""
    B, H, Tq, d = Q.shape
    Tk = K.shape[2]
    tdt = _DTYPES[dtype][1]
    dev = Q.device
    _check_tensor("Q", Q, (B, H, Tq, d), tdt, dev)
    _check_tensor("K", K, (B, H, Tk, d), tdt, dev)
    _check_tensor("V", V, (B, H, Tk, d), tdt, dev)
    _check_tensor("bias", bias, (B, H, Tk), torch.float32, dev)
    out = torch.empty_like(Q) if out is None else out
    _check_tensor("out", out, (B, H, Tq, d), tdt, dev)
    if lse is not None:
        _check_tensor("lse", lse, (B, H, Tq), torch.float32, dev)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with torch.cuda.device(dev):
        check("sga_bias_forward", lib().sga_bias_forward(B, H, Tq, Tk, d, _DTYPES[dtype][0], _KERNELS[kernel],
                                                         _ptr(Q), _ptr(K), _ptr(V), _ptr(bias), _ptr(out),
                                                         _ptr(lse), ctypes.c_float(scale), _stream(dev)))
    return out


@dataclass
class MergeConfig:
    """Head-wise temporal token merging ("HTTM ..." section 2): chunks of n_t frames, runs of n_s
    patch tokens, r_permille of each block's sources merged into the chunk's first frame."""
    B: int
    H: int
    N: int
    grid_h: int = 37
    grid_w: int = 37
    n_special: int = 5
    n_t: int = 4
    n_s: int = 37
    r_permille: int = 500
    dtype: str = "bf16"

    @property
    def T(self) -> int:
        return self.N * (self.n_special + self.grid_h * self.grid_w)

    def to_c(self) -> SgaMergeConfig:
        c = SgaMergeConfig()
        c.B, c.H, c.N, c.grid_h, c.grid_w, c.n_special = self.B, self.H, self.N, self.grid_h, self.grid_w, self.n_special
        c.head_dim, c.n_t, c.n_s, c.r_permille = 64, self.n_t, self.n_s, self.r_permille
        c.dtype = _DTYPES[self.dtype][0]
        return c


def merge_size(mcfg: MergeConfig) -> int:
    """Merged tokens per (batch, head)."""
    c = mcfg.to_c()
    m = ctypes.c_int64(0)
    check("sga_merge_size", lib().sga_merge_size(ctypes.byref(c), ctypes.byref(m)))
    return m.value


def merge(mcfg: MergeConfig, X, Y=None, out=None):
    """Merge X [B, H, T, 64] (matched by its own cosine similarity) and Y (following X's match):
    returns (X_m, Y_m or None, log_g [B, H, M], map [B, H, T]); ``out`` may hold those four."""
    dev = X.device
    tdt = _DTYPES[mcfg.dtype][1]
    shp = (mcfg.B, mcfg.H, mcfg.T, 64)
    _check_tensor("X", X, shp, tdt, dev)
    if Y is not None:
        _check_tensor("Y", Y, shp, tdt, dev)
    M = merge_size(mcfg)
    if out is None:
        Xm = torch.empty((mcfg.B, mcfg.H, M, 64), dtype=tdt, device=dev)
        Ym = torch.empty_like(Xm) if Y is not None else None
        log_g = torch.empty((mcfg.B, mcfg.H, M), dtype=torch.float32, device=dev)
        mp = torch.empty((mcfg.B, mcfg.H, mcfg.T), dtype=torch.int32, device=dev)
    else:
        Xm, Ym, log_g, mp = out
        _check_tensor("X_m", Xm, (mcfg.B, mcfg.H, M, 64), tdt, dev)
        if Y is not None:
            _check_tensor("Y_m", Ym, (mcfg.B, mcfg.H, M, 64), tdt, dev)
        _check_tensor("log_g", log_g, (mcfg.B, mcfg.H, M), torch.float32, dev)
        _check_tensor("map", mp, (mcfg.B, mcfg.H, mcfg.T), torch.int32, dev)
    c = mcfg.to_c()
    with torch.cuda.device(dev):
        check("sga_merge", lib().sga_merge(ctypes.byref(c), _ptr(X), _ptr(Y), _ptr(Xm), _ptr(Ym), _ptr(log_g),
                                           _ptr(mp), _stream(dev)))
    return Xm, Ym, log_g, mp


def unmerge(mcfg: MergeConfig, mp, Ym, out=None):
    """Every token receives the row of the merged token it belongs to: out[..., t, :] = Ym[..., map[t], :]."""
    dev = Ym.device
    tdt = _DTYPES[mcfg.dtype][1]
    out = torch.empty((mcfg.B, mcfg.H, mcfg.T, 64), dtype=tdt, device=dev) if out is None else out
    _check_tensor("out", out, (mcfg.B, mcfg.H, mcfg.T, 64), tdt, dev)
    _check_tensor("map", mp, (mcfg.B, mcfg.H, mcfg.T), torch.int32, dev)
    c = mcfg.to_c()
    with torch.cuda.device(dev):
        check("sga_unmerge", lib().sga_unmerge(ctypes.byref(c), _ptr(mp), _ptr(Ym), _ptr(out), _stream(dev)))
    return out


def merged_attention(mcfg: MergeConfig, Q, K, V, *, merge_queries=False, scale=None):
    """Attention over head-wise merged keys/values with the ln g size bias ("HTTM ..." section 2,
    "RegimeVGGT ..." Key design 2).  With merge_queries, queries are merged by their own
    similarity and the merged outputs are copied back to every query (unmerge)."""
    Km, Vm, log_g, _ = merge(mcfg, K, V)
    if not merge_queries:
        return bias_forward(Q, Km, Vm, log_g, dtype=mcfg.dtype, scale=scale)
    Qm, _, _, mq = merge(mcfg, Q)
    Om = bias_forward(Qm, Km, Vm, log_g, dtype=mcfg.dtype, scale=scale)
    return unmerge(mcfg, mq, Om)


def last_device_status(plan: "Plan") -> int:
    """``sga_last_device_status``: synchronise the current stream of the plan's device and
    return (and clear) that device's kernel status word; raises for an invalid plan."""
    with torch.cuda.device(plan.device):
        st = int(lib().sga_last_device_status(plan._h, _stream(plan.device)))
    if st in (_lib.SGA_ERR_PLAN_MISMATCH, _lib.SGA_ERR_CUDA):
        check("sga_last_device_status", st)
    return st


def device_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device's kernel status word."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib().sga_device_status(_stream(dev)))


class _Streamer:
    """Common part of the host-streaming executors (``sga_stream_*``): the library owns the
    device buffer sets and three CUDA streams (copies in, compute, copies out); ``h2d`` and
    ``d2h`` are its first and last streams, for timing events."""

    def _attach(self, create):
        self._h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            create(ctypes.byref(self._h))
            a, b, c = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
            check("sga_stream_handles", lib().sga_stream_handles(self._h, ctypes.byref(a), ctypes.byref(b),
                                                                 ctypes.byref(c)))
            self.h2d = torch.cuda.ExternalStream(a.value, device=self.device)
            self.compute = torch.cuda.ExternalStream(b.value, device=self.device)
            self.d2h = torch.cuda.ExternalStream(c.value, device=self.device)
        self._keep = []          # host tensors of queued layers, held until synchronize

    def synchronize(self):
        """Wait until every submitted layer's output is in its host buffer."""
        with torch.cuda.device(self.device):
            check("sga_stream_synchronize", lib().sga_stream_synchronize(self._h))
        self._keep.clear()

    def close(self):
        if self._h:
            lib().sga_stream_destroy(self._h)
            self._h = ctypes.c_void_p()
            self._keep.clear()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class HostStream(_Streamer):
    """Streams SGA layers from pinned host memory through one plan (``sga_stream_*``): the
    library double-buffers the device tensors and runs host-to-device copies, compute and
    device-to-host copies on three CUDA streams of its own, so layer i+1's inputs and layer
    i-1's output move while layer i computes (K and V first, so the compaction starts while Q is
    in flight).  Each output equals ``Plan.layer`` on the same inputs."""

    def __init__(self, plan: Plan, depth: int = 2):
        self.plan, self.device = plan, plan.device
        self._attach(lambda h: check("sga_stream_create", lib().sga_stream_create(plan._h, int(depth), h)))

    def submit(self, Q_host, K_host, V_host, out_host, scale=None):
        """Queue one layer: out_host <- SGA(Q_host, K_host, V_host).  Returns immediately; the
        host tensors (CPU, contiguous, pinned for overlap) must stay untouched until
        ``synchronize``."""
        cfg = self.plan.cfg
        shp = (cfg.B, cfg.H, self.plan.T, 64)
        for n, t in (("Q", Q_host), ("K", K_host), ("V", V_host), ("out", out_host)):
            _check_tensor(n, t, shp, cfg.torch_dtype, torch.device("cpu"))
        with torch.cuda.device(self.device):
            check("sga_stream_submit", lib().sga_stream_submit(
                self._h, _ptr(Q_host), _ptr(K_host), _ptr(V_host), _ptr(out_host),
                ctypes.c_float(0.0 if scale is None else float(scale))))
        self._keep.append((Q_host, K_host, V_host, out_host))
        return out_host


_PLAIN_KINDS = {"dense": _lib.SGA_PLAIN_DENSE, "frame": _lib.SGA_PLAIN_FRAME, "bias": _lib.SGA_PLAIN_BIAS}


class PlainHostStream(_Streamer):
    """The host-streaming executor for the plain attention calls (``sga_stream_create_plain``):
    kind "dense" (``dense_forward``), "frame" (``frame_forward``, N frames of L tokens) or
    "bias" (``bias_forward``, Tk keys with an fp32 bias).  Each output equals the device call
    on the same inputs."""

    def __init__(self, kind: str, B: int, H: int, Tq: int, *, Tk: int | None = None, N: int = 0, L: int = 0,
                 dtype: str = "bf16", kernel: str = "auto", depth: int = 2, device=None):
        if kind not in _PLAIN_KINDS:
            raise ValueError(f"kind must be one of {sorted(_PLAIN_KINDS)}")
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.kind, self.B, self.H, self.Tq = kind, B, H, Tq
        self.Tk = Tk if (kind == "bias" and Tk is not None) else Tq
        self.dtype = dtype
        spec = _lib.SgaPlainSpec()
        spec.kind, spec.B, spec.H, spec.Tq, spec.Tk = _PLAIN_KINDS[kind], B, H, Tq, self.Tk
        spec.N, spec.L, spec.head_dim = N, L, 64
        spec.dtype, spec.kernel = _DTYPES[dtype][0], _KERNELS[kernel]
        self._attach(lambda h: check("sga_stream_create_plain",
                                     lib().sga_stream_create_plain(ctypes.byref(spec), int(depth), h)))

    def submit(self, Q_host, K_host, V_host, out_host, bias_host=None, scale=None):
        """Queue one call: out_host <- attention(Q_host, K_host, V_host[, bias_host]).  Host
        tensors (CPU, contiguous, pinned for overlap) must stay untouched until ``synchronize``."""
        tdt, cpu = _DTYPES[self.dtype][1], torch.device("cpu")
        _check_tensor("Q", Q_host, (self.B, self.H, self.Tq, 64), tdt, cpu)
        _check_tensor("out", out_host, (self.B, self.H, self.Tq, 64), tdt, cpu)
        for n, t in (("K", K_host), ("V", V_host)):
            _check_tensor(n, t, (self.B, self.H, self.Tk, 64), tdt, cpu)
        if (self.kind == "bias") != (bias_host is not None):
            raise ValueError("bias_host is required for kind 'bias' and only for it")
        if bias_host is not None:
            _check_tensor("bias", bias_host, (self.B, self.H, self.Tk), torch.float32, cpu)
        with torch.cuda.device(self.device):
            check("sga_stream_submit_plain", lib().sga_stream_submit_plain(
                self._h, _ptr(Q_host), _ptr(K_host), _ptr(V_host), _ptr(bias_host), _ptr(out_host),
                ctypes.c_float(0.0 if scale is None else float(scale))))
        self._keep.append((Q_host, K_host, V_host, bias_host, out_host))
        return out_host


def layer_from_host(plan: Plan, Q_host, K_host, V_host, out_host=None, scale=None):
    """End-to-end call from host memory: copy pinned Q, K, V to the device, run the layer, copy
    the output back (all on the current stream)."""
    dev = plan.device
    Q = Q_host.to(dev, non_blocking=True)
    K = K_host.to(dev, non_blocking=True)
    V = V_host.to(dev, non_blocking=True)
    O = plan.layer(Q, K, V, scale=scale)
    if out_host is None:
        out_host = torch.empty(O.shape, dtype=O.dtype, pin_memory=True)
    out_host.copy_(O, non_blocking=True)
    return out_host
