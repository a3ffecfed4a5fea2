"""ctypes binding of libsga.so (the C ABI declared in include/sga.h): symbol table only."""
from __future__ import annotations

import ctypes
import os

from . import _build
from ._build import LIB, LIB_DEBUG

SGA_OK = 0
SGA_ERR_CUDA, SGA_ERR_TIMEOUT, SGA_ERR_PLAN_MISMATCH = 4, 5, 6
STATUS_NAMES = {
    0: "SGA_OK", 1: "SGA_ERR_INVALID_ARG", 2: "SGA_ERR_UNSUPPORTED", 3: "SGA_ERR_ALIGNMENT",
    4: "SGA_ERR_CUDA", 5: "SGA_ERR_TIMEOUT", 6: "SGA_ERR_PLAN_MISMATCH", 7: "SGA_ERR_SCRATCH_LIMIT",
    8: "SGA_ERR_DEBUG_CHECK",
}
SGA_BF16, SGA_F32 = 0, 1
SGA_MEAN_LOO, SGA_MEAN_GLOBAL = 0, 1
SGA_KERNEL_AUTO, SGA_KERNEL_TC, SGA_KERNEL_SIMT = 0, 1, 2

# every entry point include/sga.h declares (checked by the CPU test-suite)
EXPORTS = (
    "sga_plan_host", "sga_plan_create", "sga_plan_info", "sga_plan_copy_indices", "sga_plan_destroy",
    "sga_compact", "sga_forward", "sga_dense_forward", "sga_frame_forward", "sga_device_status",
    "sga_status_string", "sga_build_info", "sga_compact_noalloc", "sga_bias_forward",
    "sga_plan_host_general", "sga_plan_create_from_index", "sga_rope2d",
    "sga_merge_size", "sga_merge", "sga_unmerge", "sga_selftest_timeout",
    "sga_stream_create", "sga_stream_submit", "sga_stream_synchronize", "sga_stream_handles",
    "sga_stream_destroy", "sga_kept_count", "sga_last_device_status",
    "sga_stream_create_plain", "sga_stream_submit_plain", "sga_debug_report",
)


class SgaConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "B", "H", "N", "grid_h", "grid_w", "n_special", "head_dim", "s_h", "s_w",
        "phase_shift", "ref_frame_dense", "diag", "mean", "mean_mode", "dtype", "kernel", "rope")] + [
        ("rope_base", ctypes.c_float), ("rope_pos_offset", ctypes.c_int)]


class SgaGridSpec(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "N", "grid_h", "grid_w", "n_special", "sh_num", "sh_den", "sw_num", "sw_den",
        "phase_shift", "ref_frame_dense")]


class SgaMergeConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "B", "H", "N", "grid_h", "grid_w", "n_special", "head_dim", "n_t", "n_s", "r_permille", "dtype")]


class SgaPlainSpec(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("B", ctypes.c_int), ("H", ctypes.c_int), ("Tq", ctypes.c_int64),
                ("Tk", ctypes.c_int64), ("N", ctypes.c_int), ("L", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("dtype", ctypes.c_int), ("kernel", ctypes.c_int)]


SGA_PLAIN_DENSE, SGA_PLAIN_FRAME, SGA_PLAIN_BIAS = 1, 2, 3


class SgaError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call} failed: {STATUS_NAMES.get(status, status)} ({_describe(status)})")


_lib = None


def _describe(status: int) -> str:
    try:
        return lib().sga_status_string(status).decode()
    except Exception:  # pragma: no cover - only while the library is unavailable
        return "?"


def library_path() -> str:
    """The library this process loads: libsga.so, or its debug build (every kernel checks its
    indexed stores) when the environment sets SGA_LIBRARY=debug."""
    return LIB_DEBUG if os.environ.get("SGA_LIBRARY", "") == "debug" else LIB


def lib():
    """Load libsga.so (built in-tree by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{os.path.basename(path)} is not built ({path}); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        cfgp = ctypes.POINTER(SgaConfig)
        sig = {
            "sga_plan_host": (i32, [cfgp, vp, vp, vp, ctypes.POINTER(i64)]),
            "sga_plan_create": (i32, [cfgp, i32, ctypes.POINTER(vp)]),
            "sga_plan_info": (i32, [vp, ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i64)]),
            "sga_plan_copy_indices": (i32, [vp, vp, vp]),
            "sga_plan_destroy": (None, [vp]),
            "sga_compact": (i32, [vp, vp, vp, vp, vp, vp, vp, vp]),
            "sga_forward": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, vp]),
            "sga_dense_forward": (i32, [i32, i32, i64, i32, i32, i32, vp, vp, vp, vp, vp, f32, vp]),
            "sga_frame_forward": (i32, [i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, f32, vp]),
            "sga_compact_noalloc": (i32, [cfgp, vp, vp, vp, vp, vp, vp, vp]),
            "sga_bias_forward": (i32, [i32, i32, i64, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp, f32, vp]),
            "sga_plan_host_general": (i32, [ctypes.POINTER(SgaGridSpec), vp, i64, vp, vp, vp, ctypes.POINTER(i64)]),
            "sga_plan_create_from_index": (i32, [cfgp, vp, i64, i32, ctypes.POINTER(vp)]),
            "sga_rope2d": (i32, [vp, vp, vp]),
            "sga_merge_size": (i32, [ctypes.POINTER(SgaMergeConfig), ctypes.POINTER(i64)]),
            "sga_selftest_timeout": (i32, [vp]),
            "sga_merge": (i32, [ctypes.POINTER(SgaMergeConfig), vp, vp, vp, vp, vp, vp, vp]),
            "sga_unmerge": (i32, [ctypes.POINTER(SgaMergeConfig), vp, vp, vp, vp]),
            "sga_device_status": (i32, [vp]),
            "sga_last_device_status": (i32, [vp, vp]),
            "sga_kept_count": (i32, [cfgp, ctypes.POINTER(i64)]),
            "sga_status_string": (ctypes.c_char_p, [i32]),
            "sga_build_info": (ctypes.c_char_p, []),
            "sga_stream_create": (i32, [vp, i32, ctypes.POINTER(vp)]),
            "sga_stream_submit": (i32, [vp, vp, vp, vp, vp, f32]),
            "sga_stream_synchronize": (i32, [vp]),
            "sga_stream_handles": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp)]),
            "sga_stream_destroy": (None, [vp]),
            "sga_debug_report": (i32, [ctypes.POINTER(i64)] * 4),
            "sga_stream_create_plain": (i32, [ctypes.POINTER(SgaPlainSpec), i32, ctypes.POINTER(vp)]),
            "sga_stream_submit_plain": (i32, [vp, vp, vp, vp, vp, vp, f32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        # a library compiled from other sources than the ones in the tree is refused, so a
        # stale build can never stand in for the current code
        info = L.sga_build_info().decode()
        built = info.rsplit("src=", 1)[-1] if "src=" in info else "unknown"
        tree = _tree_source_hash()
        if built != tree:
            raise RuntimeError(f"libsga.so was built from other sources (library {built}, tree {tree}); "
                               "run __graft_entry__.build()")
        _lib = L
    return _lib


def _tree_source_hash() -> str:
    return _build.source_hash()


def check(call: str, status: int) -> None:
    if status != SGA_OK:
        raise SgaError(call, status)
