"""Subsampling Global Attention (SGA) for one global cross-frame attention layer of a VGGT-style
multi-view transformer, on one B300 GPU (sm_103a).

The compute runs in libsga.so (hand-written CUDA: host plan builder, compaction kernel,
tcgen05/TMEM/TMA attention kernel, CUDA-core fp32 kernel) behind the C ABI of include/sga.h.
This package is its thin Python binding.
"""
from ._lib import SgaError, lib
from .api import (SIGMA_WINDOWS, HostStream, MergeConfig, PlainHostStream, Plan, SGAConfig, bias_forward, compact_noalloc,
                  dense_forward, device_status, frame_forward, kept_count, last_device_status, layer_from_host,
                  merge, merge_size, merged_attention, plan_host, plan_host_general, sigma_window, unmerge)

__all__ = ["SGAConfig", "Plan", "HostStream", "PlainHostStream", "plan_host", "plan_host_general", "kept_count", "dense_forward",
           "frame_forward", "bias_forward", "device_status", "last_device_status", "layer_from_host",
           "compact_noalloc", "MergeConfig", "merge", "merge_size", "merged_attention", "unmerge", "sigma_window",
           "SIGMA_WINDOWS", "SgaError", "lib"]
