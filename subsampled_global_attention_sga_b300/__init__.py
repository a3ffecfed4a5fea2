"""Subsampling Global Attention (SGA) for one global cross-frame attention layer of a VGGT-style
multi-view transformer, on one B300 GPU (sm_103a).

The compute runs in libsga.so (hand-written CUDA: host plan builder, compaction kernel,
tcgen05/TMEM/TMA attention kernel, CUDA-core fp32 kernel) behind the C ABI of include/sga.h.
This package is its thin Python binding.
"""
from .api import (SIGMA_WINDOWS, HostStream, MergeConfig, Plan, SGAConfig, bias_forward, merge, merge_size, merged_attention, unmerge, compact_noalloc, dense_forward, device_status,
                  frame_forward, layer_from_host, plan_host, plan_host_general, sigma_window)
from ._lib import SgaError, lib

__all__ = ["SGAConfig", "Plan", "HostStream", "plan_host", "dense_forward", "frame_forward", "device_status",
           "layer_from_host", "compact_noalloc", "bias_forward", "plan_host_general", "MergeConfig", "merge", "merge_size", "merged_attention", "unmerge", "sigma_window", "SIGMA_WINDOWS", "SgaError", "lib"]
