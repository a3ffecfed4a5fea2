"""Seeded synthetic Q/K/V for a VGGT-style global attention layer.

This module holds the input recipe only -- none of the attention method's arithmetic -- so
that the CUDA path and the CPU oracle can be fed the very same tensors.

Recipe (the pages' datasets and trained weights are not available, so correlated Gaussians of
VGGT's shapes stand in for the projected tokens): for every batch element b, head h, frame f and
in-frame slot p,

    X[b, h, f*L + p, :] = sqrt(rho) * Z_shared[b, h, p, :] + sqrt(1 - rho) * Z_ind[b, h, f, p, :]

with Z ~ N(0, 1) i.i.d., so every entry has unit variance and two frames' tokens at the same
in-frame slot have correlation rho (0.5 by default).  Q, K and V are drawn independently from
the generator streams seed, seed + 1 and seed + 2, in fp32, then cast to the requested dtype.
"""
from __future__ import annotations

import math

import torch


def correlated_tokens(B: int, H: int, N: int, L: int, d: int, *, seed: int,
                      dtype=torch.float32, device="cpu", rho: float = 0.5,
                      scale: float = 1.0) -> torch.Tensor:
    """One [B, H, N*L, d] tensor of cross-frame-correlated Gaussian tokens."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = torch.empty((B, H, N * L, d), dtype=dtype, device=device)
    a = math.sqrt(rho) * scale
    b = math.sqrt(1.0 - rho) * scale
    for bi in range(B):
        for hi in range(H):
            shared = torch.randn((1, L, d), generator=g, device=device, dtype=torch.float32)
            ind = torch.randn((N, L, d), generator=g, device=device, dtype=torch.float32)
            x = ind.mul_(b).add_(shared, alpha=a)
            out[bi, hi].copy_(x.reshape(N * L, d))
            del shared, ind, x
    return out


def correlated_qkv(B: int, H: int, N: int, L: int, d: int = 64, *, seed: int = 0,
                   dtype=torch.float32, device="cpu", rho: float = 0.5, q_scale: float = 1.0):
    """(Q, K, V), each [B, H, N*L, d], from generator streams seed, seed+1, seed+2.

    ``q_scale`` multiplies Q only (a peaky-softmax robustness case uses 8).
    """
    q = correlated_tokens(B, H, N, L, d, seed=seed, dtype=dtype, device=device, rho=rho,
                          scale=q_scale)
    k = correlated_tokens(B, H, N, L, d, seed=seed + 1, dtype=dtype, device=device, rho=rho)
    v = correlated_tokens(B, H, N, L, d, seed=seed + 2, dtype=dtype, device=device, rho=rho)
    return q, k, v


def sample_rows(T: int, L: int, n: int, *, seed: int = 1234, kept=None) -> torch.Tensor:
    """Seeded sorted sample of n query rows in [0, T) that always contains the first and last
    row, rows of frame 0, every special-token slot of frame 1 and, when ``kept`` (a bool/uint8
    array of length T) is given, both kept and dropped rows."""
    g = torch.Generator().manual_seed(int(seed))
    forced = {0, T - 1, min(T - 1, L // 2), min(T - 1, L - 1)}
    if T > L:
        forced.update(range(L, min(T, L + 5)))
    if kept is not None:
        kept_t = torch.as_tensor(kept).bool()
        ks = torch.nonzero(kept_t).flatten()
        ds = torch.nonzero(~kept_t).flatten()
        if len(ks):
            forced.add(int(ks[-1]))
        if len(ds):
            forced.update({int(ds[0]), int(ds[-1])})
    forced = sorted(x for x in forced if 0 <= x < T)
    n_rand = max(0, min(n, T) - len(forced))
    pool = torch.randperm(T, generator=g)[: n_rand + len(forced)]
    rows = set(forced)
    for x in pool.tolist():
        if len(rows) >= min(n, T):
            break
        rows.add(int(x))
    return torch.tensor(sorted(rows), dtype=torch.int64)
