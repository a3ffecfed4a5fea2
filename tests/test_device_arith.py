"""Integer quotients that the kernels take through fp32 arithmetic instead of an integer division,
checked exhaustively on the host in the same fp32 operations.

The kernels compute floor(i / d) for a non-negative integer i as int((i + 0.5f) * (1.0f / d)).
The library is built without fast-math, so the device's `/`, `+` and `*` round to nearest, as
numpy's float32 does.  i + 1/2 lies at least 1/2 from every multiple of d.  The two roundings
move the product by under (i / d + 1) 2^-23, which stays below 1 / (2 d) while i + d < 2^22.
So the truncated product is the quotient there:

- the merge kernel: a block entry's frame, i / ws, with i below the block's entry count;
- the compaction with the 2D rotation: a token's grid row, q / grid_w, with q below the frame's
  patch count.
"""
import numpy as np


def _float_quotient(i: np.ndarray, d: int) -> np.ndarray:
    inv = np.float32(1.0) / np.float32(d)
    return ((i.astype(np.float32) + np.float32(0.5)) * inv).astype(np.int64)


def test_float_quotient_exact_for_every_block_shape():
    # every window size a merge block can have, over more entries than a block holds
    i = np.arange(4096, dtype=np.int64)
    for d in range(1, 2049):
        assert np.array_equal(_float_quotient(i, d), i // d), d


def test_float_quotient_exact_up_to_the_stated_bound():
    # grids up to 2^21 patches per frame for the rotation's row, and larger divisors
    q = np.arange(1 << 21, dtype=np.int64)
    for d in (1, 2, 3, 5, 7, 36, 37, 100, 127, 128, 129, 518, 1369, 2047, 4095, 65535):
        assert np.array_equal(_float_quotient(q, d), q // d), d


def test_float_quotient_fails_past_the_bound():
    # the bound is not loose by orders of magnitude: far past it, with d = 3, the truncated
    # product leaves the quotient
    q = np.arange((1 << 27) - (1 << 16), 1 << 27, dtype=np.int64)
    assert not np.array_equal(_float_quotient(q, 3), q // 3)


def _bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even), returned as fp32."""
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def test_merge_shortlist_window_covers_any_summation_order():
    """The tensor-core matching shortlists destinations within 2^-10 of the best approximate
    cosine: the products of bf16 values are exact in fp32, and an fp32 sum of 64 of them in any
    order lies within 2^-17 of the sum of their magnitudes (so, by Cauchy-Schwarz, approximate
    and exact cosines differ by under 2^-16).  Checked here for sequential, reversed, pairwise
    and shuffled orders on random and cancelling bf16 vectors."""
    rng = np.random.default_rng(7)
    for trial in range(400):
        x = _bf16(rng.standard_normal(64).astype(np.float32))
        b = _bf16(rng.standard_normal(64).astype(np.float32))
        if trial % 2:
            # near cancellation: products in pairs of opposite sign and almost equal size, so
            # the sum is tiny against the sum of magnitudes
            x[1::2] = _bf16(x[0::2] * np.float32(1.0 + 1e-2) * rng.choice([1.0, -1.0], 32).astype(np.float32))
            b = _bf16(np.abs(x) * np.where(np.arange(64) % 2 == 0, 1.0, -1.0).astype(np.float32)
                      * np.sign(x).astype(np.float32))
        p = (x * b).astype(np.float32)      # exact: 8-bit by 8-bit significands
        assert np.array_equal(p.astype(np.float64), x.astype(np.float64) * b.astype(np.float64))
        exact = float(np.sum(p.astype(np.float64)))
        bound = 2.0 ** -17 * float(np.sum(np.abs(p.astype(np.float64))))
        orders = [np.arange(64), np.arange(64)[::-1]] + [rng.permutation(64) for _ in range(6)]
        for order in orders:
            s = np.float32(0.0)
            for k in order:
                s = np.float32(s + p[k])
            assert abs(float(s) - exact) <= bound
        tree = p.copy()                     # pairwise order
        while tree.size > 1:
            tree = (tree[0::2] + tree[1::2]).astype(np.float32)
        assert abs(float(tree[0]) - exact) <= bound
