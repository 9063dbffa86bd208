"""The fp16 two-term split's value range, emulated on the CPU with numpy.

x = v * s with s a power of two; hi = fp16(x), lo = fp16(x - hi); the split
represents v as (hi + lo) / s.  With s taken from the largest magnitude of the
whole tensor, entries 1e-9 below it fall into fp16's subnormal range and keep
only a few bits, so output rows made of such entries lose accuracy; with s
taken per slab of mode 0 those rows are as accurate as the others.  This is
the arithmetic reason for the per-slab scales of the tensor-core path (the
GPU tests check the kernels themselves).
"""
import numpy as np


def pow2_scale(m):
    """Power of two mapping m > 0 into [2^13, 2^14)."""
    e = int(np.floor(np.log2(m)))
    return 2.0 ** (13 - e)


def split(v, s):
    x = (v.astype(np.float32) * np.float32(s)).astype(np.float32)
    hi = x.astype(np.float16)
    lo = (x - hi.astype(np.float32)).astype(np.float16)
    return (hi.astype(np.float64) + lo.astype(np.float64)) / s


def two_level(seed=3, dims=(16, 8, 8)):
    rng = np.random.default_rng(seed)
    Y = rng.uniform(0.5, 1.0, size=dims)
    Y[dims[0] // 2:] *= 1e-9
    return Y.astype(np.float32)


def mode0_rows(Yv, krp_cols):
    return Yv.reshape(Yv.shape[0], -1).astype(np.float64) @ krp_cols


def worst_row(got, ref):
    return float((np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)).max())


def test_global_scale_loses_small_rows_slab_scale_keeps_them():
    Y = two_level()
    rng = np.random.default_rng(4)
    krp = rng.uniform(0, 1, size=(Y[0].size, 5))
    ref = mode0_rows(Y, krp)
    glob = split(Y, pow2_scale(np.abs(Y).max()))
    slab = np.stack([split(Y[i], pow2_scale(np.abs(Y[i]).max())) for i in range(Y.shape[0])])
    err_glob = worst_row(mode0_rows(glob, krp), ref)
    err_slab = worst_row(mode0_rows(slab, krp), ref)
    assert err_glob > 1e-4          # far outside the 1e-5 tolerance
    assert err_slab < 1e-6          # the split's ~2^-22 per entry
    # the large rows are fine either way: the global-scale error sits in the small rows
    half = Y.shape[0] // 2
    assert worst_row(mode0_rows(glob, krp)[:half], ref[:half]) < 1e-6


def test_split_keeps_22_bits_within_2_17_of_the_scale_maximum():
    """Relative representation error of one entry, against its magnitude below the
    largest one: about 2^-22 down to 2^-17 of it, then growing as lo goes subnormal."""
    s = pow2_scale(1.0)
    rng = np.random.default_rng(5)
    for rel, bound in [(1.0, 2.0 ** -21), (2.0 ** -10, 2.0 ** -21), (2.0 ** -17, 2.0 ** -20),
                       (2.0 ** -30, 2.0 ** -7)]:
        v = (rng.uniform(0.5, 1.0, size=4096) * rel).astype(np.float32)
        err = np.abs(split(v, s) - v.astype(np.float64)) / v
        assert err.max() < bound, (rel, err.max())
