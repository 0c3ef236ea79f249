"""CPU checks of the parity tests' tolerance helpers: the distance beyond storage rounding is zero
exactly when the stored value is the rounding of the reference, and grows with the error."""
import numpy as np
import torch

from parity import partial_storage_allowance, round_to, storage_distance


def test_rounded_reference_has_zero_distance():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.3, 1.0, 7.0, 300.0)])
    x = np.concatenate([x, [0.0, 2.0 ** -130, 4.0, -4.0, 1.0, 65504.0]])
    x = x.astype(np.float32).astype(np.float64)   # the kernels round an fp32 value once
    for dt in (torch.bfloat16, torch.float16):
        xx = x if dt == torch.bfloat16 else x[np.abs(x) < 6e4]
        assert (storage_distance(round_to(xx, dt), xx, dt) == 0).all()


def test_distance_counts_what_lies_beyond_half_a_spacing():
    dt = torch.bfloat16
    # 4.0 is a power of two: spacing 2^-5 above, 2^-6 below
    o = np.array([4.0, 4.0, 4.0, 4.0, 1.5, -1.5])
    ref = np.array([4.0 + 2 ** -6, 4.0 + 2 ** -6 + 0.01, 4.0 - 2 ** -7, 4.0 - 2 ** -7 - 0.01,
                    1.5 + 2 ** -8 + 0.002, -1.5 - 2 ** -8 - 0.003])
    d = storage_distance(o, ref, dt)
    np.testing.assert_allclose(d, [0.0, 0.01, 0.0, 0.01, 0.002, 0.003], atol=1e-12)
    # a stored value one spacing off is half a spacing beyond the rounding cell
    x = np.array([0.7, -2.3, 33.0])
    r = round_to(x, dt)
    ulp = np.exp2(np.floor(np.log2(np.abs(r))) - 7)
    np.testing.assert_allclose(storage_distance(r + ulp, r, dt), ulp / 2, rtol=1e-12)


def test_partial_storage_allowance_bounds_the_merge_of_rounded_partials():
    """Merging partials rounded to bf16 moves the merged value by no more than the allowance."""
    rng = np.random.default_rng(5)
    op = rng.standard_normal((3, 400, 16)) * 3
    lp = rng.standard_normal((3, 400)) * 2
    w = np.exp(lp - lp.max(0))
    exact = (w[..., None] * op).sum(0) / w.sum(0)[..., None]
    stored = round_to(op, torch.bfloat16)
    merged = (w[..., None] * stored).sum(0) / w.sum(0)[..., None]
    allow = partial_storage_allowance(stored, lp, torch.bfloat16)
    assert (np.abs(merged - exact) <= allow * (1 + 1e-9)).all()
    assert (np.abs(merged - exact) > 0.5 * allow).any()
