"""Shared helpers for the GPU parity tests: tolerances, comparisons and row sampling.

Tolerances for attention (max |dO| <= 1e-2, mean |dO| <= 1e-3, max |dLSE| <= 1e-3, absolute,
against the float64 oracle on the same 16-bit inputs) are the ones the build targets for bf16
attention with fp32 accumulation.  The max-|dO| bound is applied on top of the unavoidable
rounding of the stored output: an element may also differ by half an ulp of the output type at
the reference value (2^-8 relative for bf16, 2^-11 for fp16), since even the exact result
rounded to bf16 misses by up to 0.0156 once |O| >= 4.  For N(0,1) workloads |O| << 1 and this
term is below 1e-3.  The layout kernels must be bit-exact.  The merge in isolation
is held to what its own arithmetic allows: output rounding to the 16-bit type (half an ulp,
2^-9 relative for bf16, 2^-12 for fp16) plus fp32 accumulation error.
"""
import numpy as np
import torch

import oracle

TOL_MAX = 1e-2
TOL_MEAN = 1e-3
TOL_LSE = 1e-3


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def half_ulp(x: np.ndarray, dtype) -> np.ndarray:
    """Half the spacing of the 16-bit output type at |x| (normal range)."""
    mant = 7 if dtype == torch.bfloat16 else 10
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    return np.exp2(np.floor(np.log2(ax)) - mant - 1)


def assert_attention_close(o_gpu, lse_gpu, o_ref, lse_ref, what="", dtype=None):
    if isinstance(o_gpu, torch.Tensor):
        dtype = o_gpu.dtype
        o = to_np(o_gpu)
    else:
        o = o_gpu
    dtype = torch.bfloat16 if dtype is None else dtype
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    excess = err - half_ulp(o_ref, dtype)
    i = np.unravel_index(np.argmax(excess), err.shape)
    assert excess.max() <= TOL_MAX, (f"{what}: |dO| = {err[i]:.3e} at |O| = {abs(o_ref[i]):.3f} "
                                     f"exceeds 1e-2 + half ulp; max |dO| = {err.max():.3e}")
    assert err.mean() <= TOL_MEAN, f"{what}: mean |dO| = {err.mean():.3e}"
    if lse_gpu is not None:
        lse = to_np(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
        lerr = np.abs(lse - lse_ref)
        assert lerr.max() <= TOL_LSE, f"{what}: max |dLSE| = {lerr.max():.3e}"
    return err.max(), err.mean()


def merge_tol(dtype) -> float:
    return 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -11


def sample_rows(Sq: int, n_random: int, seed: int, extra=()) -> np.ndarray:
    """Query rows to check at full size: both ends of every 128-row tile boundary near the start
    and end, the ragged tail, a few given rows, and seeded random rows."""
    rows = {0, 1, 127, 128, 255, 256, Sq - 1, Sq - 2, (Sq // 128) * 128 - 1, (Sq // 128) * 128}
    rows.update(int(r) for r in extra)
    rng = np.random.default_rng(seed)
    rows.update(int(r) for r in rng.integers(0, Sq, size=n_random))
    return np.array(sorted(r for r in rows if 0 <= r < Sq), dtype=np.int64)


def oracle_rows(q, k, v, rows, P=None):
    """Oracle on a subset of query rows (rows are independent in the definition)."""
    qs = q[..., torch.as_tensor(rows), :]
    if P is None:
        return oracle.attention(qs, k, v)
    return oracle.attention_chunked(qs, k, v, P)
