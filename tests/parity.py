"""Shared helpers for the GPU parity tests: tolerances, comparisons and row sampling.

Attention tolerances (max |dO| <= 1e-2, mean |dO| <= 1e-3, max |dLSE| <= 1e-3, absolute, against
the float64 oracle on the same 16-bit inputs) are the ones stated for bf16 attention with fp32
accumulation.  They bound the kernel's arithmetic, not the storage of its result: the output is
a 16-bit value, and even the exact result rounded to bf16 misses by up to half a spacing (0.0156
once |O| >= 4; mean 8.5e-4 on a sharp softmax where |O| ~ |v|).  So each element's error is the
distance from the oracle value to the set of real numbers that round (to nearest even) to the
stored GPU value -- zero when the exact result rounds to what the kernel stored -- and the max
and mean bounds apply to that distance.  For N(0,1) workloads |O| << 1 and the distance differs
from the plain |dO| by less than 1e-3.

An output merged from partials that were themselves stored in 16 bits carries one more storage
rounding per partial (the partial O has the input dtype).  Its end-to-end check against exact
attention allows, on top, the LSE-weighted half spacing of the stored partials it was merged from
(``partial_storage_allowance``); the merge itself is checked separately on the GPU's own stored
partials with the plain bound.

The layout kernels must be bit-exact.  The merge in isolation is held to what its own arithmetic
allows: output rounding to the 16-bit type (half an ulp, 2^-9 relative for bf16, 2^-12 for fp16)
plus fp32 accumulation error.
"""
import numpy as np
import torch

import oracle

TOL_MAX = 1e-2
TOL_MEAN = 1e-3
TOL_LSE = 1e-3


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def _format(dtype):
    """(mantissa bits, smallest normal exponent) of a 16-bit float type."""
    return (7, -126) if dtype == torch.bfloat16 else (10, -14)


def storage_distance(o: np.ndarray, ref: np.ndarray, dtype) -> np.ndarray:
    """Distance from ref to the set of reals that round to the stored 16-bit values o.

    The reals that round to o (to nearest) reach half a spacing to either side of it; the spacing
    away from zero is the ulp of o's binade, the spacing toward zero is half of that when o is a
    power of two (the binade below is finer), and at zero it is the smallest subnormal."""
    mant, emin = _format(dtype)
    a = np.abs(o)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** emin)))
    ulp = np.exp2(e - mant)
    d = ref - o
    away = (np.sign(d) == np.sign(o)) | (o == 0)
    pow2 = (a == np.exp2(e)) & (e > emin)
    gap = np.where(away, ulp, np.where(pow2, ulp / 2, ulp))
    return np.maximum(0.0, np.abs(d) - gap / 2)


def round_to(x: np.ndarray, dtype) -> np.ndarray:
    """float64 values rounded to the 16-bit type (round to nearest even) and back; torch goes
    through fp32 on the way, which moves only values within 2^-24 relative of a tie."""
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).to(dtype).double().numpy()


def partial_storage_allowance(op_stored, lp_ref, dtype) -> np.ndarray:
    """What storing P partials in the 16-bit type can move their merge by, at most: per row the
    LSE-weighted mean of half the spacing around each stored partial value ([P, ..., D] in,
    [..., D] out)."""
    op = to_np(op_stored) if isinstance(op_stored, torch.Tensor) else np.asarray(op_stored)
    lp = np.asarray(lp_ref, dtype=np.float64)
    mant, emin = _format(dtype)
    half = np.exp2(np.floor(np.log2(np.maximum(np.abs(op), 2.0 ** emin))) - mant) / 2
    w = np.exp(lp - lp.max(axis=0, keepdims=True))
    w = w / w.sum(axis=0, keepdims=True)
    return (w[..., None] * half).sum(axis=0)


def assert_attention_close(o_gpu, lse_gpu, o_ref, lse_ref, what="", dtype=None, allowance=0.0):
    """allowance: a further per-element error the comparison accepts (e.g. the storage of the
    partials an output was merged from); zero for outputs computed in one pass."""
    if isinstance(o_gpu, torch.Tensor):
        dtype = o_gpu.dtype
        o = to_np(o_gpu)
    else:
        o = o_gpu
    dtype = torch.bfloat16 if dtype is None else dtype
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    dist = np.maximum(0.0, storage_distance(o, o_ref, dtype) - allowance)
    i = np.unravel_index(np.argmax(dist), err.shape)
    assert dist.max() <= TOL_MAX, (f"{what}: stored {o[i]:.5f} is {dist[i]:.3e} beyond rounding "
                                   f"of the exact {o_ref[i]:.5f}; plain max |dO| = {err.max():.3e}")
    assert dist.mean() <= TOL_MEAN, (f"{what}: mean error beyond storage rounding "
                                     f"{dist.mean():.3e} (plain mean |dO| {err.mean():.3e})")
    if lse_gpu is not None:
        lse = to_np(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
        lerr = np.abs(lse - lse_ref)
        assert lerr.max() <= TOL_LSE, f"{what}: max |dLSE| = {lerr.max():.3e}"
    return dist.max(), dist.mean()


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
