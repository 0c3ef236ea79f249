"""CPU oracle for context-parallel attention: plain, slow and meant to be obviously correct.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module: only the test
suite, ``__graft_entry__.smoke()`` and the CPU-baseline legs of ``bench.py`` use it.  It shares
no code, table or helper with the CUDA library; both sides only share the seeded input drawer.

All arithmetic is float64 numpy.  16-bit inputs are converted to float64 exactly before use.

Every function follows a passage of "Scaling AI Inference Across Multiple GPUs Using NVIDIA
TensorRT with Multi-Device Inference Support" (the primary page), section "Parallelism
strategies for distributed inference":

* ``attention`` -- subsection "Context parallelism": the bidirectional (non-causal) attention
  of a diffusion transformer over the whole sequence.  The page gives no formula; the reading
  used is softmax(Q K^T * scale) V with scale = 1/sqrt(D), and LSE is the natural logarithm of
  the softmax denominator sum_j exp(scale * q.k_j).  The result is written straight from that
  definition (the usual max shift is applied before exp, which changes no value, only avoids
  overflow).
* ``attention_chunked`` -- subsection "Ring Attention" and Figure 3: each rank holds one slice
  of K and V; the slice attended by a query tile produces a partial output.  Partial c is the
  plain definition restricted to KV rows [floor(c*Skv/P), floor((c+1)*Skv/P)), normalised over
  that slice only, with its own LSE.
* ``attention_online`` -- subsection "Ring Attention": "online softmax" so that the full-size K
  and V are never materialised.  The running max m, running sum l and running accumulator are
  updated block by block, in the order the blocks arrive.
* ``lse_merge`` -- subsection "Ring Attention" (the attention output is updated as KV blocks
  stream past): combine per-chunk partials by their log-sum-exp weights.
* ``seq2head`` / ``head2seq`` -- subsection "DeepSpeed Ulysses" and Figure 4: the first
  all-to-all turns sequence sharding into head sharding (every rank ends with the full sequence
  for a disjoint subset of heads), the second turns it back.
"""
from __future__ import annotations

import math
from typing import Tuple

import numpy as np

__all__ = ["to_f64", "attention", "chunk_bounds", "attention_chunked", "attention_online",
           "lse_merge", "seq2head", "head2seq", "softmax_weights"]

# Query rows processed at once.  Rows are independent in the definition, so this only bounds
# the size of the temporary score matrix; it does not reorder any reduction.
_ROW_BLOCK_BYTES = 192 << 20


def to_f64(x) -> np.ndarray:
    """Exact conversion of a torch tensor (bf16 / fp16 / fp32 / fp64) or array to float64."""
    if hasattr(x, "detach"):
        import torch  # local: only for dtype conversion of inputs
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)


def softmax_weights(q, k, scale: float | None = None) -> np.ndarray:
    """The attention weight matrix softmax(q k^T * scale) for one head: q [Sq, D], k [Skv, D]."""
    q = to_f64(q)
    k = to_f64(k)
    if scale is None:
        scale = _default_scale(q.shape[-1])
    s = (q @ k.T) * scale
    s = s - s.max(axis=1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=1, keepdims=True)


def _attention_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """One (batch, head): q [Sq, D], k/v [Skv, D] -> (o [Sq, D], lse [Sq])."""
    Sq = q.shape[0]
    Skv = k.shape[0]
    o = np.empty((Sq, v.shape[1]), dtype=np.float64)
    lse = np.empty((Sq,), dtype=np.float64)
    rows = max(1, _ROW_BLOCK_BYTES // max(1, 8 * Skv))
    for r0 in range(0, Sq, rows):
        r1 = min(Sq, r0 + rows)
        s = (q[r0:r1] @ k.T) * scale               # logits s_ij = scale * q_i . k_j
        m = s.max(axis=1, keepdims=True)            # shift only; exp(s - m) / sum is unchanged
        e = np.exp(s - m)
        denom = e.sum(axis=1, keepdims=True)
        o[r0:r1] = (e @ v) / denom                  # O_i = sum_j softmax_ij v_j
        lse[r0:r1] = (m + np.log(denom))[:, 0]      # ln sum_j exp(s_ij)
    return o, lse


def attention(q, k, v, scale: float | None = None) -> Tuple[np.ndarray, np.ndarray]:
    """Non-causal multi-head attention.

    q: [..., Sq, D], k and v: [..., Skv, D] (any leading batch/head dims, equal for all three).
    Returns (O [..., Sq, D], LSE [..., Sq]) in float64.
    """
    q = to_f64(q)
    k = to_f64(k)
    v = to_f64(v)
    if scale is None:
        scale = _default_scale(q.shape[-1])
    lead = q.shape[:-2]
    assert k.shape[:-2] == lead and v.shape[:-2] == lead
    qf = q.reshape((-1,) + q.shape[-2:])
    kf = k.reshape((-1,) + k.shape[-2:])
    vf = v.reshape((-1,) + v.shape[-2:])
    o = np.empty(qf.shape[:-1] + (vf.shape[-1],), dtype=np.float64)
    lse = np.empty(qf.shape[:-1], dtype=np.float64)
    for i in range(qf.shape[0]):
        o[i], lse[i] = _attention_head(qf[i], kf[i], vf[i], scale)
    return o.reshape(lead + o.shape[-2:]), lse.reshape(lead + lse.shape[-1:])


def chunk_bounds(Skv: int, P: int, c: int) -> Tuple[int, int]:
    """KV rows [lo, hi) of chunk c out of P: contiguous slices, balanced by a floor split, as a
    ring rank c that holds sequence slice c would see them."""
    return (c * Skv) // P, ((c + 1) * Skv) // P


def attention_chunked(q, k, v, P: int, scale: float | None = None):
    """Per-chunk partial outputs of attention over KV split into P contiguous chunks.

    Returns (O_parts [P, ..., Sq, D], LSE_parts [P, ..., Sq]); partial c is the attention of q
    over KV rows chunk_bounds(Skv, P, c) only, normalised over those rows.
    """
    q = to_f64(q)
    k = to_f64(k)
    v = to_f64(v)
    Skv = k.shape[-2]
    assert 1 <= P <= Skv
    outs, lses = [], []
    for c in range(P):
        lo, hi = chunk_bounds(Skv, P, c)
        o_c, lse_c = attention(q, k[..., lo:hi, :], v[..., lo:hi, :], scale)
        outs.append(o_c)
        lses.append(lse_c)
    return np.stack(outs), np.stack(lses)


def attention_online(q, k, v, block: int = 128, scale: float | None = None):
    """Online-softmax attention: visit KV in blocks of ``block`` rows, in order, keeping per query
    row a running max m, running denominator l and running (unnormalised) accumulator acc.

    For each block with logits s:  m' = max(m, max_j s_j);  l = l * exp(m - m') + sum_j exp(s_j - m');
    acc = acc * exp(m - m') + sum_j exp(s_j - m') v_j;  m = m'.
    At the end O = acc / l and LSE = m + ln l.
    """
    q = to_f64(q)
    k = to_f64(k)
    v = to_f64(v)
    if scale is None:
        scale = _default_scale(q.shape[-1])
    Skv = k.shape[-2]
    m = np.full(q.shape[:-1], -np.inf)
    l = np.zeros(q.shape[:-1])
    acc = np.zeros(q.shape[:-1] + (v.shape[-1],))
    for j0 in range(0, Skv, block):
        kb = k[..., j0:j0 + block, :]
        vb = v[..., j0:j0 + block, :]
        s = np.einsum("...id,...jd->...ij", q, kb) * scale
        m_new = np.maximum(m, s.max(axis=-1))
        corr = np.exp(m - m_new)                    # exp(-inf) = 0 on the first block
        e = np.exp(s - m_new[..., None])
        l = l * corr + e.sum(axis=-1)
        acc = acc * corr[..., None] + np.einsum("...ij,...jd->...id", e, vb)
        m = m_new
    return acc / l[..., None], m + np.log(l)


def lse_merge(o_parts, lse_parts):
    """Merge P partial attention outputs by their log-sum-exp weights.

    o_parts [P, ..., D], lse_parts [P, ...].  With M = max_c LSE_c, w_c = exp(LSE_c - M):
    LSE = M + ln sum_c w_c  and  O = sum_c w_c O_c / sum_c w_c.
    Rows whose partials all have LSE = -inf (no KV rows at all) merge to O = 0, LSE = -inf.
    """
    o = to_f64(o_parts)
    lse = to_f64(lse_parts)
    M = lse.max(axis=0)
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    w = np.where(finite[None], np.exp(lse - Ms[None]), 0.0)
    W = w.sum(axis=0)
    Wsafe = np.where(finite, W, 1.0)
    out = (w[..., None] * o).sum(axis=0) / Wsafe[..., None]
    out = np.where(finite[..., None], out, 0.0)
    lse_out = np.where(finite, Ms + np.log(Wsafe), -np.inf)
    return out, lse_out


def seq2head(x, P: int) -> np.ndarray:
    """First Ulysses all-to-all, emulated on one device.

    Input [P][B][S/P][H][D]: rank p holds tokens p*S/P .. (p+1)*S/P - 1 for all H heads.
    Output [P][B][H/P][S][D]: rank g holds all S tokens, in global order, for heads
    g*H/P .. (g+1)*H/P - 1.  Element map: out[g][b][j][p*S/P + s][d] = in[p][b][s][g*H/P + j][d].
    Pure data movement: works on any dtype and returns the same dtype.
    """
    x = np.asarray(x)
    Pi, B, Sl, H, D = x.shape
    assert Pi == P and H % P == 0
    Hl = H // P
    y = x.reshape(P, B, Sl, P, Hl, D)          # [p][b][s][g][j][d]
    y = y.transpose(3, 1, 4, 0, 2, 5)          # [g][b][j][p][s][d]
    return np.ascontiguousarray(y.reshape(P, B, Hl, P * Sl, D))


def head2seq(y, P: int) -> np.ndarray:
    """Second Ulysses all-to-all: the exact inverse of ``seq2head``.

    Input [P][B][H/P][S][D] -> output [P][B][S/P][H][D],
    out[p][b][s][g*H/P + j][d] = in[g][b][j][p*S/P + s][d].
    """
    y = np.asarray(y)
    Pg, B, Hl, S, D = y.shape
    assert Pg == P and S % P == 0
    Sl = S // P
    x = y.reshape(P, B, Hl, P, Sl, D)          # [g][b][j][p][s][d]
    x = x.transpose(3, 1, 4, 0, 2, 5)          # [p][b][s][g][j][d]
    return np.ascontiguousarray(x.reshape(P, B, Sl, P * Hl, D))


def ulysses_attention(q, k, v, P: int, scale: float | None = None):
    """DeepSpeed Ulysses attention on sequence-sharded inputs, as the page's "DeepSpeed Ulysses"
    subsection (Figure 4) lays it out: all-to-all to head sharding, full-sequence attention per
    head on every rank, all-to-all back to sequence sharding.

    q, k, v [P][B][S/P][H][D] -> O [P][B][S/P][H][D] (float64), LSE [P][B][H/P][S] (rank g
    holds heads g*H/P .. (g+1)*H/P - 1, every token in global order).
    """
    qh, kh, vh = (seq2head(to_f64(t), P) for t in (q, k, v))
    Pg, B, Hl, S, D = qh.shape
    o, lse = attention(qh.reshape(Pg * B, Hl, S, D), kh.reshape(Pg * B, Hl, S, D),
                       vh.reshape(Pg * B, Hl, S, D), scale)
    return head2seq(o.reshape(Pg, B, Hl, S, D), P), lse.reshape(Pg, B, Hl, S)


def attention_ring(q, k, v, P: int, scale: float | None = None):
    """Ring Attention as the page's "Ring Attention" section (Figure 3) runs it: P ranks, rank r
    holds query rows [floor(r*Sq/P), floor((r+1)*Sq/P)) and KV block r (``chunk_bounds``); at
    ring step i = 0 .. P-1 it attends over the block it holds then, (r - i) mod P, and folds
    the partial output into its running output with the log-sum-exp merge.

    q [..., Sq, D], k/v [..., Skv, D] -> O [..., Sq, D], LSE [..., Sq] (float64).
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    Sq, Skv = q.shape[-2], k.shape[-2]
    assert 1 <= P <= Skv
    o = np.zeros(q.shape)
    lse = np.full(q.shape[:-1], -np.inf)
    for r in range(P):
        q0, q1 = (r * Sq) // P, ((r + 1) * Sq) // P
        if q1 == q0:
            continue
        qr = q[..., q0:q1, :]
        o_run, lse_run = None, None
        for i in range(P):
            c = (r - i) % P
            lo, hi = chunk_bounds(Skv, P, c)
            o_c, lse_c = attention(qr, k[..., lo:hi, :], v[..., lo:hi, :], scale)
            if o_run is None:
                o_run, lse_run = o_c, lse_c
            else:
                o_run, lse_run = lse_merge(np.stack([o_run, o_c]), np.stack([lse_run, lse_c]))
        o[..., q0:q1, :] = o_run
        lse[..., q0:q1] = lse_run
    return o, lse


# ------------------------------------------------------------------------------ e4m3 (FP8)
# The 8-bit format the pages' quantisation section recommends for attention layers (FP8): e4m3
# with 1 sign bit, 4 exponent bits (bias 7) and 3 mantissa bits, no infinities, the all-ones
# pattern (S.1111.111) NaN, largest finite value 1.75 * 2^8 = 448, subnormals m/8 * 2^-6.

E4M3_MAX = 448.0


def e4m3_decode(bits) -> np.ndarray:
    """float64 value of e4m3 bytes (NaN for S.1111.111)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 15
    m = (b & 7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7))
    val = np.where((e == 15) & ((b & 7) == 7), np.nan, val)
    return sign * val


def e4m3_round(y) -> np.ndarray:
    """Nearest e4m3 value to float64 y, ties to the even mantissa, finite overflow saturated to
    +-448 (the saturating conversion); NaN stays NaN."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    # spacing of the e4m3 grid around a: 2^-9 below 2^-6 (subnormals), 2^(e-3) in binade e
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    step = np.exp2(e - 3)
    q = np.round(a / step) * step          # numpy rounds halves to even
    q = np.minimum(q, E4M3_MAX)
    q = np.where(np.isnan(y), np.nan, q)
    return np.copysign(q, y)


def e4m3_encode(vals) -> np.ndarray:
    """Bytes of values that are exactly representable in e4m3 (output of e4m3_round)."""
    v = np.asarray(vals, dtype=np.float64)
    sign = np.signbit(v).astype(np.int64) << 7
    a = np.abs(v)
    sub = a < 2.0 ** -6
    e = np.floor(np.log2(np.where(a > 0, a, 1.0))).astype(np.int64)
    e = np.maximum(e, -6)
    m_norm = np.round((a / np.exp2(e) - 1.0) * 8).astype(np.int64)
    m_sub = np.round(a / 2.0 ** -9).astype(np.int64)
    code = np.where(sub, m_sub, ((e + 7) << 3) | m_norm)
    code = np.where(np.isnan(v), 0x7F, code)
    return (sign | np.where(np.isnan(v), 0x7F, code)).astype(np.uint8)


def e4m3_quantize(x, scale: float) -> np.ndarray:
    """Bytes of e4m3(x * (1/scale)) as the quantisation step computes it: 1/scale rounded to
    fp32, the product rounded to fp32, then rounded to e4m3."""
    inv = np.float32(1.0) / np.float32(scale)
    y = (to_f64(x).astype(np.float32) * inv).astype(np.float64)
    return e4m3_encode(e4m3_round(y))


def attention_fp8(q8, k8, v8, q_scale: float, k_scale: float, v_scale: float,
                  scale: float | None = None):
    """Exact attention on the real values the e4m3 inputs stand for (byte value times the
    tensor's scale).  v8 in the natural [..., Skv, D] order.  Returns O, LSE (float64)."""
    q = e4m3_decode(q8) * q_scale
    k = e4m3_decode(k8) * k_scale
    v = e4m3_decode(v8) * v_scale
    return attention(q, k, v, scale)


def fp8_p_rounding_bound(q8, k8, v8, q_scale: float, k_scale: float, v_scale: float,
                         scale: float | None = None) -> np.ndarray:
    """Worst-case |O error| per element from rounding the softmax weights to e4m3 before P*V.

    With p_j = exp(s_j - m) for any running max m <= max_j s_j (so p_j <= 2^8 < 448: no
    saturation), rounding to nearest e4m3 moves p_j by at most max(2^-4 p_j, 2^-10) (half a
    step: relative 2^-4 for normal values, absolute 2^-10 among subnormals).  With l = sum p_j
    >= l_min = sum exp(s_j - max s) the output O = sum p_j v_j / l moves by at most
    sum_j (2^-4 w_j + 2^-10 / l_min) |v_j| (w = softmax weights).  Shape [..., Sq, D].
    """
    q = e4m3_decode(q8) * q_scale
    k = e4m3_decode(k8) * k_scale
    v = np.abs(e4m3_decode(v8) * v_scale)
    sc = _default_scale(q.shape[-1]) if scale is None else scale
    s = np.einsum("...qd,...kd->...qk", q, k) * sc         # [..., Sq, Skv]
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    l_min = e.sum(axis=-1)
    w = e / l_min[..., None]
    return 2.0 ** -4 * (w @ v) + (2.0 ** -10 / l_min)[..., None] * v.sum(axis=-2)[..., None, :]
