"""Pins for the CPU oracle, against facts fixed by mathematics rather than by the oracle itself.

Each check below is independent of the oracle's code: hand-derived closed forms, pure-Python brute
force on tiny inputs, library routines (torch float64 SDPA / logsumexp), and invariants of the
definitions on "Scaling AI Inference Across Multiple GPUs Using NVIDIA TensorRT with
Multi-Device Inference Support" (sections "Context parallelism", "Ring Attention",
"DeepSpeed Ulysses").  ``test_planted_mistakes_are_caught`` checks that plausible bugs in the
oracle (dropped scale, wrong sign, transposed operand, missing log ...) fail these pins.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import cp_attention as oracle_mod

RNG = np.random.default_rng(12345)


# ----------------------------------------------------------------------------- pin helpers
# Each helper takes the attention / merge / layout callables to test, so the same pins can be
# run against deliberately broken copies of the oracle.

def brute_force_attention(q, k, v, scale):
    """Pure-Python softmax attention for tiny inputs (no max shift, no numpy reductions)."""
    Sq, D = q.shape
    Skv = k.shape[0]
    o = [[0.0] * v.shape[1] for _ in range(Sq)]
    lse = [0.0] * Sq
    for i in range(Sq):
        ex = []
        for j in range(Skv):
            dot = 0.0
            for d in range(D):
                dot += float(q[i, d]) * float(k[j, d])
            ex.append(math.exp(scale * dot))
        z = math.fsum(ex)
        for e in range(v.shape[1]):
            o[i][e] = math.fsum(ex[j] / z * float(v[j, e]) for j in range(Skv))
        lse[i] = math.log(z)
    return np.array(o), np.array(lse)


def pin_bruteforce(attn):
    for (Sq, Skv, D) in [(1, 1, 1), (3, 5, 2), (8, 8, 4), (5, 7, 3)]:
        q = RNG.standard_normal((Sq, D))
        k = RNG.standard_normal((Skv, D))
        v = RNG.standard_normal((Skv, D))
        scale = 1.0 / math.sqrt(D)
        o, lse = attn(q[None], k[None], v[None])
        ob, lb = brute_force_attention(q, k, v, scale)
        np.testing.assert_allclose(o[0], ob, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[0], lb, rtol=1e-12, atol=1e-12)


def pin_torch_sdpa(attn):
    g = torch.Generator().manual_seed(7)
    q = torch.randn(2, 3, 37, 16, generator=g, dtype=torch.float64)
    k = torch.randn(2, 3, 53, 16, generator=g, dtype=torch.float64)
    v = torch.randn(2, 3, 53, 16, generator=g, dtype=torch.float64)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=False)
    lse_ref = torch.logsumexp((q @ k.transpose(-1, -2)) / math.sqrt(16), dim=-1)
    o, lse = attn(q.numpy(), k.numpy(), v.numpy())
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref.numpy(), rtol=1e-12, atol=1e-12)


def pin_hand_example(attn):
    # D = 2, default scale 1/sqrt(2).  q = (sqrt(2) ln 3, 0), k_0 = (1, 0), k_1 = (0, 1):
    # logits (ln 3, 0) -> exp (3, 1) -> weights (3/4, 1/4).  v_0 = (4, 8), v_1 = (0, -4):
    # O = 3/4 (4, 8) + 1/4 (0, -4) = (3, 5);  LSE = ln(3 + 1) = ln 4.
    q = np.array([[[math.sqrt(2.0) * math.log(3.0), 0.0]]])
    k = np.array([[[1.0, 0.0], [0.0, 1.0]]])
    v = np.array([[[4.0, 8.0], [0.0, -4.0]]])
    o, lse = attn(q, k, v)
    np.testing.assert_allclose(o[0, 0], [3.0, 5.0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], math.log(4.0), rtol=0, atol=1e-14)


def pin_closed_forms(attn):
    Skv, D = 29, 8
    v = RNG.standard_normal((1, Skv, D))
    k = RNG.standard_normal((1, Skv, D))
    # Q = 0: every logit is 0 -> uniform weights: O = mean_j v_j, LSE = ln Skv.
    o, lse = attn(np.zeros((1, 3, D)), k, v)
    np.testing.assert_allclose(o[0], np.repeat(v[0].mean(0, keepdims=True), 3, 0), atol=1e-13)
    np.testing.assert_allclose(lse[0], math.log(Skv), atol=1e-13)
    # All K rows equal (u): logits all equal scale*q.u -> O = mean v, LSE = scale*q.u + ln Skv.
    u = RNG.standard_normal((D,))
    q = RNG.standard_normal((1, 4, D))
    o, lse = attn(q, np.tile(u, (1, Skv, 1)), v)
    np.testing.assert_allclose(o[0], np.repeat(v[0].mean(0, keepdims=True), 4, 0), atol=1e-13)
    np.testing.assert_allclose(lse[0], q[0] @ u / math.sqrt(D) + math.log(Skv), atol=1e-12)
    # One logit above all others by more than 800: exp of the gap underflows to 0 in float64,
    # so O is exactly that value row and LSE that logit.
    kk = np.zeros((1, Skv, D))
    kk[0, 11, 0] = 1.0
    qq = np.zeros((1, 1, D))
    qq[0, 0, 0] = 900.0 * math.sqrt(D)            # logit 900 for row 11, 0 elsewhere
    o, lse = attn(qq, kk, v)
    np.testing.assert_allclose(o[0, 0], v[0, 11], rtol=0, atol=1e-300)
    np.testing.assert_allclose(lse[0, 0], 900.0, rtol=1e-15)


def pin_invariants(attn):
    Sq, Skv, D = 6, 23, 8
    q = RNG.standard_normal((2, Sq, D))
    k = RNG.standard_normal((2, Skv, D))
    v = RNG.standard_normal((2, Skv, D))
    o, lse = attn(q, k, v)
    # weights sum to one: V = 1 gives O = 1 exactly up to rounding
    o1, _ = attn(q, k, np.ones_like(v))
    np.testing.assert_allclose(o1, 1.0, atol=1e-14)
    # permuting K and V rows together changes nothing
    perm = RNG.permutation(Skv)
    op, lp = attn(q, k[:, perm], v[:, perm])
    np.testing.assert_allclose(op, o, atol=1e-13)
    np.testing.assert_allclose(lp, lse, atol=1e-13)
    # permuting K alone (breaking the pairing) does change O
    op2, _ = attn(q, k[:, perm], v)
    assert np.abs(op2 - o).max() > 1e-3
    # shifting every key by a vector u leaves O unchanged; LSE_i moves by scale * q_i . u
    u = RNG.standard_normal((D,))
    os_, ls = attn(q, k + u, v)
    np.testing.assert_allclose(os_, o, atol=1e-12)
    np.testing.assert_allclose(ls, lse + (q @ u) / math.sqrt(D), atol=1e-12)
    # swapping query rows permutes output rows
    qperm = RNG.permutation(Sq)
    oq, lq = attn(q[:, qperm], k, v)
    np.testing.assert_allclose(oq, o[:, qperm], atol=1e-14)
    np.testing.assert_allclose(lq, lse[:, qperm], atol=1e-14)


def pin_chunking(attn, chunked, merge, online):
    Sq, Skv, D = 5, 19, 4
    q = RNG.standard_normal((2, Sq, D)) * 2.0
    k = RNG.standard_normal((2, Skv, D))
    v = RNG.standard_normal((2, Skv, D))
    o, lse = attn(q, k, v)
    for P in range(1, Skv + 1):
        op, lp = chunked(q, k, v, P)
        assert op.shape == (P, 2, Sq, D) and lp.shape == (P, 2, Sq)
        om, lm = merge(op, lp)
        np.testing.assert_allclose(om, o, atol=1e-12, err_msg=f"P={P}")
        np.testing.assert_allclose(lm, lse, atol=1e-12, err_msg=f"P={P}")
    for blk in (1, 3, 7, 128):
        oo, lo = online(q, k, v, block=blk)
        np.testing.assert_allclose(oo, o, atol=1e-12)
        np.testing.assert_allclose(lo, lse, atol=1e-12)
    # P = Skv: every partial is a single value row and its LSE that row's logit
    op, lp = chunked(q, k, v, Skv)
    expect = np.stack([np.repeat(v[:, j:j + 1], Sq, axis=1) for j in range(Skv)])
    np.testing.assert_allclose(op, expect, atol=1e-14)
    np.testing.assert_allclose(lp, np.stack([np.einsum('bsd,bd->bs', q, k[:, j]) / math.sqrt(D)
                                         for j in range(Skv)]),
                               atol=1e-13)


def pin_merge(merge):
    P, R, D = 5, 7, 3
    o = RNG.standard_normal((P, R, D))
    lse = RNG.standard_normal((P, R)) * 30.0          # wide spread, like outlier-driven chunks
    om, lm = merge(o, lse)
    # direct definition without the max shift, in extended precision via math.fsum per row
    for r in range(R):
        ws = [math.exp(lse[c, r] - 60.0) for c in range(P)]
        z = math.fsum(ws)
        for d in range(D):
            exp_o = math.fsum(ws[c] * o[c, r, d] for c in range(P)) / z
            assert abs(om[r, d] - exp_o) < 1e-12
        assert abs(lm[r] - (60.0 + math.log(z))) < 1e-12
    # P = 1 is the identity
    o1, l1 = merge(o[:1], lse[:1])
    np.testing.assert_allclose(o1, o[0], atol=0)
    np.testing.assert_allclose(l1, lse[0], atol=1e-15)
    # associativity and commutativity
    oab, lab = merge(o[:2], lse[:2])
    oabc, labc = merge(np.stack([oab, o[2]]), np.stack([lab, lse[2]]))
    o3, l3 = merge(o[:3], lse[:3])
    np.testing.assert_allclose(oabc, o3, atol=1e-13)
    np.testing.assert_allclose(labc, l3, atol=1e-13)
    perm = [3, 0, 4, 2, 1]
    op, lp = merge(o[perm], lse[perm])
    np.testing.assert_allclose(op, om, atol=1e-13)
    np.testing.assert_allclose(lp, lm, atol=1e-13)
    # P identical copies: same O, LSE + ln P
    oc, lc = merge(np.repeat(o[:1], 4, 0), np.repeat(lse[:1], 4, 0))
    np.testing.assert_allclose(oc, o[0], atol=1e-14)
    np.testing.assert_allclose(lc, lse[0] + math.log(4), atol=1e-13)
    # a partial with LSE = -inf (no mass) carries no weight
    lse_m = lse.copy()
    lse_m[1] = -np.inf
    om2, lm2 = merge(o, lse_m)
    keep = [0, 2, 3, 4]
    om3, lm3 = merge(o[keep], lse[keep])
    np.testing.assert_allclose(om2, om3, atol=1e-14)
    np.testing.assert_allclose(lm2, lm3, atol=1e-14)


def pin_layout(s2h, h2s):
    P, B, S, H, D = 4, 2, 12, 8, 3
    Sl, Hl = S // P, H // P
    # encode (b, global token t, head h, d) into each element of the sequence-sharded input
    x = np.empty((P, B, Sl, H, D), dtype=np.int64)
    for p in range(P):
        for b in range(B):
            for s in range(Sl):
                for h in range(H):
                    for d in range(D):
                        x[p, b, s, h, d] = (((b * S + p * Sl + s) * H + h) * D + d)
    y = s2h(x, P)
    assert y.shape == (P, B, Hl, S, D)
    # meaning of the first all-to-all: rank g holds the full sequence, in order, for heads
    # g*H/P .. (g+1)*H/P - 1 only (disjoint across ranks)
    for g in range(P):
        for b in range(B):
            for j in range(Hl):
                for t in range(S):
                    for d in range(D):
                        code = int(y[g, b, j, t, d])
                        dd = code % D
                        h = (code // D) % H
                        tt = (code // (D * H)) % S
                        bb = code // (D * H * S)
                        assert (bb, tt, h, dd) == (b, t, g * Hl + j, d)
    # library emulation of the all-to-all: each rank splits its shard along heads into P
    # pieces and sends piece g to rank g; rank g concatenates what it receives along sequence
    xt = torch.from_numpy(x)
    recv = [torch.cat([xt[p].split(Hl, dim=2)[g] for p in range(P)], dim=1) for g in range(P)]
    ref = torch.stack([r.permute(0, 2, 1, 3) for r in recv]).numpy()
    np.testing.assert_array_equal(y, ref)
    # the second all-to-all is the inverse
    np.testing.assert_array_equal(h2s(y, P), x)
    z = RNG.standard_normal((P, B, Hl, S, D))
    np.testing.assert_array_equal(s2h(h2s(z, P), P), z)


# ----------------------------------------------------------------------------- the pins

def test_attention_brute_force():
    pin_bruteforce(oracle.attention)


def test_attention_matches_torch_sdpa_float64():
    pin_torch_sdpa(oracle.attention)


def test_attention_hand_worked_example():
    pin_hand_example(oracle.attention)


def test_attention_closed_forms():
    pin_closed_forms(oracle.attention)


def test_attention_invariants():
    pin_invariants(oracle.attention)


def test_softmax_weight_rows_sum_to_one():
    q = RNG.standard_normal((9, 16)) * 3
    k = RNG.standard_normal((31, 16))
    w = oracle.softmax_weights(q, k)
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-14)
    assert (w >= 0).all()
    # and the oracle's output is those weights applied to V
    v = RNG.standard_normal((31, 5))
    o, _ = oracle.attention(q[None], k[None], v[None])
    np.testing.assert_allclose(o[0], w @ v, atol=1e-13)


def test_chunking_invariance_and_online_softmax():
    pin_chunking(oracle.attention, oracle.attention_chunked, oracle.lse_merge,
                 oracle.attention_online)


def test_chunk_bounds_partition():
    for Skv in (1, 7, 576 * 8, 44160):
        for P in (1, 2, 3, 8):
            if P > Skv:
                continue
            b = [oracle.chunk_bounds(Skv, P, c) for c in range(P)]
            assert b[0][0] == 0 and b[-1][1] == Skv
            assert all(b[c][1] == b[c + 1][0] for c in range(P - 1))
            sizes = [hi - lo for lo, hi in b]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1


def test_merge_definition_and_algebra():
    pin_merge(oracle.lse_merge)


def test_merge_all_empty_rows():
    o = RNG.standard_normal((3, 2, 4))
    lse = np.full((3, 2), -np.inf)
    om, lm = oracle.lse_merge(o, lse)
    assert (om == 0).all() and np.isneginf(lm).all()


def test_layout_meaning_and_round_trip():
    pin_layout(oracle.seq2head, oracle.head2seq)


def test_layout_preserves_bits_of_16bit_types():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(2, 1, 4, 4, 8, generator=g).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy()
    y = oracle.seq2head(bits, 2)
    np.testing.assert_array_equal(oracle.head2seq(y, 2), bits)


def pin_ulysses(fn):
    """Ulysses is exact: sharding the sequence, swapping to head sharding and back gives, for
    every token and head, plain full-sequence attention over the unsharded tensor (torch SDPA in
    float64 here), with the LSE of head g*H/P + j at rank g."""
    P, B, Sl, H, D = 2, 2, 3, 4, 5
    g = torch.Generator().manual_seed(11)
    q, k, v = (torch.randn(P, B, Sl, H, D, generator=g, dtype=torch.float64) for _ in range(3))
    # unshard: [P][B][Sl][H][D] -> [B][H][S][D] with token p*Sl + s
    full = [t.permute(1, 3, 0, 2, 4).reshape(B, H, P * Sl, D) for t in (q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(*full, is_causal=False)
    lse_ref = torch.logsumexp(full[0] @ full[1].transpose(-1, -2) / math.sqrt(D), dim=-1)
    ref_seq = ref.reshape(B, H, P, Sl, D).permute(2, 0, 3, 1, 4)          # [P][B][Sl][H][D]
    lse_head = lse_ref.reshape(B, P, H // P, P * Sl).permute(1, 0, 2, 3)   # [P][B][Hl][S]
    o, lse = fn(q.numpy(), k.numpy(), v.numpy(), P)
    np.testing.assert_allclose(o, ref_seq.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_head.numpy(), rtol=1e-12, atol=1e-12)


def test_ulysses_equals_unsharded_attention():
    pin_ulysses(oracle.ulysses_attention)


def pin_ring(ring):
    """Ring Attention is exact: for any P (ragged ranks and chunks, fewer queries than ranks,
    Sq != Skv) it gives the plain definition's O and LSE."""
    for (Sq, Skv, P) in ((37, 53, 4), (8, 8, 8), (3, 29, 5), (64, 40, 1), (50, 50, 7)):
        q = RNG.standard_normal((2, Sq, 8))
        k = RNG.standard_normal((2, Skv, 8))
        v = RNG.standard_normal((2, Skv, 8))
        o_ref, lse_ref = oracle.attention(q, k, v)
        o, lse = ring(q, k, v, P)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


def test_ring_equals_plain_attention():
    pin_ring(oracle.attention_ring)


def test_e4m3_decode_all_codes():
    """Every e4m3 byte against torch's float8_e4m3fn decoding (a library routine), and the
    format's landmarks by hand."""
    codes = np.arange(256, dtype=np.uint8)
    d = oracle.e4m3_decode(codes)
    t = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert (np.isnan(d) == np.isnan(t)).all()
    np.testing.assert_array_equal(np.nan_to_num(d), np.nan_to_num(t))
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0xFE) == -448.0
    assert oracle.e4m3_decode(0x38) == 1.0 and oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9 and np.isnan(oracle.e4m3_decode(0x7F))


def pin_e4m3_round(rnd):
    """Round-to-nearest-even onto the e4m3 grid with saturation: torch's conversion for values
    inside the range, hand-made ties, subnormals and overflow."""
    x = np.concatenate([RNG.standard_normal(20000) * 60, RNG.standard_normal(5000) * 0.01,
                        RNG.uniform(-448, 448, 5000)])
    got = oracle.e4m3_encode(rnd(x))
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got, ref)
    cases = {1.0625: 1.0, 1.1875: 1.25, 2.0 ** -10: 0.0, 3 * 2.0 ** -10: 2.0 ** -8,
             -1.0625: -1.0, 464.0: 448.0, 500.0: 448.0, -1e6: -448.0, 0.0: 0.0, 2.0 ** -20: 0.0,
             1.96875: 2.0, 240.0: 240.0, 248.0: 256.0}
    for v, want in cases.items():
        assert rnd(np.array([v]))[0] == want, (v, rnd(np.array([v]))[0], want)


def test_e4m3_round_and_encode():
    pin_e4m3_round(oracle.e4m3_round)


def test_e4m3_quantize_is_fp32_scale_then_round():
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(4096, generator=g) * 3).to(torch.bfloat16)
    scale = 0.0123
    got = oracle.e4m3_quantize(x, scale)
    inv = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(scale, dtype=torch.float32)
    y = x.float() * inv
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    inside = (y.abs() <= 448).numpy()   # torch turns overflow into NaN; the quantiser saturates
    assert inside.sum() > 3000 and (~inside).sum() > 50
    np.testing.assert_array_equal(got[inside], ref[inside])
    np.testing.assert_array_equal(got[~inside], np.where(y.numpy()[~inside] > 0, 0x7E, 0xFE))


def simulate_p8_error(q, k, v, lag):
    """Attention with the softmax weights rounded to e4m3 relative to a running max `lag` below
    the true max (as the kernel's lazy rescale allows), against exact attention."""
    s = q @ k.T / math.sqrt(q.shape[-1])
    m = s.max(axis=-1, keepdims=True) - lag
    p = np.exp(s - m)
    pq = oracle.e4m3_round(p)
    o_q = (pq @ v) / p.sum(axis=-1, keepdims=True)
    o = (p @ v) / p.sum(axis=-1, keepdims=True)
    return np.abs(o_q - o)


def pin_p8_bound(bound_fn):
    """The e4m3 P-rounding bound holds in direct simulation, including rows dominated by
    subnormal weights and a running max up to 8 (log2) below the true max."""
    for trial, (Sq, Skv, spread) in enumerate(((16, 64, 1.0), (16, 300, 6.0), (8, 1000, 0.3))):
        D = 16
        q = RNG.standard_normal((Sq, D)) * spread
        k = RNG.standard_normal((Skv, D))
        v = RNG.standard_normal((Skv, D))
        q8, k8, v8 = (oracle.e4m3_encode(oracle.e4m3_round(t)) for t in (q, k, v))
        qd, kd, vd = (oracle.e4m3_decode(t) for t in (q8, k8, v8))
        bound = bound_fn(q8, k8, v8, 1.0, 1.0, 1.0)
        for lag in (0.0, 3.3, 8.0 * math.log(2.0)):
            err = simulate_p8_error(qd, kd, vd, lag)
            assert (err <= bound * (1 + 1e-9) + 1e-12).all(), (trial, lag, (err - bound).max())


def test_fp8_p_rounding_bound():
    pin_p8_bound(oracle.fp8_p_rounding_bound)


def _fp8_inputs(seed, lead=(2,), Sq=7, Skv=19, D=16, spread=2.0):
    """e4m3 bytes of seeded normal draws (torch's float8_e4m3fn conversion: never a NaN code)."""
    g = torch.Generator().manual_seed(seed)
    mk = lambda n, s: (torch.randn(lead + (n, D), generator=g) * s).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    return mk(Sq, spread), mk(Skv, spread), mk(Skv, 1.0)


def pin_attention_fp8(fn):
    """FP8 attention is exact attention on the real values the bytes stand for, byte x scale
    (page section on quantisation: FP8 for attention layers).  Pinned without the oracle's own
    decoder: torch decodes the bytes, scales them and runs its float64 SDPA; then the scale
    relations that any correct placement of the three scales obeys."""
    qs, ks, vs = 0.37, 0.052, 1.9
    for seed, sc in ((1, None), (2, 0.21)):
        q8, k8, v8 = _fp8_inputs(seed)
        dec = lambda b, s: torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64) * s
        q, k, v = dec(q8, qs), dec(k8, ks), dec(v8, vs)
        scale = 1.0 / math.sqrt(q.shape[-1]) if sc is None else sc
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)
        lse_ref = torch.logsumexp((q @ k.transpose(-1, -2)) * scale, dim=-1)
        o, lse = fn(q8, k8, v8, qs, ks, vs, scale=sc)
        np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref.numpy(), rtol=1e-12, atol=1e-12)
    q8, k8, v8 = _fp8_inputs(3)
    o, lse = fn(q8, k8, v8, qs, ks, vs)
    # V's scale multiplies O and nothing else (exact: a power of two)
    o2, lse2 = fn(q8, k8, v8, qs, ks, 2.0 * vs)
    np.testing.assert_array_equal(o2, 2.0 * o)
    np.testing.assert_array_equal(lse2, lse)
    # only the product of Q's and K's scales enters the logits
    o3, lse3 = fn(q8, k8, v8, 3.0 * qs, ks / 3.0, vs)
    np.testing.assert_allclose(o3, o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse3, lse, rtol=1e-12, atol=1e-13)
    # doubling Q's scale is attention on doubled real queries (sharper softmax, not a scaled O)
    o4, lse4 = fn(q8, k8, v8, 2.0 * qs, ks, vs)
    dec = lambda b, s: torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy() * s
    o5, lse5 = oracle.attention(dec(q8, 2.0 * qs), dec(k8, ks), dec(v8, vs))
    np.testing.assert_allclose(o4, o5, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse4, lse5, rtol=1e-12, atol=1e-12)
    assert np.abs(o4 - o).max() > 1e-3


def test_attention_fp8_scales():
    pin_attention_fp8(oracle.attention_fp8)


def test_raw_fp32_and_rounded_inputs_agree_to_bf16_precision():
    """tiny workload: the fp32 draw and its bf16 rounding give outputs within bf16 input error."""
    from context_math_non_b300.inputs import WORKLOADS, draw_qkv
    (q, k, v), (qf, kf, vf) = draw_qkv(WORKLOADS["tiny"], keep_fp32=True)
    o16, l16 = oracle.attention(q, k, v)
    o32, l32 = oracle.attention(qf, kf, vf)
    assert np.abs(o16 - o32).max() < 2e-2
    assert np.abs(l16 - l32).max() < 2e-2


# ----------------------------------------------------------------------------- planted mistakes

def _mutants():
    """Broken copies of the oracle, each with one plausible mistake."""
    base = oracle_mod

    def no_scale(q, k, v, scale=None):
        return base.attention(q, k, v, scale=1.0)

    def transposed_v(q, k, v, scale=None):
        v = base.to_f64(v)
        if v.shape[-1] == v.shape[-2]:
            return base.attention(q, k, np.swapaxes(v, -1, -2), scale)
        return base.attention(q, k, v[..., ::-1, :], scale)

    def lse_without_log(q, k, v, scale=None):
        o, lse = base.attention(q, k, v, scale)
        return o, np.exp(lse)

    def unnormalised(q, k, v, scale=None):
        o, lse = base.attention(q, k, v, scale)
        return o * np.exp(lse - lse.max(axis=-1, keepdims=True))[..., None], lse

    def wrong_sign(q, k, v, scale=None):
        return base.attention(-base.to_f64(q), k, v, scale)

    def merge_wrong_sign(o, lse):
        return base.lse_merge(o, -base.to_f64(lse))

    def merge_no_log(o, lse):
        om, lm = base.lse_merge(o, lse)
        M = base.to_f64(lse).max(axis=0)
        return om, M + np.exp(lm - M) - 1.0

    def merge_plain_mean(o, lse):
        o = base.to_f64(o)
        _, lm = base.lse_merge(o, lse)
        return o.mean(axis=0), lm

    def chunk_overlap(q, k, v, P, scale=None):
        # off-by-one: chunks overlap by one row
        q, k, v = (base.to_f64(t) for t in (q, k, v))
        Skv = k.shape[-2]
        outs, lses = [], []
        for c in range(P):
            lo, hi = base.chunk_bounds(Skv, P, c)
            hi = min(Skv, hi + 1)
            o_c, l_c = base.attention(q, k[..., lo:hi, :], v[..., lo:hi, :], scale)
            outs.append(o_c)
            lses.append(l_c)
        return np.stack(outs), np.stack(lses)

    def online_no_correction(q, k, v, block=128, scale=None):
        q, k, v = (base.to_f64(t) for t in (q, k, v))
        sc = 1.0 / math.sqrt(q.shape[-1]) if scale is None else scale
        m = np.full(q.shape[:-1], -np.inf)
        l = np.zeros(q.shape[:-1])
        acc = np.zeros(q.shape[:-1] + (v.shape[-1],))
        for j0 in range(0, k.shape[-2], block):
            s = np.einsum("...id,...jd->...ij", q, k[..., j0:j0 + block, :]) * sc
            m_new = np.maximum(m, s.max(axis=-1))
            e = np.exp(s - m_new[..., None])
            l = l + e.sum(axis=-1)                       # forgot exp(m - m') on l and acc
            acc = acc + np.einsum("...ij,...jd->...id", e, v[..., j0:j0 + block, :])
            m = m_new
        return acc / l[..., None], m + np.log(l)

    def s2h_swapped(x, P):
        # transposed operand: swaps the roles of the rank and head-group indices
        x = np.asarray(x)
        Pi, B, Sl, H, D = x.shape
        y = x.reshape(P, B, Sl, P, H // P, D).transpose(0, 1, 4, 3, 2, 5)
        return np.ascontiguousarray(y.reshape(P, B, H // P, P * Sl, D))

    def s2h_head_order(x, P):
        # wrong index: head j of group g taken as j*P + g (strided split instead of blocks)
        x = np.asarray(x)
        Pi, B, Sl, H, D = x.shape
        y = x.reshape(P, B, Sl, H // P, P, D).transpose(4, 1, 3, 0, 2, 5)
        return np.ascontiguousarray(y.reshape(P, B, H // P, P * Sl, D))

    def ring_missing_step(q, k, v, P):
        # ring that stops one step early: the last block a rank would receive is never merged
        q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
        Sq, Skv = q.shape[-2], k.shape[-2]
        o = np.zeros(q.shape)
        lse = np.full(q.shape[:-1], -np.inf)
        for r in range(P):
            q0, q1 = (r * Sq) // P, ((r + 1) * Sq) // P
            if q1 == q0:
                continue
            parts = [oracle.attention(q[..., q0:q1, :], k[..., lo:hi, :], v[..., lo:hi, :])
                     for lo, hi in (oracle.chunk_bounds(Skv, P, (r - i) % P)
                                    for i in range(max(1, P - 1)))]
            om, lm = oracle.lse_merge(np.stack([a for a, _ in parts]), np.stack([b for _, b in parts]))
            o[..., q0:q1, :], lse[..., q0:q1] = om, lm
        return o, lse

    def round_toward_zero(y):
        y = np.asarray(y, dtype=np.float64)
        a = np.abs(y)
        e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6.0)
        step = np.exp2(e - 3)
        return np.copysign(np.minimum(np.floor(a / step) * step, 448.0), y)

    def p8_bound_too_tight(q8, k8, v8, qs, ks, vs):
        # relative half-step of 2^-6 instead of 2^-4 and no subnormal term
        b = oracle.fp8_p_rounding_bound(q8, k8, v8, qs, ks, vs)
        q = oracle.e4m3_decode(q8)
        k = oracle.e4m3_decode(k8)
        w = oracle.softmax_weights(q, k)
        return 2.0 ** -6 * (w @ np.abs(oracle.e4m3_decode(v8))) + 0 * b

    def ulysses_local_only(q, k, v, P):
        # no all-to-all: each rank attends over its own tokens only
        q, k, v = (np.asarray(t) for t in (q, k, v))
        Pi, B, Sl, H, D = q.shape
        tr = lambda t: t.transpose(0, 1, 3, 2, 4).reshape(P * B, H, Sl, D)
        o, lse = oracle.attention(tr(q), tr(k), tr(v))
        o = o.reshape(P, B, H, Sl, D).transpose(0, 1, 3, 2, 4)
        return o, np.zeros((P, B, H // P, P * Sl))

    def ulysses_lse_batch_major(q, k, v, P):
        # LSE returned [B][P][H/P][S] instead of rank-major
        o, lse = oracle.ulysses_attention(q, k, v, P)
        return o, np.ascontiguousarray(lse.transpose(1, 0, 2, 3))

    def fp8_no_v_scale(q8, k8, v8, qs, ks, vs, scale=None):
        return base.attention_fp8(q8, k8, v8, qs, ks, 1.0, scale)

    def fp8_q_scale_twice(q8, k8, v8, qs, ks, vs, scale=None):
        return base.attention_fp8(q8, k8, v8, qs * qs, ks, vs, scale)

    def fp8_scales_outside_softmax(q8, k8, v8, qs, ks, vs, scale=None):
        # the logits see the raw bytes; the Q and K scales multiply the output instead
        o, lse = base.attention_fp8(q8, k8, v8, 1.0, 1.0, vs, scale)
        return o * qs * ks, lse

    return [
        ("attention: no scale", lambda: pin_torch_sdpa(no_scale)),
        ("attention: transposed V", lambda: pin_bruteforce(transposed_v)),
        ("attention: LSE without log", lambda: pin_closed_forms(lse_without_log)),
        ("attention: unnormalised", lambda: pin_invariants(unnormalised)),
        ("attention: wrong sign", lambda: pin_hand_example(wrong_sign)),
        ("merge: wrong sign", lambda: pin_merge(merge_wrong_sign)),
        ("merge: no log", lambda: pin_merge(merge_no_log)),
        ("merge: plain mean", lambda: pin_merge(merge_plain_mean)),
        ("chunked: overlapping chunks", lambda: pin_chunking(
            oracle.attention, chunk_overlap, oracle.lse_merge, oracle.attention_online)),
        ("online: missing correction", lambda: pin_chunking(
            oracle.attention, oracle.attention_chunked, oracle.lse_merge, online_no_correction)),
        ("layout: swapped indices", lambda: pin_layout(s2h_swapped, oracle.head2seq)),
        ("layout: strided head split", lambda: pin_layout(s2h_head_order, oracle.head2seq)),
        ("ulysses: local attention only", lambda: pin_ulysses(ulysses_local_only)),
        ("ring: one step short", lambda: pin_ring(ring_missing_step)),
        ("e4m3: rounds toward zero", lambda: pin_e4m3_round(round_toward_zero)),
        ("e4m3: P bound too tight", lambda: pin_p8_bound(p8_bound_too_tight)),
        ("ulysses: batch-major LSE", lambda: pin_ulysses(ulysses_lse_batch_major)),
        ("fp8: V scale dropped", lambda: pin_attention_fp8(fp8_no_v_scale)),
        ("fp8: Q scale applied twice", lambda: pin_attention_fp8(fp8_q_scale_twice)),
        ("fp8: scales outside the softmax", lambda: pin_attention_fp8(fp8_scales_outside_softmax)),
    ]


@pytest.mark.parametrize("name,run", _mutants(), ids=[m[0] for m in _mutants()])
def test_planted_mistakes_are_caught(name, run):
    with pytest.raises(AssertionError):
        run()


def test_oracle_regression_values():
    """The oracle still reproduces the values its generator script committed."""
    import json
    import os
    from context_math_non_b300.inputs import WORKLOADS, draw_qkv
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle.json")
    gold = json.load(open(path))
    q, k, v = draw_qkv(WORKLOADS["tiny"])
    o, lse = oracle.attention(q, k, v)
    _, lp = oracle.attention_chunked(q, k, v, 4)
    rows = gold["rows"]
    np.testing.assert_allclose(o[0, 0, rows, :4], gold["o_head0_cols0to3"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0][:, rows], gold["lse"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lp[:, 0, 1, rows], gold["lse_parts_P4_head1"], rtol=0, atol=1e-13)
