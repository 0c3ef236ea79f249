"""GPU parity of the tcgen05 attention kernel (attn_fwd / attn_fwd_chunked) against the float64
oracle, through the C ABI.  Small shapes are compared element by element over every output;
the full-size workloads are compared on sampled query rows (all heads, all D columns, and the
LSE), which the oracle computes row by row."""
import numpy as np
import pytest
import torch

import oracle
from context_math_non_b300 import cpattn
from context_math_non_b300.inputs import WORKLOADS, draw_qkv
from parity import (assert_attention_close, oracle_rows, partial_storage_allowance, sample_rows,
                    to_np)

pytestmark = pytest.mark.gpu


def rand_qkv(B, H, Sq, Skv, D, dtype, seed, q_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, Sq, D, generator=g) * q_scale).to(dtype)
    k = torch.randn(B, H, Skv, D, generator=g).to(dtype)
    v = torch.randn(B, H, Skv, D, generator=g).to(dtype)
    return q, k, v


def run_full_and_chunked(q, k, v, P, what):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = cpattn.attn_fwd(qd, kd, vd)
    op, lp = cpattn.attn_fwd_chunked(qd, kd, vd, P)
    om, lm = cpattn.attn_lse_merge(op, lp)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    o_ref, lse_ref = oracle.attention(q, k, v)
    op_ref, lp_ref = oracle.attention_chunked(q, k, v, P)
    assert_attention_close(o, lse, o_ref, lse_ref, f"{what} attn_fwd")
    assert_attention_close(op, lp, op_ref, lp_ref, f"{what} chunked P={P}")
    # the merge on the partials as stored, then the merged result against exact attention with
    # the storage of the partials allowed for
    om_ref, lm_ref = oracle.lse_merge(to_np(op), to_np(lp))
    assert_attention_close(om, lm, om_ref, lm_ref, f"{what} merge of the stored partials")
    assert_attention_close(om, lm, o_ref, lse_ref, f"{what} chunked P={P} + merge",
                           allowance=partial_storage_allowance(op, lp_ref, q.dtype))
    return o, lse


def test_tiny_workload():
    """B=1 H=2 S=256 D=64, bf16-rounded N(0,1) draws; P=4 chunks merged and P=1."""
    (q, k, v) = draw_qkv(WORKLOADS["tiny"])
    run_full_and_chunked(q, k, v, 4, "tiny")


SMALL_CASES = [
    # B, H, Sq, Skv, D, dtype, P
    (1, 3, 1000, 1000, 128, torch.bfloat16, 3),   # ragged tiles and chunk bounds (333/333/334)
    (1, 3, 1000, 1000, 128, torch.bfloat16, 8),   # chunks of 125 rows (< one tile)
    (2, 2, 300, 777, 64, torch.float16, 5),       # Sq != Skv, D = 64, fp16
    (1, 2, 129, 5, 64, torch.bfloat16, 5),        # P = Skv: one KV row per chunk
    (1, 1, 1, 1, 128, torch.bfloat16, 1),         # single query, single key
    (1, 2, 640, 640, 128, torch.float16, 2),      # exact tiles, fp16, D = 128
    (3, 1, 200, 300, 64, torch.bfloat16, 2),      # batch > 1
    (1, 4, 576, 4608, 128, torch.bfloat16, 8),    # AllGather-KV shape: local queries, full KV
]


@pytest.mark.parametrize("B,H,Sq,Skv,D,dtype,P", SMALL_CASES)
def test_small_shapes(B, H, Sq, Skv, D, dtype, P):
    q, k, v = rand_qkv(B, H, Sq, Skv, D, dtype, seed=Sq * 31 + Skv + P)
    run_full_and_chunked(q, k, v, P, f"B{B} H{H} Sq{Sq} Skv{Skv} D{D} {dtype}")


@pytest.mark.parametrize("B,H,Sq,Skv,D,dtype,P", [c for c in SMALL_CASES if c[4] == 128])
def test_small_shapes_sm_pair_kernel(B, H, Sq, Skv, D, dtype, P):
    """The same D = 128 cases on the CTA-pair kernel (cta_group::2; not the default)."""
    prev = cpattn.attn_set_kernel_variant(1)
    try:
        q, k, v = rand_qkv(B, H, Sq, Skv, D, dtype, seed=Sq * 31 + Skv + P)
        run_full_and_chunked(q, k, v, P, f"SM-pair B{B} H{H} Sq{Sq} Skv{Skv} {dtype}")
    finally:
        cpattn.attn_set_kernel_variant(prev)


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("tail", [1, 15, 16, 17, 63, 64, 65, 112, 127])
def test_tail_tile_sizes(D, tail):
    """KV lengths whose last 128-key tile holds `tail` valid keys: the S GEMM of that tile runs
    with N rounded up to 16 and its P*V skips the all-masked 16-key steps.  Plain attention (one
    chunk), two chunks of 128 + tail keys each through chunked + merge, and the ring."""
    Skv = 256 + tail
    q, k, v = rand_qkv(1, 2, 300, Skv, D, torch.bfloat16, seed=tail * 7 + D)
    run_full_and_chunked(q, k, v, 1, f"tail {tail} D{D}")
    q2, k2, v2 = rand_qkv(1, 2, 300, 2 * (128 + tail), D, torch.bfloat16, seed=tail * 11 + D)
    run_full_and_chunked(q2, k2, v2, 2, f"2 chunks of 128 + {tail} D{D}")
    orr, lrr = cpattn.attn_fwd_ring(q2.cuda(), k2.cuda(), v2.cuda(), 2)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    o_ref, lse_ref = oracle.attention(q2, k2, v2)
    assert_attention_close(orr, lrr, o_ref, lse_ref, f"ring, 2 chunks of 128 + {tail} D{D}")


def test_pair_and_single_cta_kernels_agree():
    """D = 128: the CTA-pair and single-CTA kernels give the same result to rounding."""
    q, k, v = (t.cuda() for t in rand_qkv(1, 3, 1100, 900, 128, torch.bfloat16, seed=21))
    o1, l1 = cpattn.attn_fwd_chunked(q, k, v, 3)
    prev = cpattn.attn_set_kernel_variant(1)
    try:
        o2, l2 = cpattn.attn_fwd_chunked(q, k, v, 3)
    finally:
        cpattn.attn_set_kernel_variant(prev)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    assert (o1.float() - o2.float()).abs().max().item() <= 2 ** -7
    assert (l1 - l2).abs().max().item() <= 1e-4


def test_large_logits_no_overflow():
    """Every logit lies around 90-100, where fp32 exp overflows without the running-max shift.
    Keys are shifted by a constant vector u (q has a positive mean), which moves each row's
    logits by scale * q.u but leaves the attention weights, hence O, unchanged."""
    g = torch.Generator().manual_seed(5)
    B, H, Sq, Skv, D = 1, 2, 384, 700, 128
    q = (torch.randn(B, H, Sq, D, generator=g) + 2.0).to(torch.bfloat16)
    k = (torch.randn(B, H, Skv, D, generator=g) + 4.0).to(torch.bfloat16)
    v = torch.randn(B, H, Skv, D, generator=g).to(torch.bfloat16)
    _, lse = run_full_and_chunked(q, k, v, 3, "large logits")
    assert lse.min().item() > 80.0


def test_sharp_softmax_large_logits():
    """Q x 12: logits with standard deviation 12 (peaks near 50), so one or two keys carry most of
    each row's weight and O is close to single rows of V (|O| up to 4); the running max jumps by
    tens between tiles and chunks.  Here the 16-bit rounding of P (relative 2^-9, with P up to
    2^8 under the lazy rescale) meets |O| ~ |v|, the hardest case for the bf16 tolerance."""
    q, k, v = rand_qkv(1, 2, 384, 700, 128, torch.bfloat16, seed=5, q_scale=12.0)
    o, lse = run_full_and_chunked(q, k, v, 3, "sharp softmax")
    assert o.float().abs().max().item() > 3.0 and lse.max().item() > 30.0
    orr, lrr = cpattn.attn_fwd_ring(q.cuda(), k.cuda(), v.cuda(), 3)
    o_ref, lse_ref = oracle.attention(q, k, v)
    assert_attention_close(orr, lrr, o_ref, lse_ref, "sharp softmax ring P=3")
    qh, kh, vh = (t.to(torch.float16) for t in (q, k, v))
    oh, lh = cpattn.attn_fwd(qh.cuda(), kh.cuda(), vh.cuda())
    o_ref, lse_ref = oracle.attention(qh, kh, vh)
    assert_attention_close(oh, lh, o_ref, lse_ref, "sharp softmax fp16")


def test_many_units_per_cta():
    """A grid capped at 2 CTAs (one SM pair) walks every unit of the problem: exercises every
    barrier phase wrap, on both kernels."""
    q, k, v = rand_qkv(1, 3, 1000, 1000, 128, torch.bfloat16, seed=11)
    prev = cpattn.attn_set_max_ctas(2)
    try:
        run_full_and_chunked(q, k, v, 3, "2 CTAs, single-CTA kernel")
        pv = cpattn.attn_set_kernel_variant(1)
        try:
            run_full_and_chunked(q, k, v, 3, "2 CTAs, one SM pair")
        finally:
            cpattn.attn_set_kernel_variant(pv)
    finally:
        cpattn.attn_set_max_ctas(prev)


def test_deterministic():
    q, k, v = (t.cuda() for t in rand_qkv(1, 4, 700, 900, 128, torch.bfloat16, seed=3))
    a = cpattn.attn_fwd_chunked(q, k, v, 3)
    b = cpattn.attn_fwd_chunked(q, k, v, 3)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("shift", [0, 8])
def test_outputs_stay_in_bounds(D, shift):
    """Canary regions around o_parts / lse_parts are untouched (ragged Sq = 1000).  shift = 8
    elements puts the output 16 bytes past a 32-byte boundary: rows are then written with
    16-byte stores instead of 32-byte ones, and both paths must give the same bytes."""
    B, H, Sq, Skv, P = 1, 2, 1000, 600, 3
    q, k, v = (t.cuda() for t in rand_qkv(B, H, Sq, Skv, D, torch.bfloat16, seed=9))
    n_o, n_l, pad = P * B * H * Sq * D, P * B * H * Sq, 4096
    obuf = torch.full((n_o + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((n_l + 2 * pad,), -3.0, dtype=torch.float32, device="cuda")
    op = obuf[pad + shift:pad + shift + n_o].view(P, B, H, Sq, D)
    lp = lbuf[pad:pad + n_l].view(P, B, H, Sq)
    assert (op.data_ptr() % 32 == 0) == (shift == 0) and op.data_ptr() % 16 == 0
    cpattn.attn_fwd_chunked(q, k, v, P, op, lp)
    torch.cuda.synchronize()
    assert (obuf[:pad + shift] == 7.0).all() and (obuf[pad + shift + n_o:] == 7.0).all()
    assert (lbuf[:pad] == -3.0).all() and (lbuf[pad + n_l:] == -3.0).all()
    assert torch.isfinite(op.float()).all() and torch.isfinite(lp).all()
    ref_o, ref_l = cpattn.attn_fwd_chunked(q, k, v, P)      # fresh, 32-byte aligned outputs
    assert torch.equal(op, ref_o) and torch.equal(lp, ref_l)


# ----------------------------------------------------------------------------- full sizes

@pytest.fixture(scope="module")
def image_inputs():
    return draw_qkv(WORKLOADS["image"])


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_image_workload_sampled(image_inputs, P):
    """B=1 H=24 S=4608 D=128 bf16, KV in P chunks; sampled query rows of every head."""
    q, k, v = image_inputs
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    rows = sample_rows(4608, 24, seed=100 + P)
    if P == 1:
        o, lse = cpattn.attn_fwd(qd, kd, vd)
        o_ref, lse_ref = oracle_rows(q, k, v, rows)
        assert_attention_close(o[:, :, rows].cpu(), lse[:, :, rows].cpu(), o_ref, lse_ref,
                               "image P=1")
        return
    op, lp = cpattn.attn_fwd_chunked(qd, kd, vd, P)
    om, lm = cpattn.attn_lse_merge(op, lp)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    op_ref, lp_ref = oracle_rows(q, k, v, rows, P)
    assert_attention_close(op[:, :, :, rows].cpu(), lp[:, :, :, rows].cpu(), op_ref, lp_ref,
                           f"image chunked P={P}")
    o_ref, lse_ref = oracle.lse_merge(op_ref, lp_ref)
    assert_attention_close(om[:, :, rows].cpu(), lm[:, :, rows].cpu(), o_ref, lse_ref,
                           f"image P={P} merged",
                           allowance=partial_storage_allowance(op[:, :, :, rows], lp_ref,
                                                               q.dtype))


@pytest.mark.parametrize("name", ["video", "stress"])
def test_long_sequence_workloads_sampled(name):
    """video: B=1 H=16 S=44160 D=128, P=8 (chunks of 5520 = 43*128 + 16 rows);
    stress: B=1 H=16 S=32768, Q x4 and 1 % of K rows x8, P=8.  Sampled rows of every head."""
    w = WORKLOADS[name]
    q, k, v = draw_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    op, lp = cpattn.attn_fwd_chunked(qd, kd, vd, 8)
    om, lm = cpattn.attn_lse_merge(op, lp)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    rows = sample_rows(w.S, 40, seed=w.seed)
    op_ref, lp_ref = oracle_rows(q, k, v, rows, 8)
    assert_attention_close(op[:, :, :, rows].cpu(), lp[:, :, :, rows].cpu(), op_ref, lp_ref,
                           f"{name} chunked")
    o_ref, lse_ref = oracle_rows(q, k, v, rows)
    assert_attention_close(om[:, :, rows].cpu(), lm[:, :, rows].cpu(), o_ref, lse_ref,
                           f"{name} merged vs unchunked oracle")
    # the merge itself, fed the GPU's own partials
    om_ref, lm_ref = oracle.lse_merge(to_np(op[:, :, :, rows]), to_np(lp[:, :, :, rows]))
    assert_attention_close(om[:, :, rows].cpu(), lm[:, :, rows].cpu(), om_ref, lm_ref,
                           f"{name} merge of GPU partials")


def test_very_long_sequence_sampled():
    """One head of 262144 tokens (D = 64, bf16), KV in P = 3 ragged chunks (87381 / 87381 /
    87382 keys): long units, far offsets in O and LSE; sampled rows against the oracle, for the
    partials, their merge, and the fused ring."""
    S = 262144
    g = torch.Generator().manual_seed(262144)
    q, k, v = (torch.randn(1, 1, S, 64, generator=g).to(torch.bfloat16) for _ in range(3))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    op, lp = cpattn.attn_fwd_chunked(qd, kd, vd, 3)
    om, lm = cpattn.attn_lse_merge(op, lp)
    orr, lrr = cpattn.attn_fwd_ring(qd, kd, vd, 3)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    rows = sample_rows(S, 10, seed=9, extra=(87380, 87381, 174762, 174763))
    op_ref, lp_ref = oracle_rows(q, k, v, rows, 3)
    assert_attention_close(op[:, :, :, rows].cpu(), lp[:, :, :, rows].cpu(), op_ref, lp_ref,
                           "262144 tokens, partials")
    o_ref, lse_ref = oracle_rows(q, k, v, rows)
    assert_attention_close(om[:, :, rows].cpu(), lm[:, :, rows].cpu(), o_ref, lse_ref,
                           "262144 tokens, merged")
    assert_attention_close(orr[:, :, rows].cpu(), lrr[:, :, rows].cpu(), o_ref, lse_ref,
                           "262144 tokens, ring")
