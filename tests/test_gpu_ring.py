"""GPU parity of Ring Attention with the merge fused into the kernel (attn_fwd_ring) through the
C ABI: every query block walks the P KV chunks in ring order with its softmax state on chip.
Checked against the oracle's step-by-step ring and its plain definition, and against the
unfused GPU path (per-chunk partials + LSE merge)."""
import numpy as np
import pytest
import torch

import oracle
from context_math_non_b300 import cpattn
from context_math_non_b300.inputs import WORKLOADS, draw_qkv
from parity import assert_attention_close, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu


def rand_qkv(B, H, Sq, Skv, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Sq, D, generator=g).to(dtype)
    k = torch.randn(B, H, Skv, D, generator=g).to(dtype)
    v = torch.randn(B, H, Skv, D, generator=g).to(dtype)
    return q, k, v


CASES = [
    # B, H, Sq, Skv, D, dtype, P
    (1, 3, 1000, 1000, 128, torch.bfloat16, 3),   # ragged chunks 333/333/334, blocks straddle ranks
    (1, 3, 1000, 1000, 64, torch.float16, 8),     # chunks of 125 rows (< one tile), D = 64
    (2, 2, 300, 777, 64, torch.bfloat16, 5),      # Sq != Skv
    (1, 2, 129, 5, 128, torch.bfloat16, 5),       # P = Skv: one key per chunk
    (1, 1, 1, 1, 64, torch.bfloat16, 1),          # single query, single key
    (1, 2, 640, 640, 128, torch.float16, 1),      # P = 1 is plain attention
    (3, 1, 200, 300, 64, torch.bfloat16, 2),      # batch > 1
    (1, 4, 576, 4608, 128, torch.bfloat16, 8),    # 8 ranks of 72 local queries, 576-key chunks
    (1, 2, 3, 700, 64, torch.float16, 8),         # fewer queries than ranks
]


@pytest.mark.parametrize("B,H,Sq,Skv,D,dtype,P", CASES)
def test_ring_small_against_oracle(B, H, Sq, Skv, D, dtype, P):
    q, k, v = rand_qkv(B, H, Sq, Skv, D, dtype, seed=Sq * 7 + Skv + P)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = cpattn.attn_fwd_ring(qd, kd, vd, P)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    o_ref, lse_ref = oracle.attention_ring(q, k, v, P)
    assert_attention_close(o, lse, o_ref, lse_ref, f"ring P={P} Sq={Sq} Skv={Skv} D={D}")
    # the unfused path (partials through HBM + merge) agrees within the same tolerance
    op, lp = cpattn.attn_fwd_chunked(qd, kd, vd, P)
    om, lm = cpattn.attn_lse_merge(op, lp)
    assert_attention_close(o, lse, om.cpu().double().numpy(), lm.cpu().double().numpy(),
                           "ring vs chunked + merge")


def test_ring_p1_is_bitwise_attn_fwd():
    """With one chunk the ring walks exactly attn_fwd's tiles in attn_fwd's order."""
    q, k, v = (t.cuda() for t in rand_qkv(2, 3, 700, 900, 128, torch.bfloat16, seed=3))
    o1, l1 = cpattn.attn_fwd(q, k, v)
    o2, l2 = cpattn.attn_fwd_ring(q, k, v, 1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_ring_without_lse_and_few_ctas():
    q, k, v = (t.cuda() for t in rand_qkv(1, 4, 900, 900, 64, torch.bfloat16, seed=4))
    o_full, lse_full = cpattn.attn_fwd_ring(q, k, v, 4)
    prev = cpattn.attn_set_max_ctas(5)
    try:
        o_few, lse_few = cpattn.attn_fwd_ring(q, k, v, 4)
        o_nolse, none = cpattn.attn_fwd_ring(q, k, v, 4, want_lse=False)
    finally:
        cpattn.attn_set_max_ctas(prev)
    assert none is None
    assert torch.equal(o_full, o_few) and torch.equal(lse_full, lse_few)
    assert torch.equal(o_full, o_nolse)


def test_ring_video_sampled():
    """video: B=1 H=16 S=44160 D=128 over P=8 ring steps (chunks of 5520 = 43*128 + 16 rows)."""
    w = WORKLOADS["video"]
    q, k, v = draw_qkv(w)
    o, lse = cpattn.attn_fwd_ring(q.cuda(), k.cuda(), v.cuda(), 8)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    rows = sample_rows(w.S, 24, seed=w.seed + 1, extra=(5519, 5520, 5521, 44159 - 5520))
    o_ref, lse_ref = oracle_rows(q, k, v, rows)
    assert_attention_close(o[:, :, rows].cpu(), lse[:, :, rows].cpu(), o_ref, lse_ref,
                           "video ring P=8")


def test_ring_stress_sampled():
    """stress: B=1 H=16 S=32768, Q x4 and 1 % of K rows x8 (logits up to ~150), P = 8 ring steps:
    the running max jumps by far more than the lazy-rescale threshold between chunks."""
    w = WORKLOADS["stress"]
    q, k, v = draw_qkv(w)
    o, lse = cpattn.attn_fwd_ring(q.cuda(), k.cuda(), v.cuda(), 8)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    rows = sample_rows(w.S, 24, seed=w.seed + 3, extra=(4095, 4096, 4097))
    o_ref, lse_ref = oracle_rows(q, k, v, rows)
    assert_attention_close(o[:, :, rows].cpu(), lse[:, :, rows].cpu(), o_ref, lse_ref,
                           "stress ring P=8")


@pytest.mark.parametrize("P", [16, 64])
def test_ring_many_ranks_fp16(P):
    """Many short chunks (ragged: 2000 keys over 16 / 64 ranks), fp16, both D."""
    for D in (64, 128):
        q, k, v = rand_qkv(1, 2, 700, 2000, D, torch.float16, seed=P + D)
        o, lse = cpattn.attn_fwd_ring(q.cuda(), k.cuda(), v.cuda(), P)
        o_ref, lse_ref = oracle.attention_ring(q, k, v, P)
        assert_attention_close(o, lse, o_ref, lse_ref, f"ring P={P} D={D} fp16")
