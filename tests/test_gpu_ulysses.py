"""GPU parity of the fused Ulysses attention (attn_fwd_ulysses) through the C ABI: Q, K, V are read
and O written in the sequence-sharded layout [P][B][S/P][H][D], with both all-to-alls folded into
the kernel's addressing.  Checked against the oracle's seq2head -> attention -> head2seq chain and,
bit for bit, against the unfused GPU chain (same kernel arithmetic, different addressing)."""
import numpy as np
import pytest
import torch

import oracle
from context_math_non_b300 import cpattn
from context_math_non_b300.inputs import WORKLOADS, draw_qkv
from parity import assert_attention_close, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu


def unfused(q, k, v):
    """seq2head -> attention over [P*B, H/P, S, D] -> head2seq, all on the GPU."""
    qh, kh, vh = (cpattn.cp_layout_seq2head(t) for t in (q, k, v))
    Pg, B, Hl, S, D = qh.shape
    o_h, lse_h = cpattn.attn_fwd(qh.view(Pg * B, Hl, S, D), kh.view(Pg * B, Hl, S, D),
                                 vh.view(Pg * B, Hl, S, D))
    return cpattn.cp_layout_head2seq(o_h.view(Pg, B, Hl, S, D)), lse_h.view(Pg, B, Hl, S)


def draw(P, B, S, H, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(P, B, S // P, H, D, generator=g).to(dtype) for _ in range(3)]


# (P, B, S, H, D, dtype): S/P picks the TMA box height (128, 64, 32 or 16 tokens per box), and
# S not a multiple of 128 leaves a ragged last tile whose boxes run past the last rank.
SMALL = [
    (2, 1, 256, 4, 64, torch.bfloat16),    # S/P = 128: one box per tile half
    (2, 1, 96, 4, 128, torch.float16),     # S/P = 48: 16-token boxes, one ragged tile
    (4, 2, 320, 8, 64, torch.bfloat16),    # S/P = 80: boxes of 16, ragged tail of 64
    (3, 1, 192, 3, 128, torch.bfloat16),   # S/P = 64, three ranks, one head each
    (8, 1, 1024, 8, 128, torch.bfloat16),  # eight ranks, one head each
    (4, 1, 384, 8, 64, torch.float16),     # S/P = 96: 32-token boxes
    (1, 2, 208, 2, 128, torch.bfloat16),   # P = 1: plain [B][S][H][D] attention
]


@pytest.mark.parametrize("P,B,S,H,D,dtype", SMALL)
def test_ulysses_small_against_oracle(P, B, S, H, D, dtype):
    q, k, v = draw(P, B, S, H, D, dtype, seed=P * 1000 + S + D)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = cpattn.attn_fwd_ulysses(qd, kd, vd)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    o_ref, lse_ref = oracle.ulysses_attention(q, k, v, P)
    assert o.shape == q.shape and lse.shape == (P, B, H // P, S)
    assert_attention_close(o, lse, o_ref, lse_ref, f"ulysses P={P} S={S} D={D}")
    # the same numbers as the unfused chain, bit for bit
    o_u, lse_u = unfused(qd, kd, vd)
    assert torch.equal(o, o_u)
    assert torch.equal(lse, lse_u)


def test_ulysses_without_lse_and_many_units_per_cta():
    P, B, S, H, D = 4, 1, 512, 8, 128
    q, k, v = (t.cuda() for t in draw(P, B, S, H, D, torch.bfloat16, seed=5))
    o_full, lse_full = cpattn.attn_fwd_ulysses(q, k, v)
    prev = cpattn.attn_set_max_ctas(3)
    try:
        o_few, lse_few = cpattn.attn_fwd_ulysses(q, k, v)
        o_nolse, none = cpattn.attn_fwd_ulysses(q, k, v, want_lse=False)
    finally:
        cpattn.attn_set_max_ctas(prev)
    assert none is None
    assert torch.equal(o_full, o_few) and torch.equal(lse_full, lse_few)
    assert torch.equal(o_full, o_nolse)


def test_ulysses_leaves_padding_untouched():
    """Writes land only on the tokens of O: a canary around the output survives."""
    P, B, S, H, D = 2, 1, 96, 4, 64
    q, k, v = (t.cuda() for t in draw(P, B, S, H, D, torch.bfloat16, seed=9))
    n = q.numel()
    buf = torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    o = buf[2048:2048 + n].view(q.shape)
    cpattn.attn_fwd_ulysses(q, k, v, o=o, want_lse=False)
    assert (buf[:2048] == 7.0).all() and (buf[2048 + n:] == 7.0).all()
    o_ref, _ = cpattn.attn_fwd_ulysses(q, k, v)
    assert torch.equal(o, o_ref)


def test_ulysses_full_size_sampled():
    """[8][2][2048][32][64] fp16 (the sequence-sharded Ulysses workload): bit-equal to the
    unfused chain everywhere, and within tolerance of the oracle on sampled tokens of every
    (rank, batch, head)."""
    P = 8
    q, k, v = draw_qkv(WORKLOADS["ulysses"])
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = cpattn.attn_fwd_ulysses(qd, kd, vd)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    o_u, lse_u = unfused(qd, kd, vd)
    assert torch.equal(o, o_u)
    assert torch.equal(lse, lse_u)
    # oracle on sampled global tokens, through the oracle's own re-layout
    qo, ko, vo = (torch.from_numpy(oracle.seq2head(t.numpy(), P)) for t in (q, k, v))
    Pg, B, Hl, S, D = qo.shape
    rows = sample_rows(S, 16, seed=21, extra=(S // P - 1, S // P, 3 * S // P))
    o_ref, lse_ref = oracle_rows(*(t.reshape(Pg * B, Hl, S, D) for t in (qo, ko, vo)), rows)
    Sl = S // P
    # gather the same tokens from the sequence-sharded GPU output: token t -> rank t // Sl
    oc = o.cpu()
    got = torch.stack([oc[int(t) // Sl, :, int(t) % Sl] for t in rows], dim=2)  # [B][H][rows][D]
    got = got.reshape(B, Pg, Hl, len(rows), D).permute(1, 0, 2, 3, 4).reshape(Pg * B, Hl,
                                                                             len(rows), D)
    lse_got = lse.view(Pg * B, Hl, S)[:, :, torch.as_tensor(rows)].cpu()
    assert_attention_close(got, lse_got, o_ref, lse_ref, "ulysses full size")


def test_ulysses_bf16_d128_ragged():
    """bf16, D = 128, S/P = 112 (16-token boxes), last tile ragged; bit-equal to the unfused
    chain and within tolerance of the oracle."""
    P, B, S, H, D = 4, 2, 448, 8, 128
    q, k, v = draw(P, B, S, H, D, torch.bfloat16, seed=31)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = cpattn.attn_fwd_ulysses(qd, kd, vd)
    o_ref, lse_ref = oracle.ulysses_attention(q, k, v, P)
    assert_attention_close(o, lse, o_ref, lse_ref, "ulysses bf16 D128")
    o_u, lse_u = unfused(qd, kd, vd)
    assert torch.equal(o, o_u) and torch.equal(lse, lse_u)
