"""Seeded random configurations through every attention entry point and the layout kernels,
against the float64 oracle (through the C ABI).  Shapes are small enough for the oracle to
finish in seconds but cover ragged query and key lengths, ragged chunks, both head sizes, both
16-bit types, batch > 1 and P up to the key count."""
import numpy as np
import pytest
import torch

import oracle
from context_math_non_b300 import cpattn
from parity import assert_attention_close, partial_storage_allowance, to_np

pytestmark = pytest.mark.gpu


def _configs(n=24, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        D = int(rng.choice([64, 128]))
        dt = [torch.bfloat16, torch.float16][int(rng.integers(2))]
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        Sq = int(rng.integers(1, 700))
        Skv = int(rng.integers(1, 900))
        P = int(rng.integers(1, min(Skv, 12) + 1))
        out.append((i, B, H, Sq, Skv, D, dt, P))
    return out


@pytest.mark.parametrize("i,B,H,Sq,Skv,D,dt,P", _configs())
def test_random_attention(i, B, H, Sq, Skv, D, dt, P):
    g = torch.Generator().manual_seed(1000 + i)
    q = (torch.randn(B, H, Sq, D, generator=g) * float(1 + i % 3)).to(dt)
    k = torch.randn(B, H, Skv, D, generator=g).to(dt)
    v = torch.randn(B, H, Skv, D, generator=g).to(dt)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = cpattn.attn_fwd(qd, kd, vd)
    op, lp = cpattn.attn_fwd_chunked(qd, kd, vd, P)
    om, lm = cpattn.attn_lse_merge(op, lp)
    orr, lrr = cpattn.attn_fwd_ring(qd, kd, vd, P)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    what = f"B{B} H{H} Sq{Sq} Skv{Skv} D{D} {dt} P{P}"
    o_ref, lse_ref = oracle.attention(q, k, v)
    op_ref, lp_ref = oracle.attention_chunked(q, k, v, P)
    assert_attention_close(o, lse, o_ref, lse_ref, f"{what} attn_fwd")
    assert_attention_close(op, lp, op_ref, lp_ref, f"{what} chunked")
    om_ref, lm_ref = oracle.lse_merge(to_np(op), to_np(lp))
    assert_attention_close(om, lm, om_ref, lm_ref, f"{what} merge of stored partials")
    assert_attention_close(om, lm, o_ref, lse_ref, f"{what} chunked + merge",
                           allowance=partial_storage_allowance(op, lp_ref, dt))
    assert_attention_close(orr, lrr, o_ref, lse_ref, f"{what} ring")


def _ulysses_configs(n=8, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        P = int(rng.choice([1, 2, 4]))
        Sl = 16 * int(rng.integers(1, 9))              # (S / P) % 16 == 0
        H = P * int(rng.integers(1, 3))
        out.append((i, P, int(rng.integers(1, 3)), Sl * P, H, int(rng.choice([64, 128])),
                    [torch.bfloat16, torch.float16][int(rng.integers(2))]))
    return out


@pytest.mark.parametrize("i,P,B,S,H,D,dt", _ulysses_configs())
def test_random_ulysses(i, P, B, S, H, D, dt):
    g = torch.Generator().manual_seed(5000 + i)
    q, k, v = (torch.randn(P, B, S // P, H, D, generator=g).to(dt) for _ in range(3))
    o, lse = cpattn.attn_fwd_ulysses(q.cuda(), k.cuda(), v.cuda())
    y = cpattn.cp_layout_seq2head(q.cuda())
    z = cpattn.cp_layout_head2seq(y)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    o_ref, lse_ref = oracle.ulysses_attention(q, k, v, P)
    assert_attention_close(o, lse, o_ref, lse_ref, f"ulysses P{P} B{B} S{S} H{H} D{D} {dt}")
    bits = q.view(torch.int16).numpy()
    assert np.array_equal(y.cpu().view(torch.int16).numpy(), oracle.seq2head(bits, P))
    assert torch.equal(z.cpu(), q)
