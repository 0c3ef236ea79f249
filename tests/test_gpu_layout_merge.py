"""GPU parity of the Ulysses layout kernels (bit-exact) and of the LSE merge kernel, through the
C ABI, plus the full Ulysses chain: seq2head(Q, K, V) -> attention per head group -> head2seq."""
import numpy as np
import pytest
import torch

import oracle
from context_math_non_b300 import cpattn
from context_math_non_b300.inputs import WORKLOADS, draw_partials, draw_qkv
from parity import assert_attention_close, merge_tol, oracle_rows, sample_rows, to_np

pytestmark = pytest.mark.gpu

_BITS = {2: torch.int16, 4: torch.int32, 1: torch.int8, 8: torch.int64}


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(_BITS[t.element_size()]).numpy()


@pytest.mark.parametrize("P,B,S,H,D,dtype", [
    (8, 2, 256, 32, 64, torch.float16),    # Ulysses-like (H/P = 4 heads per rank)
    (4, 1, 512, 8, 128, torch.bfloat16),   # D = 128
    (2, 1, 64, 4, 64, torch.float64),      # 8-byte elements
    (2, 3, 48, 4, 8, torch.float16),       # batch 3
    (2, 1, 6, 4, 8, torch.float16),        # D*2 = 16 bytes: one vector per row
    (4, 3, 20, 8, 64, torch.bfloat16),
    (8, 2, 64, 16, 16, torch.float32),     # 4-byte elements
    (1, 2, 10, 3, 8, torch.float16),       # P = 1 is a pure transpose [B][S][H] -> [B][H][S]
    (3, 1, 9, 6, 24, torch.float16),       # non-power-of-two P and D
    (2, 1, 30, 2, 512, torch.float16),     # 64 vectors per row: 16-token runs, ragged last run
    (2, 2, 1030, 4, 4, torch.float32),     # one vector per row: a 515-token rank in one 1024-token run
])
def test_layout_small_bit_exact(P, B, S, H, D, dtype):
    g = torch.Generator().manual_seed(P * 100 + S)
    x = torch.randn(P, B, S // P, H, D, generator=g).to(dtype)
    y = cpattn.cp_layout_seq2head(x.cuda())
    np.testing.assert_array_equal(bits(y), oracle.seq2head(bits(x), P))
    z = cpattn.cp_layout_head2seq(y)
    assert torch.equal(z.cpu(), x)


@pytest.fixture(scope="module")
def ulysses_inputs():
    return draw_qkv(WORKLOADS["ulysses"])


def test_ulysses_layout_full_size_bit_exact(ulysses_inputs):
    """[8][2][2048][32][64] fp16 -> [8][2][4][16384][64] and back, every element."""
    P = 8
    for x in ulysses_inputs:
        xd = x.cuda()
        y = cpattn.cp_layout_seq2head(xd)
        np.testing.assert_array_equal(bits(y), oracle.seq2head(bits(x), P))
        z = cpattn.cp_layout_head2seq(y)
        assert torch.equal(z, xd)


def test_ulysses_chain_sampled(ulysses_inputs):
    """seq2head -> attention on the [P*B, H/P, S, D] view -> head2seq, checked on sampled
    tokens of every (rank, batch, head) against the oracle on the same re-laid-out inputs."""
    P = 8
    q, k, v = ulysses_inputs
    qh, kh, vh = (cpattn.cp_layout_seq2head(t.cuda()) for t in (q, k, v))
    Pg, B, Hl, S, D = qh.shape
    o_h, lse_h = cpattn.attn_fwd(qh.view(Pg * B, Hl, S, D), kh.view(Pg * B, Hl, S, D),
                                 vh.view(Pg * B, Hl, S, D))
    o_seq = cpattn.cp_layout_head2seq(o_h.view(Pg, B, Hl, S, D))
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    # oracle input: the oracle's own re-layout of the same draws
    qo, ko, vo = (torch.from_numpy(oracle.seq2head(t.numpy(), P)).reshape(Pg * B, Hl, S, D)
                  for t in (q, k, v))
    rows = sample_rows(S, 24, seed=77)
    o_ref, lse_ref = oracle_rows(qo, ko, vo, rows)
    assert_attention_close(o_h[:, :, rows].cpu(), lse_h[:, :, rows].cpu(), o_ref, lse_ref,
                           "ulysses attention per head group")
    # head2seq of the GPU output agrees bit for bit with the oracle's re-layout of it
    np.testing.assert_array_equal(bits(o_seq),
                                  oracle.head2seq(bits(o_h.view(Pg, B, Hl, S, D)), P))


@pytest.mark.parametrize("P,D,dtype", [(1, 128, torch.bfloat16), (2, 64, torch.bfloat16),
                                       (3, 128, torch.float16), (8, 128, torch.bfloat16),
                                       (13, 64, torch.float16), (8, 24, torch.bfloat16)])
def test_merge_random_partials(P, D, dtype):
    B, H, Sq = 2, 3, 301
    o_p, lse_p = draw_partials(P, B, H, Sq, D, dtype, seed=P * 7 + D)
    om, lm = cpattn.attn_lse_merge(o_p.cuda(), lse_p.cuda())
    o_ref, lse_ref = oracle.lse_merge(o_p, lse_p)
    tol = merge_tol(dtype)
    err = np.abs(to_np(om) - o_ref)
    assert (err <= tol * np.abs(o_ref) + 1e-5).all(), err.max()
    np.testing.assert_allclose(to_np(lm), lse_ref, rtol=0, atol=1e-5 * max(1, np.abs(lse_ref).max()))


def test_merge_empty_and_outlier_rows():
    """Rows whose partials are all -inf merge to O = 0, LSE = -inf; one dominant partial
    (LSE 200 above the rest) passes through unchanged."""
    P, B, H, Sq, D = 4, 1, 2, 64, 128
    o_p, lse_p = draw_partials(P, B, H, Sq, D, torch.bfloat16, seed=3)
    lse_p[:, 0, 0, :5] = -float("inf")
    lse_p[2, 0, 1, 10:20] = 200.0
    om, lm = cpattn.attn_lse_merge(o_p.cuda(), lse_p.cuda())
    om, lm = om.cpu(), lm.cpu()
    assert (om[0, 0, :5] == 0).all() and torch.isneginf(lm[0, 0, :5]).all()
    assert torch.equal(om[0, 1, 10:20], o_p[2, 0, 1, 10:20])
    o_ref, lse_ref = oracle.lse_merge(o_p, lse_p)
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(to_np(lm)[fin], lse_ref[fin], atol=1e-4)
    err = np.abs(to_np(om) - o_ref)
    assert (err <= merge_tol(torch.bfloat16) * np.abs(o_ref) + 1e-5).all()


def test_merge_without_lse_output():
    o_p, lse_p = draw_partials(3, 1, 2, 100, 64, torch.bfloat16, seed=4)
    om, lm = cpattn.attn_lse_merge(o_p.cuda(), lse_p.cuda(), want_lse=False)
    assert lm is None
    o_ref, _ = oracle.lse_merge(o_p, lse_p)
    err = np.abs(to_np(om) - o_ref)
    assert (err <= merge_tol(torch.bfloat16) * np.abs(o_ref) + 1e-5).all()


def test_watchdog_reports_timeout_and_context_survives():
    """A bounded wait that nothing ever satisfies ends with ATTN_ERR_TIMEOUT (no hang, no
    fault), the status clears on read, and the next attention call still works."""
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    cpattn.attn_watchdog_selftest(50_000_000)          # 50 ms
    assert cpattn.attn_device_status() == cpattn.ATTN_ERR_TIMEOUT
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    g = torch.Generator().manual_seed(1)
    q, k, v = (torch.randn(1, 1, 130, 64, generator=g).to(torch.bfloat16) for _ in range(3))
    o, lse = cpattn.attn_fwd(q.cuda(), k.cuda(), v.cuda())
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    o_ref, lse_ref = oracle.attention(q, k, v)
    assert_attention_close(o, lse, o_ref, lse_ref, "after watchdog")
