"""GPU parity of the e4m3 path through the C ABI: cp_absmax and cp_quantize_e4m3 bit for bit
against the oracle, and attn_fwd_fp8 against exact attention on the real values the e4m3 inputs
stand for.  The attention inputs are quantized by the oracle (never by the GPU quantizer).

Tolerance for attn_fwd_fp8 (derived in the oracle's fp8_p_rounding_bound): the only rounding
the method adds beyond the 16-bit path is P -> e4m3 before P*V, worth at most
sum_j (2^-4 w_j + 2^-10 / l_min) |v_j| per output element, plus 2e-3 for fp32 accumulation and
scale rounding; the error is measured before the bf16 storage of O (the distance from the exact
value to the reals that round to the stored one, as in the 16-bit tests).  The mean error is held to what
unbiased rounding noise gives: round-to-nearest moves p_j by a roughly uniform amount of at most
half a step, variance <= (2^-4 p_j)^2 / 3 (plus (2^-10)^2 / 3 among subnormals), so
E[dO^2] <= sum_j ((2^-4 w_j)^2 + (2^-10 / l_min)^2) v_j^2 / 3 and mean |dO| <= sqrt(mean E[dO^2]);
the test allows twice that -- a systematic bias (a wrong scale, a truncating conversion) fails
it.  LSE (summed from unrounded fp32 weights) stays
within 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from context_math_non_b300 import cpattn
from context_math_non_b300.inputs import WORKLOADS, draw_qkv
from parity import sample_rows, storage_distance, to_np

pytestmark = pytest.mark.gpu


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


@pytest.mark.parametrize("BH,S,D,dtype,transpose", [
    (2, 256, 128, torch.bfloat16, False),
    (3, 48, 128, torch.float16, False),
    (2, 256, 128, torch.bfloat16, True),
    (3, 80, 128, torch.float16, True),      # S not a multiple of the 64-token tile
    (1, 16, 64, torch.bfloat16, True),
    (2, 32, 16, torch.bfloat16, False),
])
def test_quantize_bit_exact(BH, S, D, dtype, transpose):
    g = torch.Generator().manual_seed(BH * 1000 + S + D)
    x = (torch.randn(BH, S, D, generator=g) * 4).to(dtype)
    x[0, 0, :4] = torch.tensor([600.0, -600.0, 0.0, -0.0]).to(dtype)   # saturation and zeros
    scale = 0.0173
    y = cpattn.cp_quantize_e4m3(x.cuda(), scale, transpose=transpose)
    ref = oracle.e4m3_quantize(x, scale).reshape(BH, S, D)
    if transpose:
        ref = np.ascontiguousarray(ref.transpose(0, 2, 1))
    np.testing.assert_array_equal(bits(y), ref)


def test_absmax_exact():
    g = torch.Generator().manual_seed(9)
    x = torch.randn(5, 333, 128, generator=g).to(torch.bfloat16)
    x[3, 100, 7] = -37.5
    a = cpattn.cp_absmax(x.cuda()).item()
    assert a == 37.5
    xh = torch.randn(1000 * 8, generator=g).to(torch.float16)
    assert cpattn.cp_absmax(xh.cuda()).item() == xh.abs().max().item()


def quantized_inputs(q, k, v):
    """Per-tensor scales amax/448 and the oracle's e4m3 bytes (V also transposed)."""
    scales = [float(t.float().abs().max()) / oracle.E4M3_MAX for t in (q, k, v)]
    q8, k8, v8 = (oracle.e4m3_quantize(t, s).reshape(t.shape) for t, s in zip((q, k, v), scales))
    vt8 = np.ascontiguousarray(np.swapaxes(v8, -1, -2))
    return (q8, k8, v8, vt8), scales


def check_fp8(o, lse, q8, k8, v8, scales, rows=None, what=""):
    if rows is not None:
        q8 = q8[..., rows, :]
        idx = torch.as_tensor(rows)
        o, lse = o[..., idx, :], lse[..., idx]
    o_ref, lse_ref = oracle.attention_fp8(q8, k8, v8, *scales)
    bound = oracle.fp8_p_rounding_bound(q8, k8, v8, *scales)
    og = to_np(o)
    err = storage_distance(og, o_ref, torch.bfloat16)   # error before the bf16 output rounding
    limit = bound + 2e-3
    worst = np.unravel_index(np.argmax(err - limit), err.shape)
    assert (err <= limit).all(), (f"{what}: |dO| {err[worst]:.3e} > bound {limit[worst]:.3e}")
    # expected noise of unbiased rounding of P (see the module docstring)
    q = oracle.e4m3_decode(q8) * scales[0]
    k = oracle.e4m3_decode(k8) * scales[1]
    v2 = (oracle.e4m3_decode(v8) * scales[2]) ** 2
    s = np.einsum("...qd,...kd->...qk", q, k) / np.sqrt(q.shape[-1])
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    l_min = e.sum(axis=-1, keepdims=True)
    var = ((2.0 ** -4 * e / l_min) ** 2 + (2.0 ** -10 / l_min) ** 2) @ v2 / 3.0
    noise = np.sqrt(var.mean())
    assert err.mean() <= 2 * noise, (
        f"{what}: mean |dO| {err.mean():.3e} beyond output rounding > 2 x rounding noise "
        f"{noise:.3e}")
    assert np.abs(to_np(lse) - lse_ref).max() <= 1e-3, what


FP8_CASES = [
    # B, H, Sq, Skv, P
    (1, 2, 300, 256, 1),
    (1, 3, 1000, 1024, 4),      # 256-key chunks
    (2, 2, 129, 4608, 8),       # 576-key chunks
    (1, 1, 1, 16, 1),           # one query, one 16-key tile
    (1, 2, 200, 48, 3),         # three 16-key chunks
]


@pytest.mark.parametrize("B,H,Sq,Skv,P", FP8_CASES)
def test_fp8_attention_small(B, H, Sq, Skv, P):
    g = torch.Generator().manual_seed(Sq + Skv * 3 + P)
    q = torch.randn(B, H, Sq, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(B, H, Skv, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(B, H, Skv, 128, generator=g).to(torch.bfloat16)
    (q8, k8, v8, vt8), scales = quantized_inputs(q, k, v)
    o, lse = cpattn.attn_fwd_fp8(*(torch.from_numpy(t).cuda() for t in (q8, k8, vt8)), P, *scales)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    check_fp8(o.cpu(), lse.cpu(), q8, k8, v8, scales, what=f"fp8 Sq{Sq} Skv{Skv} P{P}")


def test_fp8_attention_video_heads_sampled():
    """The video shape (S = 44160, D = 128) on 2 of its 16 heads, P = 8 ring steps of 5520 keys,
    checked on sampled rows."""
    w = WORKLOADS["video"]
    q, k, v = draw_qkv(w, H=2)
    (q8, k8, v8, vt8), scales = quantized_inputs(q, k, v)
    o, lse = cpattn.attn_fwd_fp8(*(torch.from_numpy(t).cuda() for t in (q8, k8, vt8)), 8, *scales)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    rows = sample_rows(w.S, 12, seed=w.seed + 2, extra=(5519, 5520))
    check_fp8(o.cpu(), lse.cpu(), q8, k8, v8, scales, rows=rows, what="fp8 video")


def test_fp8_gpu_quantizer_feeds_the_same_attention():
    """End to end on the device: cp_absmax -> cp_quantize_e4m3 -> attn_fwd_fp8 gives the same
    bytes, hence the same output, as the oracle-quantized inputs."""
    g = torch.Generator().manual_seed(77)
    q, k, v = (torch.randn(1, 2, 512, 128, generator=g).to(torch.bfloat16) for _ in range(3))
    (q8, k8, v8, vt8), scales = quantized_inputs(q, k, v)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    amax = [cpattn.cp_absmax(t).item() for t in (dq, dk, dv)]
    assert amax == [float(t.float().abs().max()) for t in (q, k, v)]
    gq = cpattn.cp_quantize_e4m3(dq, scales[0])
    gk = cpattn.cp_quantize_e4m3(dk, scales[1])
    gvt = cpattn.cp_quantize_e4m3(dv, scales[2], transpose=True)
    for a, b in ((gq, q8), (gk, k8), (gvt, vt8)):
        np.testing.assert_array_equal(bits(a), b)
    o1, l1 = cpattn.attn_fwd_fp8(gq, gk, gvt, 2, *scales)
    o2, l2 = cpattn.attn_fwd_fp8(*(torch.from_numpy(t).cuda() for t in (q8, k8, vt8)), 2, *scales)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fp8_attention_large_logits():
    """Q x4 and a few K rows x8 (the stress recipe): logits far above 1, the running max jumps
    between tiles; the P-rounding bound still applies (P <= 2^8 after the lazy rescale)."""
    g = torch.Generator().manual_seed(123)
    q = (torch.randn(1, 2, 256, 128, generator=g) * 4).to(torch.bfloat16)
    k = torch.randn(1, 2, 2048, 128, generator=g)
    k[:, :, torch.randperm(2048, generator=g)[:20]] *= 8
    k = k.to(torch.bfloat16)
    v = torch.randn(1, 2, 2048, 128, generator=g).to(torch.bfloat16)
    (q8, k8, v8, vt8), scales = quantized_inputs(q, k, v)
    o, lse = cpattn.attn_fwd_fp8(*(torch.from_numpy(t).cuda() for t in (q8, k8, vt8)), 4, *scales)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    check_fp8(o.cpu(), lse.cpu(), q8, k8, v8, scales, what="fp8 large logits")


def test_fp8_few_ctas_and_repeat_are_bit_equal():
    """Three CTAs walking all units (every barrier phase wraps many times) and a second launch give
    the same bytes as the default grid: the e4m3 kernel is deterministic and its per-unit state
    does not leak between units."""
    g = torch.Generator().manual_seed(41)
    q = torch.randn(2, 3, 700, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(2, 3, 1152, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(2, 3, 1152, 128, generator=g).to(torch.bfloat16)
    (q8, k8, v8, vt8), scales = quantized_inputs(q, k, v)
    args = [torch.from_numpy(t).cuda() for t in (q8, k8, vt8)]
    o1, l1 = cpattn.attn_fwd_fp8(*args, 4, *scales)
    prev = cpattn.attn_set_max_ctas(3)
    try:
        o2, l2 = cpattn.attn_fwd_fp8(*args, 4, *scales)
    finally:
        cpattn.attn_set_max_ctas(prev)
    o3, l3 = cpattn.attn_fwd_fp8(*args, 4, *scales)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)
    check_fp8(o1.cpu(), l1.cpu(), q8, k8, v8, scales, what="fp8 few CTAs")
