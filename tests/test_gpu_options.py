"""GPU parity of the calls' options against the float64 oracle, through the C ABI: an explicit
softmax scale in every attention entry point, outputs without LSE, a problem with very many heads
(thousands of units per launch), and the chunked step replayed from a CUDA graph."""
import numpy as np
import pytest
import torch

import oracle
from context_math_non_b300 import cpattn
from parity import assert_attention_close, to_np

pytestmark = pytest.mark.gpu


def _qkv(B, H, Sq, Skv, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(B, H, Sq, D, generator=g).to(dtype),
            torch.randn(B, H, Skv, D, generator=g).to(dtype),
            torch.randn(B, H, Skv, D, generator=g).to(dtype))


@pytest.mark.parametrize("scale", [0.02, 0.3])
@pytest.mark.parametrize("D", [64, 128])
def test_explicit_scale(scale, D):
    """scale > 0 replaces 1/sqrt(D): plain, chunked (each partial), ring."""
    q, k, v = _qkv(1, 2, 333, 517, D, torch.bfloat16, seed=int(scale * 1000) + D)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = cpattn.attn_fwd(qd, kd, vd, scale=scale)
    op, lp = cpattn.attn_fwd_chunked(qd, kd, vd, 3, scale=scale)
    orr, lrr = cpattn.attn_fwd_ring(qd, kd, vd, 3, scale=scale)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    o_ref, lse_ref = oracle.attention(q, k, v, scale=scale)
    op_ref, lp_ref = oracle.attention_chunked(q, k, v, 3, scale=scale)
    assert_attention_close(o, lse, o_ref, lse_ref, f"scale {scale} D{D} attn_fwd")
    assert_attention_close(op, lp, op_ref, lp_ref, f"scale {scale} D{D} chunked")
    assert_attention_close(orr, lrr, o_ref, lse_ref, f"scale {scale} D{D} ring")
    # the default scale differs: the explicit one really is used
    o_def, _ = oracle.attention(q, k, v)
    assert np.abs(o_def - o_ref).max() > 1e-2


def test_explicit_scale_ulysses_and_fp8():
    P, B, Sl, H, D, scale = 2, 1, 96, 4, 64, 0.2
    g = torch.Generator().manual_seed(31)
    q, k, v = (torch.randn(P, B, Sl, H, D, generator=g).to(torch.float16) for _ in range(3))
    o, lse = cpattn.attn_fwd_ulysses(q.cuda(), k.cuda(), v.cuda(), scale=scale)
    o_ref, lse_ref = oracle.ulysses_attention(q, k, v, P, scale=scale)
    assert_attention_close(o, lse, o_ref, lse_ref, "ulysses scale 0.2")

    import test_gpu_fp8 as tf8
    q, k, v = _qkv(1, 2, 200, 256, 128, torch.bfloat16, seed=32)
    (q8, k8, v8, vt8), scales = tf8.quantized_inputs(q, k, v)
    o8, l8 = cpattn.attn_fwd_fp8(*(torch.from_numpy(t).cuda() for t in (q8, k8, vt8)), 2,
                                 *scales, scale=0.05)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    o_ref, lse_ref = oracle.attention_fp8(q8, k8, v8, *scales, scale=0.05)
    err = np.abs(to_np(o8) - o_ref)
    bound = oracle.fp8_p_rounding_bound(q8, k8, v8, *scales, scale=0.05)
    assert (err <= bound + 2.0 ** -8 * np.abs(o_ref) + 2e-3).all(), err.max()
    assert np.abs(to_np(l8) - lse_ref).max() <= 1e-3


def test_outputs_without_lse():
    """LSE pointers left NULL: O is unchanged and nothing else is written."""
    q, k, v = _qkv(2, 2, 300, 400, 128, torch.float16, seed=41)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_with, _ = cpattn.attn_fwd(qd, kd, vd)
    o_without, lse = cpattn.attn_fwd(qd, kd, vd, want_lse=False)
    r_with, _ = cpattn.attn_fwd_ring(qd, kd, vd, 2)
    r_without, lr = cpattn.attn_fwd_ring(qd, kd, vd, 2, want_lse=False)
    assert lse is None and lr is None
    assert torch.equal(o_with, o_without) and torch.equal(r_with, r_without)


def test_many_heads():
    """B = 8, H = 256 (2048 heads), 130 queries and keys: 2048 units, 14 per CTA, ragged tiles."""
    q, k, v = _qkv(8, 256, 130, 130, 64, torch.bfloat16, seed=51)
    o, lse = cpattn.attn_fwd(q.cuda(), k.cuda(), v.cuda())
    op, lp = cpattn.attn_fwd_chunked(q.cuda(), k.cuda(), v.cuda(), 2)
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    o_ref, lse_ref = oracle.attention(q, k, v)
    op_ref, lp_ref = oracle.attention_chunked(q, k, v, 2)
    assert_attention_close(o, lse, o_ref, lse_ref, "2048 heads")
    assert_attention_close(op, lp, op_ref, lp_ref, "2048 heads, chunked")


def test_step_replays_from_a_cuda_graph():
    """The chunked step (attn_fwd_chunked + attn_lse_merge) captured once in a CUDA graph and
    replayed on new inputs written into the same buffers gives the bytes of direct calls."""
    q, k, v = _qkv(1, 4, 700, 900, 128, torch.bfloat16, seed=61)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    op = torch.empty((3, 1, 4, 700, 128), dtype=torch.bfloat16, device="cuda")
    lp = torch.empty((3, 1, 4, 700), dtype=torch.float32, device="cuda")
    o = torch.empty_like(qd)
    lse = torch.empty((1, 4, 700), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):          # warm-up outside the capture (one-time kernel set-up)
        cpattn.attn_fwd_chunked(qd, kd, vd, 3, op, lp)
        cpattn.attn_lse_merge(op, lp, o, lse)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        cpattn.attn_fwd_chunked(qd, kd, vd, 3, op, lp)
        cpattn.attn_lse_merge(op, lp, o, lse)
    q2, k2, v2 = _qkv(1, 4, 700, 900, 128, torch.bfloat16, seed=62)
    qd.copy_(q2)
    kd.copy_(k2)
    vd.copy_(v2)
    graph.replay()
    torch.cuda.synchronize()
    assert cpattn.attn_device_status() == cpattn.ATTN_OK
    o_ref, lse_ref = cpattn.attn_lse_merge(*cpattn.attn_fwd_chunked(q2.cuda(), k2.cuda(),
                                                                  v2.cuda(), 3))
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
