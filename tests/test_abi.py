"""C-ABI checks that need no GPU: the library loads, exports every function the header declares,
and rejects invalid arguments on the host (before any CUDA call) with the documented status.

Pointers passed here are fake addresses; every case below is rejected (or is an empty problem)
before the library touches the device, which is exactly what these tests pin down.
"""
import ctypes
import os
import re

import pytest

from context_math_non_b300 import cpattn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cpattn.h")

A = 0x7f0000000000          # fake, 16-byte aligned "device" addresses, far apart
B_ = 0x7f0010000000
C = 0x7f0020000000
O = 0x7f0030000000
L = 0x7f0040000000
BIG = 1 << 20


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^CPATTN_API\s+(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*"
                                 r"([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def L_():
    if not os.path.exists(cpattn.LIB_PATH):
        from context_math_non_b300.build import build
        build()
    return cpattn.lib()


def test_header_declares_the_boundary():
    fns = declared_functions()
    for name in ("attn_fwd", "attn_fwd_chunked", "attn_lse_merge", "attn_fwd_ulysses",
                 "cp_layout_seq2head", "cp_layout_head2seq", "attn_status_string", "attn_device_status",
                 "attn_watchdog_selftest"):
        assert name in fns, name


def test_library_exports_every_declared_symbol(L_):
    for name in declared_functions():
        assert hasattr(L_, name), f"libcpattn.so does not export {name}"


def test_library_exports_nothing_undeclared(L_):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", cpattn.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    ours = {s for s in exported if s.startswith(("attn_", "cp_"))}
    assert ours == set(declared_functions())


def test_status_strings(L_):
    assert cpattn.attn_status_string(0) == "ATTN_OK"
    assert cpattn.attn_status_string(5) == "ATTN_ERR_TIMEOUT"
    assert cpattn.attn_status_string(99) == "ATTN_ERR_UNKNOWN"
    assert cpattn.attn_version() >= 100


def test_max_ctas_setter(L_):
    prev = cpattn.attn_set_max_ctas(7)
    assert cpattn.attn_set_max_ctas(0) == 7
    assert cpattn.attn_set_max_ctas(prev) == 0


def fwd(L_, q=A, k=B_, v=C, o=O, lse=L, B=1, H=2, Sq=256, Skv=256, D=64, dt=0, scale=0.0):
    return L_.attn_fwd(q, k, v, o, lse, B, H, Sq, Skv, D, dt, scale, None)


def chunked(L_, P=4, q=A, k=B_, v=C, o=O, lse=L, B=1, H=2, Sq=256, Skv=256, D=64, dt=0):
    return L_.attn_fwd_chunked(q, k, v, P, o, lse, B, H, Sq, Skv, D, dt, 0.0, None)


def test_attention_argument_errors(L_):
    E, U, M = cpattn.ATTN_ERR_INVALID_ARG, cpattn.ATTN_ERR_UNSUPPORTED, cpattn.ATTN_ERR_MISALIGNED
    assert fwd(L_, q=None) == E
    assert fwd(L_, o=None) == E
    assert fwd(L_, Skv=0) == E
    assert fwd(L_, B=-1) == E
    assert fwd(L_, dt=7) == E
    assert fwd(L_, D=96) == U
    assert fwd(L_, D=256) == U
    assert fwd(L_, q=A + 8) == M
    assert fwd(L_, lse=L + 4) == M
    assert fwd(L_, o=A) == E                        # output aliases q
    assert fwd(L_, lse=B_ + 64) == E                # lse inside k
    assert chunked(L_, P=0) == E
    assert chunked(L_, P=257) == E                  # more chunks than KV rows
    assert chunked(L_, lse=None) == E               # partial LSEs are required
    assert chunked(L_, o=O, lse=O + 1024) == E      # the two outputs overlap


def test_attention_empty_problems_launch_nothing(L_):
    # zero batch / heads / queries: OK without any device work (fake pointers never touched)
    assert fwd(L_, B=0) == cpattn.ATTN_OK
    assert fwd(L_, H=0) == cpattn.ATTN_OK
    assert fwd(L_, Sq=0) == cpattn.ATTN_OK
    assert chunked(L_, Sq=0) == cpattn.ATTN_OK


def test_merge_argument_errors(L_):
    E, M = cpattn.ATTN_ERR_INVALID_ARG, cpattn.ATTN_ERR_MISALIGNED
    f = L_.attn_lse_merge
    assert f(None, L, 4, 1, 2, 8, 64, 0, O, None, None) == E
    assert f(A, L, 0, 1, 2, 8, 64, 0, O, None, None) == E
    assert f(A, L, 4, 1, 2, 8, 60, 0, O, None, None) == E          # D*2 not a multiple of 16
    assert f(A, L, 4, 1, 2, 8, 64, 3, O, None, None) == E
    assert f(A + 2, L, 4, 1, 2, 8, 64, 0, O, None, None) == M
    assert f(A, L, 4, 1, 2, 8, 64, 0, A + 64, None, None) == E     # o inside o_parts
    assert f(A, L, 4, 1, 2, 8, 64, 0, O, L, None) == E             # lse aliases lse_parts
    assert f(A, L, 4, 0, 2, 8, 64, 0, O, None, None) == cpattn.ATTN_OK


@pytest.mark.parametrize("fn", ["cp_layout_seq2head", "cp_layout_head2seq"])
def test_layout_argument_errors(L_, fn):
    E, M = cpattn.ATTN_ERR_INVALID_ARG, cpattn.ATTN_ERR_MISALIGNED
    f = getattr(L_, fn)
    assert f(None, O, 8, 2, 64, 32, 64, 2, None) == E
    assert f(A, O, 0, 2, 64, 32, 64, 2, None) == E
    assert f(A, O, 8, 2, 60, 32, 64, 2, None) == E     # S % P
    assert f(A, O, 8, 2, 64, 30, 64, 2, None) == E     # H % P
    assert f(A, O, 8, 2, 64, 32, 3, 2, None) == E      # D*elem_bytes % 16
    assert f(A, O, 8, 2, 64, 32, 64, 0, None) == E
    assert f(A + 4, O, 8, 2, 64, 32, 64, 2, None) == M
    assert f(A, A + 256, 8, 2, 64, 32, 64, 2, None) == E   # in-place / overlapping
    assert f(A, O, 8, 0, 64, 32, 64, 2, None) == cpattn.ATTN_OK
    assert f(A, O, 8, 2, 0, 32, 64, 2, None) == cpattn.ATTN_OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(cpattn, "_lib", None)
    monkeypatch.setattr(cpattn, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(cpattn.CpAttnLibraryError):
        cpattn.lib()


def uly(L_, q=A, k=B_, v=C, o=O, lse=L, P=4, B=1, S=512, H=8, D=64, dt=0):
    return L_.attn_fwd_ulysses(q, k, v, o, lse, P, B, S, H, D, dt, 0.0, None)


def test_ulysses_argument_errors(L_):
    E, U, M = cpattn.ATTN_ERR_INVALID_ARG, cpattn.ATTN_ERR_UNSUPPORTED, cpattn.ATTN_ERR_MISALIGNED
    assert uly(L_, q=None) == E
    assert uly(L_, P=0) == E
    assert uly(L_, S=510) == E                      # S not divisible by P
    assert uly(L_, H=6) == E                        # H not divisible by P
    assert uly(L_, dt=2) == E
    assert uly(L_, D=96) == U
    assert uly(L_, S=4 * 24) == U                   # S/P = 24 is not a multiple of 16
    assert uly(L_, v=C + 8) == M
    assert uly(L_, o=B_ + 4096) == E                # output inside k
    assert uly(L_, lse=O + 64) == E                 # lse inside o
    assert uly(L_, B=0) == cpattn.ATTN_OK           # empty problems touch nothing
    assert uly(L_, S=0) == cpattn.ATTN_OK


def test_probe_argument_errors(L_):
    E = cpattn.ATTN_ERR_INVALID_ARG
    f = L_.attn_probe_mma
    assert f(96, 0, 100, None) == E       # N must be 64, 128 or 256
    assert f(128, 11, 100, None) == E     # unknown mode
    assert f(128, -1, 100, None) == E
    assert f(64, 2, 100, None) == E       # the step sequences need n = 128
    assert f(128, 0, 0, None) == E        # no iterations


def ring(L_, P=4, q=A, k=B_, v=C, o=O, lse=L, B=1, H=2, Sq=256, Skv=256, D=64, dt=0):
    return L_.attn_fwd_ring(q, k, v, P, o, lse, B, H, Sq, Skv, D, dt, 0.0, None)


def test_ring_argument_errors(L_):
    E, U, M = cpattn.ATTN_ERR_INVALID_ARG, cpattn.ATTN_ERR_UNSUPPORTED, cpattn.ATTN_ERR_MISALIGNED
    assert ring(L_, P=0) == E
    assert ring(L_, P=257) == E                     # more ranks than keys
    assert ring(L_, D=96) == U
    assert ring(L_, o=A + 16) == E                  # output inside q
    assert ring(L_, lse=L + 4) == M
    assert ring(L_, Sq=0) == cpattn.ATTN_OK         # nothing to compute
    assert ring(L_, B=0, P=0) == E                  # P is still checked on an empty problem


def fp8(L_, q=A, k=B_, vt=C, P=1, qs=0.01, ks=0.01, vs=0.01, o=O, lse=L, B=1, H=2, Sq=256,
        Skv=256, D=128):
    return L_.attn_fwd_fp8(q, k, vt, P, qs, ks, vs, o, lse, B, H, Sq, Skv, D, 0.0, None)


def test_fp8_argument_errors(L_):
    E, U, M = cpattn.ATTN_ERR_INVALID_ARG, cpattn.ATTN_ERR_UNSUPPORTED, cpattn.ATTN_ERR_MISALIGNED
    assert fp8(L_, D=64) == U                      # e4m3 path is D = 128
    assert fp8(L_, Skv=250) == U                   # V^T rows must be a multiple of 16 bytes
    assert fp8(L_, P=7, Skv=256) == U              # unequal chunks
    assert fp8(L_, P=2, Skv=48) == U               # 24-key chunks: not a multiple of 16
    assert fp8(L_, qs=0.0) == E
    assert fp8(L_, vs=float("inf")) == E
    assert fp8(L_, P=0) == E
    assert fp8(L_, o=A + 1024) == E                # output inside q
    assert fp8(L_, k=B_ + 8) == M
    assert fp8(L_, Sq=0) == cpattn.ATTN_OK


def test_quantize_argument_errors(L_):
    E, M = cpattn.ATTN_ERR_INVALID_ARG, cpattn.ATTN_ERR_MISALIGNED
    f = L_.cp_quantize_e4m3
    assert f(A, 0, O, 2, 64, 100, 0.5, 0, None) == E        # D not a multiple of 16
    assert f(A, 0, O, 2, 40, 128, 0.5, 1, None) == E        # transposed: S multiple of 16
    assert f(A, 0, O, 2, 64, 96, 0.5, 1, None) == E         # transposed: D multiple of 64
    assert f(A, 0, O, 2, 64, 128, 0.0, 0, None) == E        # scale must be positive
    assert f(A, 0, A + 64, 2, 64, 128, 0.5, 0, None) == E   # output overlaps input
    assert f(A + 4, 0, O, 2, 64, 128, 0.5, 0, None) == M
    assert f(A, 0, O, 0, 64, 128, 0.5, 0, None) == cpattn.ATTN_OK
    g = L_.cp_absmax
    assert g(A, 12, 0, L, None) == E                        # n must be a multiple of 8
    assert g(A, 16, 0, L + 2, None) == M


def test_binding_rejects_wrong_dtypes():
    """The binding names the argument when a tensor has the wrong element type (checked before
    the library is called)."""
    import torch
    with pytest.raises(ValueError, match="bfloat16 or float16"):
        cpattn._dt(torch.zeros(4, dtype=torch.float32), "q")
    with pytest.raises(ValueError, match="e4m3 bytes"):
        cpattn._e4m3(torch.zeros(4, dtype=torch.bfloat16), "q")
    with pytest.raises(ValueError, match="CUDA tensor"):
        cpattn.attn_fwd(*(torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16) for _ in range(3)))


def test_alu_probe_argument_errors(L_):
    assert L_.attn_probe_alu(6, 10, None) == cpattn.ATTN_ERR_INVALID_ARG
    assert L_.attn_probe_alu(-1, 10, None) == cpattn.ATTN_ERR_INVALID_ARG
    assert L_.attn_probe_alu(0, 0, None) == cpattn.ATTN_ERR_INVALID_ARG
